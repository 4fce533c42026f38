"""Seeded synthetic workloads for split-tier paged decode attention.

Only random numbers and page placement live here (no attention, quantisation or
merge arithmetic), so tests hand the same inputs to the CPU oracle and to the
CUDA library.  The generator itself is ``synth.c`` (counter-based splitmix64,
Box-Muller in double, round-to-nearest-even to bfloat16); it is compiled on
first use with the host C compiler.

Workload shapes follow the configurations the method is measured on: GQA group
of 8 query rows per KV head, head size 256, 64-token pages, a recent tier of
BF16 tokens and an older tier of whole 8-bit pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libtpk_synth.so")
_lib = None

BF16_NAN = 0x7FC0
PAGE_TOKENS = 64
HEAD_DIM = 256
RECORD_BYTES = 35072
PACK13_RECORD_BYTES = 65552  # fixed-stride slot of a 13-bit page-head record

# tensor ids of the generator streams
TID_Q, TID_K, TID_V, TID_SIGK, TID_SIGV, TID_OUTLIER, TID_SLOTS, TID_LENS, TID_SPLIT = range(1, 10)


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library (host C compiler, no GPU needed)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, i64, i32, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.tpks_u64.restype = u64
        L.tpks_u64.argtypes = [u64, u64, u64]
        L.tpks_uniform.argtypes = [u64, u64, u64, i64, vp]
        L.tpks_normal.argtypes = [u64, u64, u64, i64, vp]
        L.tpks_normal_bf16.argtypes = [u64, u64, u64, i64, vp, i64, vp]
        L.tpks_permutation.argtypes = [u64, u64, i64, vp]
        L.tpks_randint.argtypes = [u64, u64, i64, i64, i64, vp]
        L.tpks_fill_pages.argtypes = [u64, u64, i32, i64, i32, i32, vp, vp, vp, i32]
        for f in (L.tpks_uniform, L.tpks_normal, L.tpks_normal_bf16, L.tpks_permutation,
                  L.tpks_randint, L.tpks_fill_pages):
            f.restype = None
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def uniform(seed, tid, n, offset=0):
    out = np.empty(n, np.float64)
    lib().tpks_uniform(seed, tid, offset, n, _ptr(out))
    return out


def normal(seed, tid, n, offset=0):
    out = np.empty(n, np.float64)
    lib().tpks_normal(seed, tid, offset, n, _ptr(out))
    return out


def normal_bf16(seed, tid, n, sigma=None, offset=0):
    out = np.empty(n, np.uint16)
    sig = None if sigma is None else np.ascontiguousarray(sigma, np.float64)
    lib().tpks_normal_bf16(seed, tid, offset, n, _ptr(sig), 1 if sig is None else sig.size, _ptr(out))
    return out


def permutation(seed, tid, n):
    out = np.empty(n, np.int32)
    lib().tpks_permutation(seed, tid, n, _ptr(out))
    return out


def randint(seed, tid, n, lo, hi):
    out = np.empty(n, np.int64)
    lib().tpks_randint(seed, tid, n, lo, hi, _ptr(out))
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bfloat16 bits (finite inputs)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


@dataclass
class Workload:
    """One decode step over paged histories.

    Pools are laid out [slot][H][64][256] (bfloat16 bits as uint16).  Every page
    of every request's history has a BF16 copy in the pools (the older pages are
    the input to the page conversion; the unquantised reference reads them).
    For request b, logical page p lives in slot ``pages[b][p]``; the first
    ``n8[b]`` pages form the 8-bit tier and the remaining ``n_ex[b]`` tokens the
    exact tier.
    """
    H: int
    G: int
    d: int
    seed: int
    n_tokens: np.ndarray          # [B] history length
    n8: np.ndarray                # [B] 8-bit pages
    n_ex: np.ndarray              # [B] exact-tier tokens
    pages: list                   # per request: int32 slots of its logical pages
    n_slots: int
    q: np.ndarray                 # [B][H*G][d] uint16
    k_pool: np.ndarray            # [n_slots][H][64][d] uint16
    v_pool: np.ndarray
    sigma_k: np.ndarray = None    # [H][d]
    sigma_v: np.ndarray = None
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return len(self.n_tokens)

    # --- tier views -------------------------------------------------------------
    def exact_page_table(self):
        """CSR over requests of the exact tier's slots (pages n8[b] .. end)."""
        tabs = [self.pages[b][self.n8[b]:] for b in range(self.B)]
        off = np.zeros(self.B + 1, np.int32)
        off[1:] = np.cumsum([len(t) for t in tabs])
        flat = np.concatenate(tabs).astype(np.int32) if off[-1] else np.zeros(0, np.int32)
        return flat, off

    def int8_page_table(self):
        """CSR over requests of the 8-bit tier's slots (pages 0 .. n8[b])."""
        tabs = [self.pages[b][:self.n8[b]] for b in range(self.B)]
        off = np.zeros(self.B + 1, np.int32)
        off[1:] = np.cumsum([len(t) for t in tabs])
        flat = np.concatenate(tabs).astype(np.int32) if off[-1] else np.zeros(0, np.int32)
        return flat, off

    def used_slots(self):
        return np.concatenate([np.asarray(p) for p in self.pages]) if self.B else np.zeros(0, np.int32)

    def int8_slots(self):
        s = [np.asarray(self.pages[b][:self.n8[b]]) for b in range(self.B)]
        return np.concatenate(s).astype(np.int32) if s else np.zeros(0, np.int32)

    def packed_image(self, rec_pool, pack13_pool=None):
        """One step's history packed for host-resident staging: the 8-bit records
        (from rec_pool, [n_slots][H] records) and exact-tier BF16 pages of every
        request in page order, then q and identity page tables, each part at a
        256-byte-aligned offset of one byte image.  Returns (image uint8, off) where
        off maps 'rec', 'k', 'v', 'q', 'pt', 'pt8' to byte offsets, and holds the
        CSR arrays 'req_page_off', 'req_page_off8' and the page counts.

        With pack13_pool (fixed-stride 13-bit records of the exact-tier pages,
        [n_slots][H][65552] bytes) the exact tier travels as those records instead,
        each cut to its size (header words 0 and 1) and 16-byte aligned: part 'p13'
        holds them in (page, head) order and part 'p13off' their int64 offsets
        relative to 'p13'; 'k' and 'v' are then empty."""
        H = self.H
        rb = RECORD_BYTES * H
        s8 = self.int8_slots()
        recs = (np.asarray(rec_pool, np.uint8).reshape(self.n_slots, rb)[s8].reshape(-1) if len(s8)
                else np.zeros(0, np.uint8))
        ex, off_e = self.exact_page_table()
        _, off_8 = self.int8_page_table()
        empty = np.zeros(0, np.uint8)
        p13 = p13off = empty
        if pack13_pool is not None:
            pool = np.asarray(pack13_pool, np.uint8).reshape(self.n_slots, H, PACK13_RECORD_BYTES)
            chunks, offs, pos = [], [], 0
            for slot in ex:
                for h in range(H):
                    r = pool[slot, h]
                    size = 16 + int(r[0:4].view(np.uint32)[0]) + int(r[4:8].view(np.uint32)[0])
                    offs.append(pos)
                    chunks.append(r[:size])
                    pos += (size + 15) & ~15
                    if size & 15:
                        chunks.append(np.zeros(16 - (size & 15), np.uint8))
            p13 = np.concatenate(chunks) if chunks else empty
            p13off = np.asarray(offs, np.int64).view(np.uint8)
        exact_k = self.k_pool[ex].reshape(-1).view(np.uint8) if pack13_pool is None else empty
        exact_v = self.v_pool[ex].reshape(-1).view(np.uint8) if pack13_pool is None else empty
        parts = [("rec", recs), ("k", exact_k), ("v", exact_v), ("p13", p13), ("p13off", p13off),
                 ("q", self.q.reshape(-1).view(np.uint8)),
                 ("pt", np.arange(len(ex), dtype=np.int32).view(np.uint8)),
                 ("pt8", np.arange(len(s8), dtype=np.int32).view(np.uint8))]
        off = {}
        pos = 0
        for name, a in parts:
            off[name] = pos
            pos = (pos + a.size + 255) & ~255
        img = np.zeros(max(pos, 256), np.uint8)
        for name, a in parts:
            img[off[name]:off[name] + a.size] = a
        off.update(req_page_off=off_e, req_page_off8=off_8, n_exact_pages=len(ex), n_int8_pages=len(s8),
                   nbytes=int(pos), p13_bytes=int(p13.size))
        return img, off

    def history_bytes(self):
        """Algorithmic history bytes of one hybrid step: 548 B per 8-bit token-head
        (codes and all scales), 1024 B per BF16 token-head (K and V)."""
        return int(self.H * (RECORD_BYTES * int(self.n8.sum()) + 1024 * int(self.n_ex.sum())))


def make_workload(lengths, recent, H=4, G=8, d=HEAD_DIM, seed=0, key_sigma="unit",
                  value_sigma="unit", n_outliers=4, outlier_sigma=20.0, pool_factor=1.25,
                  tid_base=0, n_threads=None):
    """Build a seeded workload.

    lengths     : history length per request (tokens)
    recent      : BF16 recent tokens R; the older pages form the 8-bit tier,
                  n8 = floor((N - R) / 64) whole pages, so R <= n_ex < R + 64
                  (n8 = 0 when N <= R).  recent=None means all-exact.
    key_sigma   : "unit", "loguniform" (per-channel std 10^U(-1,1)) or "outliers"
                  (n_outliers seeded channels per head at outlier_sigma).
    value_sigma : "unit" or "loguniform".
    """
    lengths = np.asarray(lengths, np.int64)
    B = len(lengths)
    T = PAGE_TOKENS
    if n_threads is None:
        n_threads = max(1, min(32, os.cpu_count() or 1))
    tb = tid_base
    n_pages = (lengths + T - 1) // T
    if recent is None:
        n8 = np.zeros(B, np.int64)
    else:
        n8 = np.maximum(0, (lengths - recent) // T)
    n_ex = lengths - n8 * T
    total_pages = int(n_pages.sum())
    n_slots = max(1, int(np.ceil(pool_factor * total_pages)))
    perm = permutation(seed, tb + TID_SLOTS, n_slots)
    pages, o = [], 0
    for b in range(B):
        pages.append(perm[o:o + n_pages[b]].astype(np.int32))
        o += int(n_pages[b])

    def sig(kind, tid):
        if kind == "unit":
            return None
        if kind == "loguniform":
            return 10.0 ** (2.0 * uniform(seed, tb + tid, H * d) - 1.0)
        if kind == "outliers":
            s = np.ones(H * d)
            for h in range(H):
                ch = permutation(seed, tb + TID_OUTLIER + 64 * h, d)[:n_outliers]
                s[h * d + ch] = outlier_sigma
            return s
        raise ValueError(kind)

    sk = sig(key_sigma, TID_SIGK)
    sv = sig(value_sigma, TID_SIGV)
    k_pool = np.full((n_slots, H, T, d), BF16_NAN, np.uint16)
    v_pool = np.full((n_slots, H, T, d), BF16_NAN, np.uint16)
    L = lib()
    for b in range(B):
        slots = np.ascontiguousarray(pages[b])
        L.tpks_fill_pages(seed, tb + TID_K + 16 * b, H, int(lengths[b]), d, T, _ptr(slots),
                          _ptr(sk), _ptr(k_pool), n_threads)
        L.tpks_fill_pages(seed, tb + TID_V + 16 * b, H, int(lengths[b]), d, T, _ptr(slots),
                          _ptr(sv), _ptr(v_pool), n_threads)
    q = normal_bf16(seed, tb + TID_Q, B * H * G * d).reshape(B, H * G, d)
    return Workload(H=H, G=G, d=d, seed=seed, n_tokens=lengths, n8=n8.astype(np.int64),
                    n_ex=n_ex.astype(np.int64), pages=pages, n_slots=n_slots, q=q,
                    k_pool=k_pool, v_pool=v_pool,
                    sigma_k=None if sk is None else sk.reshape(H, d),
                    sigma_v=None if sv is None else sv.reshape(H, d))


# ------------------------------------------------------------------ configs
def tiny_hybrid(seed=0):
    """1 request, 1 KV head x 8 query rows, 1024 tokens = 12 8-bit pages + 256 BF16,
    K and V with per-channel std log-uniform in [0.1, 10], q ~ N(0, 1)."""
    return make_workload([1024], 256, H=1, seed=seed, key_sigma="loguniform",
                         value_sigma="loguniform")


def exact_32k(seed=1, n_tokens=32768, H=4):
    """All-exact BF16 history of 32K tokens at a seeded permutation of slots."""
    w = make_workload([n_tokens], None, H=H, seed=seed)
    w.meta["split_at"] = int(randint(seed, TID_SPLIT, 1, 1, n_tokens - 1)[0])
    return w


def hybrid_128k(seed=2, n_tokens=131072, recent=4096, H=4):
    """128K tokens, last 4096 BF16, the rest 8-bit pages; keys with 4 outlier
    channels per head at 20x std; values and q ~ N(0, 1)."""
    return make_workload([n_tokens], recent, H=H, seed=seed, key_sigma="outliers")


def batched_hybrid(seed=3, n_req=16, lo=8192, hi=65536, recent=2048, H=4):
    """16 requests with lengths uniform in [8K, 64K], 2048 recent BF16 tokens each."""
    lengths = randint(seed, TID_LENS, n_req, lo, hi)
    return make_workload(lengths, recent, H=H, seed=seed, key_sigma="outliers")
