"""CPU oracle for split-tier paged decode attention -- test infrastructure only.

Plain double-precision C (``oracle.c``) behind thin ctypes wrappers taking numpy
arrays.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
may import this package; the library under ``tiered_paged_kv_gb300`` never does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liborc.so")
_lib = None

T_PAGE = 64
D_HEAD = 256
REC_BYTES = 35072
OFF_KC, OFF_VC, OFF_KS_CHAN, OFF_KS_TOK, OFF_VS_CHAN = 0, 16384, 32768, 33792, 34048


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        # strict IEEE float: no contraction, no fast-math
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-fno-fast-math", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        i32, vp = ctypes.c_int, ctypes.c_void_p
        L.orc_compensated_walk.argtypes = [i32, vp, vp, vp]
        L.orc_compensated_walk.restype = None
        L.orc_channel_scales.argtypes = [vp, vp, vp]
        L.orc_channel_scales.restype = i32
        L.orc_codes_given.argtypes = [vp] * 6
        L.orc_codes_given.restype = None
        L.orc_quantize_page_head.argtypes = [vp, vp, vp]
        L.orc_quantize_page_head.restype = i32
        L.orc_quantize_pages.argtypes = [i32, vp, vp, vp, vp, i32, vp]
        L.orc_quantize_pages.restype = None
        L.orc_attend.argtypes = [i32, i32, i32, vp, vp, vp, ctypes.c_double, vp, vp]
        L.orc_attend.restype = None
        L.orc_partial_exact.argtypes = [i32, i32, vp, vp, vp, vp, i32, i32, vp, vp]
        L.orc_partial_exact.restype = None
        L.orc_partial_int8.argtypes = [i32, i32, vp, vp, vp, i32, i32, vp, vp]
        L.orc_partial_int8.restype = None
        L.orc_merge.argtypes = [i32, i32, i32, vp, vp, vp, vp]
        L.orc_merge.restype = None
        L.orc_partial_int8_iq.argtypes = [i32, i32, vp, vp, vp, i32, i32, vp, vp]
        L.orc_partial_int8_iq.restype = None
        L.orc_query_codes.argtypes = [vp, vp, vp]
        L.orc_query_codes.restype = ctypes.c_float
        L.orc_hybrid_batched.argtypes = [i32, i32, i32] + [vp] * 12 + [i32, i32]
        L.orc_pack13_plane.argtypes = [vp, vp]
        L.orc_pack13_plane.restype = i32
        L.orc_unpack13_plane.argtypes = [vp, i32, vp]
        L.orc_unpack13_plane.restype = i32
        L.orc_pack13_page_head.argtypes = [vp, vp, vp]
        L.orc_pack13_page_head.restype = i32
        L.orc_unpack13_page_head.argtypes = [vp, vp, vp]
        L.orc_unpack13_page_head.restype = i32
        L.orc_pack13_pages.argtypes = [i32, vp, vp, vp, vp, i32, vp]
        L.orc_pack13_pages.restype = None
        L.orc_hybrid_batched.restype = None
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ------------------------------------------------------------------ quantiser
def channel_scales(k_page):
    """k_page: uint16 bf16 bits [64][256] -> (s float32[256], shat float64[256], n_clamped)."""
    k = _c(k_page, np.uint16)
    s = np.empty(D_HEAD, np.float32)
    sh = np.empty(D_HEAD, np.float64)
    n = lib().orc_channel_scales(_p(k), _p(s), _p(sh))
    return s, sh, n


def compensated_walk(dlo, dhi):
    """The channel walk of the compensated rounding alone: given each channel's
    log errors of its lower (dlo <= 0) and upper (dhi >= 0) float32 neighbour,
    returns take_hi (int32, 1 where the upper neighbour is stored)."""
    dlo = _c(dlo, np.float64)
    dhi = _c(dhi, np.float64)
    assert dlo.shape == dhi.shape and dlo.ndim == 1
    out = np.empty(dlo.size, np.int32)
    lib().orc_compensated_walk(dlo.size, _p(dlo), _p(dhi), _p(out))
    return out


def quantize_page_head(k_page, v_page):
    rec = np.zeros(REC_BYTES, np.uint8)
    n = lib().orc_quantize_page_head(_p(_c(k_page, np.uint16)), _p(_c(v_page, np.uint16)), _p(rec))
    return rec, n


def codes_given(k_page, v_page, ks_chan, ks_tok, vs_chan):
    rec = np.zeros(REC_BYTES, np.uint8)
    lib().orc_codes_given(_p(_c(k_page, np.uint16)), _p(_c(v_page, np.uint16)), _p(_c(ks_chan, np.float32)),
                          _p(_c(ks_tok, np.float32)), _p(_c(vs_chan, np.float32)), _p(rec))
    return rec


def quantize_pages(H, k_pool, v_pool, src_slots, dst_slots, rec_pool):
    """In place into rec_pool (uint8, [n_slots*H*35072])."""
    src = _c(src_slots, np.int32)
    dst = _c(dst_slots, np.int32)
    assert rec_pool.flags.c_contiguous and rec_pool.dtype == np.uint8
    lib().orc_quantize_pages(H, _p(_c(k_pool, np.uint16)), _p(_c(v_pool, np.uint16)), _p(src), _p(dst),
                             len(src), _p(rec_pool))


_T = np.arange(T_PAGE)[:, None]
_C = np.arange(D_HEAD)[None, :]
# byte / float positions of the swizzled record fields (see oracle.c)
KC_POS = _T * D_HEAD + (_C ^ (64 * (_T & 1)))                    # [t][c]
VC_POS = (_C * T_PAGE + (_T ^ (32 * ((_C >> 1) & 1))))          # [t][c] -> position in vc[256][64]
KS_POS = np.arange(D_HEAD) ^ (8 * ((np.arange(D_HEAD) >> 5) & 1))


def record_fields(rec):
    """Split one 35,072-byte record into logical (kc[64][256], vc[64][256] (token
    by channel), s[256], r[64], u[256]), undoing the position swizzles and the
    code bias (a code c is stored as the byte c + 128)."""
    rec = np.asarray(rec, np.uint8)
    kc = (rec[OFF_KC:OFF_VC][KC_POS].astype(np.int16) - 128).astype(np.int8)
    vc = (rec[OFF_VC:OFF_KS_CHAN][VC_POS].astype(np.int16) - 128).astype(np.int8)
    s = rec[OFF_KS_CHAN:OFF_KS_TOK].view(np.float32)[KS_POS]
    r = rec[OFF_KS_TOK:OFF_VS_CHAN].view(np.float32)
    u = rec[OFF_VS_CHAN:REC_BYTES].view(np.float32)
    return kc, vc, s, r, u


def pack_record(kc, vc, s, r, u):
    """Inverse of record_fields: logical fields -> 35,072-byte record."""
    rec = np.zeros(REC_BYTES, np.uint8)
    kcb = np.zeros(T_PAGE * D_HEAD, np.uint8)
    kcb[KC_POS] = (np.asarray(kc, np.int16) + 128).astype(np.uint8)
    vcb = np.zeros(T_PAGE * D_HEAD, np.uint8)
    vcb[VC_POS] = (np.asarray(vc, np.int16) + 128).astype(np.uint8)
    ks = np.zeros(D_HEAD, np.float32)
    ks[KS_POS] = s
    rec[OFF_KC:OFF_VC] = kcb
    rec[OFF_VC:OFF_KS_CHAN] = vcb
    rec[OFF_KS_CHAN:OFF_KS_TOK] = ks.view(np.uint8)
    rec[OFF_KS_TOK:OFF_VS_CHAN] = np.asarray(r, np.float32).view(np.uint8)
    rec[OFF_VS_CHAN:REC_BYTES] = np.asarray(u, np.float32).view(np.uint8)
    return rec


# ------------------------------------------------------------------ lossless tier
PLANE_ENC_BYTES = 26656
PLANE_RAW_BYTES = 32768
PACK13_RECORD_BYTES = 16 + 2 * PLANE_RAW_BYTES


def pack13_plane(v):
    """One 64 x 256 plane of BF16 bit patterns -> its 13-bit (or raw) encoding
    ("model quantization", "A lossless tier first")."""
    out = np.zeros(PLANE_RAW_BYTES, np.uint8)
    n = lib().orc_pack13_plane(_p(_c(v, np.uint16)), _p(out))
    return out[:n].copy()


def unpack13_plane(enc):
    enc = _c(enc, np.uint8)
    v = np.empty(T_PAGE * D_HEAD, np.uint16)
    if lib().orc_unpack13_plane(_p(enc), len(enc), _p(v)) != 0:
        raise ValueError("not a 13-bit or raw plane")
    return v.reshape(T_PAGE, D_HEAD)


def pack13_page_head(k_page, v_page):
    rec = np.zeros(PACK13_RECORD_BYTES, np.uint8)
    n = lib().orc_pack13_page_head(_p(_c(k_page, np.uint16)), _p(_c(v_page, np.uint16)), _p(rec))
    return rec[:n].copy()


def unpack13_page_head(rec):
    rec = _c(rec, np.uint8)
    k = np.empty((T_PAGE, D_HEAD), np.uint16)
    v = np.empty((T_PAGE, D_HEAD), np.uint16)
    if lib().orc_unpack13_page_head(_p(rec), _p(k), _p(v)) != 0:
        raise ValueError("malformed record")
    return k, v


def pack13_pages(H, k_pool, v_pool, src_slots, dst_slots, pack_pool):
    """In place into pack_pool (uint8, [n_slots*H*65552]): fixed-stride records."""
    src = _c(src_slots, np.int32)
    dst = _c(dst_slots, np.int32)
    assert pack_pool.flags.c_contiguous and pack_pool.dtype == np.uint8
    lib().orc_pack13_pages(H, _p(_c(k_pool, np.uint16)), _p(_c(v_pool, np.uint16)), _p(src), _p(dst), len(src),
                           _p(pack_pool))


# ------------------------------------------------------------------ attention
def attend(q, K, V, scale=None):
    """q [rows][d], K/V [n][d] (float64) -> (o [rows][d], lse [rows])."""
    q = _c(q, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    rows, d = q.shape
    n = K.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty((rows, d))
    lse = np.empty(rows)
    lib().orc_attend(n, d, rows, _p(q), _p(K if n else np.zeros((1, d))), _p(V if n else np.zeros((1, d))),
                     float(scale), _p(o), _p(lse))
    return o, lse


def partial_exact(H, G, q, k_pool, v_pool, page_table, tok_begin, tok_end):
    q = _c(q, np.uint16)
    pt = _c(page_table, np.int32) if len(page_table) else np.zeros(1, np.int32)
    o = np.empty((H * G, D_HEAD))
    lse = np.empty(H * G)
    lib().orc_partial_exact(H, G, _p(q), _p(_c(k_pool, np.uint16)), _p(_c(v_pool, np.uint16)), _p(pt),
                            int(tok_begin), int(tok_end), _p(o), _p(lse))
    return o, lse


def partial_int8(H, G, q, rec_pool, page_table8, page_begin, page_end):
    q = _c(q, np.uint16)
    pt = _c(page_table8, np.int32) if len(page_table8) else np.zeros(1, np.int32)
    o = np.empty((H * G, D_HEAD))
    lse = np.empty(H * G)
    lib().orc_partial_int8(H, G, _p(q), _p(_c(rec_pool, np.uint8)), _p(pt), int(page_begin), int(page_end),
                           _p(o), _p(lse))
    return o, lse


def query_codes(q_row, s):
    """Integer query of one row for one page ("SYCL", "Attention that reads 8-bit
    history": the integer query cache).  q_row: 256 bf16 bit patterns, s: the
    page's key channel scales in channel order -> (alpha float32, int8 codes)."""
    qi = np.empty(D_HEAD, np.int8)
    alpha = lib().orc_query_codes(_p(_c(q_row, np.uint16)), _p(_c(s, np.float32)), _p(qi))
    return np.float32(alpha), qi


def partial_int8_iq(H, G, q, rec_pool, page_table8, page_begin, page_end):
    """8-bit partial with the integer query (codes per page and row, integer dots)."""
    q = _c(q, np.uint16)
    pt = _c(page_table8, np.int32) if len(page_table8) else np.zeros(1, np.int32)
    o = np.empty((H * G, D_HEAD))
    lse = np.empty(H * G)
    lib().orc_partial_int8_iq(H, G, _p(q), _p(_c(rec_pool, np.uint8)), _p(pt), int(page_begin), int(page_end),
                              _p(o), _p(lse))
    return o, lse


def merge(o_parts, lse_parts):
    """o_parts [k][rows][d], lse_parts [k][rows] -> (o [rows][d], lse [rows])."""
    o_parts = _c(o_parts, np.float64)
    lse_parts = _c(lse_parts, np.float64)
    k, rows, d = o_parts.shape
    o = np.empty((rows, d))
    lse = np.empty(rows)
    lib().orc_merge(k, rows, d, _p(o_parts), _p(lse_parts), _p(o), _p(lse))
    return o, lse


def hybrid_batched(H, G, q, k_pool, v_pool, rec_pool, page_table, req_page_off, n_exact_tokens,
                   page_table8, req_page_off8, n_int8_pages, n_threads=1, int_query=False):
    q = _c(q, np.uint16)
    B = q.shape[0]
    o = np.empty((B, H * G, D_HEAD))
    lse = np.empty((B, H * G))
    pt = _c(page_table, np.int32) if len(page_table) else np.zeros(1, np.int32)
    pt8 = _c(page_table8, np.int32) if len(page_table8) else np.zeros(1, np.int32)
    lib().orc_hybrid_batched(B, H, G, _p(q), _p(_c(k_pool, np.uint16)), _p(_c(v_pool, np.uint16)),
                             _p(_c(rec_pool, np.uint8)), _p(pt), _p(_c(req_page_off, np.int32)),
                             _p(_c(n_exact_tokens, np.int32)), _p(pt8), _p(_c(req_page_off8, np.int32)),
                             _p(_c(n_int8_pages, np.int32)), _p(o), _p(lse), int(bool(int_query)),
                             int(n_threads))
    return o, lse


def hybrid_workload(w, rec_pool, n_threads=1, int_query=False):
    """Oracle hybrid step over a synth.Workload whose 8-bit pages are in rec_pool."""
    pt, off = w.exact_page_table()
    pt8, off8 = w.int8_page_table()
    return hybrid_batched(w.H, w.G, w.q, w.k_pool, w.v_pool, rec_pool, pt, off, w.n_ex.astype(np.int32),
                          pt8, off8, w.n8.astype(np.int32), n_threads, int_query)


def full_precision_workload(w, n_threads=1):
    """Unquantised reference: attention over the original BF16 of every token."""
    B = w.B
    pages = [np.asarray(p, np.int32) for p in w.pages]
    off = np.zeros(B + 1, np.int32)
    off[1:] = np.cumsum([len(p) for p in pages])
    flat = np.concatenate(pages)
    empty = np.zeros(B + 1, np.int32)
    rec_dummy = np.zeros(REC_BYTES, np.uint8)
    return hybrid_batched(w.H, w.G, w.q, w.k_pool, w.v_pool, rec_dummy, flat, off,
                          w.n_tokens.astype(np.int32), np.zeros(1, np.int32), empty, np.zeros(B, np.int32),
                          n_threads)
