"""Helpers shared by the GPU parity tests: move synthetic workloads to the
device, call the library through its C ABI, and compare with the oracle."""
import json
import os

import numpy as np

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth

# Parity tolerances.  Outputs: max |o_gpu - o_oracle| <= O_TOL * max |o_oracle|
# (the bar the method is held to against the oracle on the same codes).  lse
# (natural-log units), held near the precision each tier's kernel reaches:
#  - exact tier only: LSE_TOL_EXACT absolute (bf16 inputs, float32 scores;
#    observed at most 1.1e-6 over the suite);
#  - with 8-bit pages: LSE_TOL_8BIT + LSE_REL_8BIT * max|lse|, capped at 1e-3.  The
#    8-bit tier's products run on code + 1152 with the offset removed after the
#    float32 sum, which keeps about 15 bits of a score relative to its size
#    (observed at most 1e-4 + 2.7e-5 max|lse|, and 5.3e-4 in all, over the suite).
# Queries scaled far beyond unit variance have a bar of their own that grows with
# |lse| (test_extreme_query_scales).
O_TOL = 1e-3
LSE_TOL_EXACT = 1e-5
LSE_TOL_8BIT = 1e-4
LSE_REL_8BIT = 4e-5
LSE_CAP = 1e-3


def lse_bar(ol, exact_only=False):
    """The lse bar of one comparison (ol: the oracle's lse)."""
    if exact_only:
        return LSE_TOL_EXACT
    fin = np.isfinite(ol)
    m = np.abs(ol[fin]).max() if fin.any() else 0.0
    return min(LSE_CAP, LSE_TOL_8BIT + LSE_REL_8BIT * m)


# Record slots no page uses are filled with this byte: every scale reads as a NaN
# (0xffffffff), so a stray read of an unused record shows up in the output.
REC_POISON = 0xFF


def torch():
    import torch as t
    return t


def dev_u16(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def dev_i32(a):
    t = torch()
    a = np.ascontiguousarray(a, np.int32)
    if a.size == 0:
        a = np.zeros(1, np.int32)
    return t.from_numpy(a).cuda()


def dev_u8(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def dev_f32(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


class DevWorkload:
    """A synth.Workload resident on the GPU."""

    def __init__(self, w, impl=tpk.IMPL_DEFAULT):
        t = torch()
        self.w = w
        self.shape = tpk.Shape(w.H, impl=impl, kv_slots=w.n_slots, rec_slots=w.n_slots)
        self.k = dev_u16(w.k_pool)
        self.v = dev_u16(w.v_pool)
        self.q = dev_u16(w.q)
        self.rec = t.full((w.n_slots * w.H * tpk.RECORD_BYTES,), REC_POISON, dtype=t.uint8, device="cuda")
        pt, self.off = w.exact_page_table()
        pt8, self.off8 = w.int8_page_table()
        self.pt = dev_i32(pt)
        self.pt8 = dev_i32(pt8)

    def quantize_gpu(self):
        slots = dev_i32(self.w.int8_slots())
        n = len(self.w.int8_slots())
        tpk.kv_quantize_pages(self.shape, self.k, self.v, slots, slots, n, self.rec)
        return self.rec.cpu().numpy()

    def load_records(self, rec_host):
        self.rec.copy_(torch().from_numpy(np.ascontiguousarray(rec_host, np.uint8)))

    def hybrid(self):
        t = torch()
        w = self.w
        o = t.empty(w.B, w.H * w.G, 256, dtype=t.float32, device="cuda")
        lse = t.empty(w.B, w.H * w.G, dtype=t.float32, device="cuda")
        nbytes = tpk.hybrid_workspace_bytes(self.shape, w.B)
        ws = t.empty(nbytes, dtype=t.uint8, device="cuda")
        tpk.workspace_init(ws, nbytes)
        tpk.decode_hybrid_batched(self.shape, w.B, self.q, self.k, self.v, self.rec, self.pt, self.off, w.n_ex,
                                  self.pt8, self.off8, w.n8, o, lse, ws, nbytes)
        t.cuda.synchronize()
        return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def oracle_records(w):
    rec = np.full(w.n_slots * w.H * oracle.REC_BYTES, REC_POISON, np.uint8)
    s = w.int8_slots()
    oracle.quantize_pages(w.H, w.k_pool, w.v_pool, s, s, rec)
    return rec


def _record(what, err, lerr, lse_max):
    """With TPK_RECORD_ERRORS set to a file path, append each comparison's errors
    (how far inside the bars the results land)."""
    path = os.environ.get("TPK_RECORD_ERRORS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", ""), "what": what, "o_err": float(err),
                                "lse_err": float(lerr), "lse_absmax": float(lse_max)}) + "\n")


def assert_close(o, lse, oo, ol, what="", exact_only=False):
    """o, lse against the oracle's oo, ol; exact_only: no 8-bit page took part."""
    scale = max(np.abs(oo).max(), 1e-30)
    err = np.abs(o - oo).max() / scale
    fin = np.isfinite(ol)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: -inf pattern differs"
    assert np.all(lse[~fin] == ol[~fin]), f"{what}: empty rows differ"
    lerr = np.abs(lse[fin] - ol[fin]).max() if fin.any() else 0.0
    _record(what, err, lerr, np.abs(ol[fin]).max() if fin.any() else 0.0)
    bar = lse_bar(ol, exact_only)
    assert err <= O_TOL, f"{what}: max|do|/max|o| = {err:.3e} > {O_TOL}"
    assert lerr <= bar, f"{what}: max|dlse| = {lerr:.3e} > {bar:.3e}"
    return err, lerr


def split_ranges_exact(tok_begin, tok_end, S):
    """Token pieces of tpk_decode_attn_exact: page-aligned cuts of the range."""
    pg0 = tok_begin // 64
    pg1 = (tok_end + 63) // 64
    P = pg1 - pg0
    out = []
    for s in range(S):
        pa = pg0 + (P * s) // S
        pb = pg0 + (P * (s + 1)) // S
        b = max(tok_begin, pa * 64)
        e = min(tok_end, pb * 64)
        out.append((b, max(b, e)))
    return out


def split_ranges_int8(page_begin, page_end, S):
    P = page_end - page_begin
    return [(page_begin + (P * s) // S, page_begin + (P * (s + 1)) // S) for s in range(S)]
