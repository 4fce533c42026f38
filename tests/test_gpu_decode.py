"""GPU tier partials and merge against the oracle on the same inputs (same BF16
pages, same 8-bit records): outputs within 1e-3 of max|o|, lse within 1e-3,
empty partials exact, ragged ranges, splits and poisoned slots."""
import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import (DevWorkload, assert_close, dev_f32, dev_i32, oracle_records, split_ranges_exact,
                          split_ranges_int8, torch)

pytestmark = pytest.mark.gpu
IMPLS = [tpk.IMPL_SIMT, tpk.IMPL_TENSOR]


def run_exact(d, b, e, S, row_q=0):
    t = torch()
    w = d.w
    rows = w.H * w.G
    o = t.full((S, rows, 256), float("nan"), dtype=t.float32, device="cuda")
    lse = t.full((S, rows), float("nan"), dtype=t.float32, device="cuda")
    pt = dev_i32(w.pages[row_q])
    tpk.decode_attn_exact(d.shape, d.q[row_q], d.k, d.v, pt, b, e, S, o, lse)
    t.cuda.synchronize()
    return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def run_int8(d, pb, pe, S, row_q=0):
    t = torch()
    w = d.w
    rows = w.H * w.G
    o = t.full((S, rows, 256), float("nan"), dtype=t.float32, device="cuda")
    lse = t.full((S, rows), float("nan"), dtype=t.float32, device="cuda")
    pt = dev_i32(w.pages[row_q])
    tpk.decode_attn_int8(d.shape, d.q[row_q], d.rec, pt, pb, pe, S, o, lse)
    t.cuda.synchronize()
    return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("b,e,S", [(0, 1, 1), (0, 63, 1), (0, 64, 1), (0, 65, 2), (37, 1000, 3), (0, 3000, 7),
                                   (5, 5, 2), (100, 200, 9), (0, 3000, 1)])
def test_exact_partials(impl, b, e, S):
    w = synth.make_workload([3000], None, H=4, seed=11)
    d = DevWorkload(w, impl)
    o, lse = run_exact(d, b, e, S)
    for s, (tb, te) in enumerate(split_ranges_exact(b, e, S)):
        oo, ol = oracle.partial_exact(w.H, w.G, w.q[0], w.k_pool, w.v_pool, w.pages[0], tb, te)
        if te == tb:
            assert np.all(o[s] == 0) and np.all(lse[s] == -np.inf)
        else:
            assert_close(o[s], lse[s], oo, ol, f"split {s} [{tb},{te})", exact_only=True)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("kind", ["loguniform", "outliers"])
@pytest.mark.parametrize("pb,pe,S", [(0, 1, 1), (0, 12, 1), (0, 12, 5), (3, 11, 2), (4, 4, 1), (0, 40, 40),
                                     (0, 3, 8)])
def test_int8_partials_on_same_codes(impl, kind, pb, pe, S):
    w = synth.make_workload([64 * 40], 0, H=2, seed=12, key_sigma=kind, value_sigma="loguniform"
                            if kind == "loguniform" else "unit")
    rec = oracle_records(w)
    d = DevWorkload(w, impl)
    d.load_records(rec)
    o, lse = run_int8(d, pb, pe, S)
    for s, (a, b) in enumerate(split_ranges_int8(pb, pe, S)):
        oo, ol = oracle.partial_int8(w.H, w.G, w.q[0], rec, w.pages[0], a, b)
        if a == b:
            assert np.all(o[s] == 0) and np.all(lse[s] == -np.inf)
        else:
            assert_close(o[s], lse[s], oo, ol, f"split {s} pages [{a},{b})")


@pytest.mark.parametrize("impl", IMPLS)
def test_split_at_random_point_then_merge_equals_unsplit(impl):
    """Exact-tier history cut at seeded points: two calls + GPU merge vs one call."""
    w = synth.make_workload([4096 + 77], None, H=4, seed=13)
    d = DevWorkload(w, impl)
    t = torch()
    full_o, full_l = run_exact(d, 0, 4173, 1)
    for x in synth.randint(13, synth.TID_SPLIT, 4, 1, 4172):
        a_o, a_l = run_exact(d, 0, int(x), 1)
        b_o, b_l = run_exact(d, int(x), 4173, 1)
        acc_o = dev_f32(np.zeros((32, 256)))
        acc_l = dev_f32(np.full(32, -np.inf))
        parts_o = dev_f32(np.stack([a_o[0], b_o[0]]))
        parts_l = dev_f32(np.stack([a_l[0], b_l[0]]))
        tpk.merge_lse(2, 32, 256, parts_o, parts_l, acc_o, acc_l)
        t.cuda.synchronize()
        assert_close(acc_o.cpu().numpy().astype(np.float64), acc_l.cpu().numpy().astype(np.float64), full_o[0],
                     full_l[0], f"split at {x}", exact_only=True)


def merge_on_gpu(parts_o, parts_l):
    """Fold partials [k][rows][256], [k][rows] into an empty accumulator on the GPU."""
    t = torch()
    k, rows = parts_l.shape
    acc_o = dev_f32(np.zeros((rows, 256)))
    acc_l = dev_f32(np.full(rows, -np.inf))
    tpk.merge_lse(k, rows, 256, dev_f32(parts_o), dev_f32(parts_l), acc_o, acc_l)
    t.cuda.synchronize()
    return acc_o.cpu().numpy().astype(np.float64), acc_l.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("impl", IMPLS)
def test_full_exact_32k_split_at_random_point(impl):
    """The exact-tier workload at full size (32,768 tokens in 512 pages at a seeded
    permutation of slots, 4 KV heads x 8 query rows): the history cut at seeded
    uniform points in [1, N - 1], each side decoded by its own call and every
    partial merged on the GPU, against one call over the whole history (merged
    the same way) and against the oracle's unsplit attention."""
    w = synth.exact_32k(seed=1)
    N = int(w.n_tokens[0])
    d = DevWorkload(w, impl)
    u_o, u_l = merge_on_gpu(*run_exact(d, 0, N, 32))
    oo, ol = oracle.partial_exact(w.H, w.G, w.q[0], w.k_pool, w.v_pool, w.pages[0], 0, N)
    assert_close(u_o, u_l, oo, ol, "unsplit", exact_only=True)
    for x in synth.randint(1, synth.TID_SPLIT, 3, 1, N - 1):
        a_o, a_l = run_exact(d, 0, int(x), 16)
        b_o, b_l = run_exact(d, int(x), N, 16)
        m_o, m_l = merge_on_gpu(np.concatenate([a_o, b_o]), np.concatenate([a_l, b_l]))
        assert_close(m_o, m_l, u_o, u_l, f"split at {x} vs unsplit", exact_only=True)
        assert_close(m_o, m_l, oo, ol, f"split at {x} vs oracle", exact_only=True)


@pytest.mark.parametrize("impl", IMPLS)
def test_full_int8_tier_128k_split_at_random_page(impl):
    """The 8-bit tier of the 128K hybrid workload at full size (1,984 pages x 4 KV
    heads, the oracle's records) through the primitive 8-bit call: the page range cut
    at seeded pages, each side decoded by its own call and every partial merged on
    the GPU, against one call over the whole range and against the oracle."""
    w = synth.hybrid_128k(seed=2)
    P = int(w.n8[0])
    rec = oracle_records(w)
    d = DevWorkload(w, impl)
    d.load_records(rec)
    u_o, u_l = merge_on_gpu(*run_int8(d, 0, P, 38))
    oo, ol = oracle.partial_int8(w.H, w.G, w.q[0], rec, w.pages[0], 0, P)
    assert_close(u_o, u_l, oo, ol, "unsplit")
    for x in synth.randint(2, synth.TID_SPLIT, 2, 1, P - 1):
        a_o, a_l = run_int8(d, 0, int(x), 19)
        b_o, b_l = run_int8(d, int(x), P, 19)
        m_o, m_l = merge_on_gpu(np.concatenate([a_o, b_o]), np.concatenate([a_l, b_l]))
        assert_close(m_o, m_l, u_o, u_l, f"split at page {x} vs unsplit")
        assert_close(m_o, m_l, oo, ol, f"split at page {x} vs oracle")


def test_merge_matches_oracle_and_empty_is_identity():
    t = torch()
    rows = 24
    o_parts = synth.normal(1, 70, 5 * rows * 256).reshape(5, rows, 256)
    l_parts = synth.normal(1, 71, 5 * rows).reshape(5, rows) * 4.0
    l_parts[2, :7] = -np.inf
    l_parts[:, 20] = -np.inf                          # an all-empty row
    o_parts[2, :7] = np.nan                           # never read
    o_parts[:, 20] = np.nan
    acc_o0 = synth.normal(1, 72, rows * 256).reshape(rows, 256)
    acc_l0 = synth.normal(1, 73, rows) * 4.0
    acc_l0[20] = -np.inf
    acc_o0[20] = 0.0
    acc_o = dev_f32(acc_o0)
    acc_l = dev_f32(acc_l0)
    tpk.merge_lse(5, rows, 256, dev_f32(o_parts), dev_f32(l_parts), acc_o, acc_l)
    t.cuda.synchronize()
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    oo, ol = oracle.merge(np.concatenate([f32(acc_o0)[None], f32(o_parts)]),
                          np.concatenate([f32(acc_l0)[None], f32(l_parts)]))
    go = acc_o.cpu().numpy().astype(np.float64)
    gl = acc_l.cpu().numpy().astype(np.float64)
    assert np.all(go[20] == 0) and gl[20] == -np.inf
    assert_close(go, gl, oo, ol, "merge", exact_only=True)
    # an empty partial leaves the accumulator bit-identical
    before_o = acc_o.clone()
    before_l = acc_l.clone()
    tpk.merge_lse(1, rows, 256, dev_f32(np.full((1, rows, 256), np.nan)), dev_f32(np.full((1, rows), -np.inf)),
                  acc_o, acc_l)
    t.cuda.synchronize()
    assert t.equal(acc_o, before_o) and t.equal(acc_l, before_l)


@pytest.mark.parametrize("impl", IMPLS)
def test_poisoned_tail_tokens_are_not_read(impl):
    """Tokens past the range in the last page hold NaN; they must not leak."""
    w = synth.make_workload([150], None, H=1, seed=14)
    last = w.pages[0][2]
    w.k_pool[last, :, 150 - 128:] = synth.BF16_NAN
    w.v_pool[last, :, 150 - 128:] = synth.BF16_NAN
    d = DevWorkload(w, impl)
    o, lse = run_exact(d, 0, 150, 1)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    oo, ol = oracle.partial_exact(w.H, w.G, w.q[0], w.k_pool, w.v_pool, w.pages[0], 0, 150)
    assert_close(o[0], lse[0], oo, ol, "poisoned tail", exact_only=True)


@pytest.mark.parametrize("impl", IMPLS)
def test_out_of_pool_page_is_skipped_and_reported(impl):
    w = synth.make_workload([256], None, H=1, seed=15)
    d = DevWorkload(w, impl)
    tpk.get_device_status(reset=True)
    bad = np.array(w.pages[0], np.int32)
    bad[1] = w.n_slots + 3
    t = torch()
    o = t.empty((1, 8, 256), dtype=t.float32, device="cuda")
    lse = t.empty((1, 8), dtype=t.float32, device="cuda")
    tpk.decode_attn_exact(d.shape, d.q[0], d.k, d.v, dev_i32(bad), 0, 256, 1, o, lse)
    st, flags = tpk.get_device_status(reset=True)
    assert st == 4 and flags & 1
    # the result equals attention over the remaining pages
    keep = [0, 2, 3]
    pt = np.array([w.pages[0][i] for i in keep], np.int32)
    oo, ol = oracle.partial_exact(w.H, w.G, w.q[0], w.k_pool, w.v_pool, pt, 0, 192)
    assert_close(o.cpu().numpy()[0].astype(np.float64), lse.cpu().numpy()[0].astype(np.float64), oo, ol, "skip", exact_only=True)
