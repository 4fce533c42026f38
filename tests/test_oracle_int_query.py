"""Pins of the oracle's integer-query variant against closed forms, hand-worked
codes, error bounds and an independent route (the float-query partial), none of
which reuse the oracle's code.

Source: "SYCL", section "Attention that reads 8-bit history": the kernel keeps an
integer query cache (8 rows x 256 channels, 2 KB), and a two-by-two experiment
decided which products run on integers.  Reading taken where the page is silent:
the query folded with the page's key channel scales is coded per page and row
with the absmax rule of the key codes (alpha = max|q'| / 127, rint half to even,
float32 steps).
"""
import numpy as np
import pytest

import oracle
from tiered_paged_kv_gb300 import synth

D = 256
SCALE = 1.0 / 16.0


def bf16_row(values):
    v = np.asarray(values, np.float32)
    b = synth.f32_to_bf16(v)
    assert np.array_equal(synth.bf16_to_f32(b), v), "test values must be exact in bfloat16"
    return b


def test_codes_of_a_representable_row():
    """q'_c = k_c / 64 with integer k_c and max |k| = 127: 127 / m is exactly 64, so
    the codes are the integers k_c and alpha is 1/64."""
    k = (np.floor(synth.uniform(1, 70, D) * 255) - 127).astype(np.int64)
    k[17] = -127
    s = np.ones(D, np.float32)
    alpha, qi = oracle.query_codes(bf16_row(k / 64.0), s)
    assert alpha == np.float32(1 / 64)
    assert np.array_equal(qi.astype(np.int64), k)


def test_codes_fold_the_channel_scales():
    """q_c = k_c * 2^-e_c with s_c = 2^(e_c + 3): q'_c = k_c * 8, codes k_c."""
    k = (np.floor(synth.uniform(2, 70, D) * 255) - 127).astype(np.int64)
    k[200] = 127
    e = (np.floor(synth.uniform(2, 71, D) * 9) - 4).astype(np.int64)
    s = np.exp2(e + 3).astype(np.float32)
    alpha, qi = oracle.query_codes(bf16_row(k * np.exp2(-e.astype(np.float64))), s)
    assert alpha == np.float32(8)  # m = 8 * 127
    assert np.array_equal(qi.astype(np.int64), k)


def test_ties_round_half_to_even():
    """With 127 / m = 64, q = (2j + 1) / 128 lands on j + 1/2: half to even."""
    q = np.zeros(D)
    q[0] = 127 / 64
    halves = [1, 3, 5, 7, -1, -3, -5, 9]    # q * 64 = 0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 4.5
    expect = [0, 2, 2, 4, 0, -2, -2, 4]      # worked by hand
    for i, h in enumerate(halves):
        q[1 + i] = h / 128
    alpha, qi = oracle.query_codes(bf16_row(q), np.ones(D, np.float32))
    assert qi[0] == 127 and alpha == np.float32(1 / 64)
    assert list(qi[1:1 + len(halves)]) == expect
    assert not qi[1 + len(halves):].any()


def test_zero_row_gives_zero_codes():
    alpha, qi = oracle.query_codes(np.zeros(D, np.uint16), np.ones(D, np.float32))
    assert alpha == 0 and not qi.any()


def page_scales(seed):
    """Key channel scales of a page converted by the oracle's quantiser."""
    k = synth.normal_bf16(seed, 72, 64 * D).reshape(64, D)
    s, _, _ = oracle.channel_scales(k)
    return s


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_code_error_bound_and_absmax(seed):
    """|alpha qi_c - q'_c| <= alpha / 2 (plus float32 rounding), the absmax channel
    codes to +-127, and alpha is max |q'| / 127."""
    s = page_scales(seed)
    for r in range(8):
        q = synth.normal_bf16(seed, 73 + r, D)
        alpha, qi = oracle.query_codes(q, s)
        qp = synth.bf16_to_f32(q).astype(np.float64) * s.astype(np.float64)
        m = np.abs(qp).max()
        assert abs(float(alpha) - m / 127) <= 2 ** -23 * m / 127
        assert np.abs(qi.astype(np.int64)).max() == 127
        assert np.abs(qi[np.argmax(np.abs(qp))]) == 127
        err = np.abs(float(alpha) * qi.astype(np.float64) - qp)
        assert err.max() <= float(alpha) / 2 * (1 + 2 ** -20) + 2 ** -22 * m


def test_codes_are_invariant_to_a_power_of_two():
    s = page_scales(6)
    q = synth.normal_bf16(6, 80, D)
    a1, q1 = oracle.query_codes(q, s)
    a2, q2 = oracle.query_codes(synth.f32_to_bf16(synth.bf16_to_f32(q) * 8), s)
    assert np.array_equal(q1, q2) and a2 == a1 * 8


def records_with_exact_query(seed, n_pages, H, G):
    """Records with s_c = 2^(e_c + E_p) and a query q_c = k_c 2^-e_c: on every page
    q'_c = k_c 2^E_p with max |k| = 127 per row, so the integer query is exact."""
    kc = (np.floor(synth.uniform(seed, 81, n_pages * H * 64 * D) * 255) - 127).astype(np.int8)
    vc = (np.floor(synth.uniform(seed, 82, n_pages * H * 64 * D) * 255) - 127).astype(np.int8)
    kc = kc.reshape(n_pages, H, 64, D)
    vc = vc.reshape(n_pages, H, 64, D)
    e = (np.floor(synth.uniform(seed, 83, D) * 7) - 3).astype(np.int64)
    Ep = (np.floor(synth.uniform(seed, 84, n_pages * H) * 5) - 2).astype(np.int64).reshape(n_pages, H)
    r = np.exp2(np.floor(synth.uniform(seed, 85, n_pages * H * 64) * 5) - 9).reshape(n_pages, H, 64)
    u = np.exp2(np.floor(synth.uniform(seed, 86, n_pages * H * D) * 5) - 9).reshape(n_pages, H, D)
    recs = np.zeros((n_pages, H, oracle.REC_BYTES), np.uint8)
    for p in range(n_pages):
        for h in range(H):
            s = np.exp2(e + Ep[p, h]).astype(np.float32)
            recs[p, h] = oracle.pack_record(kc[p, h], vc[p, h], s, r[p, h].astype(np.float32),
                                            u[p, h].astype(np.float32))
    k = (np.floor(synth.uniform(seed, 87, H * G * D) * 255) - 127).astype(np.int64).reshape(H * G, D)
    k[:, 5] = 127
    q = synth.f32_to_bf16((k * np.exp2(-e.astype(np.float64))[None, :]).astype(np.float32))
    assert np.array_equal(synth.bf16_to_f32(q).astype(np.float64), k * np.exp2(-e.astype(np.float64))[None, :])
    return recs, q


def test_iq_partial_equals_float_partial_when_the_query_is_exact():
    """Independent route: with an exactly representable integer query the integer
    dots must give the float-query partial (dequantise, then attend)."""
    H, G, n_pages = 2, 8, 3
    recs, q = records_with_exact_query(7, n_pages, H, G)
    slots = synth.permutation(7, 88, n_pages).astype(np.int32)
    pool = np.zeros((n_pages, H, oracle.REC_BYTES), np.uint8)
    for p in range(n_pages):
        pool[slots[p]] = recs[p]
    for b, e in [(0, 3), (1, 3), (2, 2)]:
        oi, li = oracle.partial_int8_iq(H, G, q, pool.reshape(-1), slots, b, e)
        of, lf = oracle.partial_int8(H, G, q, pool.reshape(-1), slots, b, e)
        assert np.allclose(oi, of, rtol=0, atol=1e-13 * max(1.0, np.abs(of).max()))
        assert np.allclose(li, lf, rtol=0, atol=1e-12) or (b == e and np.all(np.isneginf(li)))


def test_iq_zero_query_gives_mean_value():
    """q = 0: every score is 0, so o is the mean of the dequantised values and
    lse = ln n."""
    H, G, n_pages = 1, 8, 2
    recs, _ = records_with_exact_query(8, n_pages, H, G)
    pool = recs.reshape(-1)
    q = np.zeros((H * G, D), np.uint16)
    o, lse = oracle.partial_int8_iq(H, G, q, pool, np.arange(n_pages, dtype=np.int32), 0, n_pages)
    vals = []
    for p in range(n_pages):
        _, vc, _, _, u = oracle.record_fields(recs[p, 0])
        vals.append(vc.astype(np.float64) * u.astype(np.float64)[None, :])
    mean = np.concatenate(vals).mean(axis=0)
    assert np.allclose(o, np.repeat(mean[None], G, axis=0), rtol=0, atol=1e-14)
    assert np.allclose(lse, np.log(n_pages * 64), rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", [9, 10])
def test_iq_lse_within_the_coding_bound(seed):
    """Each score moves by at most delta_t = scale r_t sum_c |kc_tc| alpha / 2 (the
    code error bound), so |lse_iq - lse_float| <= max_t delta_t per row."""
    H, G, n_pages = 1, 8, 4
    w = synth.make_workload([n_pages * 64], 0, H=H, G=G, seed=seed)
    pt = np.asarray(w.pages[0], np.int32)
    pool = np.zeros((w.n_slots, H, oracle.REC_BYTES), np.uint8)
    oracle.quantize_pages(H, w.k_pool, w.v_pool, pt, pt, pool.reshape(-1))
    q = w.q[0]
    oi, li = oracle.partial_int8_iq(H, G, q, pool.reshape(-1), pt, 0, n_pages)
    of, lf = oracle.partial_int8(H, G, q, pool.reshape(-1), pt, 0, n_pages)
    for g in range(G):
        bound = 0.0
        for p in range(n_pages):
            kc, _, s, r, _ = oracle.record_fields(pool[pt[p], 0])
            alpha, _ = oracle.query_codes(q[g], s)
            delta = SCALE * r.astype(np.float64) * np.abs(kc.astype(np.float64)).sum(axis=1) * float(alpha) / 2
            bound = max(bound, delta.max() * (1 + 1e-5))
        assert abs(li[g] - lf[g]) <= bound
        assert abs(li[g] - lf[g]) > 0  # the coding did change something
        v_max = np.abs(of[g]).max() + 1
        assert np.abs(oi[g] - of[g]).max() <= (np.exp(2 * bound) - 1) * 4 * v_max


def test_hybrid_int_query_on_all_exact_requests_is_the_float_result():
    w = synth.make_workload([130, 64, 1], None, H=2, seed=11)
    rec_pool = np.zeros(oracle.REC_BYTES, np.uint8)
    o1, l1 = oracle.hybrid_workload(w, rec_pool, int_query=True)
    o2, l2 = oracle.hybrid_workload(w, rec_pool)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_hybrid_int_query_joins_the_iq_partial_and_thread_count():
    w = synth.make_workload([5 * 64 + 37, 3 * 64], 64, H=2, seed=12)
    pool = np.zeros((w.n_slots, w.H, oracle.REC_BYTES), np.uint8)
    pt8, off8 = w.int8_page_table()
    oracle.quantize_pages(w.H, w.k_pool, w.v_pool, pt8, pt8, pool.reshape(-1))
    o1, l1 = oracle.hybrid_workload(w, pool.reshape(-1), n_threads=1, int_query=True)
    o3, l3 = oracle.hybrid_workload(w, pool.reshape(-1), n_threads=3, int_query=True)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)
    # request 0 alone: the fold of its exact partial and its integer-query partial
    b = 0
    pt, off = w.exact_page_table()
    oe, le = oracle.partial_exact(w.H, w.G, w.q[b], w.k_pool, w.v_pool, pt[off[b]:off[b + 1]], 0, int(w.n_ex[b]))
    oi, li = oracle.partial_int8_iq(w.H, w.G, w.q[b], pool.reshape(-1), pt8[off8[b]:off8[b + 1]], 0, int(w.n8[b]))
    om, lm = oracle.merge(np.stack([oe, oi]), np.stack([le, li]))
    assert np.allclose(o1[b], om, rtol=0, atol=1e-14) and np.allclose(l1[b], lm, rtol=0, atol=1e-14)
