"""Pins of the oracle's attention, tier partials and merge against closed forms,
invariants and an independent route, none of which reuse the oracle's code.

Sources: "SYCL", sections "Attention that reads 8-bit history" and "A merge that
joins the tiers"; "ActiveKV", section "The idea" (tiers joined exactly).
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from tiered_paged_kv_gb300 import synth

D = 256
SCALE = 1.0 / 16.0


def rnd(seed, *shape):
    return synth.normal(seed, 50, int(np.prod(shape))).reshape(shape)


def test_single_token_returns_value_and_score():
    q, K, V = rnd(1, 3, D), rnd(2, 1, D), rnd(3, 1, D)
    o, lse = oracle.attend(q, K, V)
    assert np.allclose(o, np.repeat(V, 3, axis=0), rtol=0, atol=1e-15)
    for r in range(3):
        assert abs(lse[r] - SCALE * float(np.dot(q[r], K[0]))) < 1e-12


def test_zero_query_gives_mean_value():
    K, V = rnd(4, 7, D), rnd(5, 7, D)
    o, lse = oracle.attend(np.zeros((2, D)), K, V)
    assert np.allclose(o, V.mean(axis=0)[None, :], atol=1e-14)
    assert np.allclose(lse, np.log(7.0), atol=1e-14)


def test_identical_keys_give_mean_value():
    q, k, V = rnd(6, 4, D), rnd(7, 1, D), rnd(8, 5, D)
    o, lse = oracle.attend(q, np.repeat(k, 5, axis=0), V)
    assert np.allclose(o, V.mean(axis=0)[None, :], atol=1e-14)
    assert np.allclose(lse, SCALE * (q @ k[0]) + np.log(5.0), atol=1e-12)


def test_two_tokens_logistic_closed_form():
    q, K, V = rnd(9, 5, D), rnd(10, 2, D), rnd(11, 2, D)
    o, lse = oracle.attend(q, K, V)
    for r in range(5):
        s1 = SCALE * float(np.dot(q[r], K[0]))
        s2 = SCALE * float(np.dot(q[r], K[1]))
        w1 = expit(s1 - s2)
        assert np.allclose(o[r], w1 * V[0] + (1 - w1) * V[1], atol=1e-13)
        assert abs(lse[r] - (max(s1, s2) + np.log1p(np.exp(-abs(s1 - s2))))) < 1e-12


def test_empty_is_zero_and_minus_inf():
    o, lse = oracle.attend(rnd(12, 2, D), np.zeros((0, D)), np.zeros((0, D)))
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_linearity_permutation_and_shift():
    q, K, V1, V2 = rnd(13, 3, D), rnd(14, 9, D), rnd(15, 9, D), rnd(16, 9, D)
    o1, l1 = oracle.attend(q, K, V1)
    o2, _ = oracle.attend(q, K, V2)
    o12, _ = oracle.attend(q, K, 2.0 * V1 - 0.5 * V2)
    assert np.allclose(o12, 2.0 * o1 - 0.5 * o2, atol=1e-13)
    perm = synth.permutation(3, 1, 9)
    op, lp = oracle.attend(q, K[perm], V1[perm])
    assert np.allclose(op, o1, atol=1e-13) and np.allclose(lp, l1, atol=1e-13)
    delta = rnd(17, 1, D)
    os_, ls = oracle.attend(q, K + delta, V1)
    assert np.allclose(os_, o1, atol=1e-12)
    assert np.allclose(ls, l1 + SCALE * (q @ delta[0]), atol=1e-12)


def test_dominant_key_selects_its_value():
    q = rnd(18, 1, D)
    K = rnd(19, 6, D) * 0.01
    K[4] = q[0] * (16.0 * 60.0 / float(q[0] @ q[0]))   # score 60 above the rest
    V = rnd(20, 6, D)
    o, _ = oracle.attend(q, K, V)
    assert np.allclose(o[0], V[4], atol=1e-20)


def test_scores_use_1_over_sqrt_d():
    """Scaling q by 16 with unit-norm keys gives weights softmax(q . k)."""
    q = rnd(21, 1, D)
    K = np.eye(D)[:3]
    V = np.eye(D)[:3]
    o, _ = oracle.attend(16.0 * q, K, V)
    e = np.exp(q[0, :3] - q[0, :3].max())
    assert np.allclose(o[0, :3], e / e.sum(), atol=1e-14)


# ---------------------------------------------------------------- merge


def _parts(seed, k, rows):
    o = rnd(seed, k, rows, D)
    lse = rnd(seed + 1, k, rows) * 3.0
    return o, lse


@pytest.mark.parametrize("split", [1, 5, 31, 63, 64, 65, 99])
def test_split_then_merge_equals_unsplit(split):
    q, K, V = rnd(22, 8, D), rnd(23, 100, D), rnd(24, 100, D)
    o, lse = oracle.attend(q, K, V)
    oa, la = oracle.attend(q, K[:split], V[:split])
    ob, lb = oracle.attend(q, K[split:], V[split:])
    om, lm = oracle.merge(np.stack([oa, ob]), np.stack([la, lb]))
    assert np.allclose(om, o, rtol=1e-12, atol=1e-13) and np.allclose(lm, lse, rtol=1e-12, atol=1e-12)


def test_merge_with_empty_partial_is_identity():
    o, lse = _parts(30, 1, 4)
    garbage = np.full((1, 4, D), np.nan)
    om, lm = oracle.merge(np.concatenate([o, garbage]), np.concatenate([lse, np.full((1, 4), -np.inf)]))
    assert np.array_equal(om, o[0]) and np.array_equal(lm, lse[0])


def test_merge_all_empty():
    om, lm = oracle.merge(np.full((3, 2, D), np.nan), np.full((3, 2), -np.inf))
    assert np.all(om == 0) and np.all(lm == -np.inf)


def test_merge_order_independent():
    o, lse = _parts(31, 6, 3)
    om, lm = oracle.merge(o, lse)
    p = synth.permutation(2, 2, 6)
    om2, lm2 = oracle.merge(o[p], lse[p])
    assert np.allclose(om, om2, rtol=1e-12, atol=1e-14) and np.allclose(lm, lm2, rtol=1e-12)


def test_merge_two_parts_closed_form():
    o, lse = _parts(32, 2, 3)
    om, lm = oracle.merge(o, lse)
    w = expit(lse[0] - lse[1])
    assert np.allclose(om, w[:, None] * o[0] + (1 - w[:, None]) * o[1], atol=1e-13)
    assert np.allclose(lm, np.logaddexp(lse[0], lse[1]), atol=1e-13)


# ---------------------------------------------------------- paged partials


def test_paged_exact_partial_equals_logical_attention():
    """Paged gather with permuted slots, token sub-range and GQA head mapping."""
    w = synth.make_workload([300], None, H=2, G=4, seed=7)
    pt = np.asarray(w.pages[0])
    K = synth.bf16_to_f32(w.k_pool[pt]).astype(np.float64)  # [pages][H][64][D]
    V = synth.bf16_to_f32(w.v_pool[pt]).astype(np.float64)
    q = synth.bf16_to_f32(w.q[0]).astype(np.float64)
    b, e = 37, 261
    o, lse = oracle.partial_exact(2, 4, w.q[0], w.k_pool, w.v_pool, pt, b, e)
    for h in range(2):
        Kh = K[:, h].reshape(-1, D)[b:e]
        Vh = V[:, h].reshape(-1, D)[b:e]
        oh, lh = oracle.attend(q[h * 4:(h + 1) * 4], Kh, Vh)
        assert np.array_equal(o[h * 4:(h + 1) * 4], oh) and np.array_equal(lse[h * 4:(h + 1) * 4], lh)


def representable_records(seed, n_pages, H):
    """Records whose dequantised values are exactly representable in bfloat16, with
    the BF16 pages holding those same values."""
    rng_c = synth.uniform(seed, 60, n_pages * H * 64 * D * 2)
    codes = np.floor(rng_c * 255).astype(np.int64) - 127
    kc = codes[: n_pages * H * 64 * D].reshape(n_pages, H, 64, D).astype(np.int8)
    vc = codes[n_pages * H * 64 * D:].reshape(n_pages, H, 64, D).astype(np.int8)
    e = synth.uniform(seed, 61, n_pages * H * (D + 64 + D))
    ex = np.floor(e * 7).astype(np.int64) - 3
    s = np.exp2(ex[: n_pages * H * D]).reshape(n_pages, H, D).astype(np.float32)
    r = np.exp2(ex[n_pages * H * D: n_pages * H * (D + 64)] - 7).reshape(n_pages, H, 64).astype(np.float32)
    u = np.exp2(ex[n_pages * H * (D + 64):] - 7).reshape(n_pages, H, D).astype(np.float32)
    recs = np.zeros((n_pages, H, oracle.REC_BYTES), np.uint8)
    kp = np.zeros((n_pages, H, 64, D), np.uint16)
    vp = np.zeros((n_pages, H, 64, D), np.uint16)
    for p in range(n_pages):
        for h in range(H):
            recs[p, h] = oracle.pack_record(kc[p, h], vc[p, h], s[p, h], r[p, h], u[p, h])
            kv = kc[p, h].astype(np.float32) * s[p, h][None, :] * r[p, h][:, None]
            vv = vc[p, h].astype(np.float32) * u[p, h][None, :]
            kp[p, h] = synth.f32_to_bf16(kv)
            vp[p, h] = synth.f32_to_bf16(vv)
            assert np.array_equal(synth.bf16_to_f32(kp[p, h]), kv)
            assert np.array_equal(synth.bf16_to_f32(vp[p, h]), vv)
    return recs, kp, vp


def test_int8_partial_equals_exact_partial_on_representable_pages():
    """Independent route through the record layout: the 8-bit partial over records
    must equal the exact partial over BF16 pages holding the dequantised values."""
    H, G, n_pages = 2, 8, 3
    recs, kp, vp = representable_records(3, n_pages, H)
    slots = synth.permutation(4, 1, n_pages).astype(np.int32)
    rec_pool = np.zeros((n_pages, H, oracle.REC_BYTES), np.uint8)
    kpool = np.zeros_like(kp)
    vpool = np.zeros_like(vp)
    for p in range(n_pages):
        rec_pool[slots[p]] = recs[p]
        kpool[slots[p]] = kp[p]
        vpool[slots[p]] = vp[p]
    q = synth.normal_bf16(5, 1, H * G * D).reshape(H * G, D)
    o8, l8 = oracle.partial_int8(H, G, q, rec_pool.reshape(-1), slots, 0, n_pages)
    oe, le = oracle.partial_exact(H, G, q, kpool, vpool, slots, 0, n_pages * 64)
    assert np.allclose(o8, oe, rtol=0, atol=1e-14 * np.abs(oe).max())
    assert np.allclose(l8, le, rtol=0, atol=1e-13)
    # a sub-range of pages
    o8, l8 = oracle.partial_int8(H, G, q, rec_pool.reshape(-1), slots, 1, 3)
    oe, le = oracle.partial_exact(H, G, q, kpool, vpool, slots, 64, 192)
    assert np.allclose(o8, oe, rtol=0, atol=1e-14 * np.abs(oe).max()) and np.allclose(l8, le, atol=1e-13)


def test_hybrid_equals_full_history_when_records_are_exact():
    """Tier split + exact merge == attention over the whole history (ActiveKV: the
    tiers are joined with exact attention arithmetic)."""
    H, G, n8 = 2, 8, 3
    recs, kp, vp = representable_records(9, n8, H)
    w = synth.make_workload([n8 * 64 + 150], 150, H=H, G=G, seed=8)
    assert w.n8[0] == n8
    rec_pool = np.zeros((w.n_slots, H, oracle.REC_BYTES), np.uint8)
    for p in range(n8):
        slot = w.pages[0][p]
        rec_pool[slot] = recs[p]
        w.k_pool[slot] = kp[p]
        w.v_pool[slot] = vp[p]
    o, lse = oracle.hybrid_workload(w, rec_pool.reshape(-1))
    of, lf = oracle.full_precision_workload(w)
    assert np.allclose(o, of, rtol=0, atol=1e-13 * np.abs(of).max()) and np.allclose(lse, lf, atol=1e-12)


def test_hybrid_all_exact_requests_and_thread_count():
    w = synth.make_workload([130, 64, 1], None, H=2, seed=10)
    rec_pool = np.zeros(oracle.REC_BYTES, np.uint8)
    o1, l1 = oracle.hybrid_workload(w, rec_pool, n_threads=1)
    o3, l3 = oracle.hybrid_workload(w, rec_pool, n_threads=3)
    of, lf = oracle.full_precision_workload(w)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)
    assert np.array_equal(o1, of) and np.array_equal(l1, lf)


def test_hybrid_result_independent_of_thread_count():
    """The oracle spreads (request, KV head, query row) items over threads; the
    result must not depend on how many threads take them."""
    w = synth.make_workload([900, 64, 300], 128, H=2, seed=11, key_sigma="outliers")
    rec = np.zeros(w.n_slots * w.H * oracle.REC_BYTES, np.uint8)
    s = w.int8_slots()
    oracle.quantize_pages(w.H, w.k_pool, w.v_pool, s, s, rec)
    for iq in (False, True):
        o1, l1 = oracle.hybrid_workload(w, rec, n_threads=1, int_query=iq)
        for nt in (5, 16, 64):
            o, l = oracle.hybrid_workload(w, rec, n_threads=nt, int_query=iq)
            assert np.array_equal(o, o1) and np.array_equal(l, l1), (iq, nt)
