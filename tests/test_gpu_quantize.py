"""GPU page conversion against the oracle ("model quantization", section "An
8-bit page format shaped for its kernel"): codes bit-exact given the oracle's
scales, the GPU's own scales within 1 ulp of the oracle's, and the format's
invariants on the GPU's own output."""
import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import REC_POISON, DevWorkload, dev_f32, dev_i32, oracle_records

pytestmark = pytest.mark.gpu

WORKLOADS = {
    "tiny_loguniform": lambda: synth.tiny_hybrid(seed=0),
    "outliers": lambda: synth.make_workload([64 * 40 + 17], 17, H=4, seed=2, key_sigma="outliers"),
    "unit": lambda: synth.make_workload([64 * 24 + 5, 64 * 9], 5, H=2, seed=7),
}


def ulp_distance(a, b):
    ai = a.view(np.int32).astype(np.int64)
    bi = b.view(np.int32).astype(np.int64)
    return np.abs(ai - bi)


def check_own_record(got, ref, what=""):
    """A record the GPU converted against the oracle's record of the same page-head
    (converted by the oracle from the same BF16 page): key channel scales within 1
    ulp, and wherever every scale agrees (all but a few page-heads of the 128K
    workload, whose conversion has 75 of 2,031,616 scales 1 ulp apart) the whole record
    identical, codes included -- given the same s_c, both sides form r_t, u_c and
    the codes by the same correctly rounded float32 steps.  A page-head whose scales
    differ has its codes covered by the given-scales tests, which fix the scales on
    both sides.  Returns the number of channel scales that differ."""
    _, _, s, r, u = oracle.record_fields(got)
    _, _, s_o, r_o, u_o = oracle.record_fields(ref)
    assert ulp_distance(s, s_o).max() <= 1, what
    n = int((s != s_o).sum())
    if n == 0:
        assert np.array_equal(got, ref), what
    return n


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_codes_bit_exact_given_oracle_scales(name):
    w = WORKLOADS[name]()
    ref = oracle_records(w)
    slots = w.int8_slots()
    H = w.H
    recs = ref.reshape(w.n_slots, H, oracle.REC_BYTES)[slots]  # [n][H][rec]
    fields = [[oracle.record_fields(recs[i, h]) for h in range(H)] for i in range(len(slots))]
    ks = np.array([[f[2] for f in row] for row in fields], np.float32)   # logical channel order
    kt = np.array([[f[3] for f in row] for row in fields], np.float32)
    vs = np.array([[f[4] for f in row] for row in fields], np.float32)
    d = DevWorkload(w)
    s = dev_i32(slots)
    tpk.kv_quantize_pages_given_scales(d.shape, d.k, d.v, s, s, len(slots), dev_f32(ks), dev_f32(kt), dev_f32(vs),
                                       d.rec)
    got = d.rec.cpu().numpy().reshape(w.n_slots, H, oracle.REC_BYTES)[slots]
    assert np.array_equal(got, recs)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_own_scales_within_one_ulp_and_invariants(name):
    w = WORKLOADS[name]()
    ref = oracle_records(w).reshape(w.n_slots, w.H, oracle.REC_BYTES)
    d = DevWorkload(w)
    got = d.quantize_gpu().reshape(w.n_slots, w.H, oracle.REC_BYTES)
    n_diff = 0
    for slot in w.int8_slots():
        for h in range(w.H):
            kc, vc, s, r, u = oracle.record_fields(got[slot, h])
            _, _, s_o, r_o, u_o = oracle.record_fields(ref[slot, h])
            n_diff += check_own_record(got[slot, h], ref[slot, h], f"slot {slot} head {h}")
            assert np.array_equal(u, u_o)          # u depends on V alone: same float32 ops
            assert kc.min() >= -127 and vc.min() >= -127
            assert np.all(np.abs(kc).max(axis=1)[r > 0] == 127)
            assert np.all(np.abs(vc).max(axis=0)[u > 0] == 127)
            clamped = (s == np.float32(2.0 ** -14)) | (s == np.float32(2.0 ** 14))
            if not clamped.any():
                assert abs(np.exp(np.log(s.astype(np.float64)).sum()) - 1.0) <= 1e-6
    print(f"{name}: {n_diff} channel scales differ from the oracle by 1 ulp")


def test_zero_rows_channels_and_clamp():
    w = synth.make_workload([128], 0, H=1, seed=3)
    for slot in w.int8_slots():
        k = w.k_pool[slot, 0]
        k[:, 5] = 0                                   # silent channel -> clamped 2^-14
        k[:, 200] = synth.f32_to_bf16(np.full(64, 2.0 ** 60, np.float32))  # far above the clamp
        k[9, :] = 0                                   # silent row -> r = 0
        w.v_pool[slot, 0][:, 7] = 0
    ref = oracle_records(w).reshape(w.n_slots, 1, oracle.REC_BYTES)
    d = DevWorkload(w)
    got = d.quantize_gpu().reshape(w.n_slots, 1, oracle.REC_BYTES)
    for slot in w.int8_slots():
        kc, vc, s, r, u = oracle.record_fields(got[slot, 0])
        _, _, s_o, r_o, u_o = oracle.record_fields(ref[slot, 0])
        assert s[5] == np.float32(2.0 ** -14) and s[200] == np.float32(2.0 ** 14)
        assert np.all(kc[:, 5] == 0) and r[9] == 0 and np.all(kc[9] == 0)
        assert u[7] == 0 and np.all(vc[:, 7] == 0)
        check_own_record(got[slot, 0], ref[slot, 0], f"slot {slot}")


def test_full_hybrid_128k_conversion():
    """Every 8-bit page of the 128K hybrid workload (1,984 pages x 4 KV heads, keys
    with outlier channels) converted in one call: each record against the oracle's
    conversion of the same page-head."""
    w = synth.hybrid_128k(seed=2)
    ref = oracle_records(w).reshape(w.n_slots, w.H, oracle.REC_BYTES)
    got = DevWorkload(w).quantize_gpu().reshape(w.n_slots, w.H, oracle.REC_BYTES)
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
    s8 = w.int8_slots()
    if not np.array_equal(got[s8], ref[s8]):
        n = sum(check_own_record(got[slot, h], ref[slot, h], f"slot {slot} head {h}")
                for slot in s8 for h in range(w.H))
        print(f"hybrid 128K: {n} channel scales differ from the oracle by 1 ulp")
        # the pages holding those page-heads, converted again with the oracle's scales
        # given: their records must then equal the oracle's byte for byte
        diff = np.array([slot for slot in s8 if not np.array_equal(got[slot], ref[slot])], np.int32)
        fields = [[oracle.record_fields(ref[slot, h]) for h in range(w.H)] for slot in diff]
        ks = np.array([[f[2] for f in row] for row in fields], np.float32)
        kt = np.array([[f[3] for f in row] for row in fields], np.float32)
        vs = np.array([[f[4] for f in row] for row in fields], np.float32)
        d = DevWorkload(w)
        sl = dev_i32(diff)
        tpk.kv_quantize_pages_given_scales(d.shape, d.k, d.v, sl, sl, len(diff), dev_f32(ks), dev_f32(kt),
                                           dev_f32(vs), d.rec)
        again = d.rec.cpu().numpy().reshape(w.n_slots, w.H, oracle.REC_BYTES)
        assert np.array_equal(again[diff], ref[diff])


def test_bad_slot_is_skipped_and_reported():
    w = synth.make_workload([128], 0, H=1, seed=4)
    d = DevWorkload(w)
    tpk.get_device_status(reset=True)
    src = dev_i32(np.array([w.n_slots + 5], np.int32))
    tpk.kv_quantize_pages(d.shape, d.k, d.v, src, src, 1, d.rec)
    st, flags = tpk.get_device_status(reset=True)
    assert st == 4 and flags & 1
    assert bool((d.rec == REC_POISON).all().item())          # nothing was written


def tie_pages(seed, n_pages):
    """Pages whose quotients land on and next to half-integers: K is a
    half-integer times s_c * r_t, V a half-integer times u_c, with the given scales
    powers of two (exact quotients: ties to even) or not (ties broken by the
    roundings of the two divisions), plus elements one bfloat16 ulp off."""
    rng = np.random.default_rng(seed)
    ks = np.where(rng.random((n_pages, 256)) < 0.5, 2.0 ** rng.integers(-3, 4, (n_pages, 256)),
                  rng.uniform(0.3, 3.0, (n_pages, 256))).astype(np.float32)
    kt = np.where(rng.random((n_pages, 64)) < 0.5, 2.0 ** rng.integers(-3, 4, (n_pages, 64)),
                  rng.uniform(0.3, 3.0, (n_pages, 64))).astype(np.float32)
    vs = np.where(rng.random((n_pages, 256)) < 0.5, 2.0 ** rng.integers(-3, 4, (n_pages, 256)),
                  rng.uniform(0.3, 3.0, (n_pages, 256))).astype(np.float32)
    half = (rng.integers(-127, 127, (n_pages, 64, 256)) + 0.5).astype(np.float32)
    kf = half * ks[:, None, :] * kt[:, :, None]
    vf = (rng.integers(-127, 127, (n_pages, 64, 256)) + 0.5).astype(np.float32) * vs[:, None, :]
    kb = synth.f32_to_bf16(kf)
    vb = synth.f32_to_bf16(vf)
    nudge = rng.random(kb.shape) < 0.1                   # one bfloat16 ulp away from the value
    kb = np.where(nudge, kb + np.where(rng.random(kb.shape) < 0.5, 1, -1).astype(np.int32), kb).astype(np.uint16)
    vb = np.where(nudge, vb + np.where(rng.random(vb.shape) < 0.5, 1, -1).astype(np.int32), vb).astype(np.uint16)
    return kb, vb, ks, kt, vs


@pytest.mark.parametrize("seed", [0, 1])
def test_codes_at_half_integer_quotients(seed):
    """Codes whose quotients are exact half-integers (the reciprocal-multiplication
    estimate cannot decide them) or next to one: bit-exact with the oracle given
    the scales, and self-consistent with the GPU's own scales."""
    n = 24
    kb, vb, ks, kt, vs = tie_pages(seed, n)
    w = synth.make_workload([64 * n], 0, H=1, seed=40 + seed)
    slots = w.int8_slots()
    for i, slot in enumerate(slots):
        w.k_pool[slot, 0] = kb[i]
        w.v_pool[slot, 0] = vb[i]
    d = DevWorkload(w)
    s = dev_i32(slots)
    tpk.kv_quantize_pages_given_scales(d.shape, d.k, d.v, s, s, n, dev_f32(ks), dev_f32(kt), dev_f32(vs), d.rec)
    got = d.rec.cpu().numpy().reshape(w.n_slots, oracle.REC_BYTES)
    for i, slot in enumerate(slots):
        ref = oracle.codes_given(w.k_pool[slot, 0], w.v_pool[slot, 0], ks[i], kt[i], vs[i])
        assert np.array_equal(got[slot], ref), f"page {i}"
    # own scales: the GPU's conversion against the oracle's conversion of the same pages
    got = d.quantize_gpu().reshape(w.n_slots, oracle.REC_BYTES)
    own = oracle_records(w).reshape(w.n_slots, oracle.REC_BYTES)
    for slot in slots:
        check_own_record(got[slot], own[slot], f"own scales, slot {slot}")


@pytest.mark.parametrize("j", [-45, -30, -20, -15, 0, 15, 20, 30])
def test_key_magnitudes_across_the_sum_paths(j):
    """Keys scaled by 4^j: the channel sums run as two packed chains when max|k|
    lies in [2^-40, 2^40) and as one scaled chain outside it; either way the
    scales stay within 1 ulp of the oracle's (which are invariant under 4^j) and
    the codes follow from them exactly."""
    w = synth.make_workload([64 * 6], 0, H=2, seed=11, key_sigma="loguniform")
    scale = np.float32(4.0 ** j)
    for slot in w.int8_slots():
        w.k_pool[slot] = synth.f32_to_bf16(synth.bf16_to_f32(w.k_pool[slot]) * scale)
    ref = oracle_records(w).reshape(w.n_slots, w.H, oracle.REC_BYTES)
    got = DevWorkload(w).quantize_gpu().reshape(w.n_slots, w.H, oracle.REC_BYTES)
    for slot in w.int8_slots():
        for h in range(w.H):
            kc, vc, s, r, u = oracle.record_fields(got[slot, h])
            check_own_record(got[slot, h], ref[slot, h], f"4^{j}, slot {slot} head {h}")
            assert np.all(np.abs(kc).max(axis=1)[r > 0] == 127)


def test_subnormal_and_near_maximum_channels():
    """Channels of subnormal bfloat16 keys, of keys near the bfloat16 maximum, and
    a channel at the single-pass bound 2^-40 / 2^40: scales within 1 ulp of the
    oracle's (clamped where the oracle clamps), codes from the scales exactly."""
    w = synth.make_workload([64 * 2], 0, H=1, seed=12)
    rng = np.random.default_rng(12)
    for slot in w.int8_slots():
        k = synth.bf16_to_f32(w.k_pool[slot, 0])
        k[:, 3] = rng.integers(-100, 100, 64) * np.float32(2.0 ** -133)     # subnormal
        k[:, 4] = rng.uniform(-1.0, 1.0, 64).astype(np.float32) * np.float32(3.0e38)
        k[:, 5] = np.float32(2.0 ** -40) * np.sign(rng.standard_normal(64)).astype(np.float32)
        k[:, 6] = np.float32(2.0 ** 40) * rng.uniform(0.5, 0.99, 64).astype(np.float32)
        w.k_pool[slot, 0] = synth.f32_to_bf16(k)
    ref = oracle_records(w).reshape(w.n_slots, 1, oracle.REC_BYTES)
    got = DevWorkload(w).quantize_gpu().reshape(w.n_slots, 1, oracle.REC_BYTES)
    for slot in w.int8_slots():
        kc, vc, s, r, u = oracle.record_fields(got[slot, 0])
        check_own_record(got[slot, 0], ref[slot, 0], f"slot {slot}")
        assert s[3] == np.float32(2.0 ** -14) and s[4] == np.float32(2.0 ** 14)


@pytest.mark.parametrize("seed", range(4))
def test_random_adversarial_pages(seed):
    """Seeded page-heads built to stress the conversion: per-channel key magnitudes
    2^U(-40, 40) and value magnitudes 2^U(-60, 60) (so some key channels clamp at
    2^+-14 and the sums take both paths), heavy-tailed entries (Gaussian over uniform), whole zero channels
    and rows, and channels rounded to eighths of their maximum (many equal
    magnitudes and exact half-integer quotients).  The GPU's own records against the oracle's: scales within 1 ulp,
    identical records where the scales agree; and with the oracle's scales given,
    identical records everywhere."""
    rng = np.random.default_rng(400 + seed)
    w = synth.make_workload([64 * 32], 0, H=2, seed=20 + seed)
    for slot in w.int8_slots():
        for h in range(w.H):
            k = rng.standard_normal((64, 256)) / np.maximum(rng.uniform(size=(64, 256)), 0.02)
            v = rng.standard_normal((64, 256))
            k *= 2.0 ** rng.uniform(-40, 40, 256)[None, :]
            v *= 2.0 ** rng.uniform(-60, 60, 256)[None, :]
            if rng.uniform() < 0.5:
                k[:, rng.integers(0, 256, 3)] = 0.0
                v[:, rng.integers(0, 256, 3)] = 0.0
            if rng.uniform() < 0.5:
                k[rng.integers(0, 64, 2), :] = 0.0
            if rng.uniform() < 0.5:  # coarse grid: many equal magnitudes and exact half quotients
                c = rng.integers(0, 256, 16)
                m = np.maximum(np.abs(k[:, c]).max(axis=0), 1e-30)
                k[:, c] = np.round(k[:, c] / m * 8) / 8 * m
                mv = np.maximum(np.abs(v[:, c]).max(axis=0), 1e-30)
                v[:, c] = np.round(v[:, c] / mv * 8) / 8 * mv
            w.k_pool[slot, h] = synth.f32_to_bf16(np.clip(k, -3e38, 3e38).astype(np.float32))
            w.v_pool[slot, h] = synth.f32_to_bf16(np.clip(v, -3e38, 3e38).astype(np.float32))
    ref = oracle_records(w).reshape(w.n_slots, w.H, oracle.REC_BYTES)
    d = DevWorkload(w)
    got = d.quantize_gpu().reshape(w.n_slots, w.H, oracle.REC_BYTES)
    for slot in w.int8_slots():
        for h in range(w.H):
            kc, vc, s, r, u = oracle.record_fields(got[slot, h])
            check_own_record(got[slot, h], ref[slot, h], f"seed {seed}, slot {slot} head {h}")
            assert kc.min() >= -127 and vc.min() >= -127
            assert np.all(np.abs(kc).max(axis=1)[r > 0] == 127)
            assert np.all(np.abs(vc).max(axis=0)[u > 0] == 127)
    # the oracle's scales given: every byte identical
    slots = w.int8_slots()
    recs = ref[slots]
    fields = [[oracle.record_fields(recs[i, h]) for h in range(w.H)] for i in range(len(slots))]
    ks = np.array([[f[2] for f in row] for row in fields], np.float32)
    kt = np.array([[f[3] for f in row] for row in fields], np.float32)
    vs = np.array([[f[4] for f in row] for row in fields], np.float32)
    s_d = dev_i32(slots)
    d2 = DevWorkload(w)
    tpk.kv_quantize_pages_given_scales(d2.shape, d2.k, d2.v, s_d, s_d, len(slots), dev_f32(ks), dev_f32(kt),
                                       dev_f32(vs), d2.rec)
    assert np.array_equal(d2.rec.cpu().numpy().reshape(w.n_slots, w.H, oracle.REC_BYTES)[slots], recs)
