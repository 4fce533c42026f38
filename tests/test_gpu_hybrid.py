"""The one-launch multi-request hybrid decode against the oracle: the tiny
hybrid, ragged multi-request batches, the all-exact 32K history, the 128K
hybrid and the 16-request batch at full size, bit-for-bit determinism, and the
hybrid error against unquantised attention reported beside the oracle's."""
import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import DevWorkload, assert_close, oracle_records

pytestmark = pytest.mark.gpu
IMPLS = [tpk.IMPL_SIMT, tpk.IMPL_TENSOR]
NT = 16  # oracle threads


def check_hybrid(w, impl, gpu_records=False, what=""):
    """GPU hybrid decode against the oracle.  The oracle always converts the pages
    itself from the BF16 inputs; with gpu_records the GPU converts them on its side
    and decodes its own records (end to end), otherwise it decodes the oracle's."""
    d = DevWorkload(w, impl)
    rec = oracle_records(w)
    if gpu_records:
        d.quantize_gpu()
    else:
        d.load_records(rec)
    o, lse = d.hybrid()
    oo, ol = oracle.hybrid_workload(w, rec, n_threads=NT)
    err = assert_close(o, lse, oo, ol, what, exact_only=int(w.n8.sum()) == 0)
    return d, o, lse, oo, ol, rec, err


@pytest.mark.parametrize("impl", IMPLS)
def test_tiny_hybrid(impl):
    check_hybrid(synth.tiny_hybrid(seed=0), impl, what="tiny")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("gpu_records", [False, True])
def test_ragged_batch(impl, gpu_records):
    lengths = [1, 63, 64, 65, 700, 2 * 64 + 7, 2000, 0, 129]
    w = synth.make_workload(lengths, 100, H=2, seed=21, key_sigma="outliers")
    check_hybrid(w, impl, gpu_records, "ragged")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("n_req", [4, 5])
def test_plan_sizes(impl, n_req):
    """Launches of up to four requests take the short plan parameter, longer
    ones the full one: both sides of the boundary."""
    lengths = [300 + 517 * i for i in range(n_req)]
    w = synth.make_workload(lengths, 128, H=2, seed=30 + n_req, key_sigma="outliers")
    check_hybrid(w, impl, what=f"{n_req} requests")


@pytest.mark.parametrize("impl", IMPLS)
def test_only_one_tier(impl):
    check_hybrid(synth.make_workload([5000, 77], None, H=2, seed=22), impl, what="all exact")
    w = synth.make_workload([64 * 30, 64 * 3], 0, H=2, seed=23)
    assert (w.n_ex == 0).all()
    check_hybrid(w, impl, what="all 8-bit")


@pytest.mark.parametrize("impl", IMPLS)
def test_deterministic(impl):
    w = synth.make_workload([20000, 3000, 9000], 1024, H=4, seed=24, key_sigma="outliers")
    d = DevWorkload(w, impl)
    d.load_records(oracle_records(w))
    a = d.hybrid()
    b = d.hybrid()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("seed", range(5))
def test_configs_at_reduced_sizes_seeds_0_to_4(seed):
    """Every workload recipe at a reduced size, seeds 0-4, both kernels (8-bit
    records from the GPU conversion): the tiny hybrid, the all-exact history, the
    outlier-key hybrid and a 4-request ragged batch."""
    for impl in IMPLS:
        check_hybrid(synth.tiny_hybrid(seed=seed), impl, gpu_records=True, what=f"tiny seed {seed}")
        check_hybrid(synth.exact_32k(seed=seed, n_tokens=4096 + 37 * seed), impl, what=f"exact seed {seed}")
        check_hybrid(synth.hybrid_128k(seed=seed, n_tokens=8192 + 64 * seed + 5, recent=512), impl,
                     gpu_records=True, what=f"hybrid seed {seed}")
        check_hybrid(synth.batched_hybrid(seed=seed, n_req=4, lo=1024, hi=6000, recent=256), impl,
                     gpu_records=True, what=f"batch seed {seed}")


@pytest.mark.parametrize("impl", IMPLS)
def test_full_exact_32k(impl):
    w = synth.exact_32k(seed=1)
    check_hybrid(w, impl, what="exact 32K")


@pytest.mark.parametrize("impl", IMPLS)
def test_full_hybrid_128k(impl):
    w = synth.hybrid_128k(seed=2)
    d, o, lse, oo, ol, rec, err = check_hybrid(w, impl, gpu_records=True, what="hybrid 128K")
    # the hybrid error against unquantised attention, GPU beside oracle
    of, lf = oracle.full_precision_workload(w, n_threads=NT)
    e_gpu = np.abs(o - of).max()
    e_orc = np.abs(oo - of).max()
    print(f"hybrid 128K: worst merged error vs unquantised: gpu {e_gpu:.4g}, oracle {e_orc:.4g} "
          f"(max|o| {np.abs(of).max():.4g}); parity {err}")
    assert abs(e_gpu - e_orc) <= 1e-3 * np.abs(oo).max()


@pytest.mark.parametrize("impl", IMPLS)
def test_full_batched_16(impl):
    w = synth.batched_hybrid(seed=3)
    check_hybrid(w, impl, gpu_records=True, what="batched 16")


@pytest.mark.parametrize("impl", IMPLS)
def test_back_to_back_launches_share_a_workspace(impl):
    """Twenty launches queued without synchronising, one workspace: every result
    must equal the first bit for bit (catches pipeline and workspace races)."""
    t = __import__("torch")
    w = synth.hybrid_128k(seed=2, n_tokens=32768, recent=1024)
    d = DevWorkload(w, impl)
    d.quantize_gpu()
    nbytes = tpk.hybrid_workspace_bytes(d.shape, w.B)
    ws = t.empty(nbytes, dtype=t.uint8, device="cuda")
    tpk.workspace_init(ws, nbytes)
    outs = []
    for _ in range(20):
        o = t.empty(w.B, w.H * w.G, 256, dtype=t.float32, device="cuda")
        lse = t.empty(w.B, w.H * w.G, dtype=t.float32, device="cuda")
        tpk.decode_hybrid_batched(d.shape, w.B, d.q, d.k, d.v, d.rec, d.pt, d.off, w.n_ex, d.pt8, d.off8, w.n8, o,
                                  lse, ws, nbytes)
        outs.append((o, lse))
    t.cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
    for o, lse in outs[1:]:
        assert t.equal(o, outs[0][0]) and t.equal(lse, outs[0][1])


@pytest.mark.parametrize("impl", IMPLS)
def test_maximum_request_count(impl):
    """256 requests in one launch (the largest plan; with 4 KV heads their 2032
    (request, head, tier) segments nearly fill the 2048 partial slots), ragged
    lengths including empty and single-token histories; 257 requests are refused."""
    rng = np.random.default_rng(60)
    lengths = rng.integers(200, 1500, 256)
    lengths[:4] = [0, 1, 64, 65]
    w = synth.make_workload(list(lengths), 100, H=4, seed=60)
    check_hybrid(w, impl, what="256 requests")
    d = DevWorkload(w, impl)
    t = __import__("torch")
    o = t.empty(257, w.H * w.G, 256, dtype=t.float32, device="cuda")
    lse = t.empty(257, w.H * w.G, dtype=t.float32, device="cuda")
    nbytes = tpk.hybrid_workspace_bytes(d.shape, 256)
    ws = t.empty(nbytes, dtype=t.uint8, device="cuda")
    off = np.concatenate([d.off, d.off[-1:]])
    off8 = np.concatenate([d.off8, d.off8[-1:]])
    with pytest.raises(tpk.TpkError):
        tpk.decode_hybrid_batched(d.shape, 257, d.q, d.k, d.v, d.rec, d.pt, off, list(w.n_ex) + [0], d.pt8, off8,
                                  list(w.n8) + [0], o, lse, ws, nbytes)


@pytest.mark.parametrize("impl", IMPLS)
def test_million_token_history(impl):
    """One request over 1,048,576 tokens (16,320 8-bit pages + 4,096 BF16 tokens),
    one KV head."""
    w = synth.make_workload([1 << 20], 4096, H=1, seed=61, key_sigma="outliers")
    check_hybrid(w, impl, gpu_records=True, what="1M tokens")


@pytest.mark.parametrize("impl", IMPLS)
def test_many_kv_heads(impl):
    """64 KV heads (512 query rows) over a ragged hybrid batch, records converted on
    the GPU: head indexing in the decode, fold and conversion kernels at large H."""
    w = synth.make_workload([700, 64 * 3 + 5], 100, H=64, seed=62, key_sigma="outliers")
    check_hybrid(w, impl, gpu_records=True, what="64 heads")


def test_maximum_kv_heads():
    """1024 KV heads, the largest shape the library takes: one short exact history
    (1024 units, one per head) and one 8-bit page per head."""
    w = synth.make_workload([64 + 40], 40, H=1024, seed=63)
    assert w.n8[0] == 1
    check_hybrid(w, tpk.IMPL_TENSOR, gpu_records=True, what="1024 heads")


def test_plan_on_this_device():
    """The plan the call makes on this GPU for the 128K hybrid: one wave of the
    tensor-core kernel (one block per SM), split 2 + 36 per head."""
    t = __import__("torch")
    sms = t.cuda.get_device_properties(0).multi_processor_count
    se, s8, units = tpk.hybrid_plan(tpk.Shape(4, impl=tpk.IMPL_TENSOR), [4096], [1984], 0)
    assert units <= 2048 and (se[0] + s8[0]) * 4 == units
    assert units >= sms // 4 * 4   # at least one full wave of the resident blocks
    if sms == 152:
        assert (se[0], s8[0], units) == (2, 36, 152)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("log2_scale", [-24, -8, 3, 6])
def test_extreme_query_scales(impl, log2_scale):
    """q times 2^k (exact in bfloat16): near-uniform weights for small k, a few
    dominant tokens for large k (lse near 1,000 nats at 2^6, in both tiers).  o is
    held to the usual bar.  The lse bar grows with |lse|: scores are float32 sums and
    the 8-bit tier's products run on code + 1152 with the offset removed after the
    sum (about 18 bits of the score kept), so the lse carries a relative error near
    1e-5 -- 1e-3 + 1e-5 |lse|.  Larger scales leave float32 itself: at 2^12 the lse
    is 65,000 nats, where one float32 ulp exceeds 1e-3."""
    w = synth.make_workload([64 * 20 + 30, 900], 200, H=2, seed=64, key_sigma="outliers")
    q = synth.bf16_to_f32(w.q).astype(np.float64) * 2.0 ** log2_scale
    w.q = synth.f32_to_bf16(q.astype(np.float32))
    assert np.array_equal(synth.bf16_to_f32(w.q).astype(np.float64), q)
    d = DevWorkload(w, impl)
    rec = oracle_records(w)
    d.load_records(rec)
    o, lse = d.hybrid()
    oo, ol = oracle.hybrid_workload(w, rec, n_threads=NT)
    assert np.abs(o - oo).max() <= 1e-3 * np.abs(oo).max()
    assert np.array_equal(np.isfinite(lse), np.isfinite(ol))
    fin = np.isfinite(ol)
    assert (np.abs(lse[fin] - ol[fin]) <= 1e-3 + 1e-5 * np.abs(ol[fin])).all()


def test_decode_timing_events_bracket_the_decode_kernel():
    """The measurement hook: events recorded around the decode launch inside a
    captured graph time the decode kernel alone (shorter than the whole step)."""
    t = __import__("torch")
    w = synth.hybrid_128k(seed=2, n_tokens=32768, recent=1024)
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    d.quantize_gpu()
    nbytes = tpk.hybrid_workspace_bytes(d.shape, w.B)
    ws = t.zeros(nbytes, dtype=t.uint8, device="cuda")
    o = t.empty(w.B, w.H * w.G, 256, dtype=t.float32, device="cuda")
    lse = t.empty(w.B, w.H * w.G, dtype=t.float32, device="cuda")
    s = t.cuda.Stream()
    step = lambda: tpk.decode_hybrid_batched(d.shape, w.B, d.q, d.k, d.v, d.rec, d.pt, d.off, w.n_ex, d.pt8,
                                             d.off8, w.n8, o, lse, ws, nbytes, s)
    before, after = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    a, b = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    with t.cuda.stream(s):
        step()
        before.record(s)
        after.record(s)
        s.synchronize()
        tpk.set_decode_timing_events(before, after)
        try:
            g = t.cuda.CUDAGraph()
            with t.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                step()
        finally:
            tpk.set_decode_timing_events()
        for _ in range(3):
            a.record(s)
            g.replay()
            b.record(s)
            s.synchronize()
            k_ms, step_ms = before.elapsed_time(after), a.elapsed_time(b)
            assert 0 < k_ms < step_ms
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
