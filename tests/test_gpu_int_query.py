"""The integer-query variant of the tensor-core decode ("SYCL", "Attention that
reads 8-bit history": the integer query cache) against the oracle's integer-query
partials on the same records: 8-bit partials with splits and ragged ranges,
hybrid batches, zero and one-hot query rows, the 128K hybrid at full size, and
its error against unquantised attention reported beside the float query's."""
import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import (DevWorkload, assert_close, dev_i32, oracle_records, split_ranges_int8, torch)

pytestmark = pytest.mark.gpu
NT = 16  # oracle threads


def iq_workload(w):
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    d.shape = tpk.Shape(w.H, impl=tpk.IMPL_TENSOR, kv_slots=w.n_slots, rec_slots=w.n_slots, int_query=1)
    return d


def status_clean():
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags


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


@pytest.mark.parametrize("kind", ["loguniform", "outliers"])
@pytest.mark.parametrize("pb,pe,S", [(0, 1, 1), (0, 12, 1), (0, 12, 5), (3, 11, 2), (4, 4, 1), (0, 40, 40),
                                     (0, 3, 8)])
def test_int8_partials_on_same_codes(kind, pb, pe, S):
    w = synth.make_workload([64 * 40], 0, H=2, seed=12, key_sigma=kind,
                            value_sigma="loguniform" if kind == "loguniform" else "unit")
    rec = oracle_records(w)
    d = iq_workload(w)
    d.load_records(rec)
    o, lse = run_int8(d, pb, pe, S)
    for s, (a, b) in enumerate(split_ranges_int8(pb, pe, S)):
        oo, ol = oracle.partial_int8_iq(w.H, w.G, w.q[0], rec, w.pages[0], a, b)
        if a == b:
            assert np.all(o[s] == 0) and np.all(lse[s] == -np.inf)
        else:
            assert_close(o[s], lse[s], oo, ol, f"split {s} pages [{a},{b})")
    status_clean()


def check_hybrid(w, gpu_records=False, what=""):
    """As in the float-query tests: the oracle converts the pages itself; with
    gpu_records the GPU decodes records it converted on its side."""
    d = iq_workload(w)
    rec = oracle_records(w)
    if gpu_records:
        d.quantize_gpu()
    else:
        d.load_records(rec)
    o, lse = d.hybrid()
    status_clean()
    oo, ol = oracle.hybrid_workload(w, rec, n_threads=NT, int_query=True)
    err = assert_close(o, lse, oo, ol, what)
    return d, o, lse, oo, ol, rec, err


def test_tiny_hybrid():
    check_hybrid(synth.tiny_hybrid(seed=0), what="tiny")


@pytest.mark.parametrize("gpu_records", [False, True])
def test_ragged_batch(gpu_records):
    lengths = [1, 63, 64, 65, 700, 2 * 64 + 7, 2000, 0, 129]
    w = synth.make_workload(lengths, 100, H=2, seed=21, key_sigma="outliers")
    check_hybrid(w, gpu_records, "ragged")


@pytest.mark.parametrize("n_req", [4, 5])
def test_plan_sizes(n_req):
    lengths = [300 + 517 * i for i in range(n_req)]
    w = synth.make_workload(lengths, 128, H=2, seed=30 + n_req, key_sigma="outliers")
    check_hybrid(w, what=f"{n_req} requests")


def test_all_8bit_and_all_exact():
    w = synth.make_workload([64 * 30, 64 * 3], 0, H=2, seed=23)
    assert (w.n_ex == 0).all()
    check_hybrid(w, what="all 8-bit")
    # no 8-bit pages: the integer query changes nothing, bit for bit
    w = synth.make_workload([5000, 77], None, H=2, seed=22)
    d = iq_workload(w)
    a = d.hybrid()
    f = DevWorkload(w, tpk.IMPL_TENSOR).hybrid()
    assert np.array_equal(a[0], f[0]) and np.array_equal(a[1], f[1])


def test_zero_and_one_hot_query_rows():
    """A zero row codes to zeros (alpha = 0: uniform weights over the 8-bit tier); a
    row with one non-zero channel codes that channel to +-127 and the rest to 0."""
    w = synth.make_workload([64 * 9 + 40, 64 * 5], 40, H=2, seed=25, key_sigma="outliers")
    w.q[0, 0] = 0
    w.q[1, 3] = 0
    w.q[1, 3, 77] = synth.f32_to_bf16(np.array([-2.5], np.float32))[0]
    w.q[0, 9] = 0
    w.q[0, 9, 200] = synth.f32_to_bf16(np.array([1e-3], np.float32))[0]
    check_hybrid(w, what="zero / one-hot rows")


def test_deterministic():
    w = synth.make_workload([20000, 3000, 9000], 1024, H=4, seed=24, key_sigma="outliers")
    d = iq_workload(w)
    d.load_records(oracle_records(w))
    a = d.hybrid()
    b = d.hybrid()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_full_hybrid_128k():
    w = synth.hybrid_128k(seed=2)
    d, o, lse, oo, ol, rec, err = check_hybrid(w, gpu_records=True, what="hybrid 128K, integer query")
    # error against unquantised attention: integer query beside float query
    of, lf = oracle.full_precision_workload(w, n_threads=NT)
    ofq, _ = oracle.hybrid_workload(w, rec, n_threads=NT)
    e_gpu = np.abs(o - of).max()
    e_orc = np.abs(oo - of).max()
    e_flt = np.abs(ofq - of).max()
    print(f"hybrid 128K: worst merged error vs unquantised: integer query gpu {e_gpu:.4g}, oracle {e_orc:.4g}; "
          f"float query oracle {e_flt:.4g} (max|o| {np.abs(of).max():.4g}); parity {err}")
    assert abs(e_gpu - e_orc) <= 1e-3 * np.abs(oo).max()


def test_full_batched_16():
    """The 16-request batch at full size (lengths uniform in [8K, 64K], 2,048 recent
    BF16 tokens each, 1.35 GB of history) through the integer-query variant, with
    the GPU's own records."""
    check_hybrid(synth.batched_hybrid(seed=3), gpu_records=True, what="batched 16, integer query")


def test_full_int8_tier_128k():
    """All 131,072 tokens 8-bit (2,048 pages x 4 KV heads), the single-tier line the
    bench times, through the integer-query variant."""
    w = synth.make_workload([131072], 0, H=4, seed=12, key_sigma="outliers")
    assert (w.n_ex == 0).all()
    check_hybrid(w, gpu_records=True, what="all 8-bit 128K, integer query")
