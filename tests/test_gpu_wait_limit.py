"""Bounded device waits.  With a short wait limit set through the C ABI's test
hook, a decode launch in which one thread block's first history item never
arrives (nothing is copied for it and nothing arrives on its barrier) gives up
waiting, reports the timeout in the device status word and returns; the context
stays usable and the next normal call matches the oracle."""
import time

import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import DevWorkload, assert_close, oracle_records

pytestmark = pytest.mark.gpu

TPK_ERR_TIMEOUT = 6
LIMIT_NS = 1_000_000  # 1 ms


@pytest.mark.parametrize("tier", ["exact", "int8"])
def test_wait_runs_out_reports_and_recovers(tier):
    w = synth.make_workload([64 * 40 + 100, 64 * 12], 1024, H=2, seed=41, key_sigma="outliers")
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    rec = oracle_records(w)
    d.load_records(rec)
    oo, ol = oracle.hybrid_workload(w, rec, n_threads=16)
    o, lse = d.hybrid()
    assert_close(o, lse, oo, ol, "before")
    se, s8, units = tpk.hybrid_plan(d.shape, w.n_ex, w.n8)
    assert se[0] >= 1 and s8[0] >= 1
    unit = 0 if tier == "exact" else int(se[0])  # request 0, KV head 0: first unit of the tier
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
    tpk.set_test_wait(LIMIT_NS, unit)
    try:
        t0 = time.perf_counter()
        d.hybrid()  # synchronises: the launch must come back
        dt = time.perf_counter() - t0
    finally:
        tpk.set_test_wait()
    st, flags = tpk.get_device_status(reset=True)
    assert st == TPK_ERR_TIMEOUT and flags & 2, (st, flags)
    # a handful of 1 ms waits ran out; the default limit (2 s) would take far longer
    assert dt < 1.0, dt
    o, lse = d.hybrid()
    assert_close(o, lse, oo, ol, "after")
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags


def test_short_limit_alone_changes_nothing():
    """A short limit with no stalled block: every wait is met well within it, the
    result is bit-identical to the default limit's and no status bit is set."""
    w = synth.make_workload([64 * 30 + 7], 512, H=2, seed=42, key_sigma="outliers")
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    d.load_records(oracle_records(w))
    o0, l0 = d.hybrid()
    tpk.set_test_wait(50_000_000, -1)
    try:
        o1, l1 = d.hybrid()
    finally:
        tpk.set_test_wait()
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
