"""The no-allocation multi-request call (library-held static scratch) against the
workspace call: same inputs, two calls in a row, results bit-identical (the
workspace call is itself checked against the oracle).  It serves callers that
cannot give the library device memory, such as a plugin whose host engine owns
every allocation.  Collected last on purpose."""
import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import DevWorkload, assert_close, oracle_records as oracle_converted_records

pytestmark = pytest.mark.gpu


def test_static_scratch_call_matches_workspace_call():
    import torch
    w = synth.make_workload([9000, 4000, 70, 33000], 1024, H=4, seed=31, key_sigma="outliers")
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    d.quantize_gpu()
    ref_o, ref_lse = d.hybrid()
    # the workspace call itself against the oracle on the GPU-converted records
    rec = oracle_converted_records(w)
    oo, ol = oracle.hybrid_workload(w, rec, n_threads=16)
    assert_close(ref_o, ref_lse, oo, ol, "workspace call")
    assert tpk.static_scratch_bytes() >= tpk.hybrid_workspace_bytes(d.shape, w.B)
    for _ in range(2):
        o = torch.full((w.B, w.H * w.G, 256), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((w.B, w.H * w.G), float("nan"), dtype=torch.float32, device="cuda")
        tpk.decode_hybrid_batched_static(d.shape, w.B, d.q, d.k, d.v, d.rec, d.pt, d.off, w.n_ex, d.pt8, d.off8,
                                         w.n8, o, lse)
        torch.cuda.synchronize()
        # both calls build the same split plan and run the same kernels with a fixed
        # fold order: the results must agree bit for bit
        assert np.array_equal(o.cpu().numpy().astype(np.float64), ref_o)
        assert np.array_equal(lse.cpu().numpy().astype(np.float64), ref_lse)
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
