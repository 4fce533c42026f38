"""Seeded random multi-request batches against the oracle: request counts, history
lengths (down to a single token), recent-window sizes (all-exact and all-8-bit
requests among them), KV head counts and key / value distributions drawn per case,
so that unit cuts, ragged tails and tier boundaries land at varied places.  Half the
cases decode records the GPU converted itself, the other half the oracle's."""
import numpy as np
import pytest

import oracle
from tiered_paged_kv_gb300 import synth
import tiered_paged_kv_gb300 as tpk
from tpk_testutil import DevWorkload, assert_close, oracle_records

pytestmark = pytest.mark.gpu
NT = 16  # oracle threads


def random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    n_req = int(rng.integers(1, 10))
    # lengths: a mix of tiny (< one page), page-ragged and a few thousand tokens
    kinds = rng.integers(0, 3, n_req)
    lengths = np.where(kinds == 0, rng.integers(1, 64, n_req),
                       np.where(kinds == 1, rng.integers(64, 700, n_req), rng.integers(700, 5000, n_req)))
    choice = int(rng.integers(0, 4))
    recent = [None, 0, int(rng.integers(1, 300)), int(rng.integers(300, 900))][choice]
    H = int(rng.choice([1, 2, 3, 4]))
    key_sigma = ["unit", "loguniform", "outliers"][int(rng.integers(0, 3))]
    value_sigma = ["unit", "loguniform"][int(rng.integers(0, 2))]
    w = synth.make_workload(lengths.astype(np.int64), recent, H=H, seed=50 + seed, key_sigma=key_sigma,
                            value_sigma=value_sigma, tid_base=0)
    what = (f"seed {seed}: {n_req} requests, lengths {lengths.tolist()}, recent {recent}, H {H}, "
            f"keys {key_sigma}, values {value_sigma}")
    return w, what


@pytest.mark.parametrize("impl", [tpk.IMPL_SIMT, tpk.IMPL_TENSOR])
@pytest.mark.parametrize("seed", range(24))
def test_random_batch_matches_oracle(impl, seed):
    w, what = random_case(seed)
    d = DevWorkload(w, impl)
    rec = oracle_records(w)
    if seed % 2:
        d.quantize_gpu()
    else:
        d.load_records(rec)
    o, lse = d.hybrid()
    oo, ol = oracle.hybrid_workload(w, rec, n_threads=NT)
    assert_close(o, lse, oo, ol, what, exact_only=int(w.n8.sum()) == 0)
