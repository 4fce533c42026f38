"""The multi-request call's split plan on the host (tpk_hybrid_plan, no GPU): unit
budget, per-segment bounds, proportionality, the largest plans and the 128K
hybrid's plan on 152 resident blocks."""
import numpy as np
import pytest

import tiered_paged_kv_gb300 as tpk

MAX_UNITS = 2048


def pages(n_tokens):
    return (np.asarray(n_tokens) + 63) // 64


def check_plan(H, ne, n8, resident):
    ne = np.asarray(ne, np.int64)
    n8 = np.asarray(n8, np.int64)
    se, s8, units = tpk.hybrid_plan(tpk.Shape(H), ne, n8, resident)
    assert units == H * int(se.sum() + s8.sum()) <= MAX_UNITS
    for b in range(len(ne)):
        if ne[b] > 0:
            assert 1 <= se[b] <= pages(ne[b])
        elif n8[b] > 0:
            assert se[b] == 0
        else:
            assert se[b] == 1 and s8[b] == 0      # an empty request: one empty unit
        if n8[b] > 0:
            assert 1 <= s8[b] <= n8[b]
        else:
            assert s8[b] == 0
    return se, s8, units


def test_hybrid_128k_on_one_wave():
    se, s8, units = check_plan(4, [4096], [1984], 152)
    assert units == 152 and (se[0], s8[0]) == (2, 36)


@pytest.mark.parametrize("resident", [1, 7, 152, 304, 2048])
def test_budget_fills_whole_waves(resident):
    """Long segments: the units per head are the budget, a whole number of waves."""
    H = 4
    se, s8, units = check_plan(H, [200000, 150000, 90000], [3000, 2500, 1000], resident)
    per_head = units // H
    waves = max(1, -(-max(-(-resident // H), 4 * 6) * H // resident))
    assert per_head == max(6, min(MAX_UNITS, waves * resident) // H)


def test_units_follow_bytes():
    """Segments far from their bounds get units in proportion to their bytes (within
    one unit of the ideal share)."""
    H = 2
    ne = np.array([64000, 16000, 32000, 8000])
    n8 = np.array([4000, 1000, 2000, 500])
    se, s8, units = check_plan(H, ne, n8, 600)
    bytes_ = np.concatenate([1024.0 * ne, 35072.0 * n8])
    got = np.concatenate([se, s8]).astype(float)
    ideal = got.sum() * bytes_ / bytes_.sum()
    assert np.abs(got - ideal).max() < 1.0 + 1e-9


def test_random_batches_respect_every_bound():
    rng = np.random.default_rng(7)
    for _ in range(300):
        B = int(rng.integers(1, 257))
        H = int(rng.choice([1, 2, 4, 8]))
        if B * 2 * H > MAX_UNITS:
            H = max(1, MAX_UNITS // (2 * B))
        ne = rng.integers(0, 5000, B) * rng.integers(0, 2, B)
        n8 = rng.integers(0, 800, B) * rng.integers(0, 2, B)
        check_plan(H, ne, n8, int(rng.choice([152, 304, 1])))


def test_largest_plans():
    # 256 requests x 4 heads x 2 tiers = 2048 segments: exactly one unit each
    se, s8, units = check_plan(4, [300] * 256, [10] * 256, 152)
    assert units == 2048 and (se == 1).all() and (s8 == 1).all()
    # 1024 heads, one request with both tiers
    se, s8, units = check_plan(1024, [40], [1], 152)
    assert units == 2048
    # a single page per segment caps the split
    se, s8, units = check_plan(1, [64], [1], 2048)
    assert (se[0], s8[0]) == (1, 1)


def test_plans_that_cannot_fit_are_refused():
    with pytest.raises(tpk.TpkError):
        tpk.hybrid_plan(tpk.Shape(8), [300] * 256, [10] * 256, 152)   # 4096 segments
    with pytest.raises(tpk.TpkError):
        tpk.hybrid_plan(tpk.Shape(4), [1] * 257, [0] * 257, 152)     # too many requests
    with pytest.raises(tpk.TpkError):
        tpk.hybrid_plan(tpk.Shape(4), [-1], [0], 152)
