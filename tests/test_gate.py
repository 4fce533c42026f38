"""The economic gate's host logic against hand-computed cases ("Judge a
representation by the bytes it stops moving", "My approach": bytes saved per
token against GPU time added, at each target size, with a transfer model fitted
to measured copies)."""
import math

import pytest

from tiered_paged_kv_gb300 import gate


def test_link_fit_recovers_latency_and_rate():
    # copies of 10 us latency at 200 GB/s (200,000 bytes per us)
    pts = [(b, 10.0 + b / 200e3) for b in (1e6, 4e6, 3.2e7, 1e8, 3e8)]
    m = gate.fit_link(pts)
    assert math.isclose(m.latency_us, 10.0, rel_tol=1e-9)
    assert math.isclose(m.rate_GBps, 200.0, rel_tol=1e-9)
    assert math.isclose(m.copy_us(2e8), 1010.0, rel_tol=1e-12)
    assert math.isclose(m.transfer_us(2e8), 1000.0, rel_tol=1e-12)


def test_link_fit_least_squares_with_noise():
    # symmetric noise about the line t = 5 + b / 100e3: the fit is the line itself
    pts = [(1e6, 15.0 + 1.0), (1e6, 15.0 - 1.0), (1e8, 1005.0 + 2.0), (1e8, 1005.0 - 2.0)]
    m = gate.fit_link(pts)
    assert math.isclose(m.latency_us, 5.0, rel_tol=1e-9)
    assert math.isclose(m.rate_GBps, 100.0, rel_tol=1e-9)


def test_link_fit_refusals():
    with pytest.raises(ValueError):
        gate.fit_link([(1e6, 10.0)])
    with pytest.raises(ValueError):
        gate.fit_link([(1e6, 10.0), (1e6, 12.0)])
    with pytest.raises(ValueError):
        gate.fit_link([(1e6, 10.0), (2e6, 9.0)])


LINK = gate.LinkModel(latency_us=10.0, rate_GBps=200.0)


def test_long_context_accepts_a_slower_kernel_that_moves_fewer_bytes():
    # 16 layers; the candidate halves the bytes (1e9 -> 5e8 per layer) but its
    # kernels take 50 us more per layer: saved 5e8 * 16 / 2e5 = 40,000 us, added
    # 800 us, net +39,200 us per token
    base = gate.Candidate("exact", 1e9, 100.0)
    cand = gate.Candidate("hybrid", 5e8, 150.0)
    assert math.isclose(gate.net_saving_us(LINK, base, cand, layers=16), 39200.0, rel_tol=1e-12)
    assert gate.accept(LINK, base, cand, layers=16)


def test_short_context_rejects_the_same_trade():
    # at a small size the bytes saved are worth less than the kernel time added:
    # saved 5e5 / 2e5 = 2.5 us, added 15 us, net -12.5 us
    base = gate.Candidate("exact", 1e6, 10.0)
    cand = gate.Candidate("hybrid", 5e5, 25.0)
    assert math.isclose(gate.net_saving_us(LINK, base, cand), -12.5, rel_tol=1e-12)
    assert not gate.accept(LINK, base, cand)


def test_faster_and_smaller_always_accepted_and_zero_net_rejected():
    base = gate.Candidate("exact", 4e8, 90.0)
    assert gate.accept(LINK, base, gate.Candidate("c", 3e8, 60.0))
    # bytes saved worth exactly the time added: net 0 is not a gain
    same = gate.Candidate("c", 4e8 - 2e5 * 7.0, 97.0)
    assert math.isclose(gate.net_saving_us(LINK, base, same), 0.0, abs_tol=1e-9)
    assert not gate.accept(LINK, base, same)


def test_step_prediction_link_bound_and_kernel_bound():
    # copy 10 + 2e8 / 2e5 = 1010 us per layer; kernels 60 us: 1010 + 15 * 1010 + 60
    c = gate.Candidate("hybrid", 2e8, 60.0)
    assert math.isclose(gate.predict_step_us(LINK, c, 16), 16220.0, rel_tol=1e-12)
    # kernels longer than the copy: 1010 + 15 * 2000 + 2000
    k = gate.Candidate("slow", 2e8, 2000.0)
    assert math.isclose(gate.predict_step_us(LINK, k, 16), 33010.0, rel_tol=1e-12)
    # one layer: copy then kernels
    assert math.isclose(gate.predict_step_us(LINK, c, 1), 1070.0, rel_tol=1e-12)
    with pytest.raises(ValueError):
        gate.predict_step_us(LINK, c, 0)


def test_per_tile_ratio():
    base = gate.Candidate("exact", 1e9, 100.0)
    cand = gate.Candidate("hybrid", 5e8, 60.0)
    # 100 us over 1000 tiles against 60 us over 400 tiles: 0.15 / 0.1
    assert math.isclose(gate.per_tile_ratio(base, cand, 1000, 400), 1.5, rel_tol=1e-12)
