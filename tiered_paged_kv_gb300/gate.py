"""The economic gate for compressed history formats (host logic only).

"Judge a representation by the bytes it stops moving", sections "My approach"
and "What I built": once the attention history lives in host memory, a decode
step is bound by the bytes that cross the host link, so a candidate format is
judged on the whole step at the target context size -- the transfer time its
smaller history saves per token against the GPU time its kernels add -- with a
transfer model derived from the link's measured behaviour.  A candidate is
accepted at a size when that net is positive there.

The transfer model is a line fitted to measured copies: latency + bytes / rate.
A candidate is described per layer and decode step by the bytes it moves over
the link and the device time of its kernels (decode, plus any per-step unpack,
plus its page conversion amortised over the tokens of a page).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Iterable, Sequence


@dataclass(frozen=True)
class LinkModel:
    """Host-to-device copy time = latency_us + bytes / rate."""

    latency_us: float
    rate_GBps: float

    def copy_us(self, nbytes: float) -> float:
        return self.latency_us + nbytes / (self.rate_GBps * 1e3)

    def transfer_us(self, nbytes: float) -> float:
        """Time of the bytes alone (what moving nbytes fewer saves in one copy)."""
        return nbytes / (self.rate_GBps * 1e3)


def fit_link(samples: Iterable[Sequence[float]]) -> LinkModel:
    """Least-squares line through measured (bytes, microseconds) copy samples."""
    pts = [(float(b), float(t)) for b, t in samples]
    if len(pts) < 2:
        raise ValueError("need at least two copy samples")
    n = len(pts)
    mb = sum(b for b, _ in pts) / n
    mt = sum(t for _, t in pts) / n
    sbb = sum((b - mb) ** 2 for b, _ in pts)
    if sbb == 0.0:
        raise ValueError("copy samples need at least two sizes")
    slope = sum((b - mb) * (t - mt) for b, t in pts) / sbb  # us per byte
    if slope <= 0.0:
        raise ValueError("copy time does not grow with size")
    return LinkModel(latency_us=mt - slope * mb, rate_GBps=1e-3 / slope)


@dataclass(frozen=True)
class Candidate:
    """One history format at one context size, per layer and decode step."""

    name: str
    link_bytes: float  # bytes crossing the host link
    device_us: float   # GPU time of its kernels (decode, per-step unpack, amortised conversion)


def net_saving_us(link: LinkModel, base: Candidate, cand: Candidate, layers: int = 1) -> float:
    """Per decode step (one token): transfer time the candidate saves by the bytes
    it stops moving, minus the GPU time it adds, over `layers` layers."""
    saved = link.transfer_us((base.link_bytes - cand.link_bytes) * layers)
    added = (cand.device_us - base.device_us) * layers
    return saved - added


def accept(link: LinkModel, base: Candidate, cand: Candidate, layers: int = 1) -> bool:
    """The gate's rule: accept when the net saving is positive."""
    return net_saving_us(link, base, cand, layers) > 0.0


def predict_step_us(link: LinkModel, cand: Candidate, layers: int) -> float:
    """Host-resident step with two device slots: layer l + 1 is copied while layer l
    decodes, so after the first copy each layer costs the longer of its copy and
    the previous layer's kernels, and the last layer's kernels end the step."""
    if layers < 1:
        raise ValueError("layers < 1")
    c = link.copy_us(cand.link_bytes)
    return c + (layers - 1) * max(c, cand.device_us) + cand.device_us


def per_tile_ratio(base: Candidate, cand: Candidate, base_tiles: float, cand_tiles: float) -> float:
    """Device time per tile of the candidate over the base's (the per-tile speed a
    kernel-only rule would compare; reported beside the gate, not used by it)."""
    return (cand.device_us / cand_tiles) / (base.device_us / base_tiles)
