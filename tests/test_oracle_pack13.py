"""Pins of the oracle's lossless 13-bit tier: hand-worked encodings, the 32-entry
boundary, exact round trips over every kind of BF16 value, sizes, and the pool
layout.

Source: "model quantization", section "A lossless tier first": 13 bits per value
(an 18.7 % saving) with a raw fallback when a plane needs more than a 32-entry
table.  Reading taken where the page is silent: a plane is one page-head's keys
(or values), and the table holds the plane's distinct BF16 exponent fields, so a
value is its sign and mantissa (one byte) plus a 5-bit table index.
"""
import numpy as np
import pytest

import oracle
from tiered_paged_kv_gb300 import synth

N = 64 * 256


def bits(values):
    v = np.asarray(values, np.float32)
    b = synth.f32_to_bf16(v)
    assert np.array_equal(synth.bf16_to_f32(b), v)
    return b


def plane_of(head_values):
    p = np.zeros(N, np.uint16)
    p[:len(head_values)] = head_values
    return p


def test_hand_worked_plane():
    """1.0 = 0x3F80 (exp 127), -2.0 = 0xC000 (exp 128, sign), 0.5 = 0x3F00 (exp 126),
    3.0 = 0x4040 (exp 128, mantissa 0x40), 0.0 (exp 0): table [0, 126, 127, 128]."""
    enc = oracle.pack13_plane(plane_of(bits([1.0, -2.0, 0.5, 3.0])))
    assert len(enc) == 26656
    assert list(enc[:32]) == [0, 126, 127, 128] + [0] * 28
    sm = enc[32:32 + N]
    assert list(sm[:5]) == [0x00, 0x80, 0x00, 0x40, 0x00] and not sm[5:].any()
    lo4 = enc[32 + N:32 + N + N // 2]
    assert list(lo4[:3]) == [0x32, 0x31, 0x00] and not lo4[3:].any()  # indices 2, 3 | 1, 3 | 0, 0
    assert not enc[32 + N + N // 2:].any()                             # no index reaches 16


def test_hand_worked_high_index_bit():
    """2^k for k = -10 .. 10 (exponents 117 .. 137) and zero: 22 table entries; 2^10
    sits at index 21 = 0b10101 (nibble 5, high bit 1)."""
    vals = [2.0 ** k for k in range(-10, 11)]
    enc = oracle.pack13_plane(plane_of(bits(vals)))
    assert list(enc[:22]) == [0] + list(range(117, 138)) and not enc[22:32].any()
    lo4 = enc[32 + N:32 + N + N // 2]
    hi1 = enc[32 + N + N // 2:]
    idx = [((lo4[i // 2] >> (4 * (i % 2))) & 15) | (((hi1[i // 8] >> (i % 8)) & 1) << 4) for i in range(22)]
    assert idx == list(range(1, 22)) + [0]
    # index >= 16 means exponent >= 132, i.e. 2^5 .. 2^10: values 15 .. 20
    assert hi1[1] == 0b10000000 and hi1[2] == 0b00011111 and hi1[0] == 0


def exponent_plane(n_exponents, seed):
    """A plane whose values use exactly n_exponents distinct exponent fields."""
    e = np.arange(n_exponents) + 100
    pick = synth.randint(seed, 90, N, 0, n_exponents - 1)  # bounds inclusive
    pick[:n_exponents] = np.arange(n_exponents)
    mant = synth.randint(seed, 91, N, 0, 127)
    sign = synth.randint(seed, 92, N, 0, 1)
    return ((sign << 15) | (e[pick] << 7) | mant).astype(np.uint16)


@pytest.mark.parametrize("n,encoded", [(1, True), (31, True), (32, True), (33, False), (200, False)])
def test_table_boundary(n, encoded):
    p = exponent_plane(n, n)
    enc = oracle.pack13_plane(p)
    assert len(enc) == (26656 if encoded else 32768)
    if not encoded:
        assert np.array_equal(enc.view(np.uint16), p)  # raw: the BF16 values themselves
    assert np.array_equal(oracle.unpack13_plane(enc).reshape(-1), p)


def test_every_kind_of_value_round_trips():
    specials = np.array([0x0000, 0x8000, 0x0001, 0x807F, 0x007F, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x7F81,
                         0x0080, 0x7F7F, 0xFF7F, 0x3F80], np.uint16)
    p = plane_of(specials)
    enc = oracle.pack13_plane(p)
    assert len(enc) == 26656
    assert np.array_equal(oracle.unpack13_plane(enc).reshape(-1), p)
    everything = np.arange(65536, dtype=np.uint16)
    for part in everything.reshape(4, N):
        assert np.array_equal(oracle.unpack13_plane(oracle.pack13_plane(part)).reshape(-1), part)


@pytest.mark.parametrize("kind", ["unit", "outliers", "loguniform"])
def test_page_heads_of_the_workloads_round_trip(kind):
    w = synth.make_workload([64 * 6], 0, H=2, seed=93, key_sigma=kind,
                            value_sigma="loguniform" if kind == "loguniform" else "unit")
    for slot in w.pages[0]:
        for h in range(w.H):
            rec = oracle.pack13_page_head(w.k_pool[slot, h], w.v_pool[slot, h])
            kb, vb = rec[:4].view(np.uint32)[0], rec[4:8].view(np.uint32)[0]
            assert kb in (26656, 32768) and vb in (26656, 32768) and len(rec) == 16 + kb + vb
            assert not rec[8:16].any()
            k, v = oracle.unpack13_page_head(rec)
            assert np.array_equal(k, w.k_pool[slot, h]) and np.array_equal(v, w.v_pool[slot, h])


def test_thirteen_bits_per_value():
    enc = oracle.pack13_plane(exponent_plane(20, 5))
    assert (len(enc) - 32) * 8 == 13 * N           # plus the 32-byte table
    assert abs(1 - len(enc) / 32768 - 0.187) < 0.001


def test_malformed_size_is_refused():
    with pytest.raises(ValueError):
        oracle.unpack13_plane(np.zeros(1000, np.uint8))


def test_pool_layout():
    w = synth.make_workload([64 * 5], 0, H=2, seed=94, key_sigma="outliers")
    src = np.asarray(w.pages[0], np.int32)
    dst = synth.permutation(94, 95, len(src)).astype(np.int32)
    pool = np.full(len(src) * w.H * oracle.PACK13_RECORD_BYTES, 0xAB, np.uint8)
    oracle.pack13_pages(w.H, w.k_pool, w.v_pool, src, dst, pool)
    recs = pool.reshape(len(src), w.H, oracle.PACK13_RECORD_BYTES)
    for i in range(len(src)):
        for h in range(w.H):
            r = recs[dst[i], h]
            one = oracle.pack13_page_head(w.k_pool[src[i], h], w.v_pool[src[i], h])
            assert np.array_equal(r[:len(one)], one) and not r[len(one):].any()
