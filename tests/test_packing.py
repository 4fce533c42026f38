"""The host-resident history image (Workload.packed_image): parts at 256-byte
aligned offsets, each holding the step's bytes in page order (records of the 8-bit
pages, BF16 K and V of the exact pages, q, identity page tables), for multi-request
and single-tier histories."""
import numpy as np
import pytest

import oracle
from tiered_paged_kv_gb300 import synth


@pytest.mark.parametrize("lengths,recent", [([700, 64 * 5 + 3, 1], 100), ([64 * 9], None), ([64 * 9], 0)])
def test_packed_image_layout(lengths, recent):
    w = synth.make_workload(lengths, recent, H=2, seed=70)
    rec = (np.arange(w.n_slots * w.H * oracle.REC_BYTES) % 251).astype(np.uint8)   # distinct bytes per slot
    img, off = w.packed_image(rec)
    for name in ("rec", "k", "v", "q", "pt", "pt8"):
        assert off[name] % 256 == 0
    s8 = w.int8_slots()
    ex, off_e = w.exact_page_table()
    rb = w.H * oracle.REC_BYTES
    recs = img[off["rec"]:off["rec"] + len(s8) * rb].reshape(len(s8), rb)
    for i, slot in enumerate(s8):
        assert np.array_equal(recs[i], rec[slot * rb:(slot + 1) * rb])
    kb = w.k_pool[ex].reshape(-1).view(np.uint8)
    assert np.array_equal(img[off["k"]:off["k"] + kb.size], kb)
    vb = w.v_pool[ex].reshape(-1).view(np.uint8)
    assert np.array_equal(img[off["v"]:off["v"] + vb.size], vb)
    qb = w.q.reshape(-1).view(np.uint8)
    assert np.array_equal(img[off["q"]:off["q"] + qb.size], qb)
    pt = img[off["pt"]:off["pt"] + 4 * len(ex)].view(np.int32)
    pt8 = img[off["pt8"]:off["pt8"] + 4 * len(s8)].view(np.int32)
    assert np.array_equal(pt, np.arange(len(ex))) and np.array_equal(pt8, np.arange(len(s8)))
    assert np.array_equal(off["req_page_off"], off_e) and off["n_exact_pages"] == len(ex)
    assert off["n_int8_pages"] == len(s8) and off["nbytes"] % 256 == 0 and img.size >= off["nbytes"]


@pytest.mark.parametrize("lengths,recent", [([700, 64 * 5 + 3, 1], 100), ([64 * 9], None)])
def test_packed_image_with_13bit_exact_tier(lengths, recent):
    """The exact tier as compacted 13-bit records: each record cut to its size,
    16-byte aligned, in (page, head) order, with int64 offsets; no BF16 K or V."""
    w = synth.make_workload(lengths, recent, H=2, seed=71, key_sigma="outliers")
    rec = np.zeros(w.n_slots * w.H * oracle.REC_BYTES, np.uint8)
    ex, _ = w.exact_page_table()
    p13 = np.zeros(w.n_slots * w.H * oracle.PACK13_RECORD_BYTES, np.uint8)
    oracle.pack13_pages(w.H, w.k_pool, w.v_pool, ex, ex, p13)
    # one plane stored raw: more than 32 exponent fields in the first exact page's keys
    slot0 = ex[0]
    raw_keys = np.arange(64 * 256, dtype=np.uint16).reshape(64, 256)
    one = oracle.pack13_page_head(raw_keys, w.v_pool[slot0, 1])
    p13.reshape(w.n_slots, w.H, -1)[slot0, 1, :len(one)] = one
    img, off = w.packed_image(rec, p13)
    assert off["k"] == off["v"] == off["p13"] and off["p13"] % 256 == 0 and off["p13off"] % 256 == 0
    offs = img[off["p13off"]:off["p13off"] + 8 * len(ex) * w.H].view(np.int64)
    assert (offs % 16 == 0).all() and offs[0] == 0
    pool = p13.reshape(w.n_slots, w.H, -1)
    for i, slot in enumerate(ex):
        for h in range(w.H):
            r = pool[slot, h]
            size = 16 + int(r[:4].view(np.uint32)[0]) + int(r[4:8].view(np.uint32)[0])
            at = off["p13"] + offs[i * w.H + h]
            assert np.array_equal(img[at:at + size], r[:size])
            k, v = oracle.unpack13_page_head(img[at:at + size])
            assert np.array_equal(k, raw_keys if (slot == slot0 and h == 1) else w.k_pool[slot, h])
            assert np.array_equal(v, w.v_pool[slot, h])
    assert off["p13_bytes"] == int(offs[-1]) + ((size + 15) & ~15)
    n = len(ex) * w.H   # every plane encoded except the one raw key plane
    assert off["p13_bytes"] == n * (16 + 2 * 26656) + (32768 - 26656)
