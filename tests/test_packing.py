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
