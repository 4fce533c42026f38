"""The lossless 13-bit tier on the GPU ("model quantization", "A lossless tier
first"): records bit-identical to the oracle's, unpacking restores every bit
(fixed-stride pools and compacted host images alike), raw fallback planes, special
values, malformed records and out-of-pool slots reported, the full 128K history,
and the exact decode over unpacked pages equal to the decode over the originals."""
import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import DevWorkload, dev_i32, dev_u8, torch

pytestmark = pytest.mark.gpu
R = tpk.PACK13_RECORD_BYTES


def with_special_pages(w):
    """Overwrite three exact pages: keys with more than 32 exponent fields (raw),
    values with exactly 32 (encoded); every special BF16 pattern (signed zeros,
    subnormals, infinities, NaNs); a constant page (one exponent)."""
    ex, _ = w.exact_page_table()
    a, b, c = ex[:3]
    w.k_pool[a, 0] = np.arange(64 * 256, dtype=np.uint16).reshape(64, 256) * 3
    e = (np.arange(64 * 256) % 32 + 100).astype(np.uint16)
    w.v_pool[a, 0] = ((e << 7) | (np.arange(64 * 256) % 128).astype(np.uint16)).reshape(64, 256)
    specials = np.array([0x0000, 0x8000, 0x0001, 0x807F, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x7F81, 0x0080,
                         0x7F7F, 0xFF7F], np.uint16)
    w.k_pool[b, -1] = np.resize(specials, 64 * 256).reshape(64, 256)
    w.v_pool[c, 0] = 0x3F80
    return w


def gpu_pack(w, d):
    slots = w.exact_page_table()[0]
    pool = torch().full((w.n_slots * w.H * R,), 0xCD, dtype=torch().uint8, device="cuda")
    s = dev_i32(slots)
    tpk.kv_pack13_pages(d.shape, d.k, d.v, s, s, len(slots), pool, w.n_slots)
    torch().cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
    return pool


def record_size(r):
    return 16 + int(r[:4].view(np.uint32)[0]) + int(r[4:8].view(np.uint32)[0])


@pytest.mark.parametrize("kind", ["unit", "outliers", "loguniform"])
def test_pack_matches_the_oracle_and_unpack_restores_every_bit(kind):
    w = with_special_pages(synth.make_workload([64 * 12 + 5, 64 * 3], None, H=2, seed=80, key_sigma=kind,
                                               value_sigma="loguniform" if kind == "loguniform" else "unit"))
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    pool = gpu_pack(w, d)
    host = pool.cpu().numpy().reshape(w.n_slots, w.H, R)
    ex, _ = w.exact_page_table()
    ref = np.zeros(w.n_slots * w.H * R, np.uint8)
    oracle.pack13_pages(w.H, w.k_pool, w.v_pool, ex, ex, ref)
    ref = ref.reshape(w.n_slots, w.H, R)
    n_raw = 0
    for slot in ex:
        for h in range(w.H):
            size = record_size(ref[slot, h])
            assert np.array_equal(host[slot, h, :size], ref[slot, h, :size]), (slot, h)
            n_raw += (size - 16 - 2 * 26656) // (32768 - 26656)
    assert n_raw >= 1
    # unpack into poisoned pools at other slots
    t = torch()
    k2 = t.full_like(d.k, -1)
    v2 = t.full_like(d.v, -1)
    dst = synth.permutation(81, 1, w.n_slots)[:len(ex)].astype(np.int32)
    offs = (np.repeat(ex.astype(np.int64), w.H) * w.H + np.tile(np.arange(w.H), len(ex))) * R
    tpk.kv_unpack13_pages(d.shape, pool, pool.numel(), dev_u8(offs.view(np.uint8)), dev_i32(dst), len(ex), k2, v2)
    t.cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
    k2h = k2.cpu().numpy().view(np.uint16).reshape(w.k_pool.shape)
    v2h = v2.cpu().numpy().view(np.uint16).reshape(w.v_pool.shape)
    assert np.array_equal(k2h[dst], w.k_pool[ex]) and np.array_equal(v2h[dst], w.v_pool[ex])


def test_unpack_from_a_compacted_image_and_decode_matches():
    """The host-resident form: compacted records staged as one image; the exact
    decode over the unpacked pages equals the decode over the originals bit for bit."""
    t = torch()
    w = synth.make_workload([3000, 64 * 7 + 1, 64], None, H=4, seed=82, key_sigma="outliers")
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    pool = gpu_pack(w, d)
    img, off = w.packed_image(np.zeros(16, np.uint8), pool.cpu().numpy())
    dimg = dev_u8(img)
    ne = off["n_exact_pages"]
    offs = dimg[off["p13off"]:off["p13off"] + 8 * ne * w.H]
    k2 = t.zeros(ne * w.H * 64 * 256, dtype=t.int16, device="cuda")
    v2 = t.zeros_like(k2)
    shape2 = tpk.Shape(w.H, impl=tpk.IMPL_TENSOR, kv_slots=ne, rec_slots=1)
    src = dimg[off["p13"]:]
    tpk.kv_unpack13_pages(shape2, src, off["p13_bytes"], offs, dev_i32(np.arange(ne)), ne, k2, v2)
    t.cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
    ex, off_e = w.exact_page_table()
    assert np.array_equal(k2.cpu().numpy().view(np.uint16).reshape(ne, w.H, 64, 256), w.k_pool[ex])
    a = d.hybrid()
    o = t.empty(w.B, w.H * w.G, 256, dtype=t.float32, device="cuda")
    lse = t.empty(w.B, w.H * w.G, dtype=t.float32, device="cuda")
    nb = tpk.hybrid_workspace_bytes(shape2, w.B)
    ws = t.empty(nb, dtype=t.uint8, device="cuda")
    tpk.decode_hybrid_batched(shape2, w.B, d.q, k2, v2, t.zeros(16, dtype=t.uint8, device="cuda"),
                              dev_i32(np.arange(ne)), off_e, w.n_ex, dev_i32(np.zeros(1)), np.zeros(w.B + 1, np.int32),
                              np.zeros(w.B, np.int32), o, lse, ws, nb)
    t.cuda.synchronize()
    assert np.array_equal(o.cpu().numpy(), a[0].astype(np.float32)) and np.array_equal(lse.cpu().numpy(),
                                                                                         a[1].astype(np.float32))


def test_malformed_records_and_bad_slots_are_reported_and_skipped():
    t = torch()
    w = synth.make_workload([64 * 4], None, H=2, seed=83)
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    pool = gpu_pack(w, d)
    ex, _ = w.exact_page_table()
    host = pool.cpu().numpy().reshape(w.n_slots, w.H, R)
    host[ex[1], 0, 0:4] = np.array([123, 0, 0, 0], np.uint8)    # key-plane size neither 26656 nor 32768
    pool.copy_(t.from_numpy(host.reshape(-1)))
    offs = ((np.repeat(ex.astype(np.int64), w.H) * w.H + np.tile(np.arange(w.H), len(ex))) * R)
    offs[5] += 8                                                  # misaligned record (page 2, head 1)
    k2 = t.full_like(d.k, 7)
    v2 = t.full_like(d.v, 7)
    tpk.kv_unpack13_pages(d.shape, pool, pool.numel(), dev_u8(offs.view(np.uint8)), dev_i32(ex), len(ex), k2, v2)
    t.cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert flags == 4 and tpk.STATUS_NAMES[st] == "TPK_ERR_FORMAT"
    k2h = k2.cpu().numpy().view(np.uint16).reshape(w.k_pool.shape)
    for i, slot in enumerate(ex):
        for h in range(w.H):
            bad = (i == 1 and h == 0) or (i == 2 and h == 1)
            assert np.array_equal(k2h[slot, h], np.full((64, 256), 7, np.uint16) if bad else w.k_pool[slot, h])
    # a destination outside the pool, and a record extent past src_bytes
    dst = ex.copy()
    dst[0] = w.n_slots
    tpk.kv_unpack13_pages(d.shape, pool, int(offs[0]) + 100, dev_u8(offs[:2].view(np.uint8)), dev_i32(dst[:1]), 1,
                          k2, v2)
    t.cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert flags & 1
    dst[0] = ex[0]
    tpk.kv_unpack13_pages(d.shape, pool, int(offs[0]) + 100, dev_u8(offs[:2].view(np.uint8)), dev_i32(dst[:1]), 1,
                          k2, v2)
    t.cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert flags == 4


def test_full_exact_history_round_trip():
    """The 131,072-token all-BF16 history (4 KV heads, 2048 pages): pack, unpack,
    every bit back; the compacted size is reported."""
    t = torch()
    w = synth.make_workload([131072], None, H=4, seed=12, key_sigma="outliers")
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    pool = gpu_pack(w, d)
    ex, _ = w.exact_page_table()
    host = pool.cpu().numpy().reshape(w.n_slots, w.H, R)
    sizes = np.array([[record_size(host[s, h]) for h in range(w.H)] for s in ex])
    k2 = t.zeros_like(d.k)
    v2 = t.zeros_like(d.v)
    offs = (np.repeat(ex.astype(np.int64), w.H) * w.H + np.tile(np.arange(w.H), len(ex))) * R
    tpk.kv_unpack13_pages(d.shape, pool, pool.numel(), dev_u8(offs.view(np.uint8)), dev_i32(ex), len(ex), k2, v2)
    t.cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
    used = t.from_numpy(ex.astype(np.int64)).cuda()   # the pool's other slots are not part of the history
    view = lambda x: x.view(w.n_slots, -1).index_select(0, used)
    assert t.equal(view(k2), view(d.k)) and t.equal(view(v2), view(d.v))
    frac = sizes.sum() / (len(ex) * w.H * 65536)
    print(f"13-bit image of the 128K history: {sizes.sum() / 1e6:.1f} MB = {frac:.4f} of BF16")
    assert frac < 0.82


def test_many_heads_round_trip():
    t = torch()
    w = synth.make_workload([64 * 3 + 7], None, H=64, seed=84, key_sigma="loguniform")
    d = DevWorkload(w, tpk.IMPL_TENSOR)
    pool = gpu_pack(w, d)
    ex, _ = w.exact_page_table()
    ref = np.zeros(w.n_slots * w.H * R, np.uint8)
    oracle.pack13_pages(w.H, w.k_pool, w.v_pool, ex, ex, ref)
    host = pool.cpu().numpy().reshape(w.n_slots, w.H, R)
    ref = ref.reshape(w.n_slots, w.H, R)
    for slot in ex:
        for h in range(w.H):
            n = record_size(ref[slot, h])
            assert np.array_equal(host[slot, h, :n], ref[slot, h, :n])
    k2, v2 = t.zeros_like(d.k), t.zeros_like(d.v)
    offs = (np.repeat(ex.astype(np.int64), w.H) * w.H + np.tile(np.arange(w.H), len(ex))) * R
    tpk.kv_unpack13_pages(d.shape, pool, pool.numel(), dev_u8(offs.view(np.uint8)), dev_i32(ex), len(ex), k2, v2)
    t.cuda.synchronize()
    st, flags = tpk.get_device_status(reset=True)
    assert st == 0, flags
    k2h = k2.cpu().numpy().view(np.uint16).reshape(w.k_pool.shape)
    v2h = v2.cpu().numpy().view(np.uint16).reshape(w.v_pool.shape)
    assert np.array_equal(k2h[ex], w.k_pool[ex]) and np.array_equal(v2h[ex], w.v_pool[ex])
