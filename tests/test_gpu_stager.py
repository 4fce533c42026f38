"""Host-resident staging: per-layer histories in pinned host memory pass through
two device slots of a stager while the previous layer decodes; every layer's
output must equal the decode of the same history resident in HBM (bit for bit,
same kernels on the same bytes) and the oracle; calls out of the slot lifecycle
are refused."""
import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import DevWorkload, assert_close, dev_u16, oracle_records, torch

pytestmark = pytest.mark.gpu


def pinned(a):
    return torch().from_numpy(np.ascontiguousarray(a)).pin_memory()


def slot_views(dev_ptr_tensor, off, w):
    """Typed device views of one staged slot (a uint8 tensor)."""
    t = torch()
    s = dev_ptr_tensor
    H, G = w.H, w.G
    n8, ne = off["n_int8_pages"], off["n_exact_pages"]
    rec = s[off["rec"]:off["rec"] + n8 * H * tpk.RECORD_BYTES]
    k = s[off["k"]:off["k"] + ne * H * 64 * 256 * 2]
    v = s[off["v"]:off["v"] + ne * H * 64 * 256 * 2]
    q = s[off["q"]:off["q"] + w.B * H * G * 256 * 2]
    pt = s[off["pt"]:off["pt"] + max(ne, 1) * 4]
    pt8 = s[off["pt8"]:off["pt8"] + max(n8, 1) * 4]
    return rec, k, v, q, pt, pt8


def decode_from_slot(slot_t, off, w, impl, o, lse, ws, nbytes, stream):
    rec, k, v, q, pt, pt8 = slot_views(slot_t, off, w)
    shape = tpk.Shape(w.H, impl=impl, kv_slots=max(off["n_exact_pages"], 1), rec_slots=max(off["n_int8_pages"], 1))
    tpk.decode_hybrid_batched(shape, w.B, q, k, v, rec, pt, off["req_page_off"], w.n_ex, pt8, off["req_page_off8"],
                              w.n8, o, lse, ws, nbytes, stream)


@pytest.mark.parametrize("impl", [tpk.IMPL_SIMT, tpk.IMPL_TENSOR])
def test_layers_through_two_slots(impl):
    t = torch()
    L = 6
    layers = []
    for l in range(L):
        w = synth.make_workload([2500 + 300 * l, 900], 300, H=2, seed=200 + l, key_sigma="outliers")
        rec = oracle_records(w)
        img, off = w.packed_image(rec)
        layers.append((w, rec, pinned(img), off))
    slot_bytes = max(off["nbytes"] for _, _, _, off in layers)
    slots = [t.empty(slot_bytes, dtype=t.uint8, device="cuda") for _ in range(2)]
    stream = t.cuda.Stream()
    outs = []
    with tpk.Stager(slots, slot_bytes) as st:
        shape0 = tpk.Shape(2, impl=impl)
        nbytes = tpk.hybrid_workspace_bytes(shape0, 2)
        ws = t.empty(nbytes, dtype=t.uint8, device="cuda")
        pending = st.stage([(layers[0][2], 0, layers[0][3]["nbytes"])])
        for l in range(L):
            w, _, img, off = layers[l]
            nxt = st.stage([(layers[l + 1][2], 0, layers[l + 1][3]["nbytes"])]) if l + 1 < L else None
            slot, _ = pending
            st.acquire(slot, stream)
            o = t.empty(w.B, w.H * w.G, 256, dtype=t.float32, device="cuda")
            lse = t.empty(w.B, w.H * w.G, dtype=t.float32, device="cuda")
            with t.cuda.stream(stream):
                decode_from_slot(slots[slot], off, w, impl, o, lse, ws, nbytes, stream)
            st.release(slot, stream)
            outs.append((o, lse))
            pending = nxt
        stream.synchronize()
    for l, (w, rec, _, _) in enumerate(layers):
        o = outs[l][0].cpu().numpy().astype(np.float64)
        lse = outs[l][1].cpu().numpy().astype(np.float64)
        d = DevWorkload(w, impl)
        d.load_records(rec)
        ro, rl = d.hybrid()
        assert np.array_equal(o, ro) and np.array_equal(lse, rl), f"layer {l}: staged != resident"
        oo, ol = oracle.hybrid_workload(w, rec, n_threads=8)
        assert_close(o, lse, oo, ol, f"layer {l}")


@pytest.mark.parametrize("impl", [tpk.IMPL_SIMT, tpk.IMPL_TENSOR])
def test_full_size_128k_layers_through_two_slots(impl):
    """The host-resident workload at its full layer size: four layers of the 128K
    hybrid history image (1,984 8-bit pages x 4 KV heads + 4,096 BF16 tokens, 295 MB
    each), each layer with a query of its own, staged from pinned host memory
    through two slots, each layer staged while the previous one decodes (the order
    the bench times).  Every layer equals the resident decode of its history and
    query bit for bit, and the oracle within the parity bar."""
    import dataclasses

    t = torch()
    w = synth.hybrid_128k(seed=2)
    rec = oracle_records(w)
    img0, off = w.packed_image(rec)
    L = 4
    qs, imgs = [], []
    for l in range(L):
        q = synth.normal_bf16(300 + l, 0, w.q.size).reshape(w.q.shape)
        img = img0.copy()
        img[off["q"]:off["q"] + q.nbytes] = q.view(np.uint8).reshape(-1)
        qs.append(q)
        imgs.append(pinned(img))
    del img0, img
    nb = off["nbytes"]
    slots = [t.empty(nb, dtype=t.uint8, device="cuda") for _ in range(2)]
    stream = t.cuda.Stream()
    nbytes = tpk.hybrid_workspace_bytes(tpk.Shape(w.H, impl=impl), w.B)
    ws = t.empty(nbytes, dtype=t.uint8, device="cuda")
    outs = []
    with tpk.Stager(slots, nb) as st:
        pending = st.stage([(imgs[0], 0, nb)])
        for l in range(L):
            nxt = st.stage([(imgs[l + 1], 0, nb)]) if l + 1 < L else None
            slot, _ = pending
            st.acquire(slot, stream)
            o = t.full((w.B, w.H * w.G, 256), float("nan"), dtype=t.float32, device="cuda")
            lse = t.full((w.B, w.H * w.G), float("nan"), dtype=t.float32, device="cuda")
            with t.cuda.stream(stream):
                decode_from_slot(slots[slot], off, w, impl, o, lse, ws, nbytes, stream)
            st.release(slot, stream)
            outs.append((o, lse))
            pending = nxt
        stream.synchronize()
    del slots, imgs
    d = DevWorkload(w, impl)
    d.load_records(rec)
    for l in range(L):
        o = outs[l][0].cpu().numpy().astype(np.float64)
        lse = outs[l][1].cpu().numpy().astype(np.float64)
        d.q = dev_u16(qs[l])
        ro, rl = d.hybrid()
        assert np.array_equal(o, ro) and np.array_equal(lse, rl), f"layer {l}: staged != resident"
        oo, ol = oracle.hybrid_workload(dataclasses.replace(w, q=qs[l]), rec, n_threads=8)
        assert_close(o, lse, oo, ol, f"layer {l}")
    st_, flags = tpk.get_device_status(reset=True)
    assert st_ == 0, flags


def test_lifecycle_is_enforced():
    t = torch()
    slots = [t.empty(4096, dtype=t.uint8, device="cuda") for _ in range(2)]
    src = pinned(np.arange(4096, dtype=np.uint8))
    stream = t.cuda.Stream()
    with tpk.Stager(slots, 4096) as st:
        with pytest.raises(tpk.TpkError):
            st.acquire(0, stream)                       # nothing staged
        s0, p0 = st.stage([(src, 0, 4096)])
        assert s0 == 0 and p0 == slots[0].data_ptr()
        with pytest.raises(tpk.TpkError):
            st.release(s0, stream)                      # staged, not acquired
        s1, _ = st.stage([(src, 0, 1024)])
        assert s1 == 1
        with pytest.raises(tpk.TpkError):
            st.stage([(src, 0, 16)])                    # slot 0 not released yet
        st.acquire(s0, stream)
        with pytest.raises(tpk.TpkError):
            st.acquire(s0, stream)                      # already acquired
        st.release(s0, stream)
        with pytest.raises(tpk.TpkError):
            st.stage([(src, 4000, 200)])                # outside the slot
        pageable = np.zeros(64, np.uint8)
        with pytest.raises(tpk.TpkError):
            st.stage([(pageable.ctypes.data, 0, 64)])   # not pinned
        s2, _ = st.stage([(src, 0, 4096)])              # slot 0 again, after its release
        assert s2 == 0
        st.acquire(s2, stream)
        st.release(s2, stream)
        stream.synchronize()
        assert np.array_equal(slots[0].cpu().numpy(), np.arange(4096, dtype=np.uint8))
    with pytest.raises(tpk.TpkError):
        tpk.Stager([slots[0], src], 4096)               # a host buffer is not a slot
