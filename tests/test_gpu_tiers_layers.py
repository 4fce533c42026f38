"""Incremental conversion across several layers ("model quantization", "An 8-bit
page format shaped for its kernel": conversion only for pages fully written in
every layer, served exact until published; "ActiveKV", "The idea": host memory
holds the authoritative copy of the history).

Four layers share the requests' page tables; histories grow by ragged amounts and
one layer lags behind the others for a while.  At every step: no page is in the
8-bit table before every layer has written it and every layer's record of it is
converted -- in the device pool and in the pinned host image alike -- each
layer's decode through the step's tables matches the oracle on the oracle's own
records, and the host image's records, staged back through the stager, decode
bit-identically to the device-resident ones."""
import dataclasses

import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import REC_POISON, assert_close, dev_u16, torch

pytestmark = pytest.mark.gpu

L = 4


def layer_workloads(final, H, seed):
    """One workload per layer, every layer's pages moved into layer 0's slots (the
    layers share the page tables); unused slots stay poisoned."""
    w0 = synth.make_workload(final, None, H=H, seed=seed, key_sigma="outliers")
    out = [w0]
    for l in range(1, L):
        wl = synth.make_workload(final, None, H=H, seed=seed + l, key_sigma="outliers")
        k = np.full_like(w0.k_pool, synth.BF16_NAN)
        v = np.full_like(w0.v_pool, synth.BF16_NAN)
        for b in range(w0.B):
            k[w0.pages[b]] = wl.k_pool[wl.pages[b]]
            v[w0.pages[b]] = wl.v_pool[wl.pages[b]]
        out.append(dataclasses.replace(w0, k_pool=k, v_pool=v, q=wl.q))
    return out


def split_view(w, n_tokens, n8):
    pages = [list(w.pages[b][: (n_tokens[b] + 63) // 64]) for b in range(w.B)]
    return dataclasses.replace(w, n_tokens=np.asarray(n_tokens, np.int64), n8=np.asarray(n8, np.int64),
                               n_ex=np.asarray(n_tokens, np.int64) - 64 * np.asarray(n8, np.int64), pages=pages)


def test_layers_publish_together_and_host_image_is_authoritative():
    t = torch()
    final = [64 * 30 + 5, 64 * 22 + 33, 64 * 10]
    recent = 200
    H = 2
    ws_ = layer_workloads(final, H, seed=70)
    w0 = ws_[0]
    G, B = w0.G, w0.B
    max_pages = max(len(p) for p in w0.pages)
    RB = H * tpk.RECORD_BYTES
    shape = tpk.Shape(H, impl=tpk.IMPL_TENSOR, kv_slots=w0.n_slots, rec_slots=w0.n_slots)
    k = [dev_u16(w.k_pool) for w in ws_]
    v = [dev_u16(w.v_pool) for w in ws_]
    q = [dev_u16(w.q) for w in ws_]
    rec = [t.full((w0.n_slots * RB,), REC_POISON, dtype=t.uint8, device="cuda") for _ in range(L)]
    host = [t.full((w0.n_slots * RB,), REC_POISON, dtype=t.uint8).pin_memory() for _ in range(L)]
    nbytes = tpk.Tiers.device_bytes(B, max_pages)
    scratch = t.empty(nbytes, dtype=t.uint8, device="cuda")
    ws_bytes = tpk.hybrid_workspace_bytes(shape, B)
    wsp = t.empty(ws_bytes, dtype=t.uint8, device="cuda")
    conv, dec = t.cuda.Stream(), t.cuda.Stream()
    # the oracle's own records of every page the loop can publish, per layer
    last8 = [max(0, (f - recent) // 64) for f in final]
    rec_orc = []
    for w in ws_:
        r = np.full(w0.n_slots * RB, REC_POISON, np.uint8)
        s8 = np.concatenate([np.asarray(w.pages[b][:last8[b]]) for b in range(B)]).astype(np.int32)
        oracle.quantize_pages(H, w.k_pool, w.v_pool, s8, s8, r)
        rec_orc.append(r.reshape(w0.n_slots, H, oracle.REC_BYTES))
    # a staging slot big enough for every layer's published records
    slot_bytes = max(sum(last8), 1) * RB
    slots = [t.empty(slot_bytes, dtype=t.uint8, device="cuda") for _ in range(2)]
    n = [min(f, 600 + 250 * b) for b, f in enumerate(final)]
    lag_layer, lag = 2, 150
    checked_pages = scale_ulp_pages = 0
    with tpk.Tiers(shape, B, max_pages, recent, k, v, rec, scratch, nbytes, host_rec_pools=host) as tiers, \
            tpk.Stager(slots, slot_bytes) as st:
        for step in range(14):
            lagging = 3 <= step < 9
            written = []
            for b in range(B):
                lw = [n[b]] * L
                if lagging:
                    lw[lag_layer] = max(n[b] - lag, 0)
                written.append(lw)
            # (the lagging layer stays above the pages already converted: those were
            # older than the recent window, 200 tokens, when they started)
            for b in range(B):
                tiers.update(b, n[b], w0.pages[b][: (n[b] + 63) // 64], layer_written=written[b])
            plan = tiers.step(conv, dec)
            n8, n_ex = plan["n_int8_pages"], plan["n_exact_tokens"]
            for b in range(B):
                assert 64 * n8[b] + n_ex[b] == n[b]
                assert 64 * n8[b] <= max(0, n[b] - recent)
                assert 64 * n8[b] <= min(written[b]), (step, b, n8[b], written[b])
            # every page in the 8-bit table is converted in every layer, in the device
            # pool and in the host image
            pt8 = np.concatenate([np.asarray(w0.pages[b][:n8[b]]) for b in range(B)]).astype(np.int64)
            for l in range(L):
                got_d = rec[l].cpu().numpy().reshape(w0.n_slots, H, oracle.REC_BYTES)
                got_h = host[l].numpy().reshape(w0.n_slots, H, oracle.REC_BYTES)
                for slot in pt8:
                    for h in range(H):
                        assert np.array_equal(got_h[slot, h], got_d[slot, h]), (step, l, slot, h)
                        if np.array_equal(got_h[slot, h], rec_orc[l][slot, h]):
                            continue
                        # otherwise only a near tie may move a channel scale by one ulp
                        _, _, s_g, r_g, u_g = oracle.record_fields(got_h[slot, h])
                        _, _, s_o, r_o, u_o = oracle.record_fields(rec_orc[l][slot, h])
                        d = np.abs(s_g.view(np.int32).astype(np.int64) - s_o.view(np.int32).astype(np.int64))
                        assert d.max() <= 1 and d.max() > 0, (step, l, slot, h)
                        scale_ulp_pages += 1
                    checked_pages += 1
            # each layer's decode through the step's tables against the oracle
            for l in range(L):
                o = t.empty(B, H * G, 256, dtype=t.float32, device="cuda")
                lse = t.empty(B, H * G, dtype=t.float32, device="cuda")
                with t.cuda.stream(dec):
                    tpk.decode_hybrid_batched(shape, B, q[l], k[l], v[l], rec[l], plan["page_table"],
                                              plan["req_page_off"], n_ex, plan["page_table8"],
                                              plan["req_page_off8"], n8, o, lse, wsp, ws_bytes, dec)
                dec.synchronize()
                oo, ol = oracle.hybrid_workload(split_view(ws_[l], n, n8), rec_orc[l].reshape(-1), n_threads=8)
                og, lg = o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
                assert_close(og, lg, oo, ol, f"step {step} layer {l}")
                # the host image's records of this layer, staged through the stager into
                # a device slot (published pages in table order), decode bit-identically
                if len(pt8):
                    regions = [(host[l].data_ptr() + int(s) * RB, i * RB, RB) for i, s in enumerate(pt8)]
                    slot, _ = st.stage(regions)
                    st.acquire(slot, dec)
                    ident = t.arange(len(pt8), dtype=t.int32, device="cuda")
                    o2 = t.empty_like(o)
                    l2 = t.empty_like(lse)
                    shape2 = tpk.Shape(H, impl=tpk.IMPL_TENSOR, kv_slots=w0.n_slots, rec_slots=len(pt8))
                    with t.cuda.stream(dec):
                        tpk.decode_hybrid_batched(shape2, B, q[l], k[l], v[l], slots[slot], plan["page_table"],
                                                  plan["req_page_off"], n_ex, ident, plan["req_page_off8"], n8, o2,
                                                  l2, wsp, ws_bytes, dec)
                    st.release(slot, dec)
                    dec.synchronize()
                    assert np.array_equal(o2.cpu().numpy(), o.cpu().numpy()) and \
                        np.array_equal(l2.cpu().numpy(), lse.cpu().numpy()), (step, l)
            n = [min(f, x + 83 + 29 * b) for b, (f, x) in enumerate(zip(final, n))]
        # catch up: every eligible page converted and published in every layer
        for b in range(B):
            tiers.update(b, n[b], w0.pages[b][: (n[b] + 63) // 64])
        tiers.step(conv, dec)
        tiers.sync()
        plan = tiers.step(conv, dec)
        assert list(plan["n_int8_pages"]) == [max(0, (x - recent) // 64) for x in n] and plan["converting"] == 0
    st_, flags = tpk.get_device_status(reset=True)
    assert st_ == 0, flags
    assert checked_pages > 0
    assert scale_ulp_pages <= max(2, checked_pages // 50), (scale_ulp_pages, checked_pages)


def test_layer_written_bounds_are_checked():
    t = torch()
    w = synth.make_workload([64 * 10], None, H=1, seed=71)
    shape = tpk.Shape(1, kv_slots=w.n_slots, rec_slots=w.n_slots)
    k = [dev_u16(w.k_pool) for _ in range(2)]
    v = [dev_u16(w.v_pool) for _ in range(2)]
    rec = [t.zeros(w.n_slots * tpk.RECORD_BYTES, dtype=t.uint8, device="cuda") for _ in range(2)]
    nbytes = tpk.Tiers.device_bytes(1, 10)
    scratch = t.empty(nbytes, dtype=t.uint8, device="cuda")
    s = t.cuda.Stream()
    with tpk.Tiers(shape, 1, 10, 64, k, v, rec, scratch, nbytes) as tiers:
        slots = list(w.pages[0])
        # layer 1 has written 3 pages: only those convert
        tiers.update(0, 640, slots, layer_written=[640, 3 * 64 + 10])
        plan = tiers.step(s, s)
        assert plan["started"] == 3
        with pytest.raises(tpk.TpkError):
            tiers.update(0, 640, slots, layer_written=[640, 64])      # below the converted pages
        with pytest.raises(tpk.TpkError):
            tiers.update(0, 640, slots, layer_written=[641, 640])     # beyond the history
        tiers.update(0, 640, slots, layer_written=[640, 640])
        plan = tiers.step(s, s)
        assert plan["started"] == 6
