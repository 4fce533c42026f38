"""Incremental conversion and publication during decode: histories grow step by
step; pages older than the recent window are converted on a side stream and join
the 8-bit tier only once their conversion has finished.  Every step's decode
(through the tier manager's page tables) must match the oracle on the same split
and the same records, the split must always cover the history with at least the
recent tokens exact, and every eligible page must be published in the end."""
import dataclasses

import numpy as np
import pytest

import oracle
import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import synth
from tpk_testutil import REC_POISON, assert_close, dev_u16, oracle_records, torch

pytestmark = pytest.mark.gpu


def split_view(w, n_tokens, n8):
    """The workload restricted to history prefixes n_tokens[b] with n8[b] 8-bit pages."""
    pages = [list(w.pages[b][: (n_tokens[b] + 63) // 64]) for b in range(w.B)]
    return dataclasses.replace(w, n_tokens=np.asarray(n_tokens, np.int64), n8=np.asarray(n8, np.int64),
                               n_ex=np.asarray(n_tokens, np.int64) - 64 * np.asarray(n8, np.int64), pages=pages)


@pytest.mark.parametrize("impl", [tpk.IMPL_SIMT, tpk.IMPL_TENSOR])
def test_histories_grow_and_pages_are_published(impl):
    t = torch()
    final = [64 * 40 + 5, 64 * 25 + 33, 64 * 12]
    recent = 200
    w = synth.make_workload(final, None, H=2, seed=50, key_sigma="outliers")
    H, G, B = w.H, w.G, w.B
    max_pages = max(len(p) for p in w.pages)
    shape = tpk.Shape(H, impl=impl, kv_slots=w.n_slots, rec_slots=w.n_slots)
    k = dev_u16(w.k_pool)
    v = dev_u16(w.v_pool)
    q = dev_u16(w.q)
    rec = t.full((w.n_slots * H * tpk.RECORD_BYTES,), REC_POISON, dtype=t.uint8, device="cuda")
    nbytes = tpk.Tiers.device_bytes(B, max_pages)
    scratch = t.empty(nbytes, dtype=t.uint8, device="cuda")
    ws_bytes = tpk.hybrid_workspace_bytes(shape, B)
    ws = t.empty(ws_bytes, dtype=t.uint8, device="cuda")
    conv, dec = t.cuda.Stream(), t.cuda.Stream()
    n = [min(f, 700 + 300 * b) for b, f in enumerate(final)]   # starting lengths
    published_total = 0
    # the oracle's records of every page the loop can publish: the whole pages older
    # than the recent window at the final lengths
    rec_orc = oracle_records(split_view(w, final, [max(0, (f - recent) // 64) for f in final]))
    with tpk.Tiers(shape, B, max_pages, recent, k, v, rec, scratch, nbytes) as tiers:
        for step in range(16):
            for b in range(B):
                tiers.update(b, n[b], w.pages[b][: (n[b] + 63) // 64])
            plan = tiers.step(conv, dec)
            published_total += plan["published"]
            n8, n_ex = plan["n_int8_pages"], plan["n_exact_tokens"]
            for b in range(B):
                assert 64 * n8[b] + n_ex[b] == n[b]
                assert n_ex[b] >= min(n[b], recent)                # the recent tokens stay exact
                assert 64 * n8[b] <= max(0, n[b] - recent)          # only whole pages older than the window
            o = t.empty(B, H * G, 256, dtype=t.float32, device="cuda")
            lse = t.empty(B, H * G, dtype=t.float32, device="cuda")
            with t.cuda.stream(dec):
                tpk.decode_hybrid_batched(shape, B, q, k, v, rec, plan["page_table"], plan["req_page_off"], n_ex,
                                          plan["page_table8"], plan["req_page_off8"], n8, o, lse, ws, ws_bytes, dec)
            dec.synchronize()
            view = split_view(w, n, n8)
            # the same pages through the oracle's own records (the GPU converted them on
            # its side)
            oo, ol = oracle.hybrid_workload(view, rec_orc, n_threads=8)
            assert_close(o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), oo, ol,
                         f"step {step}")
            n = [min(f, x + 97 + 31 * b) for b, (f, x) in enumerate(zip(final, n))]
        tiers.sync()
        for b in range(B):
            tiers.update(b, n[b], w.pages[b][: (n[b] + 63) // 64])
        plan = tiers.step(conv, dec)
        published_total += plan["published"]
        tiers.sync()
        plan = tiers.step(conv, dec)      # conversions started by the previous step are published now
        published_total += plan["published"]
        eligible = [max(0, (x - recent) // 64) for x in n]
        assert list(plan["n_int8_pages"]) == eligible
        assert published_total == sum(eligible) and plan["converting"] == 0
    # the published records are the oracle's conversion of the same pages
    ref = np.zeros(w.n_slots * H * oracle.REC_BYTES, np.uint8)
    s8 = np.concatenate([np.asarray(w.pages[b][:eligible[b]]) for b in range(B)]).astype(np.int32)
    oracle.quantize_pages(H, w.k_pool, w.v_pool, s8, s8, ref)
    got = rec.cpu().numpy().reshape(w.n_slots, H, oracle.REC_BYTES)
    ref = ref.reshape(w.n_slots, H, oracle.REC_BYTES)
    for slot in s8:
        for h in range(H):
            _, _, s_g, _, _ = oracle.record_fields(got[slot, h])
            _, _, s_o, _, _ = oracle.record_fields(ref[slot, h])
            assert np.abs(s_g.view(np.int32).astype(np.int64) - s_o.view(np.int32).astype(np.int64)).max() <= 1


def test_moving_a_converted_page_is_refused():
    t = torch()
    w = synth.make_workload([64 * 10], None, H=1, seed=51)
    shape = tpk.Shape(1, kv_slots=w.n_slots, rec_slots=w.n_slots)
    k, v = dev_u16(w.k_pool), dev_u16(w.v_pool)
    rec = t.zeros(w.n_slots * tpk.RECORD_BYTES, dtype=t.uint8, device="cuda")
    nbytes = tpk.Tiers.device_bytes(1, 10)
    scratch = t.empty(nbytes, dtype=t.uint8, device="cuda")
    s = t.cuda.Stream()
    with tpk.Tiers(shape, 1, 10, 64, k, v, rec, scratch, nbytes) as tiers:
        slots = list(w.pages[0])
        tiers.update(0, 64 * 10, slots)
        plan = tiers.step(s, s)
        assert plan["started"] == 9
        moved = list(slots)
        moved[0] = slots[1]
        with pytest.raises(tpk.TpkError):
            tiers.update(0, 64 * 10, moved)
        with pytest.raises(tpk.TpkError):
            tiers.update(0, 64 * 9, slots[:9])              # histories do not shrink
        with pytest.raises(tpk.TpkError):
            tiers.update(0, 64 * 11, slots + [w.n_slots])   # outside the pool
