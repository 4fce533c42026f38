"""The C-ABI library loads, exports every entry point its header declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

import tiered_paged_kv_gb300 as tpk
from tiered_paged_kv_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tpk.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return tpk.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tpk_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tpk_kv_quantize_pages", "tpk_decode_attn_exact", "tpk_decode_attn_int8", "tpk_merge_lse",
              "tpk_decode_hybrid_batched"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_version(L):
    assert b"sm_103a" in L.tpk_version()


def err(L):
    return L.tpk_last_error_string().decode()


def test_unsupported_shapes_are_rejected(L):
    for kw, code in [({"group": 4}, 2), ({"head_dim": 128}, 2), ({"page_tokens": 32}, 2), ({"sm_scale": 0.1}, 2),
                     ({"impl": 7}, 1), ({"int_query": 2}, 1), ({"int_query": 1, "impl": tpk.IMPL_SIMT}, 2)]:
        s = tpk.Shape(4, **kw)
        st = L.tpk_decode_attn_exact(ctypes.byref(s), 16, 16, 16, 16, 0, 64, 1, 16, 16, None)
        assert st == code, (kw, st, err(L))
    s = tpk.Shape(0)
    assert L.tpk_decode_attn_int8(ctypes.byref(s), 16, 16, 16, 0, 1, 1, 16, 16, None) == 1
    s = tpk.Shape(1025)   # more KV heads than the library takes
    assert L.tpk_decode_attn_int8(ctypes.byref(s), 16, 16, 16, 0, 1, 1, 16, 16, None) == 1
    assert L.tpk_decode_attn_exact(None, 16, 16, 16, 16, 0, 64, 1, 16, 16, None) == 1


def test_bad_ranges_and_pointers_are_rejected(L):
    s = tpk.Shape(4)
    assert L.tpk_decode_attn_exact(ctypes.byref(s), 16, 16, 16, 16, 10, 5, 1, 16, 16, None) == 1
    assert "token range" in err(L)
    assert L.tpk_decode_attn_exact(ctypes.byref(s), 16, 16, 16, 16, 0, 64, 0, 16, 16, None) == 1
    assert L.tpk_decode_attn_exact(ctypes.byref(s), 16, 16, 16, 16, 0, 64, 5000, 16, 16, None) == 1
    assert L.tpk_decode_attn_exact(ctypes.byref(s), None, 16, 16, 16, 0, 64, 1, 16, 16, None) == 1
    assert L.tpk_decode_attn_exact(ctypes.byref(s), 24, 16, 16, 16, 0, 64, 1, 16, 16, None) == 1
    assert "aligned" in err(L)
    assert L.tpk_decode_attn_int8(ctypes.byref(s), 16, 16, 16, 3, 2, 1, 16, 16, None) == 1
    assert L.tpk_merge_lse(1, 8, 128, 16, 16, 16, 16, None) == 2
    assert L.tpk_merge_lse(-1, 8, 256, 16, 16, 16, 16, None) == 1
    assert L.tpk_kv_quantize_pages(ctypes.byref(s), 16, 16, 16, 16, -1, 16, None) == 1
    assert L.tpk_kv_quantize_pages_given_scales(ctypes.byref(s), 16, 16, 16, 16, 1, None, 16, 16, 16, None) == 1


def test_pack13_arguments_are_validated_before_any_device_call(L):
    s = tpk.Shape(4)
    assert L.tpk_kv_pack13_pages(ctypes.byref(s), 16, 16, 16, 16, -1, 16, 0, None) == 1
    assert L.tpk_kv_pack13_pages(ctypes.byref(s), 16, 16, 16, 16, 0, 16, 0, None) == 0   # nothing to do
    assert L.tpk_kv_pack13_pages(ctypes.byref(s), 16, 16, 16, 16, 1, 16, -2, None) == 1
    assert L.tpk_kv_pack13_pages(ctypes.byref(s), 16, None, 16, 16, 1, 16, 0, None) == 1
    assert L.tpk_kv_pack13_pages(ctypes.byref(s), 16, 16, 16, 16, 1, 24, 0, None) == 1
    assert "aligned" in err(L)
    assert L.tpk_kv_unpack13_pages(ctypes.byref(s), 16, -1, 16, 16, 1, 16, 16, None) == 1
    assert L.tpk_kv_unpack13_pages(ctypes.byref(s), 16, 0, None, 16, 1, 16, 16, None) == 1
    assert L.tpk_kv_unpack13_pages(ctypes.byref(s), 8, 0, 16, 16, 1, 16, 16, None) == 1
    assert L.tpk_kv_unpack13_pages(ctypes.byref(s), 16, 0, 16, 16, -3, 16, 16, None) == 1
    assert L.tpk_kv_unpack13_pages(ctypes.byref(tpk.Shape(4, group=4)), 16, 0, 16, 16, 1, 16, 16, None) == 2


def test_timing_events_come_in_pairs(L):
    assert L.tpk_set_decode_timing_events(ctypes.c_void_p(16), None) == 1
    assert L.tpk_set_decode_timing_events(None, None) == 0
    # the bounded-wait test hook: refusals, then back to the defaults
    assert L.tpk_set_test_wait(0, -2) == 1
    assert L.tpk_set_test_wait(61 * 10 ** 9, -1) == 1
    assert L.tpk_set_test_wait(10 ** 6, 3) == 0
    assert L.tpk_set_test_wait(0, -1) == 0


def test_hybrid_host_metadata_is_validated(L):
    s = tpk.Shape(2)
    need = L.tpk_hybrid_workspace_bytes(ctypes.byref(s), 2)
    assert need > 0
    import numpy as np
    off = np.array([0, 1, 2], np.int32)
    off8 = np.array([0, 0, 0], np.int32)
    nex = np.array([64, 100], np.int32)   # request 1 needs 2 pages, its table holds 1
    n8 = np.array([0, 0], np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = L.tpk_decode_hybrid_batched(ctypes.byref(s), 2, 16, 16, 16, 16, 16, p(off), p(nex), 16, p(off8), p(n8),
                                     16, 16, 16, need, None)
    assert st == 1 and "page table" in err(L)
    st = L.tpk_decode_hybrid_batched(ctypes.byref(s), 2, 16, 16, 16, 16, 16, p(off), p(nex), 16, p(off8), p(n8),
                                     16, 16, 16, need - 1, None)
    assert st == 5
    st = L.tpk_decode_hybrid_batched(ctypes.byref(s), 0, 16, 16, 16, 16, 16, p(off), p(nex), 16, p(off8), p(n8),
                                     16, 16, 16, need, None)
    assert st == 1
    nex[0] = -1
    st = L.tpk_decode_hybrid_batched(ctypes.byref(s), 2, 16, 16, 16, 16, 16, p(off), p(nex), 16, p(off8), p(n8),
                                     16, 16, 16, need, None)
    assert st == 1


def test_package_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(tpk, "_lib", None)
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        tpk.lib()


def test_stager_arguments_are_validated_before_any_device_call(L):
    out = ctypes.c_void_p(1)
    slots = (ctypes.c_void_p * 2)(16, 32)
    assert L.tpk_stager_create(0, slots, 1024, ctypes.byref(out)) == 1 and out.value is None
    assert L.tpk_stager_create(2, None, 1024, ctypes.byref(out)) == 1
    assert L.tpk_stager_create(2, slots, 0, ctypes.byref(out)) == 1
    assert L.tpk_stager_create(2, slots, 1024, None) == 1
    assert L.tpk_stager_stage(None, 0, None, None, None, None, None) == 1
    assert L.tpk_stager_acquire(None, 0, None) == 1
    assert L.tpk_stager_release(None, 0, None) == 1
    assert L.tpk_stager_sync(None) == 1
    assert L.tpk_stager_destroy(None) == 0


def test_tier_manager_arguments_are_validated_before_any_device_call(L):
    out = ctypes.c_void_p(1)
    s = tpk.Shape(2)
    assert L.tpk_tiers_device_bytes(0, 4) == 0 and L.tpk_tiers_device_bytes(2, 0) == 0
    need = L.tpk_tiers_device_bytes(2, 4)
    assert need > 0
    assert L.tpk_tiers_create(ctypes.byref(s), 2, 4, 0, 16, 16, 16, 256, need, None) == 1
    assert L.tpk_tiers_create(None, 2, 4, 0, 16, 16, 16, 256, need, ctypes.byref(out)) == 1 and out.value is None
    assert L.tpk_tiers_create(ctypes.byref(s), 0, 4, 0, 16, 16, 16, 256, need, ctypes.byref(out)) == 1
    assert L.tpk_tiers_create(ctypes.byref(s), 2, 4, -1, 16, 16, 16, 256, need, ctypes.byref(out)) == 1
    assert L.tpk_tiers_create(ctypes.byref(s), 2, 4, 0, None, 16, 16, 256, need, ctypes.byref(out)) == 1
    assert L.tpk_tiers_create(ctypes.byref(s), 2, 4, 0, 16, 16, 16, 256, need - 1, ctypes.byref(out)) == 5
    assert L.tpk_tiers_create(ctypes.byref(s), 2, 4, 0, 16, 16, 16, 260, need, ctypes.byref(out)) == 1
    assert L.tpk_tiers_update(None, 0, 10, None) == 1
    assert L.tpk_tiers_step(None, None, None, None) == 1
    assert L.tpk_tiers_sync(None) == 1
    assert L.tpk_tiers_destroy(None) == 0
