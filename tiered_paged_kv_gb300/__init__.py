"""tiered_paged_kv_gb300 -- split-tier paged decode attention on GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/tpk.h`` (``libtpk.so``).  Every
function here only marshals arguments: device buffers are passed as raw
pointers (torch tensors are accepted and their ``data_ptr()`` is used), streams
as ``torch.cuda.Stream`` or raw handles.  All computation runs in the library's
CUDA kernels; there is no CPU fallback, and loading fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build_mod

__all__ = [
    "Shape", "TpkError", "lib", "RECORD_BYTES", "IMPL_DEFAULT", "IMPL_SIMT", "IMPL_TENSOR",
    "kv_quantize_pages", "kv_quantize_pages_given_scales", "decode_attn_exact", "decode_attn_int8",
    "merge_lse", "hybrid_workspace_bytes", "workspace_init", "decode_hybrid_batched", "hybrid_plan",
    "set_decode_timing_events",
    "get_device_status",
    "static_scratch_bytes", "decode_hybrid_batched_static", "Stager", "Tiers", "TiersPlan",
    "PACK13_RECORD_BYTES", "PACK13_PLANE_ENC", "PACK13_PLANE_RAW", "kv_pack13_pages", "kv_unpack13_pages",
]

RECORD_BYTES = 35072
PACK13_RECORD_BYTES, PACK13_PLANE_ENC, PACK13_PLANE_RAW = 65552, 26656, 32768
IMPL_DEFAULT, IMPL_SIMT, IMPL_TENSOR = 0, 1, 2
STATUS_NAMES = {0: "TPK_OK", 1: "TPK_ERR_INVALID", 2: "TPK_ERR_UNSUPPORTED", 3: "TPK_ERR_CUDA",
                4: "TPK_ERR_BOUNDS", 5: "TPK_ERR_NOMEM", 6: "TPK_ERR_TIMEOUT", 7: "TPK_ERR_FORMAT"}


class Shape(ctypes.Structure):
    _fields_ = [("kv_heads", ctypes.c_int), ("group", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("page_tokens", ctypes.c_int), ("sm_scale", ctypes.c_float), ("impl", ctypes.c_int),
                ("kv_slots", ctypes.c_int64), ("rec_slots", ctypes.c_int64), ("int_query", ctypes.c_int)]

    def __init__(self, kv_heads, group=8, head_dim=256, page_tokens=64, sm_scale=0.0, impl=IMPL_DEFAULT,
                 kv_slots=0, rec_slots=0, int_query=0):
        super().__init__(kv_heads, group, head_dim, page_tokens, sm_scale, impl, kv_slots, rec_slots,
                         int(int_query))


class TiersPlan(ctypes.Structure):
    _fields_ = [("page_table", ctypes.c_void_p), ("req_page_off", ctypes.POINTER(ctypes.c_int32)),
                ("n_exact_tokens", ctypes.POINTER(ctypes.c_int32)), ("page_table8", ctypes.c_void_p),
                ("req_page_off8", ctypes.POINTER(ctypes.c_int32)), ("n_int8_pages", ctypes.POINTER(ctypes.c_int32)),
                ("pages_published", ctypes.c_int), ("pages_started", ctypes.c_int),
                ("pages_converting", ctypes.c_int)]


class TpkError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def lib():
    """Load libtpk.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build_mod.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libtpk.so not built ({path}); run tiered_paged_kv_gb300.build.build()")
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sp = ctypes.POINTER(Shape)
        L.tpk_version.restype = ctypes.c_char_p
        L.tpk_last_error_string.restype = ctypes.c_char_p
        L.tpk_kv_quantize_pages.argtypes = [sp, vp, vp, vp, vp, i32, vp, vp]
        L.tpk_kv_quantize_pages_given_scales.argtypes = [sp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp]
        i64 = ctypes.c_int64
        L.tpk_kv_pack13_pages.argtypes = [sp, vp, vp, vp, vp, i32, vp, i64, vp]
        L.tpk_kv_unpack13_pages.argtypes = [sp, vp, i64, vp, vp, i32, vp, vp, vp]
        L.tpk_decode_attn_exact.argtypes = [sp, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.tpk_decode_attn_int8.argtypes = [sp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.tpk_merge_lse.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp]
        L.tpk_hybrid_workspace_bytes.argtypes = [sp, i32]
        L.tpk_hybrid_workspace_bytes.restype = sz
        L.tpk_workspace_init.argtypes = [vp, sz, vp]
        L.tpk_decode_hybrid_batched.argtypes = [sp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.tpk_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), i32, vp]
        L.tpk_set_decode_timing_events.argtypes = [vp, vp]
        L.tpk_set_decode_timing_events.restype = i32
        L.tpk_set_test_wait.argtypes = [ctypes.c_uint64, i32]
        L.tpk_set_test_wait.restype = i32
        ip = ctypes.POINTER(ctypes.c_int32)
        L.tpk_hybrid_plan.argtypes = [sp, i32, ip, ip, i32, ip, ip, ip]
        L.tpk_hybrid_plan.restype = i32
        L.tpk_static_scratch_bytes.argtypes = []
        L.tpk_static_scratch_bytes.restype = sz
        L.tpk_decode_hybrid_batched_static.argtypes = [sp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        pp = ctypes.POINTER(ctypes.c_void_p)
        L.tpk_stager_create.argtypes = [i32, pp, sz, pp]
        L.tpk_stager_destroy.argtypes = [vp]
        L.tpk_stager_stage.argtypes = [vp, i32, pp, ctypes.POINTER(sz), ctypes.POINTER(sz),
                                       ctypes.POINTER(i32), pp]
        L.tpk_stager_acquire.argtypes = [vp, i32, vp]
        L.tpk_stager_release.argtypes = [vp, i32, vp]
        L.tpk_stager_sync.argtypes = [vp]
        L.tpk_stager_copy_ms.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_float)]
        for name in ("tpk_stager_create", "tpk_stager_destroy", "tpk_stager_stage", "tpk_stager_acquire",
                     "tpk_stager_release", "tpk_stager_sync", "tpk_stager_copy_ms"):
            getattr(L, name).restype = i32
        L.tpk_tiers_device_bytes.argtypes = [i32, i32]
        L.tpk_tiers_device_bytes.restype = sz
        L.tpk_tiers_create.argtypes = [sp, i32, i32, i32, vp, vp, vp, vp, sz, pp]
        L.tpk_tiers_update.argtypes = [vp, i32, i32, vp]
        L.tpk_tiers_create_layers.argtypes = [sp, i32, i32, i32, i32, pp, pp, pp, pp, vp, sz, pp]
        L.tpk_tiers_update_layers.argtypes = [vp, i32, i32, vp, vp]
        L.tpk_tiers_step.argtypes = [vp, vp, vp, ctypes.POINTER(TiersPlan)]
        L.tpk_tiers_sync.argtypes = [vp]
        L.tpk_tiers_destroy.argtypes = [vp]
        for name in ("tpk_tiers_create", "tpk_tiers_update", "tpk_tiers_step", "tpk_tiers_sync",
                     "tpk_tiers_destroy", "tpk_tiers_create_layers", "tpk_tiers_update_layers"):
            getattr(L, name).restype = i32
        for name in ("tpk_kv_quantize_pages", "tpk_kv_quantize_pages_given_scales", "tpk_kv_pack13_pages",
                     "tpk_kv_unpack13_pages", "tpk_decode_attn_exact",
                     "tpk_decode_attn_int8", "tpk_merge_lse", "tpk_workspace_init", "tpk_decode_hybrid_batched",
                     "tpk_get_device_status", "tpk_decode_hybrid_batched_static"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot take a device pointer from {type(x)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _host_i32(a):
    """(array kept alive by the caller, its address) of a host int32 array; an
    int32 C-contiguous ndarray is passed as it is, anything else is copied."""
    if isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous:
        return a, a.ctypes.data
    arr = np.ascontiguousarray(np.asarray(a), dtype=np.int32)
    return arr, arr.ctypes.data


def _check(status):
    if status != 0:
        raise TpkError(status, lib().tpk_last_error_string().decode())


def kv_quantize_pages(shape, k_pool, v_pool, src_slots, dst_slots, n_pages, rec_pool, stream=None):
    _check(lib().tpk_kv_quantize_pages(ctypes.byref(shape), _ptr(k_pool), _ptr(v_pool), _ptr(src_slots),
                                       _ptr(dst_slots), int(n_pages), _ptr(rec_pool), _stream(stream)))


def kv_quantize_pages_given_scales(shape, k_pool, v_pool, src_slots, dst_slots, n_pages, ks_chan, ks_tok,
                                   vs_chan, rec_pool, stream=None):
    _check(lib().tpk_kv_quantize_pages_given_scales(ctypes.byref(shape), _ptr(k_pool), _ptr(v_pool),
                                                    _ptr(src_slots), _ptr(dst_slots), int(n_pages), _ptr(ks_chan),
                                                    _ptr(ks_tok), _ptr(vs_chan), _ptr(rec_pool), _stream(stream)))


def kv_pack13_pages(shape, k_pool, v_pool, src_slots, dst_slots, n_pages, pack_pool, pack_slots=0, stream=None):
    _check(lib().tpk_kv_pack13_pages(ctypes.byref(shape), _ptr(k_pool), _ptr(v_pool), _ptr(src_slots),
                                     _ptr(dst_slots), int(n_pages), _ptr(pack_pool), int(pack_slots),
                                     _stream(stream)))


def kv_unpack13_pages(shape, src, src_bytes, rec_offsets, dst_slots, n_pages, k_pool, v_pool, stream=None):
    _check(lib().tpk_kv_unpack13_pages(ctypes.byref(shape), _ptr(src), int(src_bytes), _ptr(rec_offsets),
                                       _ptr(dst_slots), int(n_pages), _ptr(k_pool), _ptr(v_pool), _stream(stream)))


def decode_attn_exact(shape, q, k_pool, v_pool, page_table, tok_begin, tok_end, num_splits, o_part, lse_part,
                      stream=None):
    _check(lib().tpk_decode_attn_exact(ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                       int(tok_begin), int(tok_end), int(num_splits), _ptr(o_part), _ptr(lse_part),
                                       _stream(stream)))


def decode_attn_int8(shape, q, rec_pool, page_table8, page_begin, page_end, num_splits, o_part, lse_part,
                     stream=None):
    _check(lib().tpk_decode_attn_int8(ctypes.byref(shape), _ptr(q), _ptr(rec_pool), _ptr(page_table8),
                                      int(page_begin), int(page_end), int(num_splits), _ptr(o_part), _ptr(lse_part),
                                      _stream(stream)))


def merge_lse(n_parts, rows, head_dim, o_parts, lse_parts, o_acc, lse_acc, stream=None):
    _check(lib().tpk_merge_lse(int(n_parts), int(rows), int(head_dim), _ptr(o_parts), _ptr(lse_parts), _ptr(o_acc),
                               _ptr(lse_acc), _stream(stream)))


def hybrid_workspace_bytes(shape, n_req):
    return int(lib().tpk_hybrid_workspace_bytes(ctypes.byref(shape), int(n_req)))


def workspace_init(ws, ws_bytes, stream=None):
    _check(lib().tpk_workspace_init(_ptr(ws), int(ws_bytes), _stream(stream)))


def decode_hybrid_batched(shape, n_req, q, k_pool, v_pool, rec_pool, page_table, req_page_off, n_exact_tokens,
                          page_table8, req_page_off8, n_int8_pages, o, lse, ws, ws_bytes, stream=None):
    """req_page_off, n_exact_tokens, req_page_off8, n_int8_pages are host arrays."""
    a, pa = _host_i32(req_page_off)
    b, pb = _host_i32(n_exact_tokens)
    c, pc = _host_i32(req_page_off8)
    d, pd = _host_i32(n_int8_pages)
    _check(lib().tpk_decode_hybrid_batched(ctypes.byref(shape), int(n_req), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                           _ptr(rec_pool), _ptr(page_table), pa, pb, _ptr(page_table8), pc, pd,
                                           _ptr(o), _ptr(lse), _ptr(ws), int(ws_bytes), _stream(stream)))


def static_scratch_bytes():
    return int(lib().tpk_static_scratch_bytes())


def decode_hybrid_batched_static(shape, n_req, q, k_pool, v_pool, rec_pool, page_table, req_page_off,
                                 n_exact_tokens, page_table8, req_page_off8, n_int8_pages, o, lse, stream=None):
    """As decode_hybrid_batched, with the library's fixed device scratch instead of
    a caller workspace (for callers that cannot allocate device memory)."""
    a, pa = _host_i32(req_page_off)
    b, pb = _host_i32(n_exact_tokens)
    c, pc = _host_i32(req_page_off8)
    d, pd = _host_i32(n_int8_pages)
    _check(lib().tpk_decode_hybrid_batched_static(ctypes.byref(shape), int(n_req), _ptr(q), _ptr(k_pool),
                                                  _ptr(v_pool), _ptr(rec_pool), _ptr(page_table), pa, pb,
                                                  _ptr(page_table8), pc, pd, _ptr(o), _ptr(lse), _stream(stream)))


def hybrid_plan(shape, n_exact_tokens, n_int8_pages, resident_blocks=0):
    """The split plan of decode_hybrid_batched: (splits_exact, splits_int8, n_units)."""
    ne = np.ascontiguousarray(n_exact_tokens, np.int32)
    n8 = np.ascontiguousarray(n_int8_pages, np.int32)
    se = np.zeros(len(ne), np.int32)
    s8 = np.zeros(len(ne), np.int32)
    units = ctypes.c_int32(0)
    ip = ctypes.POINTER(ctypes.c_int32)
    _check(lib().tpk_hybrid_plan(ctypes.byref(shape), len(ne), ne.ctypes.data_as(ip), n8.ctypes.data_as(ip),
                                 int(resident_blocks), se.ctypes.data_as(ip), s8.ctypes.data_as(ip),
                                 ctypes.byref(units)))
    return se, s8, units.value


def set_decode_timing_events(before=None, after=None):
    """Record two torch.cuda.Event (timing enabled) around every decode-kernel
    launch until called with no events (see tpk_set_decode_timing_events)."""
    _check(lib().tpk_set_decode_timing_events(before.cuda_event if before is not None else None,
                                              after.cuda_event if after is not None else None))


def set_test_wait(wait_limit_ns=0, stall_unit=-1):
    """Test hook of the bounded device waits (see tpk_set_test_wait): every decode
    wait gives up after wait_limit_ns (0: the default two seconds); stall_unit >= 0
    leaves that decode block's first item unissued so its waits run out."""
    _check(lib().tpk_set_test_wait(int(wait_limit_ns), int(stall_unit)))


def get_device_status(reset=True, stream=None):
    """Returns (status, flags); status is a tpk_status, not raised."""
    flags = ctypes.c_int(0)
    st = lib().tpk_get_device_status(ctypes.byref(flags), 1 if reset else 0, _stream(stream))
    return st, flags.value


class Stager:
    """Host-resident history staging through n caller-owned device slots (see
    tpk_stager_* in include/tpk.h).  `slots` are device buffers (tensors or raw
    pointers) of `slot_bytes` each; the stager keeps references to them."""

    def __init__(self, slots, slot_bytes):
        self._keep = list(slots)
        arr = (ctypes.c_void_p * len(slots))(*[_ptr(x) for x in slots])
        h = ctypes.c_void_p()
        _check(lib().tpk_stager_create(len(slots), arr, int(slot_bytes), ctypes.byref(h)))
        self._h = h

    def stage(self, regions):
        """regions: [(host_src, slot_offset, nbytes)], host_src a pinned tensor or a
        raw pointer.  Returns (slot index, slot device address)."""
        n = len(regions)
        src = (ctypes.c_void_p * max(n, 1))(*[_ptr(r[0]) for r in regions])
        off = (ctypes.c_size_t * max(n, 1))(*[int(r[1]) for r in regions])
        nb = (ctypes.c_size_t * max(n, 1))(*[int(r[2]) for r in regions])
        slot = ctypes.c_int(-1)
        dev = ctypes.c_void_p()
        _check(lib().tpk_stager_stage(self._h, n, src, off, nb, ctypes.byref(slot), ctypes.byref(dev)))
        return slot.value, dev.value

    def acquire(self, slot, stream=None):
        _check(lib().tpk_stager_acquire(self._h, int(slot), _stream(stream)))

    def release(self, slot, stream=None):
        _check(lib().tpk_stager_release(self._h, int(slot), _stream(stream)))

    def sync(self):
        _check(lib().tpk_stager_sync(self._h))

    def copy_ms(self, slot):
        """Device time (ms) of the copies of the slot's latest staging (waits for them)."""
        ms = ctypes.c_float(0.0)
        _check(lib().tpk_stager_copy_ms(self._h, int(slot), ctypes.byref(ms)))
        return ms.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            h, self._h = self._h, None
            _check(lib().tpk_stager_destroy(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class Tiers:
    """Incremental conversion and publication during decode (see tpk_tiers_* in
    include/tpk.h).  `scratch` is a device buffer of at least
    Tiers.device_bytes(n_req, max_pages) bytes; the pools must outlive the object."""

    @staticmethod
    def device_bytes(n_req, max_pages):
        return int(lib().tpk_tiers_device_bytes(int(n_req), int(max_pages)))

    def __init__(self, shape, n_req, max_pages, recent_tokens, k_pool, v_pool, rec_pool, scratch, scratch_bytes,
                 host_rec_pools=None):
        """One layer: k_pool, v_pool, rec_pool are device buffers.  Several layers
        (tpk_tiers_create_layers): lists of one buffer per layer, and optionally
        host_rec_pools, pinned host record pools that receive every converted record."""
        self._keep = (shape, k_pool, v_pool, rec_pool, scratch, host_rec_pools)
        self.n_req = int(n_req)
        h = ctypes.c_void_p()
        if isinstance(k_pool, (list, tuple)):
            n = len(k_pool)
            self.n_layers = n
            arr = lambda xs: (ctypes.c_void_p * n)(*[_ptr(x) for x in xs])
            host = arr(host_rec_pools) if host_rec_pools is not None else None
            _check(lib().tpk_tiers_create_layers(ctypes.byref(shape), n, self.n_req, int(max_pages),
                                                 int(recent_tokens), arr(k_pool), arr(v_pool), arr(rec_pool), host,
                                                 _ptr(scratch), int(scratch_bytes), ctypes.byref(h)))
        else:
            self.n_layers = 1
            _check(lib().tpk_tiers_create(ctypes.byref(shape), self.n_req, int(max_pages), int(recent_tokens),
                                          _ptr(k_pool), _ptr(v_pool), _ptr(rec_pool), _ptr(scratch),
                                          int(scratch_bytes), ctypes.byref(h)))
        self._h = h

    def update(self, b, n_tokens, page_slots, layer_written=None):
        """layer_written: tokens each layer has written (None: all n_tokens)."""
        arr, p = _host_i32(page_slots)
        if layer_written is None:
            _check(lib().tpk_tiers_update(self._h, int(b), int(n_tokens), p))
        else:
            lw, plw = _host_i32(layer_written)
            _check(lib().tpk_tiers_update_layers(self._h, int(b), int(n_tokens), p, plw))

    def step(self, conv_stream=None, decode_stream=None):
        """Returns a dict: device page tables (raw pointers) and host numpy copies of
        the CSR offsets and counts, plus the publication counters."""
        plan = TiersPlan()
        _check(lib().tpk_tiers_step(self._h, _stream(conv_stream), _stream(decode_stream), ctypes.byref(plan)))
        n = self.n_req
        return {"page_table": plan.page_table, "page_table8": plan.page_table8,
                "req_page_off": np.ctypeslib.as_array(plan.req_page_off, (n + 1,)).copy(),
                "n_exact_tokens": np.ctypeslib.as_array(plan.n_exact_tokens, (n,)).copy(),
                "req_page_off8": np.ctypeslib.as_array(plan.req_page_off8, (n + 1,)).copy(),
                "n_int8_pages": np.ctypeslib.as_array(plan.n_int8_pages, (n,)).copy(),
                "published": plan.pages_published, "started": plan.pages_started,
                "converting": plan.pages_converting}

    def sync(self):
        _check(lib().tpk_tiers_sync(self._h))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            h, self._h = self._h, None
            _check(lib().tpk_tiers_destroy(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
