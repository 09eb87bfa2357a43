"""Thin Python binding of the C ABI in ``include/hs.h``.

Functions carry the C names and only marshal arguments: every step of the
resolve path runs in the CUDA kernels of ``libhs.so``.  Device buffers may be
passed as torch tensors (their ``data_ptr()`` is used) or as raw integer
addresses; streams as ``torch.cuda.Stream`` objects, raw handles, or ``None``
for torch's current stream.  A failing call raises :class:`HsError`.

:class:`Pool` wraps a pool handle with numpy views of the host records and
zero-copy torch views of the device metadata.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _native

HS_OK = 0
HS_ERR_INVALID_ARG = -1
HS_ERR_CUDA = -2
HS_ERR_NOMEM = -3
HS_ERR_DEVICE_INPUT = -4
HS_ERR_TIMEOUT = -5
HS_ERR_UNSUPPORTED = -6

HS_HOST_ALLOC_AUTO = 0
HS_HOST_ALLOC_PINNED = 1
HS_HOST_ALLOC_VMM_NUMA = 2
HS_HOST_ALLOC_THP_REGISTERED = 3

HS_OVERLAP_AUTO = 0
HS_OVERLAP_ON = 1
HS_OVERLAP_OFF = 2

HS_STATUS_POS_RANGE = 0x1
HS_STATUS_POS_DUP = 0x2
HS_STATUS_REQ_RANGE = 0x4
HS_STATUS_REQ_BUSY = 0x8
HS_STATUS_PLAN = 0x10
HS_STATUS_META = 0x20


class HsError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {hs_strerror(code)} ({code})")


def _lib():
    return _native.load()


def _check(rc: int, what: str) -> None:
    if rc != HS_OK:
        raise HsError(rc, what)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def hs_strerror(code: int) -> str:
    return _lib().hs_strerror(code).decode()


def hs_kernels_per_call() -> int:
    return int(_lib().hs_kernels_per_call())


def hs_plan_bytes(n_req: int, k: int) -> int:
    return int(_lib().hs_plan_bytes(n_req, k))


def hs_create_pool(n_requests, n_layers, n_positions, record_bytes, slots, max_k,
                   layer_anchor=None, host_limit_bytes=0, host_alloc=HS_HOST_ALLOC_AUTO,
                   launch_overlap=HS_OVERLAP_AUTO) -> int:
    anchors = None
    if layer_anchor is not None:
        anchors = (ctypes.c_int32 * len(layer_anchor))(*layer_anchor)
    d = _native.PoolDesc(n_requests, n_layers, n_positions, record_bytes, slots, max_k,
                         ctypes.cast(anchors, ctypes.c_void_p) if anchors is not None else None,
                         host_limit_bytes, host_alloc, launch_overlap)
    h = ctypes.c_void_p()
    _check(_lib().hs_create_pool(ctypes.byref(d), ctypes.byref(h)), "hs_create_pool")
    return h.value


def hs_destroy_pool(pool: int) -> None:
    _check(_lib().hs_destroy_pool(pool), "hs_destroy_pool")


def hs_host_records(pool: int, req: int, layer: int) -> int:
    p = ctypes.c_void_p()
    _check(_lib().hs_host_records(pool, req, layer, ctypes.byref(p)), "hs_host_records")
    return p.value


def hs_device_views(pool: int, layer: int) -> _native.Views:
    v = _native.Views()
    _check(_lib().hs_device_views(pool, layer, ctypes.byref(v)), "hs_device_views")
    return v


def hs_device_host_numa(device: int) -> int:
    """Host NUMA node closest to `device`, -1 when none is reported."""
    return int(_lib().hs_device_host_numa(device))


def hs_touch_records(pool: int, req: int = -1, layer: int = -1, stream=None) -> None:
    _check(_lib().hs_touch_records(pool, req, layer, _stream(stream)), "hs_touch_records")


def hs_warm_pool(pool: int) -> None:
    _check(_lib().hs_warm_pool(pool), "hs_warm_pool")


def hs_pool_info(pool: int) -> dict:
    i = _native.PoolInfo()
    _check(_lib().hs_pool_info(pool, ctypes.byref(i)), "hs_pool_info")
    return {f: int(getattr(i, f)) for f, _ in _native.PoolInfo._fields_}


def hs_resolve(pool, layer, n_req, req_ids, sel, k, out, plan=None, stream=None) -> None:
    _check(_lib().hs_resolve(pool, layer, n_req, _ptr(req_ids), _ptr(sel), k, _ptr(out),
                             _ptr(plan), _stream(stream)), "hs_resolve")


def hs_resolve_anchor(pool, layer, n_req, req_ids, sel, k, out, plan_out, stream=None) -> None:
    _check(_lib().hs_resolve_anchor(pool, layer, n_req, _ptr(req_ids), _ptr(sel), k, _ptr(out),
                                    _ptr(plan_out), _stream(stream)), "hs_resolve_anchor")


HS_MEASURE_NO_FETCH = 0x1
HS_STAMPS = ("ENTRY", "LOADED", "HASHED", "PROBED", "DECIDED", "CHECKED", "VERDICT", "COMMITTED",
             "F_ISSUE", "F_ISSUED", "F_WAITED", "F_LANDED", "F_STORED", "ATTEMPTS", "EXIT",
             "LEAD_FETCHED")
HS_STAMP = {name: i for i, name in enumerate(HS_STAMPS)}


def hs_measure_stamp_slots() -> int:
    return int(_lib().hs_measure_stamp_slots())


def hs_resolve_measure(pool, layer, n_req, req_ids, sel, k, out, flags=0, times=None,
                       stream=None) -> None:
    """Measurement variant of hs_resolve: HS_MEASURE_NO_FETCH skips the miss
    fetch; `times` (device u64 [n_req][hs_measure_stamp_slots()]) receives
    stage timestamps."""
    _check(_lib().hs_resolve_measure(pool, layer, n_req, _ptr(req_ids), _ptr(sel), k, _ptr(out),
                                     flags, _ptr(times), _stream(stream)), "hs_resolve_measure")


def hs_prefetch_plan(pool, anchor_layer, target_layer, n_req, req_ids, sel, k, plan,
                     stream=None) -> None:
    _check(_lib().hs_prefetch_plan(pool, anchor_layer, target_layer, n_req, _ptr(req_ids),
                                   _ptr(sel), k, _ptr(plan), _stream(stream)), "hs_prefetch_plan")


def hs_prefetch_copy(pool, target_layer, n_req, k, plan, stream=None) -> None:
    _check(_lib().hs_prefetch_copy(pool, target_layer, n_req, k, _ptr(plan), _stream(stream)),
           "hs_prefetch_copy")


def hs_stats(pool, layer: int = -1, check: bool = True) -> dict:
    """Counters of `layer` (-1: all).  With check=False a status error is
    returned in the dict instead of raised."""
    s = _native.Stats()
    rc = _lib().hs_stats(pool, layer, ctypes.byref(s))
    if rc not in (HS_OK, HS_ERR_DEVICE_INPUT) or (check and rc != HS_OK):
        raise HsError(rc, f"hs_stats (status 0x{s.status:x})")
    d = {f: int(getattr(s, f)) for f, _ in _native.Stats._fields_}
    d["rc"] = rc
    return d


def hs_reset(pool) -> None:
    _check(_lib().hs_reset(pool), "hs_reset")


def hs_link_probe(nbytes: int, reps: int = 10, record_bytes: int = 1152,
                  host_alloc: int = HS_HOST_ALLOC_AUTO):
    """(H2D memcpy GB/s, scattered-record GPU-load GB/s), best of `reps`,
    over a host buffer of `nbytes` allocated the `host_alloc` way."""
    a, b = ctypes.c_double(), ctypes.c_double()
    _check(_lib().hs_link_probe(nbytes, reps, record_bytes, host_alloc, ctypes.byref(a),
                                ctypes.byref(b)), "hs_link_probe")
    return a.value, b.value


def hs_sparse_attention(q, cache, cache_rows, idx, n_req, k, heads, scale, out,
                        stream=None) -> None:
    """Attention of q [n_req][heads][576] bf16 over the published rows idx
    [n_req][k] of a layer's cache; fp32 out [n_req][heads][512]."""
    _check(_lib().hs_sparse_attention(_ptr(q), _ptr(cache), cache_rows, _ptr(idx), n_req, k,
                                      heads, scale, _ptr(out), _stream(stream)),
           "hs_sparse_attention")


def hs_sparse_attention_heads(q, cache, cache_rows, idx, n_req, k, heads, scale, out,
                              stream=None) -> None:
    """Attention of q [n_req][heads][128] bf16 over the published rows idx
    [n_req][k] of a layer's cache of per-head token records (keys of every
    head, then values; heads * 512 bytes); fp32 out [n_req][heads][128]."""
    _check(_lib().hs_sparse_attention_heads(_ptr(q), _ptr(cache), cache_rows, _ptr(idx), n_req,
                                            k, heads, scale, _ptr(out), _stream(stream)),
           "hs_sparse_attention_heads")


HS_ATTN_STATUS_TIMEOUT = 0x1


def hs_attention_status() -> int:
    """HS_ATTN_STATUS_* bits set by attention calls since the last query
    (synchronises the device, clears the bits)."""
    v = ctypes.c_uint32()
    _check(_lib().hs_attention_status(ctypes.byref(v)), "hs_attention_status")
    return int(v.value)


HS_NOALLOC_MAX_REQUESTS = 4096


def hs_resolve_noalloc(state: dict, n_req, req_ids, sel, k, out, status=None, stream=None) -> None:
    """Resolve one layer whose state the caller owns, allocating nothing.

    ``state`` maps the hs_layer_state fields to values: sizes as ints,
    arrays as torch tensors or device addresses.  See include/hs.h for the
    scratch array it shares between calls."""
    st = _native.LayerState(
        state["n_requests"], state["n_positions"], state["record_bytes"], state["slots"],
        _ptr(state["host_records"]), _ptr(state["cache"]), _ptr(state["page_table"]),
        _ptr(state["slot_pos"]), _ptr(state["stamps"]), _ptr(state["lru"]),
        _ptr(state["resolves"]))
    _check(_lib().hs_resolve_noalloc(ctypes.byref(st), n_req, _ptr(req_ids), _ptr(sel), k,
                                     _ptr(out), _ptr(status), _stream(stream)),
           "hs_resolve_noalloc")


class _CudaArray:
    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


class Pool:
    """A pool handle plus host and device views."""

    def __init__(self, n_requests, n_layers, n_positions, record_bytes, slots, max_k,
                 layer_anchor=None, host_limit_bytes=0, host_alloc=HS_HOST_ALLOC_AUTO,
                 launch_overlap=HS_OVERLAP_AUTO):
        self.R, self.NL, self.L = n_requests, n_layers, n_positions
        self.W, self.B, self.max_k = record_bytes, slots, max_k
        self.handle = hs_create_pool(n_requests, n_layers, n_positions, record_bytes, slots,
                                     max_k, layer_anchor, host_limit_bytes, host_alloc,
                                     launch_overlap)

    @classmethod
    def for_workload(cls, w, host_limit_bytes=0, host_alloc=HS_HOST_ALLOC_AUTO,
                     launch_overlap=HS_OVERLAP_AUTO):
        return cls(w.n_requests, w.n_layers, w.n_positions, w.record_bytes, w.slots, w.k,
                   list(w.anchors), host_limit_bytes, host_alloc, launch_overlap)

    def info(self) -> dict:
        return hs_pool_info(self.handle)

    def touch(self, req=-1, layer=-1, stream=None):
        hs_touch_records(self.handle, req, layer, stream)

    def warm(self):
        """Touch every record, resolve synthetic steps, reset (before first use)."""
        hs_warm_pool(self.handle)

    def close(self):
        if self.handle:
            hs_destroy_pool(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def host_records(self, req, layer) -> np.ndarray:
        """numpy uint8 view [L][W] of the pinned host records of (req, layer)."""
        addr = hs_host_records(self.handle, req, layer)
        buf = (ctypes.c_uint8 * (self.L * self.W)).from_address(addr)
        return np.frombuffer(buf, np.uint8).reshape(self.L, self.W)

    def views(self, layer):
        """torch tensors (zero-copy) over the device arrays of `layer`."""
        import torch
        v = hs_device_views(self.handle, layer)
        R, B, L, W = self.R, self.B, self.L, self.W

        def t(ptr, shape, ts):
            return torch.as_tensor(_CudaArray(ptr, shape, ts), device="cuda")
        return {"cache": t(v.cache, (R * B, W), "|u1"),
                "page_table": t(v.page_table, (R, L), "<i4"),
                "slot_pos": t(v.slot_pos, (R, B), "<i4"),
                "stamps": t(v.stamps, (R, B), "<u4"),
                "lru": t(v.lru, (R, B), "<u2"),
                "resolves": t(v.resolves, (R,), "<u4")}

    def resolve(self, layer, sel, out, req_ids=None, plan=None, stream=None, n_req=None):
        n = sel.shape[0] if n_req is None else n_req
        hs_resolve(self.handle, layer, n, req_ids, sel, sel.shape[-1], out, plan, stream)

    def resolve_anchor(self, layer, sel, out, plan_out, req_ids=None, stream=None):
        hs_resolve_anchor(self.handle, layer, sel.shape[0], req_ids, sel, sel.shape[-1], out,
                          plan_out, stream)

    def resolve_measure(self, layer, sel, out, flags=0, times=None, req_ids=None, stream=None):
        hs_resolve_measure(self.handle, layer, sel.shape[0], req_ids, sel, sel.shape[-1], out,
                           flags, times, stream)

    def prefetch_plan(self, anchor_layer, target_layer, sel, plan, req_ids=None, stream=None):
        hs_prefetch_plan(self.handle, anchor_layer, target_layer, sel.shape[0], req_ids, sel,
                         sel.shape[-1], plan, stream)

    def prefetch_copy(self, target_layer, n_req, k, plan, stream=None):
        hs_prefetch_copy(self.handle, target_layer, n_req, k, plan, stream)

    def stats(self, layer=-1, check=True):
        return hs_stats(self.handle, layer, check)

    def reset(self):
        hs_reset(self.handle)
