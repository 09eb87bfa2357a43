"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/hs.h declares, and its host-side argument checks
reject bad input before touching CUDA."""
import ctypes
import os
import re

import pytest

from hierarchical_kv_cache_resolve_gb300 import _native, hs

HEADER = os.path.join(_native.INCLUDE, "hs.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hs_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _native.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_native.EXPORTS)


def test_library_is_built_for_sm_103a_only():
    assert _native.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(_native.LIB)


def test_host_only_helpers(lib):
    assert hs.hs_plan_bytes(8, 2048) == 16 + 8 * (16 + 8 * 2048)
    assert hs.hs_plan_bytes(0, 5) == 16
    assert hs.hs_strerror(hs.HS_OK) == "ok"
    assert "invalid" in hs.hs_strerror(hs.HS_ERR_INVALID_ARG)
    assert hs.hs_kernels_per_call() == 1


def _desc(**kw):
    d = dict(n_requests=2, n_layers=2, n_positions=1000, record_bytes=128, slots=64,
             max_k=32, layer_anchor=None, host_limit_bytes=0, host_alloc=0, launch_overlap=0)
    d.update(kw)
    return _native.PoolDesc(**d)


@pytest.mark.parametrize("bad", [
    dict(n_requests=0), dict(n_layers=0), dict(n_positions=0), dict(n_positions=1 << 31),
    dict(record_bytes=100), dict(record_bytes=0), dict(slots=0), dict(slots=40000),
    dict(max_k=0), dict(max_k=65), dict(host_alloc=-1), dict(host_alloc=4),
    dict(launch_overlap=-1), dict(launch_overlap=3)])
def test_create_pool_rejects_bad_descriptors(lib, bad):
    h = ctypes.c_void_p(1234)
    rc = lib.hs_create_pool(ctypes.byref(_desc(**bad)), ctypes.byref(h))
    assert rc == hs.HS_ERR_INVALID_ARG
    assert h.value is None


def test_create_pool_rejects_bad_anchor_map(lib):
    a = (ctypes.c_int32 * 2)(1, 1)   # layer 0 may not share a later layer
    d = _desc(layer_anchor=ctypes.cast(a, ctypes.c_void_p))
    h = ctypes.c_void_p()
    assert lib.hs_create_pool(ctypes.byref(d), ctypes.byref(h)) == hs.HS_ERR_INVALID_ARG


def test_create_pool_refuses_over_host_limit(lib):
    d = _desc(host_limit_bytes=1000)
    h = ctypes.c_void_p()
    assert lib.hs_create_pool(ctypes.byref(d), ctypes.byref(h)) == hs.HS_ERR_NOMEM
    assert lib.hs_create_pool(None, ctypes.byref(h)) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_create_pool(ctypes.byref(d), None) == hs.HS_ERR_INVALID_ARG


def test_attention_argument_checks(lib):
    f = lib.hs_sparse_attention
    assert f(16, 16, 10, 16, 1, 10, 8, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG   # heads
    assert f(16, 16, 10, 16, 1, 0, 16, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG   # k = 0
    assert f(16, 16, 0, 16, 1, 10, 16, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG   # no rows
    assert f(8, 16, 10, 16, 1, 10, 16, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG   # alignment
    assert f(16, 16, 10, 16, 1, 10, 16, 1.0, 8, None) == hs.HS_ERR_INVALID_ARG
    assert f(None, 16, 10, 16, 1, 10, 16, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG
    assert f(16, 16, 10, 16, 70000, 10, 16, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG
    assert f(16, 16, 10, 16, 0, 10, 16, 1.0, 16, None) == hs.HS_OK   # n_req = 0: no-op
    assert lib.hs_attention_status(None) == hs.HS_ERR_INVALID_ARG


def test_attention_heads_argument_checks(lib):
    f = lib.hs_sparse_attention_heads
    assert f(16, 16, 10, 16, 1, 10, 0, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG   # heads
    assert f(16, 16, 10, 16, 1, 10, 9, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG
    assert f(16, 16, 10, 16, 1, 0, 8, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG    # k = 0
    assert f(16, 16, 0, 16, 1, 10, 8, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG    # no rows
    assert f(8, 16, 10, 16, 1, 10, 8, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG    # alignment
    assert f(16, 8, 10, 16, 1, 10, 8, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG
    assert f(16, 16, 10, 16, 1, 10, 8, 1.0, 8, None) == hs.HS_ERR_INVALID_ARG
    assert f(16, 16, 10, None, 1, 10, 8, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG
    assert f(16, 16, 10, 16, 70000, 10, 8, 1.0, 16, None) == hs.HS_ERR_INVALID_ARG
    assert f(16, 16, 10, 16, 0, 10, 8, 1.0, 16, None) == hs.HS_OK   # n_req = 0: no-op


def test_calls_on_null_pool_are_rejected(lib):
    v = _native.Views()
    s = _native.Stats()
    p = ctypes.c_void_p()
    assert lib.hs_resolve(None, 0, 1, None, 16, 1, 16, None, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_prefetch_plan(None, 0, 0, 1, None, 16, 1, 16, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_prefetch_copy(None, 0, 1, 1, 16, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_stats(None, -1, ctypes.byref(s)) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_device_views(None, 0, ctypes.byref(v)) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_host_records(None, 0, 0, ctypes.byref(p)) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_reset(None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_destroy_pool(None) == hs.HS_OK
    assert lib.hs_link_probe(8, 0, 1152, 0, None, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_link_probe(1 << 20, 1, 1152, 7, None, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_pool_info(None, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_touch_records(None, -1, -1, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_warm_pool(None) == hs.HS_ERR_INVALID_ARG


def test_noalloc_refuses_misaligned_pointers_before_any_cuda_call(lib):
    """hs_resolve_noalloc checks the alignment its kernel's accesses need
    (16-byte records and slots, 4-byte int32 arrays, 2-byte LRU order) and
    refuses before touching CUDA (no device here)."""
    def state(**kw):
        f = dict(n_requests=2, n_positions=100, record_bytes=64, slots=8, host_records=4096,
                 cache=8192, page_table=12288, slot_pos=16384, stamps=20480, lru=24576,
                 resolves=28672)
        f.update(kw)
        return _native.LayerState(**f)

    call = lib.hs_resolve_noalloc
    for bad in (dict(host_records=4104), dict(cache=8200), dict(page_table=12290),
                dict(slot_pos=16385), dict(stamps=20482), dict(lru=24577), dict(resolves=28673)):
        assert call(ctypes.byref(state(**bad)), 1, None, 32768, 4, 36864, None, None) == \
            hs.HS_ERR_INVALID_ARG, bad
    s = state()
    assert call(ctypes.byref(s), 1, None, 32770, 4, 36864, None, None) == hs.HS_ERR_INVALID_ARG
    assert call(ctypes.byref(s), 1, None, 32768, 4, 36866, None, None) == hs.HS_ERR_INVALID_ARG
    assert call(ctypes.byref(s), 1, 40962, 32768, 4, 36864, None, None) == hs.HS_ERR_INVALID_ARG
    assert call(ctypes.byref(s), 1, None, 32768, 4, 36864, 45058, None) == hs.HS_ERR_INVALID_ARG
