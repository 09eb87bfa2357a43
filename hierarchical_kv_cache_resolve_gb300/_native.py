"""Builds and loads ``libhs.so``, the CUDA library behind ``include/hs.h``.

The library is compiled in-tree for sm_103a only (GB300) with nvcc; no other
architecture and no CPU implementation exist.  Loading fails loudly when the
library cannot be built or found.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
CSRC = os.path.join(_PKG, "csrc")
INCLUDE = os.path.join(_ROOT, "include")
BUILD = os.path.join(_PKG, "_build")
LIB = os.path.join(BUILD, "libhs.so")
SOURCES = ("api.cu", "hostmem.cu", "resolve.cu", "copy.cu", "noalloc.cu", "attention.cu",
           "attention_heads.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

_lock = threading.Lock()
_lib = None


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the hs CUDA library cannot be built")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, "hs_internal.cuh"), os.path.join(INCLUDE, "hs.h")]
    return files


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit in parallel, then link ``libhs.so``."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE, "-I", CSRC]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + common
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, err in results:
            print(err)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def load() -> ctypes.CDLL:
    """Load (building first if needed) and type the library's entry points."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(LIB)
        _declare(lib)
        _lib = lib
        return lib


# ---- ctypes mirrors of include/hs.h ------------------------------------------

class PoolDesc(ctypes.Structure):
    _fields_ = [("n_requests", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("n_positions", ctypes.c_int64), ("record_bytes", ctypes.c_int32),
                ("slots", ctypes.c_int32), ("max_k", ctypes.c_int32),
                ("layer_anchor", ctypes.c_void_p), ("host_limit_bytes", ctypes.c_uint64),
                ("host_alloc", ctypes.c_int32), ("launch_overlap", ctypes.c_int32)]


class PoolInfo(ctypes.Structure):
    _fields_ = [("host_alloc", ctypes.c_int32), ("device", ctypes.c_int32),
                ("device_numa", ctypes.c_int32), ("host_numa_first", ctypes.c_int32),
                ("host_numa_last", ctypes.c_int32), ("launch_overlap", ctypes.c_int32),
                ("host_bytes", ctypes.c_uint64), ("host_mapped_bytes", ctypes.c_uint64),
                ("host_granularity", ctypes.c_uint64), ("device_bytes", ctypes.c_uint64),
                ("host_huge_bytes", ctypes.c_uint64), ("warmup_us", ctypes.c_uint64)]


class Stats(ctypes.Structure):
    _fields_ = [("resolves", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("misses", ctypes.c_uint64), ("fetched_bytes", ctypes.c_uint64),
                ("prefetched_bytes", ctypes.c_uint64), ("plan_hits", ctypes.c_uint64),
                ("plan_mismatches", ctypes.c_uint64), ("status", ctypes.c_uint32)]


class Views(ctypes.Structure):
    _fields_ = [("cache", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("slot_pos", ctypes.c_void_p), ("stamps", ctypes.c_void_p),
                ("lru", ctypes.c_void_p), ("resolves", ctypes.c_void_p)]


class LayerState(ctypes.Structure):
    _fields_ = [("n_requests", ctypes.c_int32), ("n_positions", ctypes.c_int64),
                ("record_bytes", ctypes.c_int32), ("slots", ctypes.c_int32),
                ("host_records", ctypes.c_void_p), ("cache", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("slot_pos", ctypes.c_void_p),
                ("stamps", ctypes.c_void_p), ("lru", ctypes.c_void_p),
                ("resolves", ctypes.c_void_p)]


EXPORTS = ("hs_create_pool", "hs_destroy_pool", "hs_host_records", "hs_device_views",
           "hs_pool_info", "hs_device_host_numa", "hs_touch_records", "hs_warm_pool",
           "hs_resolve", "hs_resolve_anchor", "hs_resolve_measure", "hs_measure_stamp_slots", "hs_plan_bytes",
           "hs_prefetch_plan", "hs_prefetch_copy",
           "hs_stats", "hs_reset", "hs_link_probe", "hs_kernels_per_call", "hs_strerror",
           "hs_resolve_noalloc", "hs_sparse_attention", "hs_sparse_attention_heads",
           "hs_attention_status")


def _declare(lib):
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    P = ctypes.c_void_p
    sig = {
        "hs_create_pool": ([ctypes.POINTER(PoolDesc), ctypes.POINTER(vp)], ctypes.c_int),
        "hs_destroy_pool": ([P], ctypes.c_int),
        "hs_host_records": ([P, i32, i32, ctypes.POINTER(vp)], ctypes.c_int),
        "hs_device_views": ([P, i32, ctypes.POINTER(Views)], ctypes.c_int),
        "hs_pool_info": ([P, ctypes.POINTER(PoolInfo)], ctypes.c_int),
        "hs_device_host_numa": ([i32], ctypes.c_int),
        "hs_touch_records": ([P, i32, i32, vp], ctypes.c_int),
        "hs_warm_pool": ([P], ctypes.c_int),
        "hs_resolve": ([P, i32, i32, vp, vp, i32, vp, vp, vp], ctypes.c_int),
        "hs_resolve_anchor": ([P, i32, i32, vp, vp, i32, vp, vp, vp], ctypes.c_int),
        "hs_resolve_measure": ([P, i32, i32, vp, vp, i32, vp, i32, vp, vp], ctypes.c_int),
        "hs_measure_stamp_slots": ([], i32),
        "hs_plan_bytes": ([i32, i32], ctypes.c_size_t),
        "hs_prefetch_plan": ([P, i32, i32, i32, vp, vp, i32, vp, vp], ctypes.c_int),
        "hs_prefetch_copy": ([P, i32, i32, i32, vp, vp], ctypes.c_int),
        "hs_stats": ([P, i32, ctypes.POINTER(Stats)], ctypes.c_int),
        "hs_reset": ([P], ctypes.c_int),
        "hs_link_probe": ([ctypes.c_size_t, i32, i32, i32, ctypes.POINTER(ctypes.c_double),
                           ctypes.POINTER(ctypes.c_double)], ctypes.c_int),
        "hs_kernels_per_call": ([], i32),
        "hs_strerror": ([ctypes.c_int], ctypes.c_char_p),
        "hs_resolve_noalloc": ([ctypes.POINTER(LayerState), i32, vp, vp, i32, vp, vp, vp],
                               ctypes.c_int),
        "hs_sparse_attention": ([vp, vp, i64, vp, i32, i32, i32, ctypes.c_float, vp, vp],
                                ctypes.c_int),
        "hs_sparse_attention_heads": ([vp, vp, i64, vp, i32, i32, i32, ctypes.c_float, vp, vp],
                                      ctypes.c_int),
        "hs_attention_status": ([ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
