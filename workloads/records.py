"""Python side of the seeded record generator (``records.c``).

``fill(dst_ptr, ...)`` writes the records of one (request, layer) into a host
buffer, for example the pinned host pool; ``gen(...)`` returns the records of
an explicit list of positions as a numpy ``uint8`` array ``[n][W]``.  Both
follow the counter-based definition stated in ``records.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import Workload

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "records.c")
_LIB = os.path.join(_HERE, "librecords.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``records.c`` into ``librecords.so`` next to it (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O3", "-std=gnu11", "-fPIC", "-shared", "-pthread",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # a separately built copy (e.g. the sanitizer build of the
            # tests) may be named in the environment
            path = os.environ.get("HS_RECORDS_LIB")
            if not path:
                build()
                path = _LIB
            lib = ctypes.CDLL(path)
            lib.wl_gen_records.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64]
            lib.wl_gen_records.restype = None
            lib.wl_fill_records.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int]
            lib.wl_fill_records.restype = ctypes.c_int
            _lib = lib
    return _lib


def stream_id(w: Workload, r: int, l: int) -> int:
    return r * w.n_layers + l


def gen(w: Workload, r: int, l: int, positions) -> np.ndarray:
    """Records ``[n][W]`` (uint8) of request r, layer l at ``positions``."""
    pos = np.ascontiguousarray(positions, dtype=np.int32).reshape(-1)
    if pos.size and (pos.min() < 0 or pos.max() >= w.n_positions):
        raise ValueError("position out of range")
    out = np.empty((pos.size, w.record_bytes), np.uint8)
    _load().wl_gen_records(out.ctypes.data, pos.ctypes.data, pos.size,
                           w.record_bytes, w.value_format, w.seed,
                           stream_id(w, r, l))
    return out


def fill(dst_ptr: int, w: Workload, r: int, l: int, pos0: int = 0,
         n: int | None = None, threads: int | None = None) -> None:
    """Write records ``[pos0, pos0 + n)`` of (r, l) to the host address ``dst_ptr``."""
    if n is None:
        n = w.n_positions - pos0
    if threads is None:
        threads = max(1, len(os.sched_getaffinity(0)))
    _load().wl_fill_records(ctypes.c_void_p(dst_ptr), pos0, n, w.record_bytes,
                            w.value_format, w.seed, stream_id(w, r, l), threads)


def decode(w: Workload, rec: np.ndarray) -> np.ndarray:
    """View records as float64 values (fp16 or bf16 elements)."""
    u16 = np.ascontiguousarray(rec).view(np.uint16)
    if w.value_format == 0:
        return u16.view(np.float16).astype(np.float64)
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
