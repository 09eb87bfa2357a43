"""Python driver of the CPU oracle (``hs_oracle.c``) -- test infrastructure.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this module.  It never touches the CUDA library: the oracle and the
GPU path share nothing but the seeded input generators in ``workloads``.

:class:`Pair` holds the state of one (request, layer) pair in numpy arrays
(slot -> position, stamps, page table, resolve count, optional cache mirror)
and calls the C functions on it.  :class:`Layered` keeps one Pair per
(request, layer) of a workload and replays whole traces.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hs_oracle.c")
_LIB = os.path.join(_HERE, "libhs_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_RANGE, ERR_DUP, ERR_STATE = 0, 1, 2, 3, 4
# counter slots of a pair
C_HITS, C_MISSES, C_FETCHED, C_PLAN_HITS, C_PLAN_MISMATCH, C_PREFETCHED, C_RESOLVES = range(7)


def build(force: bool = False) -> str:
    """Compile the oracle into ``libhs_oracle.so`` beside its source (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


class _PairC(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("W", ctypes.c_int32), ("L", ctypes.c_int64),
                ("slot_pos", ctypes.c_void_p), ("stamp", ctypes.c_void_p),
                ("pt", ctypes.c_void_p), ("t", ctypes.c_void_p),
                ("cache", ctypes.c_void_p), ("host", ctypes.c_void_p),
                ("counters", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # a separately built copy (e.g. the sanitizer build of the
            # tests) may be named in the environment
            path = os.environ.get("HS_ORACLE_LIB")
            if not path:
                build()
                path = _LIB
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER(_PairC)
            vp, i32 = ctypes.c_void_p, ctypes.c_int32
            lib.ora_validate.argtypes = [P, vp, i32]
            lib.ora_plan.argtypes = [P, vp, i32, vp, vp, vp, vp]
            lib.ora_prefetch_copy.argtypes = [P, vp, vp, i32]
            lib.ora_resolve.argtypes = [P, vp, i32, i32, vp, vp, vp, vp, i32]
            lib.ora_run.argtypes = [P, vp, i32, i32, i32, i32, vp, vp]
            for f in (lib.ora_validate, lib.ora_plan, lib.ora_prefetch_copy,
                      lib.ora_resolve, lib.ora_run):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


class Pair:
    """Oracle state of one (request, layer): B slots over L positions."""

    def __init__(self, B: int, L: int, W: int, host: np.ndarray | None = None,
                 mirror: bool = False):
        self.B, self.L, self.W = int(B), int(L), int(W)
        self.slot_pos = np.full(B, -1, np.int32)
        self.stamp = np.zeros(B, np.uint32)
        self.pt = np.full(L, -1, np.int32)
        self.t = np.zeros(1, np.uint32)
        self.counters = np.zeros(7, np.uint64)
        self.host = None if host is None else np.ascontiguousarray(host, np.uint8)
        if self.host is not None and self.host.shape != (L, W):
            raise ValueError("host records must be [L][W]")
        self.cache = np.zeros((B, W), np.uint8) if mirror else None
        self._c = _PairC(self.B, self.W, self.L, _ptr(self.slot_pos), _ptr(self.stamp),
                         _ptr(self.pt), _ptr(self.t), _ptr(self.cache), _ptr(self.host),
                         _ptr(self.counters))

    def copy(self) -> "Pair":
        q = Pair.__new__(Pair)
        q.B, q.L, q.W = self.B, self.L, self.W
        q.slot_pos, q.stamp, q.pt = self.slot_pos.copy(), self.stamp.copy(), self.pt.copy()
        q.t, q.counters, q.host = self.t.copy(), self.counters.copy(), self.host
        q.cache = None if self.cache is None else self.cache.copy()
        q._c = _PairC(q.B, q.W, q.L, _ptr(q.slot_pos), _ptr(q.stamp), _ptr(q.pt),
                      _ptr(q.t), _ptr(q.cache), _ptr(q.host), _ptr(q.counters))
        return q

    def validate(self, sel) -> int:
        sel = np.ascontiguousarray(sel, np.int32)
        return _load().ora_validate(ctypes.byref(self._c), _ptr(sel), sel.size)

    def plan(self, sel):
        """Read-only: (rc, hit_slot[k], miss_idx[m], victim[m])."""
        sel = np.ascontiguousarray(sel, np.int32)
        k = sel.size
        hit = np.empty(max(k, 1), np.int32)
        miss = np.empty(max(k, 1), np.int32)
        vic = np.empty(max(k, 1), np.int32)
        m = np.zeros(1, np.int32)
        rc = _load().ora_plan(ctypes.byref(self._c), _ptr(sel), k, _ptr(hit), _ptr(miss),
                              _ptr(vic), _ptr(m))
        if rc:
            return rc, None, None, None
        return rc, hit[:k].copy(), miss[:m[0]].copy(), vic[:m[0]].copy()

    def prefetch_plan(self, sel):
        """Plan pairs (positions, slots) the next resolve of ``sel`` will fill."""
        rc, _, miss, vic = self.plan(sel)
        if rc:
            return rc, None, None
        sel = np.asarray(sel, np.int32)
        return rc, sel[miss].astype(np.int32), vic.astype(np.int32)

    def prefetch_copy(self, plan_pos, plan_slot) -> int:
        pp = np.ascontiguousarray(plan_pos, np.int32)
        ps = np.ascontiguousarray(plan_slot, np.int32)
        return _load().ora_prefetch_copy(ctypes.byref(self._c), _ptr(pp), _ptr(ps), pp.size)

    def resolve(self, sel, out_base: int = 0, plan=None):
        """One resolve: returns (rc, out[k], m)."""
        sel = np.ascontiguousarray(sel, np.int32)
        out = np.empty(max(sel.size, 1), np.int32)
        m = np.zeros(1, np.int32)
        if plan is None:
            pp = ps = None
            pm = -1
        else:
            pp = np.ascontiguousarray(plan[0], np.int32)
            ps = np.ascontiguousarray(plan[1], np.int32)
            pm = pp.size
        rc = _load().ora_resolve(ctypes.byref(self._c), _ptr(sel), sel.size, out_base,
                                 _ptr(out), _ptr(m), _ptr(pp), _ptr(ps), pm)
        return rc, out[:sel.size].copy(), int(m[0])

    def run(self, sels: np.ndarray, out_base: int = 0):
        """Resolves of ``sels[T][k]`` back to back: returns (rc, out[T][k], m[T])."""
        sels = np.ascontiguousarray(sels, np.int32)
        T, k = sels.shape
        out = np.empty((T, k), np.int32)
        m = np.empty(T, np.int32)
        rc = _load().ora_run(ctypes.byref(self._c), _ptr(sels), T, k, k, out_base,
                             _ptr(out), _ptr(m))
        return rc, out, m

    # convenience views
    @property
    def hits(self):
        return int(self.counters[C_HITS])

    @property
    def misses(self):
        return int(self.counters[C_MISSES])

    @property
    def fetched_bytes(self):
        return int(self.counters[C_FETCHED])
