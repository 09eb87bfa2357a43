"""Replacement-policy study on selection traces -- CPU only, test/analysis code.

The Pith review's Fig. 6 compares per-step top-k miss rates of several
cache configurations on one selection trace: LRU at several B against
staging only the current top-k ("Swap-vanilla", B = k); its reference list
cites Belady's offline-optimal replacement as the bound for such studies.
This module replays a trace ``sel[T][k]`` of one (request, layer) under:

* ``lru_misses``  -- the resolve method itself (the C oracle), any B >= k;
* ``min_misses``  -- offline farthest-next-use replacement: when m new
  positions must enter a full cache, evict the m resident positions (not
  selected at this step) whose next selection lies farthest in the future
  (never = infinitely far; ties to the smaller position).  This is Belady's
  MIN applied to a step that must hold its whole selection at once;
* ``topk_only``   -- B = k LRU, which keeps exactly the current selection.

Misses count selected positions not resident before the step (the first
step's k are all misses).  Pinned by tests/test_policy.py: exhaustive
search over every eviction choice on tiny traces finds no schedule with
fewer misses than ``min_misses``, and ``min_misses <= lru_misses`` always.
"""
from __future__ import annotations

import heapq

import numpy as np

from .oracle import OK, Pair


def lru_misses(sel: np.ndarray, B: int, L: int) -> np.ndarray:
    """Per-step misses of the resolve method's LRU with B slots."""
    p = Pair(B, L, 16)
    rc, _, m = p.run(np.ascontiguousarray(sel, np.int32))
    if rc != OK:
        raise ValueError(f"oracle rejected the trace ({rc})")
    return m.astype(np.int64)


def topk_only(sel: np.ndarray, L: int) -> np.ndarray:
    """Per-step misses when only the current top-k is staged (B = k)."""
    return lru_misses(sel, sel.shape[1], L)


def _next_use(sel: np.ndarray):
    """nxt[t][i]: next step > t at which sel[t][i] is selected (or T)."""
    T = sel.shape[0]
    last = {}
    nxt = np.full(sel.shape, T, np.int64)
    for t in range(T - 1, -1, -1):
        for i, p in enumerate(sel[t].tolist()):
            nxt[t, i] = last.get(p, T)
        for p in sel[t].tolist():
            last[p] = t
    return nxt


def min_misses(sel: np.ndarray, B: int) -> np.ndarray:
    """Per-step misses of offline farthest-next-use replacement."""
    T, k = sel.shape
    if B < k:
        raise ValueError("B must be at least k")
    nxt = _next_use(sel)
    resident = {}          # position -> next use
    heap = []              # (-next_use, position), lazily invalidated
    out = np.zeros(T, np.int64)
    for t in range(T):
        cur = sel[t].tolist()
        cur_set = set(cur)
        new = [p for p in cur if p not in resident]
        out[t] = len(new)
        # refresh next uses of the selected positions
        for i, p in enumerate(cur):
            resident[p] = int(nxt[t, i])
        need = len(resident) - B
        held = []
        while need > 0:
            nu, p = heapq.heappop(heap)
            nu = -nu
            if p not in resident or resident[p] != nu:
                continue           # stale entry
            if p in cur_set:
                held.append((-nu, p))
                continue           # this step's selection cannot be evicted
            del resident[p]
            need -= 1
        for h in held:
            heapq.heappush(heap, h)
        for i, p in enumerate(cur):
            heapq.heappush(heap, (-int(nxt[t, i]), p))
    return out


def study(sel: np.ndarray, L: int, slots) -> dict:
    """Steady-state miss rates (steps 1..T-1) per policy and B."""
    k = sel.shape[1]
    res = {}
    for B in slots:
        res[("lru", B)] = lru_misses(sel, B, L)[1:].sum() / (k * (sel.shape[0] - 1))
        res[("min", B)] = min_misses(sel, B)[1:].sum() / (k * (sel.shape[0] - 1))
    return res


def main():
    """Fig. 6 analogue on the synthetic traces: steady-state miss rates."""
    from workloads import configs, traces

    for w in (configs.DSA_MLA, configs.QUEST_PAGES, configs.NO_LOCALITY):
        sel = traces.stream(w, 0, 0)
        slots = [w.k, (3 * w.k) // 2, 2 * w.k, 3 * w.k, 4 * w.k]
        r = study(sel, w.n_positions, slots)
        print(f"{w.name} (request 0, layer 0, {sel.shape[0]} steps, k={w.k})")
        print("| B | LRU (this method) | farthest-next-use (offline bound) |")
        print("|---|---|---|")
        for B in slots:
            tag = " (top-k only)" if B == w.k else ""
            print(f"| {B}{tag} | {100 * r[('lru', B)]:.2f} % | {100 * r[('min', B)]:.2f} % |")
        print()


if __name__ == "__main__":
    main()
