"""Pins of the replacement-policy study (oracle/policy.py)."""
import itertools

import numpy as np
import pytest

from oracle import policy
from workloads import configs, traces


def _brute_min(sel, B):
    """Fewest total misses over every possible eviction schedule."""
    best = [None]

    def go(t, resident, misses):
        if best[0] is not None and misses >= best[0]:
            return
        if t == len(sel):
            best[0] = misses
            return
        cur = list(sel[t])
        new = [p for p in cur if p not in resident]
        res = resident | set(cur)
        need = len(res) - B
        if need <= 0:
            go(t + 1, frozenset(res), misses + len(new))
            return
        cand = sorted(resident - set(cur))
        for ev in itertools.combinations(cand, need):
            go(t + 1, frozenset(res - set(ev)), misses + len(new))

    go(0, frozenset(), 0)
    return best[0]


def test_min_equals_exhaustive_search_on_tiny_traces():
    rng = np.random.default_rng(5)
    for _ in range(300):
        L = int(rng.integers(3, 8))
        k = int(rng.integers(1, 3))
        B = int(rng.integers(k, k + 3))
        T = int(rng.integers(1, 7))
        sel = np.array([rng.choice(L, k, replace=False) for _ in range(T)], np.int32)
        assert policy.min_misses(sel, B).sum() == _brute_min(sel.tolist(), B)


def test_min_never_worse_than_lru():
    rng = np.random.default_rng(6)
    for _ in range(200):
        L = int(rng.integers(5, 60))
        k = int(rng.integers(1, 6))
        B = int(rng.integers(k, 3 * k + 2))
        T = int(rng.integers(1, 25))
        sel = np.array([rng.choice(L, k, replace=False) for _ in range(T)], np.int32)
        assert policy.min_misses(sel, B).sum() <= policy.lru_misses(sel, B, L).sum()


def test_cache_holding_everything_misses_each_position_once():
    rng = np.random.default_rng(7)
    sel = np.array([rng.choice(30, 6, replace=False) for _ in range(20)], np.int32)
    distinct = len(np.unique(sel))
    assert policy.min_misses(sel, 40).sum() == distinct
    assert policy.lru_misses(sel, 40, 30).sum() == distinct


def test_study_orders_policies_on_the_dsa_mla_trace():
    w = configs.DSA_MLA.with_(steps=64)
    sel = traces.stream(w, 0, 0)
    r = policy.study(sel, w.n_positions, [w.k, 2 * w.k])
    assert r[("lru", w.k)] > r[("lru", 2 * w.k)] >= r[("min", 2 * w.k)]
    assert r[("lru", w.k)] >= r[("min", w.k)]
