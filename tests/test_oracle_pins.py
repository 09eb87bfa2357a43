"""Pins of the CPU oracle against facts that do not come from the oracle.

* a hand-worked trace (tests/golden/micro_lru.txt);
* brute-force replay (tests/bruteforce.py): exhaustive over tiny traces and
  on random ones;
* closed-form special cases (cold start, repeated selection, disjoint
  selections with B = k, B >= L);
* invariants after every resolve: h + m = k, every selected position
  resident, page table and slot map mutually inverse, occupancy <= B, every
  cached record byte-equal to its host record;
* rejection of invalid selections with the state left untouched.
"""
import itertools
import os

import numpy as np
import pytest

from oracle.oracle import ERR_ARG, ERR_DUP, ERR_RANGE, OK, Pair
from tests.bruteforce import BrutePair

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "micro_lru.txt")


def _ints(s):
    return [int(x) for x in s.split(",")]


def load_golden():
    steps, L, B = [], None, None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = dict(kv.split("=", 1) for kv in line.split())
        if "L" in f:
            L, B = int(f["L"]), int(f["B"])
            continue
        steps.append({k: _ints(v) for k, v in f.items()})
    return L, B, steps


def test_golden_hand_worked_trace():
    L, B, steps = load_golden()
    p = Pair(B, L, 16)
    for st in steps:
        rc, out, m = p.resolve(st["sel"])
        assert rc == OK
        assert out.tolist() == st["out"]
        assert m == st["m"][0]
        assert p.slot_pos.tolist() == st["slot_pos"]
        assert p.stamp.tolist() == st["stamp"]
        pt = np.full(L, -1)
        for b, q in enumerate(st["slot_pos"]):
            if q >= 0:
                pt[q] = b
        assert p.pt.tolist() == pt.tolist()


def _compare(p: Pair, bp: BrutePair, L):
    assert p.slot_pos.tolist() == bp.slot_pos
    assert p.stamp.tolist() == bp.stamp
    assert p.pt.tolist() == bp.page_table(L)
    assert p.hits == bp.hits and p.misses == bp.misses


def _selections(L, kmax):
    for k in range(1, kmax + 1):
        yield from itertools.permutations(range(L), k)


@pytest.mark.parametrize("L,B,length", [(4, 1, 4), (4, 2, 3), (5, 2, 3), (4, 3, 2)])
def test_bruteforce_exhaustive(L, B, length):
    sels = list(_selections(L, B))
    n = 0
    for trace in itertools.product(sels, repeat=length):
        p, bp = Pair(B, L, 16), BrutePair(B)
        for sel in trace:
            rc, out, m = p.resolve(list(sel))
            o2, m2 = bp.resolve(list(sel))
            assert rc == OK and out.tolist() == o2 and m == m2
        _compare(p, bp, L)
        n += 1
    assert n == len(sels) ** length


def test_bruteforce_random():
    rng = np.random.default_rng(12345)
    for _ in range(3000):
        B = int(rng.integers(1, 9))
        L = int(rng.integers(B, 33))
        T = int(rng.integers(1, 11))
        p, bp = Pair(B, L, 16), BrutePair(B)
        base = int(rng.integers(0, 4)) * B
        for _t in range(T):
            k = int(rng.integers(1, B + 1))
            sel = rng.choice(L, size=k, replace=False).tolist()
            rc, out, m = p.resolve(sel, out_base=base)
            o2, m2 = bp.resolve(sel, out_base=base)
            assert rc == OK and out.tolist() == o2 and m == m2
            _compare(p, bp, L)


def test_cold_start_fills_slots_in_selection_order():
    rng = np.random.default_rng(1)
    B, L, k = 128, 4096, 64
    p = Pair(B, L, 16)
    sel = rng.choice(L, size=k, replace=False)
    rc, out, m = p.resolve(sel)
    assert rc == OK and m == k
    assert out.tolist() == list(range(k))
    assert (p.stamp[:k] == 1).all() and (p.stamp[k:] == 0).all()


def test_repeated_selection_hits_from_step_two():
    rng = np.random.default_rng(2)
    B, L, k = 16, 100, 10
    p = Pair(B, L, 16)
    sel = rng.choice(L, size=k, replace=False)
    first = p.resolve(sel)[1]
    for t in range(2, 8):
        rc, out, m = p.resolve(sel)
        assert rc == OK and m == 0
        assert out.tolist() == first.tolist()
        assert (p.stamp[first] == 2 * t).all()


def test_disjoint_selections_with_b_equal_k_always_miss():
    B = k = 8
    L = 200
    p = Pair(B, L, 16)
    for t in range(20):
        sel = np.arange(t * k, (t + 1) * k)[::-1] % L
        rc, out, m = p.resolve(sel)
        assert rc == OK and m == k
        # every slot is rewritten; victims taken in slot order (all stamps tie)
        assert sorted(out.tolist()) == list(range(B))
        assert out.tolist() == list(range(B))


def test_cache_larger_than_context_never_evicts():
    rng = np.random.default_rng(3)
    L, B, k = 20, 24, 6
    p = Pair(B, L, 16)
    seen = set()
    for _ in range(50):
        sel = rng.choice(L, size=k, replace=False)
        new = len(set(sel.tolist()) - seen)
        rc, out, m = p.resolve(sel)
        assert rc == OK and m == new
        seen |= set(sel.tolist())
        assert int((p.slot_pos >= 0).sum()) == len(seen)
    assert p.misses == len(seen)


def check_invariants(p: Pair, sel, m):
    k = len(sel)
    assert 0 <= m <= k
    assert (p.pt[np.asarray(sel)] >= 0).all(), "a selected position is not resident"
    occ = np.nonzero(p.slot_pos >= 0)[0]
    assert (p.pt[p.slot_pos[occ]] == occ).all(), "page table and slot map disagree"
    assert int((p.pt >= 0).sum()) == occ.size, "stale page-table entries"
    assert occ.size <= p.B
    assert len(set(p.slot_pos[occ].tolist())) == occ.size, "position in two slots"
    if p.cache is not None:
        assert (p.cache[occ] == p.host[p.slot_pos[occ]]).all(), "cache differs from host"


def test_invariants_on_random_traces():
    rng = np.random.default_rng(4)
    for trial in range(40):
        B = int(rng.integers(2, 40))
        L = int(rng.integers(B, 300))
        W = 16
        host = rng.integers(0, 256, size=(L, W), dtype=np.uint8)
        p = Pair(B, L, W, host=host, mirror=True)
        total = 0
        for _ in range(30):
            k = int(rng.integers(1, B + 1))
            sel = rng.choice(L, size=k, replace=False)
            rc, out, m = p.resolve(sel, out_base=3 * B)
            assert rc == OK
            total += k
            assert p.hits + p.misses == total
            assert p.fetched_bytes == p.misses * W
            assert (out - 3 * B == p.pt[sel]).all()
            check_invariants(p, sel, m)


@pytest.mark.parametrize("sel,code", [
    ([1, 2, 2], ERR_DUP), ([0, 100], ERR_RANGE), ([-1, 3], ERR_RANGE),
    (list(range(9)), ERR_ARG), ([], ERR_ARG)])
def test_invalid_selection_rejected_state_untouched(sel, code):
    p = Pair(8, 100, 16)
    p.resolve([5, 6, 7])
    before = (p.slot_pos.copy(), p.stamp.copy(), p.pt.copy(), p.t.copy(), p.counters.copy())
    rc, out, m = p.resolve(sel)
    assert rc == code
    assert (out == -1).all() and m == -1
    after = (p.slot_pos, p.stamp, p.pt, p.t, p.counters)
    for a, b in zip(before, after):
        assert (a == b).all()
