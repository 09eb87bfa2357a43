"""Shared machinery of the GPU parity tests: drive a workload through the C
ABI and compare with the CPU oracle on the same seeded inputs.

Nothing the oracle computes comes from the GPU: both sides read the selection
traces and host records of ``workloads``; the GPU results are only compared.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from hierarchical_kv_cache_resolve_gb300 import hs
from oracle.oracle import OK, Pair
from workloads import records, traces


def fill_selected(pool: hs.Pool, w, sel, requests=None):
    """Write the host records of every position the trace selects.

    Positions never selected are never read by either side, so they are left
    as allocated.  sel is [T][R][N_l][k]."""
    requests = range(w.n_requests) if requests is None else requests

    def one(rl):
        r, l = rl
        pos = np.unique(sel[:, r, l, :])
        view = pool.host_records(r, l)
        view[pos] = records.gen(w, r, l, pos)

    jobs = [(r, l) for r in requests for l in range(w.n_layers)]
    with ThreadPoolExecutor(16) as ex:
        list(ex.map(one, jobs))


def fill_all(pool: hs.Pool, w):
    for r in range(w.n_requests):
        for l in range(w.n_layers):
            records.fill(pool.host_records(r, l).ctypes.data, w, r, l)


def device_trace(sel):
    """[T][R][N_l][k] -> device [T][N_l][R][k] so each (step, layer) is contiguous."""
    return torch.from_numpy(np.ascontiguousarray(sel.transpose(0, 2, 1, 3))).cuda()


class OracleRun:
    """Oracle pairs for (request, layer), replayed step by step."""

    def __init__(self, w, pairs=None):
        self.w = w
        self.pairs = pairs if pairs is not None else [(r, l) for r in range(w.n_requests)
                                                      for l in range(w.n_layers)]
        self.state = {rl: Pair(w.slots, w.n_positions, w.record_bytes) for rl in self.pairs}

    def step(self, sel_t):
        """sel_t [R][N_l][k] -> {(r, l): (out, m)}"""
        res = {}
        for (r, l), p in self.state.items():
            rc, out, m = p.resolve(sel_t[r, l], out_base=r * self.w.slots)
            assert rc == OK
            res[(r, l)] = (out, m)
        return res


def run_oracle_all(w, sel, pairs=None):
    """Whole trace per pair (C loop): {(r, l): (Pair, out[T][k], m[T])}."""
    pairs = pairs if pairs is not None else [(r, l) for r in range(w.n_requests)
                                             for l in range(w.n_layers)]

    def one(rl):
        r, l = rl
        p = Pair(w.slots, w.n_positions, w.record_bytes)
        rc, out, m = p.run(sel[:, r, l, :], out_base=r * w.slots)
        assert rc == OK
        return rl, (p, out, m)

    with ThreadPoolExecutor(16) as ex:
        return dict(ex.map(one, pairs))


def lru_of(stamps: np.ndarray) -> np.ndarray:
    """Slots in ascending (stamp, slot) order."""
    return np.lexsort((np.arange(stamps.size), stamps)).astype(np.uint16)


def check_metadata(pool: hs.Pool, w, layer, r, pair_state: Pair, t_expected):
    v = pool.views(layer)
    slot_pos = v["slot_pos"][r].cpu().numpy()
    stamps = v["stamps"][r].cpu().numpy()
    lru = v["lru"][r].cpu().numpy()
    pt = v["page_table"][r].cpu().numpy()
    assert np.array_equal(slot_pos, pair_state.slot_pos), (layer, r, "slot_pos")
    assert np.array_equal(stamps, pair_state.stamp), (layer, r, "stamps")
    assert np.array_equal(pt, pair_state.pt), (layer, r, "page_table")
    assert np.array_equal(lru, lru_of(pair_state.stamp)), (layer, r, "lru order")
    assert int(v["resolves"][r]) == t_expected


def check_cache(pool: hs.Pool, w, layer, r, slot_pos: np.ndarray, sample=None):
    """Every occupied slot (or a sample) holds the host record of its position."""
    occ = np.nonzero(slot_pos >= 0)[0]
    if sample is not None and occ.size > sample:
        occ = np.sort(np.random.default_rng(layer * 1000 + r).choice(occ, sample, replace=False))
    if occ.size == 0:
        return
    cache = pool.views(layer)["cache"]
    rows = torch.from_numpy(occ + r * w.slots).cuda()
    got = cache.index_select(0, rows).cpu().numpy()
    want = records.gen(w, r, layer, slot_pos[occ])
    assert np.array_equal(got, want), (layer, r, "cache contents")
