"""The anchor's miss plan (hs_resolve_anchor) and the measurement entry point's
argument checks.

The pages describe the shared layers' miss plans as the anchor's, replayed
("Inference Systems Infrastructure Notes (6): HiSparse", section 4 "Exact
Layer-Wise Prefetching").  The reading built here: a layer that has seen the
same selections as its anchor holds the same slots in the same recency order,
so the pairs the anchor's resolve commits are that layer's plan.  These tests
check that directly -- byte for byte against the plan hs_prefetch_plan
computes from the shared layer's own metadata -- and check rejected requests
and bad arguments.
"""
import numpy as np
import pytest
import torch

from hierarchical_kv_cache_resolve_gb300 import hs
from oracle.oracle import OK, Pair
from tests.gpu_harness import check_cache, check_metadata, fill_selected
from workloads import configs

pytestmark = pytest.mark.gpu


def _shared_trace(w, seed):
    rng = np.random.default_rng(seed)
    sel = np.empty((w.steps, w.n_requests, w.n_layers, w.k), np.int32)
    prev = None
    for t in range(w.steps):
        for r in range(w.n_requests):
            if prev is None:
                s = rng.choice(w.n_positions, w.k, replace=False)
            else:
                keep = rng.choice(prev[r], w.k // 2, replace=False)
                rest = rng.permutation(np.setdiff1d(np.arange(w.n_positions), keep))[: w.k - keep.size]
                s = rng.permutation(np.concatenate([keep, rest]))
            sel[t, r, :] = s
        prev = sel[t, :, 0].copy()
    return sel


def _entries(plan, R, k):
    """[R] of (m, req, pos[m], slot[m]) from a plan buffer."""
    buf = plan.cpu().numpy()
    out = []
    for i in range(R):
        e = buf[16 + i * (16 + 8 * k): 16 + (i + 1) * (16 + 8 * k)].view(np.int32)
        m = int(e[0])
        out.append((m, int(e[1]), e[4: 4 + m].copy(), e[4 + k: 4 + k + m].copy()))
    return out


def test_anchor_plan_equals_the_shared_layers_own_plan():
    w = configs.TINY.with_(n_requests=4, n_layers=3, n_positions=5000, k=96, slots=160,
                           steps=14, layer_anchor=(0, 0, 0))
    sel = _shared_trace(w, seed=5)
    R, k = w.n_requests, w.k
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.empty((3, R, k), dtype=torch.int32, device="cuda")
        anchor_plan = torch.empty(hs.hs_plan_bytes(R, k), dtype=torch.uint8, device="cuda")
        own_plan = torch.empty_like(anchor_plan)
        for t in range(w.steps):
            s = torch.from_numpy(np.ascontiguousarray(sel[t, :, 0])).cuda()
            # layer 1's own plan, from its metadata, before the anchor moves
            pool.prefetch_plan(0, 1, s, own_plan)
            pool.resolve_anchor(0, s, out[0], anchor_plan)
            a, b = _entries(anchor_plan, R, k), _entries(own_plan, R, k)
            for i in range(R):
                assert a[i][0] == b[i][0] and a[i][1] == b[i][1] == i, (t, i)
                assert np.array_equal(a[i][2], b[i][2]) and np.array_equal(a[i][3], b[i][3]), (t, i)
            hdr = anchor_plan[:16].cpu().numpy().view(np.int32)
            assert hdr[1] == R and hdr[2] == k and hdr[3] == 0     # n_req, k, layer
            # the anchor's plan replayed into layers 1 and 2
            for l in (1, 2):
                pool.prefetch_copy(l, R, k, anchor_plan)
                pool.resolve(l, s, out[l], plan=anchor_plan)
            got = out.cpu().numpy()
            assert np.array_equal(got[0], got[1]) and np.array_equal(got[0], got[2])
        for l in (1, 2):
            st = pool.stats(l)
            assert st["plan_mismatches"] == 0 and st["fetched_bytes"] == 0
            assert st["plan_hits"] == st["misses"] > 0
        orc = {r: Pair(w.slots, w.n_positions, w.record_bytes) for r in range(R)}
        for t in range(w.steps):
            for r in range(R):
                assert orc[r].resolve(sel[t, r, 0], out_base=r * w.slots)[0] == OK
        for l in range(3):
            for r in range(R):
                check_metadata(pool, w, l, r, orc[r], w.steps)
                # layer l's slots hold layer l's records
                check_cache(pool, w, l, r, orc[r].slot_pos)


def test_anchor_plan_of_a_rejected_request_is_empty():
    w = configs.TINY.with_(n_requests=3, n_layers=2, n_positions=3000, k=40, slots=64,
                           steps=2, layer_anchor=(0, 0))
    R, k = w.n_requests, w.k
    rng = np.random.default_rng(9)
    sel = np.stack([rng.choice(w.n_positions, k, replace=False) for _ in range(R)]).astype(np.int32)
    sel[1, 5] = sel[1, 4]                       # request 1 repeats a position
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel[None, :, None, :].repeat(2, axis=2))
        out = torch.empty((2, R, k), dtype=torch.int32, device="cuda")
        plan = torch.full((hs.hs_plan_bytes(R, k),), 0x7F, dtype=torch.uint8, device="cuda")
        s = torch.from_numpy(sel).cuda()
        pool.resolve_anchor(0, s, out[0], plan)
        e = _entries(plan, R, k)
        assert e[1][0] == 0 and e[1][1] == 1
        assert e[0][0] == k and e[2][0] == k    # cold start: every position misses
        pool.prefetch_copy(1, R, k, plan)
        pool.resolve(1, s, out[1], plan=plan)
        got = out.cpu().numpy()
        assert (got[:, 1] == -1).all()
        st = pool.stats(check=False)
        assert st["status"] & hs.HS_STATUS_POS_DUP
        assert pool.stats(1, check=False)["plan_mismatches"] == 0


def test_measure_and_anchor_argument_checks():
    w = configs.TINY.with_(n_requests=2, n_layers=1, k=32, slots=64)
    with hs.Pool.for_workload(w) as pool:
        s = torch.zeros((2, 32), dtype=torch.int32, device="cuda")
        out = torch.empty_like(s)
        times = torch.zeros((2, hs.hs_measure_stamp_slots()), dtype=torch.int64, device="cuda")
        for bad in (dict(flags=2), dict(flags=-1)):
            with pytest.raises(hs.HsError) as e:
                pool.resolve_measure(0, s, out, **bad)
            assert e.value.code == hs.HS_ERR_INVALID_ARG
        with pytest.raises(hs.HsError) as e:
            hs.hs_resolve_measure(pool.handle, 0, 2, None, s, 32, out, 0, times.data_ptr() + 4)
        assert e.value.code == hs.HS_ERR_INVALID_ARG
        plan = torch.empty(hs.hs_plan_bytes(2, 32) + 16, dtype=torch.uint8, device="cuda")
        for addr in (None, plan.data_ptr() + 8):
            with pytest.raises(hs.HsError) as e:
                hs.hs_resolve_anchor(pool.handle, 0, 2, None, s, 32, out, addr)
            assert e.value.code == hs.HS_ERR_INVALID_ARG
        assert hs.hs_measure_stamp_slots() == 8 * 16
        torch.cuda.synchronize()
        assert pool.stats()["resolves"] == 0      # nothing was enqueued
