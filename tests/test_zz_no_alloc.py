"""The allocation-free resolve (hs_resolve_noalloc) against hs_resolve.

hs_resolve_noalloc serves callers that cannot allocate device memory when
they resolve (an engine whose caching allocator owns all free device memory,
or a latency-critical loop where cudaMalloc would synchronise the device):
the caller owns the layer state and the call keeps its scratch in a fixed
array inside the library.  This test drives both entry points through the C
ABI from the same empty state over two calls in a row and requires identical
published slots, metadata and slot contents.  It sorts last so that a run
stopping at the first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

from hierarchical_kv_cache_resolve_gb300 import hs
from tests.gpu_harness import fill_selected
from workloads import configs

pytestmark = pytest.mark.gpu


def _trace(w, seed):
    rng = np.random.default_rng(seed)
    sel = np.empty((w.steps, w.n_requests, 1, w.k), np.int32)
    for t in range(w.steps):
        for r in range(w.n_requests):
            keep = sel[t - 1, r, 0, : w.k // 2] if t else np.zeros(0, np.int32)
            rest = rng.permutation(np.setdiff1d(np.arange(w.n_positions), keep))[: w.k - keep.size]
            sel[t, r, 0] = rng.permutation(np.concatenate([keep, rest]))
    return sel


def _empty_state(w, host_addr):
    R, B, L, W = w.n_requests, w.slots, w.n_positions, w.record_bytes
    dev = "cuda"
    return {
        "n_requests": R, "n_positions": L, "record_bytes": W, "slots": B,
        "host_records": host_addr,
        "cache": torch.zeros((R * B, W), dtype=torch.uint8, device=dev),
        "page_table": torch.full((R, L), -1, dtype=torch.int32, device=dev),
        "slot_pos": torch.full((R, B), -1, dtype=torch.int32, device=dev),
        "stamps": torch.zeros((R, B), dtype=torch.int32, device=dev),
        "lru": torch.arange(B, dtype=torch.int32, device=dev).to(torch.int16).repeat(R, 1),
        "resolves": torch.zeros((R,), dtype=torch.int32, device=dev),
    }


def test_noalloc_matches_pool_resolve_on_two_calls():
    w = configs.TINY.with_(n_requests=3, n_layers=1, n_positions=3000, record_bytes=144,
                           slots=96, k=40, steps=2)
    sel = _trace(w, seed=31)
    R, B, k = w.n_requests, w.slots, w.k
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        # with one layer the pool's host records are [R][L][W], the layout the
        # caller-owned state describes; pinned mapped memory is readable by the
        # GPU at its host address
        state = _empty_state(w, pool.host_records(0, 0).ctypes.data)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out_pool = torch.empty((R, k), dtype=torch.int32, device="cuda")
        out_free = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
        sels = [torch.from_numpy(np.ascontiguousarray(sel[t, :, 0])).cuda() for t in range(2)]
        for t in range(2):
            s = sels[t]
            pool.resolve(0, s, out_pool)
            torch.cuda.synchronize()
            if t == 1:
                # the first call has done the one-time set-up; the second must
                # not change the device's free memory or torch's reserve
                free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
            hs.hs_resolve_noalloc(state, R, None, s, k, out_free, status)
            torch.cuda.synchronize()
            if t == 1:
                assert torch.cuda.mem_get_info()[0] == free0
                assert torch.cuda.memory_reserved() == reserved0
            assert torch.equal(out_pool, out_free), t
            v = pool.views(0)
            assert np.array_equal(v["page_table"].cpu().numpy(), state["page_table"].cpu().numpy())
            assert np.array_equal(v["slot_pos"].cpu().numpy(), state["slot_pos"].cpu().numpy())
            assert np.array_equal(v["stamps"].cpu().numpy().view(np.int32),
                                  state["stamps"].cpu().numpy())
            assert np.array_equal(v["lru"].cpu().numpy().view(np.int16), state["lru"].cpu().numpy())
            assert np.array_equal(v["resolves"].cpu().numpy().view(np.int32),
                                  state["resolves"].cpu().numpy())
            occ = np.nonzero(v["slot_pos"].cpu().numpy().reshape(-1) >= 0)[0]
            rows = torch.from_numpy(occ).cuda()
            assert torch.equal(v["cache"].index_select(0, rows), state["cache"].index_select(0, rows))
        assert int(status.item()) == 0
        assert pool.stats()["resolves"] == 2 * R

        # a rejected request is reported through the caller's status word
        bad = sel[1, :, 0].copy()
        bad[2, 1] = bad[2, 0]
        hs.hs_resolve_noalloc(state, R, None, torch.from_numpy(bad).cuda(), k, out_free, status)
        torch.cuda.synchronize()
        assert int(status.item()) & hs.HS_STATUS_POS_DUP
        assert (out_free[2] == -1).all()

        # misaligned caller pointers: refused before anything is enqueued
        # (the kernel's 16-, 4- and 2-byte accesses would fault on them)
        before = out_free.clone()
        for name, shift in (("cache", 8), ("host_records", 4), ("page_table", 2),
                            ("stamps", 1), ("lru", 1)):
            base = state[name]
            addr = base if isinstance(base, int) else base.data_ptr()
            with pytest.raises(hs.HsError) as e:
                hs.hs_resolve_noalloc(dict(state, **{name: addr + shift}), R, None, s, k,
                                      out_free, status)
            assert e.value.code == hs.HS_ERR_INVALID_ARG, name
        with pytest.raises(hs.HsError) as e:
            hs.hs_resolve_noalloc(state, R, None, s, k, out_free.data_ptr() + 2, status)
        assert e.value.code == hs.HS_ERR_INVALID_ARG
        torch.cuda.synchronize()
        assert torch.equal(out_free, before)

        # more requests than the scratch array holds: refused before any launch
        big = dict(state, n_requests=hs.HS_NOALLOC_MAX_REQUESTS + 1)
        with pytest.raises(hs.HsError) as e:
            hs.hs_resolve_noalloc(big, 1, None, s, k, out_free, status)
        assert e.value.code == hs.HS_ERR_UNSUPPORTED
