"""Edge cases of the GPU path, each against the CPU oracle or a fixed fact."""
import numpy as np
import pytest
import torch

from hierarchical_kv_cache_resolve_gb300 import hs
from oracle.oracle import OK, Pair
from tests.gpu_harness import check_cache, check_metadata, fill_selected
from workloads import configs, records, traces

pytestmark = pytest.mark.gpu


def _small(**kw):
    base = dict(n_requests=3, n_layers=2, n_positions=3000, record_bytes=144, slots=96,
                k=40, steps=10)
    base.update(kw)
    return configs.TINY.with_(**base)


def _random_trace(w, seed=0):
    rng = np.random.default_rng(seed)
    sel = np.empty((w.steps, w.n_requests, w.n_layers, w.k), np.int32)
    for t in range(w.steps):
        for r in range(w.n_requests):
            for l in range(w.n_layers):
                sel[t, r, l] = rng.choice(w.n_positions, w.k, replace=False)
    return sel


def _oracles(w):
    return {(r, l): Pair(w.slots, w.n_positions, w.record_bytes)
            for r in range(w.n_requests) for l in range(w.n_layers)}


def test_bad_positions_abort_only_their_request():
    w = _small()
    sel = _random_trace(w)
    orc = _oracles(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.empty((w.n_requests, w.k), dtype=torch.int32, device="cuda")
        for t in range(3):
            s = torch.from_numpy(np.ascontiguousarray(sel[t, :, 0])).cuda()
            pool.resolve(0, s, out)
            for r in range(w.n_requests):
                orc[(r, 0)].resolve(sel[t, r, 0], out_base=r * w.slots)
        before = {r: (pool.views(0)["slot_pos"][r].cpu().numpy(),
                      pool.views(0)["page_table"][r].cpu().numpy()) for r in range(w.n_requests)}
        for bad, bit in (("dup", hs.HS_STATUS_POS_DUP), ("range", hs.HS_STATUS_POS_RANGE),
                         ("neg", hs.HS_STATUS_POS_RANGE)):
            s = sel[3, :, 0].copy()
            if bad == "dup":
                s[1, 7] = s[1, 3]
            elif bad == "range":
                s[1, 0] = w.n_positions
            else:
                s[1, 5] = -3
            pool.resolve(0, torch.from_numpy(s).cuda(), out)
            st = pool.stats(0, check=False)
            assert st["rc"] == hs.HS_ERR_DEVICE_INPUT and st["status"] & bit
            got = out.cpu().numpy()
            assert (got[1] == -1).all()
            for r in (0, 2):
                rc, o, _ = orc[(r, 0)].resolve(s[r], out_base=r * w.slots)
                assert rc == OK and np.array_equal(got[r], o)
            assert np.array_equal(pool.views(0)["slot_pos"][1].cpu().numpy(), before[1][0])
            assert np.array_equal(pool.views(0)["page_table"][1].cpu().numpy(), before[1][1])
        assert pool.stats(0)["status"] == 0   # cleared by the previous read
        for r in range(w.n_requests):
            check_metadata(pool, w, 0, r, orc[(r, 0)], int(orc[(r, 0)].t[0]))


def test_bad_request_ids_and_empty_call():
    w = _small()
    sel = _random_trace(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.full((2, w.k), 7, dtype=torch.int32, device="cuda")
        ids = torch.tensor([2, w.n_requests], dtype=torch.int32, device="cuda")
        s = torch.from_numpy(np.ascontiguousarray(sel[0, [2, 0], 1])).cuda()
        pool.resolve(1, s, out, req_ids=ids)
        st = pool.stats(1, check=False)
        assert st["status"] & hs.HS_STATUS_REQ_RANGE
        got = out.cpu().numpy()
        assert (got[1] == -1).all()
        p = Pair(w.slots, w.n_positions, w.record_bytes)
        rc, o, _ = p.resolve(sel[0, 2, 1], out_base=2 * w.slots)
        assert np.array_equal(got[0], o)
        # n_req = 0 enqueues nothing
        hs.hs_resolve(pool.handle, 1, 0, None, s, w.k, out)
        assert pool.stats(1)["resolves"] == 1


def test_request_resolved_twice_in_one_launch_is_detected():
    """Two rows naming the same request race for it: one claims the pair and
    resolves it, the other is refused (-1, HS_STATUS_REQ_BUSY) and changes
    nothing."""
    w = _small(n_requests=2, n_layers=1, k=200, slots=400, n_positions=20000, steps=1)
    sel = _random_trace(w, seed=9)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        one = np.ascontiguousarray(sel[0, 1, 0])
        s = torch.from_numpy(np.stack([one, one])).cuda()
        ids = torch.tensor([1, 1], dtype=torch.int32, device="cuda")
        out = torch.empty((2, w.k), dtype=torch.int32, device="cuda")
        pool.resolve(0, s, out, req_ids=ids)
        st = pool.stats(0, check=False)
        got = out.cpu().numpy()
        refused = [i for i in range(2) if (got[i] == -1).all()]
        p = Pair(w.slots, w.n_positions, w.record_bytes)
        _, want, _ = p.resolve(one, out_base=1 * w.slots)
        if st["status"] & hs.HS_STATUS_REQ_BUSY:
            assert len(refused) == 1
            assert np.array_equal(got[1 - refused[0]], want)
            assert st["resolves"] == 1
            check_metadata(pool, w, 0, 1, p, 1)
        else:
            # the two clusters did not overlap in time: both ran, one after
            # the other, and the second found every position resident
            assert not refused and st["resolves"] == 2
            assert st["misses"] == w.k and st["hits"] == w.k


def test_permuted_request_subsets():
    w = _small(n_requests=6, steps=12)
    sel = _random_trace(w, seed=5)
    orc = _oracles(w)
    rng = np.random.default_rng(11)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        for t in range(w.steps):
            for l in range(w.n_layers):
                ids = rng.permutation(w.n_requests)[: rng.integers(1, w.n_requests + 1)]
                s = torch.from_numpy(np.ascontiguousarray(sel[t, ids, l])).cuda()
                out = torch.empty((ids.size, w.k), dtype=torch.int32, device="cuda")
                pool.resolve(l, s, out, req_ids=torch.from_numpy(ids.astype(np.int32)).cuda())
                got = out.cpu().numpy()
                for i, r in enumerate(ids):
                    rc, o, _ = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)
                    assert rc == OK and np.array_equal(got[i], o)
        for (r, l), p in orc.items():
            check_metadata(pool, w, l, r, p, int(p.t[0]))
            check_cache(pool, w, l, r, p.slot_pos)


@pytest.mark.parametrize("shape", [dict(k=96, slots=96), dict(k=1, slots=96),
                                   dict(k=40, slots=64, n_positions=50),
                                   dict(k=33, slots=33, record_bytes=16),
                                   dict(k=64, slots=200, record_bytes=4096)])
def test_shapes(shape):
    w = _small(**shape)
    sel = _random_trace(w, seed=3)
    orc = _oracles(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.empty((w.n_requests, w.k), dtype=torch.int32, device="cuda")
        for t in range(w.steps):
            for l in range(w.n_layers):
                pool.resolve(l, torch.from_numpy(np.ascontiguousarray(sel[t, :, l])).cuda(), out)
                got = out.cpu().numpy()
                for r in range(w.n_requests):
                    rc, o, _ = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)
                    assert rc == OK and np.array_equal(got[r], o)
        for (r, l), p in orc.items():
            check_metadata(pool, w, l, r, p, w.steps)
            check_cache(pool, w, l, r, p.slot_pos)
        if w.slots >= w.n_positions:
            # the cache holds the whole context: no record is ever evicted
            assert pool.stats()["misses"] == sum(
                len(np.unique(sel[:, r, l])) for r in range(w.n_requests)
                for l in range(w.n_layers))


@pytest.mark.parametrize("overlap", [hs.HS_OVERLAP_ON, hs.HS_OVERLAP_OFF])
@pytest.mark.parametrize("cluster", ["1", "2", "3", "4", "5", "7", "8"])
def test_every_cluster_size(cluster, overlap, monkeypatch):
    """Leader-only (1 CTA) and 1 to 7 followers give the same result, with
    launch overlap and without it (then the leader also fetches the misses
    of its own share of the selection)."""
    monkeypatch.setenv("HS_CLUSTER", cluster)
    w = _small(n_requests=4, k=300, slots=512, n_positions=5000, steps=12)
    sel = _random_trace(w, seed=17)
    # give consecutive steps some overlap so that hits, misses and evictions mix
    for t in range(1, w.steps):
        sel[t, :, :, :150] = sel[t - 1, :, :, 150:]
        for r in range(w.n_requests):
            for l in range(w.n_layers):
                keep = set(sel[t, r, l, :150].tolist())
                fresh = [p for p in np.random.default_rng(t * 97 + r).permutation(w.n_positions)
                         if p not in keep][:150]
                sel[t, r, l, 150:] = fresh
    orc = _oracles(w)
    with hs.Pool.for_workload(w, launch_overlap=overlap) as pool:
        assert pool.info()["launch_overlap"] == overlap
        fill_selected(pool, w, sel)
        out = torch.empty((w.n_requests, w.k), dtype=torch.int32, device="cuda")
        for t in range(w.steps):
            for l in range(w.n_layers):
                pool.resolve(l, torch.from_numpy(np.ascontiguousarray(sel[t, :, l])).cuda(), out)
                got = out.cpu().numpy()
                for r in range(w.n_requests):
                    rc, o, _ = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)
                    assert rc == OK and np.array_equal(got[r], o), (cluster, t, r, l)
        for (r, l), p in orc.items():
            check_metadata(pool, w, l, r, p, w.steps)
            check_cache(pool, w, l, r, p.slot_pos)


def test_largest_supported_slots_and_rejection():
    w = _small(n_requests=2, n_layers=1, k=2048, slots=11000, n_positions=60000,
               record_bytes=64, steps=6)
    sel = _random_trace(w, seed=8)
    orc = _oracles(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.empty((w.n_requests, w.k), dtype=torch.int32, device="cuda")
        for t in range(w.steps):
            pool.resolve(0, torch.from_numpy(np.ascontiguousarray(sel[t, :, 0])).cuda(), out)
            got = out.cpu().numpy()
            for r in range(w.n_requests):
                rc, o, _ = orc[(r, 0)].resolve(sel[t, r, 0], out_base=r * w.slots)
                assert np.array_equal(got[r], o)
        for r in range(w.n_requests):
            check_metadata(pool, w, 0, r, orc[(r, 0)], w.steps)
    with pytest.raises(hs.HsError) as e:
        hs.Pool(1, 1, 100000, 64, 30000, 2048)
    assert e.value.code == hs.HS_ERR_UNSUPPORTED


def _run_group(pool, w, sel, plan_fn):
    """Layer 0 anchors layers 1 and 2; plan_fn(t, layer, plan tensor) may
    corrupt the plan between plan and copy."""
    R, k = w.n_requests, w.k
    out = torch.empty((3, R, k), dtype=torch.int32, device="cuda")
    plan = torch.empty(hs.hs_plan_bytes(R, k), dtype=torch.uint8, device="cuda")
    res = []
    for t in range(w.steps):
        s = torch.from_numpy(np.ascontiguousarray(sel[t, :, 0])).cuda()
        pool.resolve(0, s, out[0])
        for l in (1, 2):
            if plan_fn is not None:
                pool.prefetch_plan(0, l, s, plan)
                plan_fn(t, l, plan)
                pool.prefetch_copy(l, R, k, plan)
                pool.resolve(l, s, out[l], plan=plan)
            else:
                pool.resolve(l, s, out[l])
        res.append(out.cpu().numpy().copy())
    return res


def test_corrupted_plans_stay_exact():
    w = _small(n_layers=3, layer_anchor=(0, 0, 0), steps=16, k=48, slots=64)
    sel = _random_trace(w, seed=21)
    for l in (1, 2):
        sel[:, :, l] = sel[:, :, 0]
    rng = np.random.default_rng(4)
    R, k = w.n_requests, w.k
    entry = 16 + 8 * k

    def corrupt(t, l, plan):
        buf = plan.cpu().numpy()
        kind = (t + l) % 5
        for i in range(R):
            e = buf[16 + i * entry: 16 + (i + 1) * entry].view(np.int32)
            m = int(e[0])
            pos, slot = e[4: 4 + k], e[4 + k: 4 + 2 * k]
            if kind == 0 and m > 1:
                slot[:m] = np.roll(slot[:m], 1)
            elif kind == 1:
                e[0] = m // 2
            elif kind == 2:
                e[0] = k
                pos[:] = rng.integers(0, w.n_positions, k)
                slot[:] = rng.integers(0, w.slots, k)
            elif kind == 3 and m > 0:
                slot[0] = w.slots + 5          # invalid pair: flagged, never written
        if kind == 4:
            buf[12:16] = np.array([7], np.int32).view(np.uint8)   # wrong layer in header
        plan.copy_(torch.from_numpy(buf))

    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        base = _run_group(pool, w, sel, None)
        meta = {(r, l): (pool.views(l)["slot_pos"][r].cpu().numpy(),
                         pool.views(l)["page_table"][r].cpu().numpy(),
                         pool.views(l)["stamps"][r].cpu().numpy())
                for r in range(R) for l in range(3)}
        pool.reset()
        st = pool.stats()
        assert st["resolves"] == 0 and st["misses"] == 0
        pre = _run_group(pool, w, sel, corrupt)
        for a, b in zip(base, pre):
            assert np.array_equal(a, b)
        for (r, l), (sp, pt, stamps) in meta.items():
            assert np.array_equal(pool.views(l)["slot_pos"][r].cpu().numpy(), sp)
            assert np.array_equal(pool.views(l)["page_table"][r].cpu().numpy(), pt)
            assert np.array_equal(pool.views(l)["stamps"][r].cpu().numpy(), stamps)
            check_cache(pool, w, l, r, sp)
        st = pool.stats(check=False)
        assert st["plan_mismatches"] > 0 and st["status"] & hs.HS_STATUS_PLAN


def test_anchor_plan_replayed_into_a_diverged_layer_stays_exact():
    """The anchor's miss plan replayed into two layers that share its
    selection, one of which is given its own selection at a few steps, so
    its history (and from then on its misses and victims) differs from the
    anchor's: the copy writes slots that layer does not want, the consuming
    resolve re-fetches what does not match and refills what the copy
    overwrote, and every output, slot map, page table and slot content is
    the oracle's.  The layer that keeps the anchor's history matches every
    plan pair."""
    w = _small(n_layers=3, layer_anchor=(0, 0, 0), steps=16, k=48, slots=64)
    sel = _random_trace(w, seed=23)
    own = sel[:, :, 2].copy()
    sel[:, :, 1] = sel[:, :, 0]
    sel[:, :, 2] = sel[:, :, 0]
    for t in (5, 6, 11):
        sel[t, :, 2] = own[t]
    R, k = w.n_requests, w.k
    orc = _oracles(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.empty((3, R, k), dtype=torch.int32, device="cuda")
        plan = torch.empty(hs.hs_plan_bytes(R, k), dtype=torch.uint8, device="cuda")
        side = torch.cuda.Stream()
        main = torch.cuda.current_stream()
        for t in range(w.steps):
            s = [torch.from_numpy(np.ascontiguousarray(sel[t, :, l])).cuda() for l in range(3)]
            pool.resolve_anchor(0, s[0], out[0], plan)
            for l in (1, 2):
                ev = torch.cuda.Event()
                ev.record(main)
                side.wait_event(ev)
                pool.prefetch_copy(l, R, k, plan, stream=side)
                ev2 = torch.cuda.Event()
                ev2.record(side)
                main.wait_event(ev2)
                pool.resolve(l, s[l], out[l], plan=plan)
            got = out.cpu().numpy()
            for l in range(3):
                for r in range(R):
                    want = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)[1]
                    assert np.array_equal(got[l, r], want), (t, l, r)
        for (r, l), p in orc.items():
            check_metadata(pool, w, l, r, p, w.steps)
            check_cache(pool, w, l, r, p.slot_pos)
        s1, s2 = pool.stats(1), pool.stats(2)
        assert s1["status"] == 0 and s2["status"] == 0
        assert s1["plan_mismatches"] == 0 and s1["plan_hits"] == s1["misses"]
        assert s1["fetched_bytes"] == 0
        assert s2["plan_mismatches"] > 0 and s2["fetched_bytes"] > 0


def test_cuda_graph_replay_matches_oracle():
    w = configs.DSA_MLA.with_(n_requests=4, n_positions=20000, steps=20)
    from workloads import traces
    sel = traces.generate(w)
    orc = _oracles(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        static_sel = torch.empty((w.n_layers, w.n_requests, w.k), dtype=torch.int32,
                                 device="cuda")
        out = torch.empty_like(static_sel)
        dsel = torch.from_numpy(np.ascontiguousarray(sel.transpose(0, 2, 1, 3))).cuda()
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        static_sel.copy_(dsel[0])
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for l in range(w.n_layers):
                pool.resolve(l, static_sel[l], out[l], stream=s)
        # capture records without running: the pool is still empty
        assert pool.stats()["resolves"] == 0
        for t in range(w.steps):
            static_sel.copy_(dsel[t])
            g.replay()
            got = out.cpu().numpy()
            for (r, l), p in orc.items():
                rc, o, _ = p.resolve(sel[t, r, l], out_base=r * w.slots)
                assert np.array_equal(got[l, r], o)
        for (r, l), p in orc.items():
            check_metadata(pool, w, l, r, p, w.steps)
            check_cache(pool, w, l, r, p.slot_pos, sample=256)


def test_pools_of_different_sizes_coexist():
    """A small pool created after a large one must not shrink the large
    pool's launch limits."""
    big = _small(n_requests=2, n_layers=1, k=2048, slots=4096, n_positions=20000,
                 record_bytes=64, steps=3)
    small = _small(n_requests=2, n_layers=1, k=16, slots=32, n_positions=500, steps=3)
    sel_b, sel_s = _random_trace(big, seed=1), _random_trace(small, seed=2)
    with hs.Pool.for_workload(big) as pb, hs.Pool.for_workload(small) as ps:
        fill_selected(pb, big, sel_b)
        fill_selected(ps, small, sel_s)
        ob = torch.empty((2, big.k), dtype=torch.int32, device="cuda")
        os_ = torch.empty((2, small.k), dtype=torch.int32, device="cuda")
        orc_b, orc_s = _oracles(big), _oracles(small)
        for t in range(3):
            pb.resolve(0, torch.from_numpy(np.ascontiguousarray(sel_b[t, :, 0])).cuda(), ob)
            ps.resolve(0, torch.from_numpy(np.ascontiguousarray(sel_s[t, :, 0])).cuda(), os_)
            gb, gs = ob.cpu().numpy(), os_.cpu().numpy()
            for r in range(2):
                assert np.array_equal(gb[r], orc_b[(r, 0)].resolve(sel_b[t, r, 0], out_base=r * big.slots)[1])
                assert np.array_equal(gs[r], orc_s[(r, 0)].resolve(sel_s[t, r, 0], out_base=r * small.slots)[1])


@pytest.mark.parametrize("kind", [hs.HS_HOST_ALLOC_PINNED, hs.HS_HOST_ALLOC_VMM_NUMA,
                                  hs.HS_HOST_ALLOC_THP_REGISTERED])
def test_link_probe_reports_bandwidth(kind):
    h2d, gather = hs.hs_link_probe(256 << 20, reps=3, record_bytes=1152, host_alloc=kind)
    assert h2d > 1.0 and gather > 1.0


def _thread_mempolicy():
    """The calling thread's NUMA policy mode (get_mempolicy), None where
    the syscall is unknown."""
    import ctypes
    import os
    nr = {"aarch64": 236, "x86_64": 239}.get(os.uname().machine)
    if nr is None:
        return None
    mode = ctypes.c_int(-1)
    mask = (ctypes.c_ulong * 16)()
    libc = ctypes.CDLL(None, use_errno=True)
    if libc.syscall(ctypes.c_long(nr), ctypes.byref(mode), mask, ctypes.c_ulong(1025),
                    None, ctypes.c_ulong(0)) != 0:
        return None
    return mode.value, tuple(mask)


@pytest.mark.parametrize("kind", [hs.HS_HOST_ALLOC_PINNED, hs.HS_HOST_ALLOC_VMM_NUMA,
                                  hs.HS_HOST_ALLOC_THP_REGISTERED])
def test_pool_with_each_host_allocation(kind):
    """Both host allocations hold the records the kernels fetch: the same
    trace gives the oracle's slots and slot contents either way."""
    w = configs.TINY.with_(n_requests=3, n_layers=2, steps=12)
    sel = traces.generate(w)
    orc = _oracles(w)
    policy = _thread_mempolicy()
    with hs.Pool.for_workload(w, host_alloc=kind) as pool:
        # the pool is placed on the device's node; the caller's policy is back
        assert _thread_mempolicy() == policy
        info = pool.info()
        assert info["host_alloc"] == kind
        assert info["launch_overlap"] == hs.HS_OVERLAP_ON   # a small pool overlaps by default
        assert info["warmup_us"] == 0
        assert info["host_bytes"] == w.host_bytes and info["host_mapped_bytes"] >= w.host_bytes
        if kind == hs.HS_HOST_ALLOC_VMM_NUMA and info["device_numa"] >= 0 \
                and info["host_numa_first"] >= 0:
            assert info["host_numa_first"] == info["device_numa"]
        fill_selected(pool, w, sel)
        # touch some records, then warm the whole pool: the warm-up resolves
        # synthetic steps and leaves the pool as created
        pool.touch(1, 0)
        pool.touch(-1, 1)
        pool.touch(2, -1)
        pool.warm()
        assert pool.info()["warmup_us"] > 0
        st = pool.stats()
        assert st["resolves"] == 0 and st["misses"] == 0 and st["status"] == 0
        for l in range(w.n_layers):
            v = pool.views(l)
            assert (v["slot_pos"] == -1).all() and (v["page_table"] == -1).all()
            assert (v["resolves"] == 0).all()
        out = torch.empty((w.n_requests, w.k), dtype=torch.int32, device="cuda")
        for t in range(w.steps):
            for l in range(w.n_layers):
                pool.resolve(l, torch.from_numpy(np.ascontiguousarray(sel[t, :, l])).cuda(), out)
                got = out.cpu().numpy()
                for r in range(w.n_requests):
                    want = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)[1]
                    assert np.array_equal(got[r], want), (t, r, l)
        for (r, l), p in orc.items():
            check_cache(pool, w, l, r, p.slot_pos)


def test_host_records_layout():
    w = _small()
    with hs.Pool.for_workload(w) as pool:
        a = pool.host_records(1, 1)
        assert a.shape == (w.n_positions, w.record_bytes)
        per = w.n_positions * w.record_bytes
        # layer-major, host[l][r][pos][W]: a layer's requests are adjacent
        assert pool.host_records(2, 1).ctypes.data - a.ctypes.data == per
        assert a.ctypes.data - pool.host_records(1, 0).ctypes.data == w.n_requests * per
        assert pool.host_records(0, 0).ctypes.data + w.n_layers * w.n_requests * per == \
            pool.host_records(w.n_requests - 1, w.n_layers - 1).ctypes.data + per
        a[:] = records.gen(w, 1, 1, np.arange(w.n_positions))
        assert np.array_equal(pool.host_records(1, 1)[17], records.gen(w, 1, 1, [17])[0])


@pytest.mark.parametrize("cluster", ["1", "4", ""])
@pytest.mark.parametrize("tight", [False, True])
@pytest.mark.parametrize("overlap", [hs.HS_OVERLAP_ON, hs.HS_OVERLAP_OFF])
def test_back_to_back_resolves_of_one_layer(cluster, tight, overlap, monkeypatch):
    """Many resolves of the same pairs enqueued back to back with no host
    synchronisation.  Each launch starts while the previous one still runs
    and decides on metadata that launch is about to change; the decision
    must be found stale and taken again, so every step's published slots,
    the final metadata and the slot contents equal the oracle's.  With
    B = k every slot that is not selected is evicted at every step."""
    monkeypatch.setenv("HS_CLUSTER", cluster)
    from workloads import traces
    w = configs.DSA_MLA.with_(n_requests=3, n_layers=1, n_positions=12000, k=256,
                              slots=256 if tight else 512, steps=30, local_window=600)
    sel = traces.generate(w)
    orc = _oracles(w)
    with hs.Pool.for_workload(w, launch_overlap=overlap) as pool:
        fill_selected(pool, w, sel)
        dsel = torch.from_numpy(np.ascontiguousarray(sel[:, :, 0])).cuda()   # [T][R][k]
        out = torch.empty((w.steps, w.n_requests, w.k), dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        for t in range(w.steps):
            pool.resolve(0, dsel[t], out[t])
        got = out.cpu().numpy()
        misses = 0
        for t in range(w.steps):
            for r in range(w.n_requests):
                rc, o, m = orc[(r, 0)].resolve(sel[t, r, 0], out_base=r * w.slots)
                assert rc == OK and np.array_equal(got[t, r], o), (t, r)
                misses += m
        st = pool.stats(0)
        assert st["resolves"] == w.steps * w.n_requests and st["misses"] == misses
        for r in range(w.n_requests):
            check_metadata(pool, w, 0, r, orc[(r, 0)], w.steps)
            check_cache(pool, w, 0, r, orc[(r, 0)].slot_pos)


def test_interleaved_layers_without_synchronisation():
    """Launch orders that alternate layers and repeat them (0 0 1 0 1 1 ...)
    with no host synchronisation: overlapping launches of other layers keep
    their early decisions, those of the same layer take them again."""
    from workloads import traces
    w = configs.DSA_MLA.with_(n_requests=2, n_layers=2, n_positions=10000, k=192, slots=384,
                              steps=24, local_window=500)
    sel = traces.generate(w)
    orc = _oracles(w)
    order = [0, 0, 1, 0, 1, 1]
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        dsel = torch.from_numpy(np.ascontiguousarray(sel.transpose(0, 2, 1, 3))).cuda()
        launches = []   # (t, layer) in launch order; step t of a layer uses sel[t]
        nxt = [0, 0]
        while min(nxt) < w.steps:
            for l in order:
                if nxt[l] < w.steps:
                    launches.append((nxt[l], l))
                    nxt[l] += 1
        out = torch.empty((len(launches), w.n_requests, w.k), dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        for i, (t, l) in enumerate(launches):
            pool.resolve(l, dsel[t, l], out[i])
        got = out.cpu().numpy()
        for i, (t, l) in enumerate(launches):
            for r in range(w.n_requests):
                rc, o, _ = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)
                assert rc == OK and np.array_equal(got[i, r], o), (i, t, r, l)
        for (r, l), p in orc.items():
            check_metadata(pool, w, l, r, p, w.steps)
            check_cache(pool, w, l, r, p.slot_pos)


def test_more_requests_than_one_wave_back_to_back():
    """400 requests (more clusters than the SMs hold at once) over two layers,
    all launches enqueued back to back without synchronisation, against the
    oracle: later waves start while earlier launches still run."""
    w = _small(n_requests=400, n_layers=2, k=48, slots=64, n_positions=900, steps=6,
               record_bytes=64)
    sel = _random_trace(w, seed=21)
    # some reuse between consecutive steps so that hits and evictions mix
    for t in range(1, w.steps):
        sel[t, :, :, :24] = sel[t - 1, :, :, 24:]
        rng = np.random.default_rng(t)
        for r in range(w.n_requests):
            for l in range(w.n_layers):
                keep = set(sel[t, r, l, :24].tolist())
                fresh = [p for p in rng.permutation(w.n_positions) if p not in keep][:24]
                sel[t, r, l, 24:] = fresh
    orc = _oracles(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        dsel = torch.from_numpy(np.ascontiguousarray(sel.transpose(0, 2, 1, 3))).cuda()
        out = torch.empty((w.steps, w.n_layers, w.n_requests, w.k), dtype=torch.int32,
                          device="cuda")
        torch.cuda.synchronize()
        for t in range(w.steps):
            for l in range(w.n_layers):
                pool.resolve(l, dsel[t, l], out[t, l])
        got = out.cpu().numpy()
        for t in range(w.steps):
            for l in range(w.n_layers):
                for r in range(w.n_requests):
                    rc, o, _ = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)
                    assert rc == OK and np.array_equal(got[t, l, r], o), (t, l, r)
        for (r, l), p in list(orc.items())[::37]:
            check_metadata(pool, w, l, r, p, w.steps)
            check_cache(pool, w, l, r, p.slot_pos)
        st = pool.stats()
        assert st["status"] == 0 and st["resolves"] == w.steps * w.n_layers * w.n_requests


def test_permuted_request_subsets_back_to_back():
    """Random subsets and orders of the requests, every launch enqueued
    without synchronisation: each launch decides early over pairs that the
    launch before it may or may not be resolving."""
    w = _small(n_requests=6, n_layers=2, steps=16)
    sel = _random_trace(w, seed=15)
    orc = _oracles(w)
    rng = np.random.default_rng(12)
    plan = []
    for t in range(w.steps):
        for l in range(w.n_layers):
            plan.append((t, l, rng.permutation(w.n_requests)[: rng.integers(1, w.n_requests + 1)]))
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        bufs = []
        for t, l, ids in plan:
            s = torch.from_numpy(np.ascontiguousarray(sel[t, ids, l])).cuda()
            d_ids = torch.from_numpy(ids.astype(np.int32)).cuda()
            bufs.append((s, d_ids, torch.empty((ids.size, w.k), dtype=torch.int32, device="cuda")))
        torch.cuda.synchronize()
        for (t, l, ids), (s, d_ids, out) in zip(plan, bufs):
            pool.resolve(l, s, out, req_ids=d_ids)
        for (t, l, ids), (s, d_ids, out) in zip(plan, bufs):
            got = out.cpu().numpy()
            for i, r in enumerate(ids):
                rc, o, _ = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)
                assert rc == OK and np.array_equal(got[i], o), (t, l, r)
        for (r, l), p in orc.items():
            check_metadata(pool, w, l, r, p, int(p.t[0]))
            check_cache(pool, w, l, r, p.slot_pos)


def test_one_selection_buffer_rewritten_between_resolves():
    """A single device selection buffer, rewritten by a copy kernel before
    every resolve (the static-buffer pattern of captured graphs), with no
    host synchronisation: each resolve sees its own step's selection."""
    from workloads import traces
    w = configs.DSA_MLA.with_(n_requests=3, n_layers=2, n_positions=9000, k=160, slots=320,
                              steps=20, local_window=400)
    sel = traces.generate(w)
    orc = _oracles(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        dsel = torch.from_numpy(np.ascontiguousarray(sel.transpose(0, 2, 1, 3))).cuda()
        static = torch.empty((w.n_requests, w.k), dtype=torch.int32, device="cuda")
        out = torch.empty((w.steps, w.n_layers, w.n_requests, w.k), dtype=torch.int32,
                          device="cuda")
        torch.cuda.synchronize()
        for t in range(w.steps):
            for l in range(w.n_layers):
                static.copy_(dsel[t, l])
                pool.resolve(l, static, out[t, l])
        got = out.cpu().numpy()
        for t in range(w.steps):
            for l in range(w.n_layers):
                for r in range(w.n_requests):
                    rc, o, _ = orc[(r, l)].resolve(sel[t, r, l], out_base=r * w.slots)
                    assert rc == OK and np.array_equal(got[t, l, r], o), (t, l, r)
        for (r, l), p in orc.items():
            check_metadata(pool, w, l, r, p, w.steps)
            check_cache(pool, w, l, r, p.slot_pos)
