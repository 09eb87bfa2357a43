"""GPU path against the CPU oracle, bit for bit, on the five seeded workloads.

Every step: the published slot of every selected entry of every
(request, layer) and the per-layer miss count.  Periodically and at the last
step: page table, slot map, stamps, LRU order and resolve count of every
pair.  At the end: the bytes of every occupied slot (or a fixed sample for
the largest workloads) against the host record of the position it holds,
and the cumulative counters.  The launch configuration is the one the
benchmark times (hs_resolve picks the cluster size from the request count).
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from hierarchical_kv_cache_resolve_gb300 import hs
from tests.gpu_harness import (OracleRun, check_cache, check_metadata, device_trace,
                               fill_selected)
from workloads import configs, traces

pytestmark = pytest.mark.gpu


def _oracle_step(orc: OracleRun, sel_t, pool_ex):
    items = list(orc.state.items())

    def one(item):
        (r, l), p = item
        rc, out, m = p.resolve(sel_t[r, l], out_base=r * orc.w.slots)
        assert rc == 0
        return (r, l), (out, m)

    return dict(pool_ex.map(one, items))


def run_and_compare(w, meta_every=1, cache_sample=None, prefetch=False, sel=None,
                    overlap=hs.HS_OVERLAP_AUTO):
    if sel is None:
        sel = traces.generate(w)
    T, R, NL, k = sel.shape
    orc = OracleRun(w)
    ex = ThreadPoolExecutor(16)
    with hs.Pool.for_workload(w, launch_overlap=overlap) as pool:
        want = overlap if overlap != hs.HS_OVERLAP_AUTO else (
            hs.HS_OVERLAP_ON if w.host_bytes <= 16 << 30 else hs.HS_OVERLAP_OFF)
        assert pool.info()["launch_overlap"] == want
        fill_selected(pool, w, sel)
        dsel = device_trace(sel)
        out = torch.empty((NL, R, k), dtype=torch.int32, device="cuda")
        main = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        plans = {}
        replay = prefetch == "replay"
        if prefetch:
            nb = hs.hs_plan_bytes(R, k)
            for l in range(NL):
                # "plan": one plan per shared layer (hs_prefetch_plan);
                # "replay": one per anchor, written by its resolve
                if (w.anchors[l] != l) != replay:
                    plans[l] = torch.empty(nb, dtype=torch.uint8, device="cuda")
        shared = {l for l in range(NL) if w.anchors[l] != l} if prefetch else set()
        prev = {l: 0 for l in range(NL)}
        for t in range(T):
            for l in range(NL):
                a = w.anchors[l]
                if l in shared:
                    plan = plans[a] if replay else plans[l]
                    if not replay:
                        pool.prefetch_plan(a, l, dsel[t, l], plan, stream=main)
                    ev = torch.cuda.Event()
                    ev.record(main)
                    side.wait_event(ev)
                    pool.prefetch_copy(l, R, k, plan, stream=side)
                    ev2 = torch.cuda.Event()
                    ev2.record(side)
                    main.wait_event(ev2)
                    pool.resolve(l, dsel[t, l], out[l], plan=plan, stream=main)
                elif replay and l in plans:
                    pool.resolve_anchor(l, dsel[t, l], out[l], plans[l], stream=main)
                else:
                    pool.resolve(l, dsel[t, l], out[l], stream=main)
            ores = _oracle_step(orc, sel[t], ex)
            got = out.cpu().numpy()
            for (r, l), (o, m) in ores.items():
                assert np.array_equal(got[l, r], o), (t, r, l)
            for l in range(NL):
                st = pool.stats(l)
                misses = sum(ores[(r, l)][1] for r in range(R))
                assert st["misses"] - prev[l] == misses, (t, l)
                prev[l] = st["misses"]
            if (t % meta_every == 0) or t == T - 1:
                for (r, l), p in orc.state.items():
                    check_metadata(pool, w, l, r, p, t + 1)
        for (r, l), p in orc.state.items():
            check_cache(pool, w, l, r, p.slot_pos, sample=cache_sample)
        for l in range(NL):
            st = pool.stats(l)
            ps = [orc.state[(r, l)] for r in range(R)]
            assert st["resolves"] == T * R
            assert st["hits"] == sum(p.hits for p in ps)
            assert st["misses"] == sum(p.misses for p in ps)
            assert st["status"] == 0
            if l in shared:
                assert st["plan_mismatches"] == 0
                assert st["plan_hits"] == st["misses"]
                assert st["prefetched_bytes"] == st["misses"] * w.record_bytes
                assert st["fetched_bytes"] == 0
            else:
                assert st["fetched_bytes"] == sum(p.fetched_bytes for p in ps)
    ex.shutdown()
    return orc


def test_tiny_every_step():
    run_and_compare(configs.TINY, meta_every=1)


def test_tiny_with_ragged_request_set():
    """Several requests with a k that is not a multiple of the warp size."""
    w = configs.TINY.with_(n_requests=5, n_layers=2, k=45, slots=77, steps=40)
    run_and_compare(w, meta_every=1)


@pytest.mark.slow
def test_dsa_mla_full():
    run_and_compare(configs.DSA_MLA, meta_every=16)


@pytest.mark.slow
def test_no_locality_full():
    run_and_compare(configs.NO_LOCALITY, meta_every=16)


@pytest.mark.slow
def test_quest_pages_full():
    run_and_compare(configs.QUEST_PAGES, meta_every=32, cache_sample=512)


@pytest.mark.slow
def test_quest_page_records_full():
    """Page-granular records (64 KiB per record, k = 128 pages, B = 256)."""
    run_and_compare(configs.QUEST_PAGE_RECORDS, meta_every=32, cache_sample=64)


@pytest.mark.slow
def test_tight_prefetch_full_with_prefetch():
    run_and_compare(configs.TIGHT_PREFETCH, meta_every=32, cache_sample=256, prefetch=True)


@pytest.mark.slow
def test_tight_prefetch_full_with_anchor_replay():
    """The anchor's resolve writes its miss plan; the copy-only kernel
    replays it into the three layers sharing the anchor's selection, whose
    resolves consume it: every plan pair matches, nothing is fetched twice."""
    run_and_compare(configs.TIGHT_PREFETCH, meta_every=32, cache_sample=256, prefetch="replay")


def test_tight_prefetch_small_with_and_without_prefetch():
    w = configs.TIGHT_PREFETCH.with_(n_requests=6, n_positions=20000, k=512, slots=512,
                                     steps=24)
    for overlap in (hs.HS_OVERLAP_ON, hs.HS_OVERLAP_OFF):
        run_and_compare(w, meta_every=4, prefetch=False, overlap=overlap)
        run_and_compare(w, meta_every=4, prefetch=True, overlap=overlap)
        run_and_compare(w, meta_every=4, prefetch="replay", overlap=overlap)


def test_dsa_mla_small_without_overlap():
    """Launch overlap off on an 8-request, 8-CTA-cluster shape: the leader
    fetches the misses of one eighth of each selection."""
    w = configs.DSA_MLA.with_(n_positions=20000, k=1024, slots=2048, steps=16,
                              local_window=1500)
    run_and_compare(w, meta_every=4, overlap=hs.HS_OVERLAP_OFF)


@pytest.mark.slow
def test_dsa_mla_full_as_the_benchmark_runs_it():
    """The benchmark's own launch configuration at full size: one CUDA graph
    of the four layers' resolves per step, replayed step after step with no
    host synchronisation (consecutive launches overlap) and the L2 flushed
    between steps; every step's published slots, then the final metadata
    and sampled slot contents, against the oracle."""
    w = configs.DSA_MLA
    T = 24
    sel = traces.generate(w)[:T]
    R, NL, k = w.n_requests, w.n_layers, w.k
    orc = OracleRun(w)
    ex = ThreadPoolExecutor(16)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        dsel = device_trace(sel)                                   # [T][NL][R][k]
        out = torch.empty((T, NL, R, k), dtype=torch.int32, device="cuda")
        flush = torch.empty(64 << 20, dtype=torch.int32, device="cuda")
        cap = torch.cuda.Stream()
        graphs = []
        for t in range(T):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for l in range(NL):
                    hs.hs_resolve(pool.handle, l, R, None, dsel[t, l], k, out[t, l], None, cap)
            graphs.append(g)
        torch.cuda.synchronize()
        for t in range(T):
            flush.fill_(t)
            graphs[t].replay()
        got = out.cpu().numpy()
        for t in range(T):
            ores = _oracle_step(orc, sel[t], ex)
            for (r, l), (o, m) in ores.items():
                assert np.array_equal(got[t, l, r], o), (t, r, l)
        for (r, l), p in orc.state.items():
            check_metadata(pool, w, l, r, p, T)
            check_cache(pool, w, l, r, p.slot_pos, sample=512)
        st = pool.stats()
        assert st["status"] == 0 and st["resolves"] == T * R * NL
    ex.shutdown()


@pytest.mark.slow
def test_tight_prefetch_full_as_the_benchmark_runs_it():
    """The headline's own launch configuration at full size (64 requests x
    8 layers, 59.2 GB pool, launch overlap off by the pool policy, the
    leader fetching its share): one CUDA graph of the eight layers' resolves
    per step, replayed step after step with no host synchronisation and the
    L2 flushed between steps; every step's published slots, then the final
    metadata and sampled slot contents, against the oracle."""
    w = configs.TIGHT_PREFETCH
    T = 12
    sel = traces.generate(w)[:T]
    R, NL, k = w.n_requests, w.n_layers, w.k
    orc = OracleRun(w)
    ex = ThreadPoolExecutor(16)
    with hs.Pool.for_workload(w) as pool:
        info = pool.info()
        assert info["launch_overlap"] == hs.HS_OVERLAP_OFF
        # past the translation reach the pool takes huge pages when the kernel
        # backs nearly all of it with them; the bench warms it once written
        assert info["host_alloc"] in (hs.HS_HOST_ALLOC_THP_REGISTERED, hs.HS_HOST_ALLOC_PINNED)
        if info["host_alloc"] == hs.HS_HOST_ALLOC_THP_REGISTERED:
            assert info["host_huge_bytes"] >= info["host_mapped_bytes"] // 10 * 9
        fill_selected(pool, w, sel)
        pool.warm()
        dsel = device_trace(sel)
        out = torch.empty((T, NL, R, k), dtype=torch.int32, device="cuda")
        flush = torch.empty(64 << 20, dtype=torch.int32, device="cuda")
        cap = torch.cuda.Stream()
        graphs = []
        for t in range(T):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for l in range(NL):
                    hs.hs_resolve(pool.handle, l, R, None, dsel[t, l], k, out[t, l], None, cap)
            graphs.append(g)
        torch.cuda.synchronize()
        for t in range(T):
            flush.fill_(t)
            graphs[t].replay()
        got = out.cpu().numpy()
        for t in range(T):
            ores = _oracle_step(orc, sel[t], ex)
            for (r, l), (o, m) in ores.items():
                assert np.array_equal(got[t, l, r], o), (t, r, l)
        for (r, l), p in orc.state.items():
            check_metadata(pool, w, l, r, p, T)
            check_cache(pool, w, l, r, p.slot_pos, sample=64)
        st = pool.stats()
        assert st["status"] == 0 and st["resolves"] == T * R * NL
        assert st["fetched_bytes"] == sum(p.fetched_bytes for p in orc.state.values())
    ex.shutdown()


@pytest.mark.parametrize("source", ["plan", "replay"])
def test_tight_prefetch_scheduled_like_the_overlap_benchmark(source):
    """Exact prefetch in the schedule of the overlap benchmark: at each
    anchor the plans and copies of the layers sharing its selection run on a
    side stream, concurrently with the anchor's resolve and with the
    attention and GEMMs of the layers in between; the main stream waits for
    a layer's copy before the GEMM ahead of that layer's plan-consuming
    resolve; no host synchronisation from the first step to the last.  Every
    step's published slots, the final metadata and cache, the counters, and
    the attention each layer ran over its slots (bit-identical to the same
    kernel over the host records of the selection, gathered densely)."""
    from workloads import records

    w = configs.TIGHT_PREFETCH.with_(n_requests=8, n_positions=30000, k=512, slots=512,
                                     steps=12)
    sel = traces.generate(w)
    T, R, NL, k = sel.shape
    heads = 16
    scale = 576 ** -0.5
    orc = OracleRun(w)
    ex = ThreadPoolExecutor(16)
    g = torch.Generator().manual_seed(11)
    q = torch.randn((R, heads, 576), generator=g).to(torch.bfloat16).cuda()
    a = torch.randn((2048, 2048), generator=g).to(torch.bfloat16).cuda()
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        dsel = device_trace(sel)
        out = torch.empty((T, NL, R, k), dtype=torch.int32, device="cuda")
        att = torch.empty((T, NL, R, heads, 512), dtype=torch.float32, device="cuda")
        replay = source == "replay"
        shared = [l for l in range(NL) if w.anchors[l] != l]
        plans = {l: torch.empty(hs.hs_plan_bytes(R, k), dtype=torch.uint8, device="cuda")
                 for l in range(NL) if (w.anchors[l] != l) != replay}
        caches = [pool.views(l)["cache"] for l in range(NL)]
        main, side = torch.cuda.current_stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        for t in range(T):
            evs = {}
            for l in range(NL):
                if w.anchors[l] == l:
                    if replay:
                        # the anchor's resolve writes the plan; the copies
                        # replay it from there on, beside the compute
                        pool.resolve_anchor(l, dsel[t, l], out[t, l], plans[l], stream=main)
                    ready = torch.cuda.Event()
                    ready.record(main)
                    side.wait_event(ready)
                    for l2 in shared:
                        if w.anchors[l2] == l:
                            if not replay:
                                pool.prefetch_plan(l, l2, dsel[t, l2], plans[l2], stream=side)
                            pool.prefetch_copy(l2, R, k, plans[l if replay else l2], stream=side)
                            evs[l2] = torch.cuda.Event()
                            evs[l2].record(side)
                    if not replay:
                        pool.resolve(l, dsel[t, l], out[t, l], stream=main)
                else:
                    pool.resolve(l, dsel[t, l], out[t, l],
                                 plan=plans[w.anchors[l] if replay else l], stream=main)
                hs.hs_sparse_attention(q, caches[l], R * w.slots, out[t, l], R, k, heads,
                                       scale, att[t, l], stream=main)
                if l + 1 in evs:
                    main.wait_event(evs[l + 1])
                a @ a
        torch.cuda.synchronize()
        assert hs.hs_attention_status() == 0
        got = out.cpu().numpy()
        for t in range(T):
            ores = _oracle_step(orc, sel[t], ex)
            for (r, l), (o, m) in ores.items():
                assert np.array_equal(got[t, l, r], o), (t, r, l)
        for (r, l), p in orc.state.items():
            check_metadata(pool, w, l, r, p, T)
            check_cache(pool, w, l, r, p.slot_pos)
        for l in range(NL):
            st = pool.stats(l)
            assert st["status"] == 0 and st["resolves"] == T * R
            if l in shared:
                assert st["plan_mismatches"] == 0 and st["fetched_bytes"] == 0
                assert st["prefetched_bytes"] == st["misses"] * w.record_bytes
        # what each layer's attention read was the selection's records
        idx = torch.arange(R * k, dtype=torch.int32, device="cuda").reshape(R, k)
        ref = torch.empty((R, heads, 512), dtype=torch.float32, device="cuda")
        for t in range(T):
            for l in range(NL):
                host = np.concatenate([records.gen(w, r, l, sel[t, r, l]) for r in range(R)])
                dense = torch.from_numpy(host).cuda()
                hs.hs_sparse_attention(q, dense, R * k, idx, R, k, heads, scale, ref)
                assert torch.equal(att[t, l].view(torch.int32), ref.view(torch.int32)), (t, l)
    ex.shutdown()
