"""The measurement variants of the resolve (hs_resolve_measure) against the
CPU oracle.

Without the fetch (HS_MEASURE_NO_FETCH) every metadata step must still give
the oracle's published slots, page tables, slot maps, stamps, LRU orders and
hit / miss counts, with no byte fetched; with stage timestamps the resolve
must give exactly the plain resolve's results (slot contents included) and
stamps in the order the kernel's stages run.
"""
import numpy as np
import pytest
import torch

from hierarchical_kv_cache_resolve_gb300 import hs
from tests.gpu_harness import OracleRun, check_cache, check_metadata, device_trace, fill_selected
from workloads import configs, traces

pytestmark = pytest.mark.gpu

W_SMALL = configs.DSA_MLA.with_(n_requests=5, n_layers=2, n_positions=24000, k=512, slots=1024,
                                steps=10, local_window=1000)


def _run(w, flags, with_times):
    sel = traces.generate(w)
    T, R, NL, k = sel.shape
    orc = OracleRun(w)
    stamps = []
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        dsel = device_trace(sel)
        out = torch.empty((NL, R, k), dtype=torch.int32, device="cuda")
        slots = hs.hs_measure_stamp_slots()
        for t in range(T):
            for l in range(NL):
                times = None
                if with_times:
                    times = torch.zeros((R, slots), dtype=torch.int64, device="cuda")
                pool.resolve_measure(l, dsel[t, l], out[l], flags=flags, times=times)
                if with_times:
                    stamps.append(times.cpu().numpy().reshape(R, 8, 16))
            res = orc.step(sel[t])
            got = out.cpu().numpy()
            for (r, l), (o, m) in res.items():
                assert np.array_equal(got[l, r], o), (t, r, l)
        for (r, l), p in orc.state.items():
            check_metadata(pool, w, l, r, p, T)
            if not flags & hs.HS_MEASURE_NO_FETCH:
                check_cache(pool, w, l, r, p.slot_pos)
        for l in range(NL):
            st = pool.stats(l)
            ps = [orc.state[(r, l)] for r in range(R)]
            assert st["resolves"] == T * R and st["status"] == 0
            assert st["hits"] == sum(p.hits for p in ps)
            assert st["misses"] == sum(p.misses for p in ps)
            if flags & hs.HS_MEASURE_NO_FETCH:
                assert st["fetched_bytes"] == 0
            else:
                assert st["fetched_bytes"] == sum(p.fetched_bytes for p in ps)
    return stamps


def test_no_fetch_metadata_equals_oracle():
    _run(W_SMALL, hs.HS_MEASURE_NO_FETCH, with_times=False)


def test_no_fetch_single_cta_per_request():
    """More requests than a wave of 2-CTA clusters: the cluster size drops
    and the leader alone runs every step (no fetch either way)."""
    _run(W_SMALL.with_(n_requests=90, n_positions=6000, k=128, slots=256, steps=4,
                       local_window=400), hs.HS_MEASURE_NO_FETCH, with_times=False)


def test_stamps_keep_results_and_order_stages():
    S = hs.HS_STAMP
    stamps = _run(W_SMALL, 0, with_times=True)
    R = W_SMALL.n_requests
    # the cluster size the pool chose: the CTAs that stamped an entry
    C = 1
    while C < 8 and stamps[0][0, C, S["ENTRY"]] > 0:
        C += 1
    assert C == 7   # 5 requests with launch overlap: clusters of 7
    for a in stamps:
        for r in range(R):
            ld = a[r, 0]
            assert ld[S["ATTEMPTS"]] >= 1
            seq = [ld[S[x]] for x in ("ENTRY", "LOADED", "HASHED", "PROBED", "DECIDED", "CHECKED",
                                      "VERDICT", "COMMITTED", "EXIT")]
            assert all(x > 0 for x in seq) and seq == sorted(seq), seq
            for c in range(1, C):
                f = a[r, c]
                seq = [f[S[x]] for x in ("ENTRY", "F_ISSUED", "F_WAITED", "VERDICT", "F_LANDED",
                                         "F_STORED", "EXIT")]
                assert all(x > 0 for x in seq) and seq == sorted(seq), (c, seq)
            for c in range(C, 8):
                assert not a[r, c].any()


def test_stamps_without_fetch():
    stamps = _run(W_SMALL.with_(steps=4), hs.HS_MEASURE_NO_FETCH, with_times=True)
    S = hs.HS_STAMP
    for a in stamps:
        for r in range(W_SMALL.n_requests):
            ld = a[r, 0]
            assert ld[S["ENTRY"]] <= ld[S["DECIDED"]] <= ld[S["COMMITTED"]] <= ld[S["EXIT"]]
            assert a[r, 1, S["F_LANDED"]] == 0   # followers move nothing
