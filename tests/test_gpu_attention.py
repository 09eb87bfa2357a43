"""The sparse attention consumer (hs_sparse_attention) over published slots.

* against the fp64 oracle attention (oracle/attention.py) on the host
  records of the selected positions, per request and head.  Tolerance: the
  kernel rounds the probabilities to bf16 before P V while the normaliser
  sums them unrounded, so each output element is off by at most
  2^-9 * sum_j p_j |V_j| / sum_j p_j <= 2^-9 * max_j |V_j| (plus fp32
  accumulation error, far smaller); the test allows 4x that bound;
* attention over the published slots is bit-identical to attention over the
  same records copied straight from the host pool in selection order -- the
  exactness claim, on the GPU;
* rows outside the cache (a rejected request publishes -1) are masked;
* ragged key counts (one key, a partial pipeline stage, a split boundary),
  several head groups and batch sizes that change the split of the keys;
  repeated calls are bit-identical and raise no status bit.
"""
import numpy as np
import pytest
import torch

from hierarchical_kv_cache_resolve_gb300 import hs
from oracle.attention import sparse_attention
from tests.gpu_harness import fill_selected
from workloads import configs, records

pytestmark = pytest.mark.gpu

SCALE = 1.0 / np.sqrt(576.0)


def _bf16_round(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _bf16_to_f64(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _setup(R=4, k=300, heads=32, steps=2, seed=3):
    w = configs.DSA_MLA.with_(n_requests=R, n_layers=1, n_positions=20000, k=k, slots=512,
                              steps=steps, local_window=2000)
    rng = np.random.default_rng(seed)
    sel = np.stack([np.stack([rng.choice(w.n_positions, k, replace=False)[None] for _ in range(R)])
                    for _ in range(steps)]).astype(np.int32)     # [T][R][1][k]
    q16 = _bf16_round(rng.standard_normal((R, heads, 576)).astype(np.float32))
    return w, sel, q16


def _attend(cache, rows, idx, q16, R, k, heads):
    q = torch.from_numpy(q16.view(np.int16)).cuda()
    out = torch.full((R, heads, 512), float("nan"), dtype=torch.float32, device="cuda")
    hs.hs_sparse_attention(q, cache, rows, idx, R, k, heads, SCALE, out)
    torch.cuda.synchronize()
    assert hs.hs_attention_status() == 0
    return out.cpu().numpy()


def test_attention_matches_fp64_oracle_and_host_gather():
    R, k, heads = 4, 300, 32
    w, sel, q16 = _setup(R, k, heads)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.empty((R, k), dtype=torch.int32, device="cuda")
        for t in range(sel.shape[0]):
            pool.resolve(0, torch.from_numpy(np.ascontiguousarray(sel[t, :, 0])).cuda(), out)
        cache = pool.views(0)["cache"]
        got = _attend(cache, cache.shape[0], out, q16, R, k, heads)
        # the same records gathered from the host pool, in selection order
        host = np.concatenate([records.gen(w, r, 0, sel[-1, r, 0]) for r in range(R)])
        dense = torch.from_numpy(host).cuda()
        idx = torch.arange(R * k, dtype=torch.int32, device="cuda").reshape(R, k)
        direct = _attend(dense, R * k, idx, q16, R, k, heads)
        assert np.array_equal(got.view(np.uint32), direct.view(np.uint32))
        q = _bf16_to_f64(q16)
        for r in range(R):
            rec = host[r * k:(r + 1) * k]
            vmax = np.abs(records.decode(w, rec)[:, :512]).max()
            for h in range(heads):
                ref = sparse_attention(rec, 1, q[r, h])[0]   # scores q.K / sqrt(576)
                assert np.max(np.abs(got[r, h] - ref)) <= 4 * 2.0 ** -9 * vmax, (r, h)


def test_masked_rows():
    R, k, heads = 2, 200, 16
    w, sel, q16 = _setup(R, k, heads, steps=1, seed=5)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.empty((R, k), dtype=torch.int32, device="cuda")
        pool.resolve(0, torch.from_numpy(np.ascontiguousarray(sel[0, :, 0])).cuda(), out)
        cache = pool.views(0)["cache"]
        idx = out.clone()
        idx[0] = -1                      # a rejected request: every key masked
        idx[1, ::3] = cache.shape[0]     # out of range: masked
        got = _attend(cache, cache.shape[0], idx, q16, R, k, heads)
        assert np.all(got[0] == 0)
        keep = np.ones(k, bool)
        keep[::3] = False
        rec = records.gen(w, 1, 0, sel[0, 1, 0][keep])
        vmax = np.abs(records.decode(w, rec)[:, :512]).max()
        q = _bf16_to_f64(q16)
        for h in range(heads):
            ref = sparse_attention(rec, 1, q[1, h])[0]
            assert np.max(np.abs(got[1, h] - ref)) <= 4 * 2.0 ** -9 * vmax


@pytest.mark.parametrize("R,k,heads", [(1, 1, 16), (3, 33, 48), (2, 65, 16), (5, 1000, 16),
                                       (40, 96, 16), (1, 2048, 128)])
def test_ragged_shapes_against_oracle(R, k, heads):
    w = configs.DSA_MLA.with_(n_requests=1, n_layers=1, n_positions=5000)
    rng = np.random.default_rng(R * 1000 + k + heads)
    rows = 4096
    table = records.gen(w, 0, 0, np.arange(rows))          # a dense cache of records
    idx = np.stack([rng.choice(rows, k, replace=False) for _ in range(R)]).astype(np.int32)
    if k > 4:
        idx[0, 1::5] = -1                                    # masked keys
    q16 = _bf16_round(rng.standard_normal((R, heads, 576)).astype(np.float32))
    cache = torch.from_numpy(table).cuda()
    didx = torch.from_numpy(idx).cuda()
    got = _attend(cache, rows, didx, q16, R, k, heads)
    again = _attend(cache, rows, didx, q16, R, k, heads)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))
    q = _bf16_to_f64(q16)
    for r in range(R):
        rec = table[idx[r][idx[r] >= 0]]
        vmax = np.abs(records.decode(w, rec)[:, :512]).max()
        for h in range(heads):
            ref = sparse_attention(rec, 1, q[r, h])[0]
            assert np.max(np.abs(got[r, h] - ref)) <= 4 * 2.0 ** -9 * vmax, (r, h)


def test_many_heads_and_requests_sampled():
    """64 requests x 128 heads: one split per (request, 16 heads), more CTAs
    than fit at once; a sample of (request, head) against the oracle and the
    whole output finite."""
    R, k, heads = 64, 512, 128
    w = configs.DSA_MLA.with_(n_requests=1, n_layers=1, n_positions=5000)
    rng = np.random.default_rng(77)
    rows = 8192
    table = records.gen(w, 0, 0, np.arange(rows) % w.n_positions)
    idx = np.stack([rng.choice(rows, k, replace=False) for _ in range(R)]).astype(np.int32)
    q16 = _bf16_round(rng.standard_normal((R, heads, 576)).astype(np.float32))
    got = _attend(torch.from_numpy(table).cuda(), rows, torch.from_numpy(idx).cuda(), q16,
                  R, k, heads)
    assert np.isfinite(got).all()
    q = _bf16_to_f64(q16)
    for r in (0, 17, 63):
        rec = table[idx[r]]
        vmax = np.abs(records.decode(w, rec)[:, :512]).max()
        for h in (0, 15, 16, 77, 127):
            ref = sparse_attention(rec, 1, q[r, h])[0]
            assert np.max(np.abs(got[r, h] - ref)) <= 4 * 2.0 ** -9 * vmax, (r, h)


def test_closed_forms_on_the_gpu():
    """A zero query weighs every published row the same (the mean of the
    values, in fp32), and rows that are all the same record give that
    record's values exactly."""
    R, k, heads = 2, 200, 16
    w = configs.DSA_MLA.with_(n_requests=1, n_layers=1, n_positions=5000)
    rows = 1024
    table = records.gen(w, 0, 0, np.arange(rows))
    rng = np.random.default_rng(3)
    idx = np.stack([rng.choice(rows, k, replace=False) for _ in range(R)]).astype(np.int32)
    zero = np.zeros((R, heads, 576), np.uint16)
    got = _attend(torch.from_numpy(table).cuda(), rows, torch.from_numpy(idx).cuda(), zero,
                  R, k, heads)
    for r in range(R):
        mean = records.decode(w, table[idx[r]])[:, :512].mean(0)
        for h in range(heads):
            assert np.allclose(got[r, h], mean, rtol=1e-5, atol=1e-6), (r, h)
    same = np.full((R, k), 7, np.int32)
    q16 = _bf16_round(rng.standard_normal((R, heads, 576)).astype(np.float32))
    got = _attend(torch.from_numpy(table).cuda(), rows, torch.from_numpy(same).cuda(), q16,
                  R, k, heads)
    v = records.decode(w, table[7:8])[0, :512].astype(np.float32)
    assert np.array_equal(got, np.broadcast_to(v, got.shape))
