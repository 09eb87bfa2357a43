"""The per-head sparse attention consumer (hs_sparse_attention_heads) over
published slots of token records made of per-head key and value blocks.

* against the fp64 oracle attention (oracle/attention.py, per-head layout)
  on the host records of the selected positions.  Tolerance: the kernel's
  products of bf16 values are exact in fp32; each score sums 128 of them in
  fp32 (error at most 128 * 2^-24 * sum_d |q_d K_d|, below 1e-3 of a unit
  score for the magnitudes here), exp2 and the sums over at most 2048 keys
  are fp32 too, so the outputs are within about 1e-4 * max|V| of the exact
  value; the tests allow 2e-3 * max|V|;
* attention over the published slots is bit-identical to attention over the
  same records copied straight from the host pool in selection order (the
  exactness claim, on the GPU);
* rows outside the cache are masked and a request with every row masked
  gets zeros;
* ragged key counts (one key, a partial batch, split boundaries), head
  counts 1 to 8 and batch sizes that change the split of the keys.
"""
import numpy as np
import pytest
import torch

from hierarchical_kv_cache_resolve_gb300 import hs
from oracle.attention import sparse_attention
from tests.gpu_harness import fill_selected
from workloads import configs, records

pytestmark = pytest.mark.gpu

SCALE = 1.0 / np.sqrt(128.0)
TOL = 2e-3


def _bf16_round(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _bf16_to_f64(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _attend(cache, rows, idx, q16, R, k, heads):
    q = torch.from_numpy(q16.view(np.int16)).cuda()
    out = torch.full((R, heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    hs.hs_sparse_attention_heads(q, cache, rows, idx, R, k, heads, SCALE, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _vmax(rec, heads):
    v = _bf16_to_f64(np.ascontiguousarray(rec).view(np.uint16))[:, heads * 128:]
    return np.abs(v).max()


def test_heads_over_published_slots_match_oracle_and_host_gather():
    R, k, heads = 4, 300, 8
    w = configs.QUEST_PAGES.with_(n_requests=R, n_layers=1, n_positions=20000, k=k, slots=512,
                                  steps=3)
    rng = np.random.default_rng(4)
    sel = np.stack([np.stack([rng.choice(w.n_positions, k, replace=False)[None]
                              for _ in range(R)]) for _ in range(3)]).astype(np.int32)
    q16 = _bf16_round(rng.standard_normal((R, heads, 128)).astype(np.float32))
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        out = torch.empty((R, k), dtype=torch.int32, device="cuda")
        for t in range(sel.shape[0]):
            pool.resolve(0, torch.from_numpy(np.ascontiguousarray(sel[t, :, 0])).cuda(), out)
        cache = pool.views(0)["cache"]
        got = _attend(cache, cache.shape[0], out, q16, R, k, heads)
        host = np.concatenate([records.gen(w, r, 0, sel[-1, r, 0]) for r in range(R)])
        dense = torch.from_numpy(host).cuda()
        idx = torch.arange(R * k, dtype=torch.int32, device="cuda").reshape(R, k)
        direct = _attend(dense, R * k, idx, q16, R, k, heads)
        assert np.array_equal(got.view(np.uint32), direct.view(np.uint32))
        q = _bf16_to_f64(q16)
        for r in range(R):
            rec = host[r * k:(r + 1) * k]
            ref = sparse_attention(rec, 1, q[r], heads=heads, scale=SCALE)
            assert np.max(np.abs(got[r] - ref)) <= TOL * _vmax(rec, heads), r


@pytest.mark.parametrize("R,k,heads", [(1, 1, 8), (3, 33, 8), (2, 65, 4), (5, 1000, 8),
                                       (40, 96, 2), (1, 2048, 8), (7, 513, 1), (33, 2048, 8)])
def test_heads_ragged_shapes_against_oracle(R, k, heads):
    rng = np.random.default_rng(R * 1000 + k + heads)
    rows = R * k + 17
    W = heads * 512
    vals = _bf16_round(rng.standard_normal((rows, W // 2)).astype(np.float32))
    cache = torch.from_numpy(vals.view(np.uint8).reshape(rows, W)).cuda()
    idx_h = np.stack([rng.choice(rows, k, replace=False) for _ in range(R)]).astype(np.int32)
    idx = torch.from_numpy(idx_h).cuda()
    q16 = _bf16_round(rng.standard_normal((R, heads, 128)).astype(np.float32))
    got = _attend(cache, rows, idx, q16, R, k, heads)
    again = _attend(cache, rows, idx, q16, R, k, heads)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))
    q = _bf16_to_f64(q16)
    recs = vals.view(np.uint8).reshape(rows, W)
    for r in range(R):
        rec = recs[idx_h[r]]
        ref = sparse_attention(rec, 1, q[r], heads=heads, scale=SCALE)
        assert np.max(np.abs(got[r] - ref)) <= TOL * _vmax(rec, heads), r


def test_heads_masked_rows():
    R, k, heads = 3, 200, 8
    rng = np.random.default_rng(8)
    rows = 1000
    vals = _bf16_round(rng.standard_normal((rows, heads * 256)).astype(np.float32))
    recs = vals.view(np.uint8).reshape(rows, heads * 512)
    cache = torch.from_numpy(recs).cuda()
    idx_h = np.stack([rng.choice(rows, k, replace=False) for _ in range(R)]).astype(np.int32)
    idx_h[0] = -1                     # a rejected request: every row masked
    idx_h[1, ::3] = rows              # out of range: masked
    q16 = _bf16_round(rng.standard_normal((R, heads, 128)).astype(np.float32))
    got = _attend(cache, rows, torch.from_numpy(idx_h).cuda(), q16, R, k, heads)
    assert np.all(got[0] == 0)
    q = _bf16_to_f64(q16)
    for r in (1, 2):
        rec = recs[idx_h[r][(idx_h[r] >= 0) & (idx_h[r] < rows)]]
        ref = sparse_attention(rec, 1, q[r], heads=heads, scale=SCALE)
        assert np.max(np.abs(got[r] - ref)) <= TOL * _vmax(rec, heads), r


def test_heads_closed_forms_on_the_gpu():
    """A zero query averages each head's values; identical rows give their
    value exactly."""
    R, k, heads = 2, 700, 8
    rng = np.random.default_rng(21)
    rows = R * k
    vals = _bf16_round((rng.integers(-8, 9, size=(rows, heads * 256)) / 4).astype(np.float32))
    recs = vals.view(np.uint8).reshape(rows, heads * 512)
    cache = torch.from_numpy(recs).cuda()
    idx = torch.arange(rows, dtype=torch.int32, device="cuda").reshape(R, k)
    zero = np.zeros((R, heads, 128), np.uint16)
    got = _attend(cache, rows, idx, zero, R, k, heads)
    V = _bf16_to_f64(vals)[:, heads * 128:].reshape(R, k, heads, 128)
    assert np.allclose(got, V.mean(1), rtol=0, atol=1e-5)
    same = torch.from_numpy(np.repeat(recs[:1], rows, 0)).cuda()
    q16 = _bf16_round(rng.standard_normal((R, heads, 128)).astype(np.float32))
    got = _attend(same, rows, idx, q16, R, k, heads)
    want = _bf16_to_f64(vals[0])[heads * 128:].reshape(heads, 128)
    for r in range(R):
        assert np.array_equal(got[r], want.astype(np.float32)), r


def test_quest_decode_steps_with_the_per_head_consumer():
    """Decode steps of the Quest page process: every layer's resolve, then the
    per-head consumer over the slots it published, no host synchronisation
    until the end.  Every step's published slots against the oracle, and
    every step's attention bit-identical to the same kernel over the host
    records of the selection gathered densely."""
    from tests.gpu_harness import OracleRun, device_trace
    from workloads import traces
    w = configs.QUEST_PAGES.with_(n_requests=4, n_layers=2, n_positions=8192, k=512,
                                  slots=1024, steps=10)
    sel = traces.generate(w)                     # [T][R][N_l][k]
    T, R, NL, k = sel.shape
    heads = 8
    rng = np.random.default_rng(31)
    q16 = _bf16_round(rng.standard_normal((R, heads, 128)).astype(np.float32))
    q = torch.from_numpy(q16.view(np.int16)).cuda()
    orc = OracleRun(w)
    with hs.Pool.for_workload(w) as pool:
        fill_selected(pool, w, sel)
        dsel = device_trace(sel)                  # [T][N_l][R][k]
        out = torch.empty((T, NL, R, k), dtype=torch.int32, device="cuda")
        att = torch.empty((T, NL, R, heads, 128), dtype=torch.float32, device="cuda")
        caches = [pool.views(l)["cache"] for l in range(NL)]
        torch.cuda.synchronize()
        for t in range(T):
            for l in range(NL):
                pool.resolve(l, dsel[t, l], out[t, l])
                hs.hs_sparse_attention_heads(q, caches[l], caches[l].shape[0], out[t, l], R, k,
                                             heads, SCALE, att[t, l])
        got = out.cpu().numpy()
        for t in range(T):
            for (r, l), (o, m) in orc.step(sel[t]).items():
                assert np.array_equal(got[t, l, r], o), (t, r, l)
        idx = torch.arange(R * k, dtype=torch.int32, device="cuda").reshape(R, k)
        ref = torch.empty((R, heads, 128), dtype=torch.float32, device="cuda")
        for t in range(T):
            for l in range(NL):
                host = np.concatenate([records.gen(w, r, l, sel[t, r, l]) for r in range(R)])
                dense = torch.from_numpy(host).cuda()
                hs.hs_sparse_attention_heads(q, dense, R * k, idx, R, k, heads, SCALE, ref)
                assert torch.equal(att[t, l].view(torch.int32), ref.view(torch.int32)), (t, l)
        assert pool.stats()["status"] == 0
