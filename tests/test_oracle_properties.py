"""Further pins of the oracle: exactness, policy direction, footprint identity
and exact layer-wise prefetch."""
import numpy as np
import pytest

from oracle.attention import query_dims, sparse_attention
from oracle.oracle import OK, Pair
from workloads import configs, records, traces


def _host(w, r=0, l=0, n=None):
    n = w.n_positions if n is None else n
    buf = np.empty((n, w.record_bytes), np.uint8)
    records.fill(buf.ctypes.data, w, r, l, 0, n)
    return buf


@pytest.mark.parametrize("w", [configs.TINY,
                               configs.DSA_MLA.with_(n_positions=8192, steps=12),
                               configs.QUEST_PAGES.with_(steps=10)])
def test_attention_over_published_slots_equals_host_attention(w):
    """Exactness: gathering through the published slots changes nothing."""
    host = _host(w)
    sel = traces.stream(w, 0, 0)
    p = Pair(w.slots, w.n_positions, w.record_bytes, host=host, mirror=True)
    rng = np.random.default_rng(7)
    h, d = query_dims(w.record_bytes // 2)
    for t in range(sel.shape[0]):
        rc, out, m = p.resolve(sel[t])
        assert rc == OK
        q = rng.standard_normal((h, d))
        a = sparse_attention(p.cache[out], w.value_format, q)
        b = sparse_attention(host[sel[t]], w.value_format, q)
        assert np.array_equal(a, b)
        # and against a dense reference restricted to the same positions
        c = sparse_attention(host[np.sort(sel[t])], w.value_format, q)
        assert np.allclose(a, c, rtol=1e-12, atol=1e-12)


def test_attention_layout_sanity():
    """A one-hot query picks the record with the largest matching key."""
    rec = np.zeros((3, 128), np.uint8)
    vals = np.zeros((3, 64), np.float16)
    vals[0, 0], vals[1, 0], vals[2, 0] = 0.5, 8.0, -1.0
    rec[:] = vals.view(np.uint8)
    q = np.zeros(64)
    q[0] = 64.0
    out = sparse_attention(rec, 0, q)
    assert out.shape == (1, 64)
    assert abs(out[0, 0] - 8.0) < 1e-6


def test_top_k_only_staging_misses_more_than_b_2k():
    """Policy direction (Pith review, Fig. 6): B = k misses more than B = 2k."""
    w = configs.DSA_MLA
    sel = traces.stream(w, 0, 0)
    rates = {}
    for B in (w.k, 2 * w.k):
        p = Pair(B, w.n_positions, 16)
        rc, out, m = p.run(sel)
        assert rc == OK
        rates[B] = m[1:].sum() / (w.k * (w.steps - 1))
    assert rates[w.k] > rates[2 * w.k]
    # with 87% retention the steady-state miss rate at B = 2k is at most the
    # fraction of new positions per step
    assert rates[2 * w.k] <= 1 - np.floor(0.87 * w.k) / w.k + 1e-9


def test_uniform_selection_misses_almost_everything():
    w = configs.NO_LOCALITY.with_(steps=16)
    sel = traces.stream(w, 0, 0)
    p = Pair(w.slots, w.n_positions, 16)
    rc, out, m = p.run(sel)
    assert rc == OK
    assert m[1:].mean() / w.k > 0.99


def test_hbm_footprint_independent_of_context():
    """N_l x B x W per request, whatever L_ctx (HiSparse notes, section 2)."""
    a = configs.DSA_MLA
    b = a.with_(n_positions=1 << 20)
    per_req = a.n_layers * a.slots * a.record_bytes
    assert a.cache_bytes == b.cache_bytes == a.n_requests * per_req
    # the page's 128K example: 13.09 GB at full residency shrinks by L/B
    assert abs(13.09 * 4096 / 131072 - 0.409) < 1e-3
    assert a.n_positions // a.slots == 32


def _run_group(w, with_prefetch, plan_override=None):
    """One request, one anchor layer plus shared layers, oracle only."""
    sel = traces.stream(w, 0, 0)
    L, B, W = w.n_positions, w.slots, w.record_bytes
    hosts = [_host(w, 0, l, L) for l in range(3)]
    pairs = [Pair(B, L, W, host=hosts[l], mirror=True) for l in range(3)]
    outs = []
    for t in range(sel.shape[0]):
        rc, out, _ = pairs[0].resolve(sel[t])
        assert rc == OK
        outs.append(out)
        for l in (1, 2):
            plan = None
            if with_prefetch:
                rc, pp, ps = pairs[l].prefetch_plan(sel[t])
                assert rc == OK
                if plan_override is not None:
                    pp, ps = plan_override(t, pp, ps)
                pairs[l].prefetch_copy(pp, ps)
                plan = (pp, ps)
            rc, o2, _ = pairs[l].resolve(sel[t], plan=plan)
            assert rc == OK
            outs.append(o2)
    return pairs, outs


def test_prefetch_plan_replays_the_anchor_and_changes_nothing():
    w = configs.TIGHT_PREFETCH.with_(n_positions=6000, k=256, slots=256, steps=20)
    base, o_base = _run_group(w, False)
    pre, o_pre = _run_group(w, True)
    for a, b in zip(o_base, o_pre):
        assert np.array_equal(a, b)
    for a, b in zip(base, pre):
        assert np.array_equal(a.slot_pos, b.slot_pos)
        assert np.array_equal(a.stamp, b.stamp)
        assert np.array_equal(a.pt, b.pt)
        assert np.array_equal(a.cache, b.cache)
    # the shared layers' plans matched the resolves exactly: nothing left to fetch
    for b in pre[1:]:
        assert b.counters[4] == 0 and b.fetched_bytes == 0
        assert b.counters[3] == b.misses
        assert b.counters[5] == b.misses * w.record_bytes
    # shared layers mirror the anchor: same published slots as the anchor
    for t in range(w.steps):
        assert np.array_equal(o_pre[3 * t], o_pre[3 * t + 1])


def test_wrong_plan_still_exact():
    """A plan that does not match (shuffled, truncated, pointing at hit slots)
    is repaired by the resolve: the final state equals the no-prefetch run."""
    w = configs.TIGHT_PREFETCH.with_(n_positions=3000, k=64, slots=96, steps=25)
    base, _ = _run_group(w, False)
    rng = np.random.default_rng(9)

    def corrupt(t, pp, ps):
        kind = t % 4
        if kind == 0 and pp.size > 1:
            return pp, np.roll(ps, 1)
        if kind == 1:
            return pp[: pp.size // 2], ps[: ps.size // 2]
        if kind == 2:
            bad = rng.integers(0, w.slots, size=pp.size + 3).astype(np.int32)
            pos = rng.integers(0, w.n_positions, size=pp.size + 3).astype(np.int32)
            return pos, bad
        return pp, ps

    pre, _ = _run_group(w, True, plan_override=corrupt)
    for a, b in zip(base, pre):
        assert np.array_equal(a.slot_pos, b.slot_pos)
        assert np.array_equal(a.pt, b.pt)
        assert np.array_equal(a.stamp, b.stamp)
        occ = a.slot_pos >= 0
        assert np.array_equal(a.cache[occ], b.cache[occ])
    assert sum(int(b.counters[4]) for b in pre[1:]) > 0


def _bf16_records(vals):
    """uint8 records of bf16 values (vals exactly representable in bf16)."""
    v = np.ascontiguousarray(vals, np.float32)
    u = (v.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((u.astype(np.uint32) << 16).view(np.float32), v)
    return u.view(np.uint8).reshape(v.shape[0], -1)


def test_mla_attention_closed_forms():
    """576-element MLA records (K = all 576, V = the first 512, scores
    q.K / sqrt(576)): closed forms independent of the oracle's code."""
    rng = np.random.default_rng(5)
    vals = rng.integers(-8, 9, size=(5, 576)).astype(np.float32) / 4   # exact in bf16
    rec = _bf16_records(vals)
    # a zero query weighs every key the same: the mean of the values
    out = sparse_attention(rec, 1, np.zeros(576))
    assert np.allclose(out[0], vals[:, :512].astype(np.float64).mean(0), rtol=0, atol=1e-12)
    # identical keys: the common value, whatever the query
    same = _bf16_records(np.repeat(vals[:1], 4, 0))
    out = sparse_attention(same, 1, rng.standard_normal(576))
    assert np.allclose(out[0], vals[0, :512], rtol=0, atol=1e-12)
    # two keys whose scores differ by delta: weights 1 / (1 + e^delta) and
    # e^delta / (1 + e^delta), with the 1/sqrt(576) = 1/24 scale applied
    two = np.zeros((2, 576), np.float32)
    two[0, 512] = 1.0                       # a key-only element (not part of V)
    two[:, :512] = vals[:2, :512]
    q = np.zeros(576)
    q[512] = 24.0 * 1.5                     # score of key 0: 1.5, of key 1: 0
    out = sparse_attention(_bf16_records(two), 1, q)
    w0 = np.exp(1.5) / (1 + np.exp(1.5))
    assert np.allclose(out[0], w0 * vals[0, :512] + (1 - w0) * vals[1, :512], rtol=0, atol=1e-12)


def test_quest_attention_heads_are_independent():
    """2048-element Quest token records: 8 heads of 128, K in [0, 1024) and
    V in [1024, 2048), head-major; a query touching only head 3 leaves the
    other heads' weights uniform."""
    rng = np.random.default_rng(9)
    vals = rng.integers(-4, 5, size=(3, 2048)).astype(np.float32) / 2
    rec = _bf16_records(vals)
    q = np.zeros((8, 128))
    q[3, 0] = np.sqrt(128.0) * 2.0          # head 3's scores: 2 * K[:, 3*128]
    out = sparse_attention(rec, 1, q)
    assert out.shape == (8, 128)
    V = vals[:, 1024:].reshape(3, 8, 128).astype(np.float64)
    for h in range(8):
        if h == 3:
            s = 2.0 * vals[:, 3 * 128].astype(np.float64)
            p = np.exp(s - s.max())
            p /= p.sum()
            want = p @ V[:, 3]
        else:
            want = V[:, h].mean(0)
        assert np.allclose(out[h], want, rtol=0, atol=1e-12), h


@pytest.mark.parametrize("heads", [1, 2, 4, 8])
def test_per_head_records_closed_forms(heads):
    """Token records of `heads` key blocks of 128 then `heads` value blocks:
    the layout round-trips from blocks assembled by hand, and each head's
    attention has the closed forms of plain softmax attention (zero query:
    mean of its values; a query on one key element: the logistic weights of
    the score gap; identical keys: the common value), with the scale given."""
    from oracle.attention import split_kv_heads
    rng = np.random.default_rng(10 + heads)
    n = 3
    Kb = rng.integers(-4, 5, size=(n, heads, 128)).astype(np.float32) / 2
    Vb = rng.integers(-4, 5, size=(n, heads, 128)).astype(np.float32) / 2
    rec = _bf16_records(np.concatenate([Kb.reshape(n, -1), Vb.reshape(n, -1)], axis=1))
    K, V = split_kv_heads(rec, 1, heads)
    assert np.array_equal(K, Kb.transpose(1, 0, 2)) and np.array_equal(V, Vb.transpose(1, 0, 2))
    # zero query: every head averages its values
    out = sparse_attention(rec, 1, np.zeros((heads, 128)), heads=heads)
    assert np.allclose(out, Vb.astype(np.float64).mean(0), rtol=0, atol=1e-12)
    # head h looks at key element 5 with weight 3 under scale 0.5: scores
    # 1.5 * K[:, h, 5]; the other heads stay uniform
    h = heads - 1
    q = np.zeros((heads, 128))
    q[h, 5] = 3.0
    out = sparse_attention(rec, 1, q, heads=heads, scale=0.5)
    s = 1.5 * Kb[:, h, 5].astype(np.float64)
    p = np.exp(s - s.max())
    p /= p.sum()
    assert np.allclose(out[h], p @ Vb[:, h].astype(np.float64), rtol=0, atol=1e-12)
    for g in range(heads - 1):
        assert np.allclose(out[g], Vb[:, g].astype(np.float64).mean(0), rtol=0, atol=1e-12)
    # identical keys in every record: the (identical) value, whatever the query
    same = _bf16_records(np.repeat(np.concatenate([Kb[:1].reshape(1, -1),
                                                   Vb[:1].reshape(1, -1)], axis=1), 4, 0))
    out = sparse_attention(same, 1, rng.standard_normal((heads, 128)), heads=heads)
    assert np.allclose(out, Vb[0], rtol=0, atol=1e-12)


def test_per_head_layout_of_eight_heads_is_the_quest_layout():
    """heads = 8 splits a 2048-element record exactly as the Quest reading
    does: K in [0, 1024), V in [1024, 2048), head-major."""
    from oracle.attention import split_kv_heads
    rng = np.random.default_rng(12)
    vals = rng.integers(-4, 5, size=(2, 2048)).astype(np.float32) / 2
    K, V = split_kv_heads(_bf16_records(vals), 1, 8)
    for h in range(8):
        assert np.array_equal(K[h], vals[:, 128 * h:128 * (h + 1)])
        assert np.array_equal(V[h], vals[:, 1024 + 128 * h:1024 + 128 * (h + 1)])
