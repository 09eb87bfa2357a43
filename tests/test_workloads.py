"""The seeded input generators: traces and host records behave as stated."""
import numpy as np
import pytest

from workloads import configs, records, traces


def _splitmix64(z):
    m = (1 << 64) - 1
    z = (z + 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def _py_record(w, r, l, pos):
    """Re-derivation of one record from the generator's stated definition."""
    m = (1 << 64) - 1
    s = r * w.n_layers + l
    key = _splitmix64(_splitmix64(w.seed) ^ (((s + 1) * 0x9E3779B97F4A7C15) & m))
    npair = w.record_bytes // 4
    vals = []
    for j in range(npair):
        h = _splitmix64((key + pos * npair + j) & m)
        u1, u2 = h >> 40, (h >> 16) & 0xFFFFFF
        if w.value_format == 0:
            vals += [(u1 + 0.5) / 2**23 - 1, (u2 + 0.5) / 2**23 - 1]
        else:
            a, b = (u1 + 0.5) / 2**24, (u2 + 0.5) / 2**24
            rad = np.sqrt(-2 * np.log(a))
            vals += [rad * np.cos(2 * np.pi * b), rad * np.sin(2 * np.pi * b)]
    return np.array(vals)


@pytest.mark.parametrize("w", [configs.TINY, configs.DSA_MLA, configs.QUEST_PAGES])
def test_records_follow_stated_definition(w):
    got = records.decode(w, records.gen(w, 1 % w.n_requests, 0, [0, 5, w.n_positions - 1]))
    for i, pos in enumerate([0, 5, w.n_positions - 1]):
        want = _py_record(w, 1 % w.n_requests, 0, pos)
        # float32 math then rounding to a 16-bit float: within one unit in the
        # last place of the 16-bit format
        ulp = np.abs(want) * (2.0 ** -10 if w.value_format == 0 else 2.0 ** -7)
        assert np.all(np.abs(got[i] - want) <= ulp + 1e-7)


def test_record_value_distributions():
    w = configs.DSA_MLA
    x = records.decode(w, records.gen(w, 0, 0, np.arange(4000)))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    w = configs.TINY
    x = records.decode(w, records.gen(w, 0, 0, np.arange(4000)))
    assert x.min() >= -1 and x.max() <= 1 and abs(x.std() - (1 / 3) ** 0.5) < 0.01


def test_fill_matches_gen_and_streams_differ():
    w = configs.DSA_MLA
    buf = np.empty((300, w.record_bytes), np.uint8)
    records.fill(buf.ctypes.data, w, 2, 3, pos0=1000, n=300, threads=3)
    assert np.array_equal(buf, records.gen(w, 2, 3, np.arange(1000, 1300)))
    assert not np.array_equal(buf, records.gen(w, 2, 2, np.arange(1000, 1300)))


@pytest.mark.parametrize("w", [configs.TINY, configs.DSA_MLA.with_(steps=40),
                               configs.TIGHT_PREFETCH.with_(n_requests=2, steps=20),
                               configs.NO_LOCALITY.with_(steps=8),
                               configs.QUEST_PAGES.with_(n_requests=2, steps=20),
                               configs.QUEST_PAGE_RECORDS.with_(n_requests=2, steps=20)])
def test_trace_shape_range_distinct(w):
    s = traces.generate(w)
    assert s.shape == (w.steps, w.n_requests, w.n_layers, w.k) and s.dtype == np.int32
    assert s.min() >= 0 and s.max() < w.n_positions
    for t in range(w.steps):
        for r in range(w.n_requests):
            for l in range(w.n_layers):
                assert np.unique(s[t, r, l]).size == w.k
    again = traces.generate(w)
    assert np.array_equal(s, again)


def test_retention_and_locality():
    w = configs.DSA_MLA.with_(steps=30)
    s = traces.stream(w, 0, 1)
    n_keep = int(np.floor(0.87 * w.k))
    for t in range(1, w.steps):
        kept = np.intersect1d(s[t], s[t - 1]).size
        # new draws avoid this step's set only, so they may re-pick a position
        # dropped from step t-1
        assert kept >= n_keep
    # new positions near a kept one: at least 70% lie within the window of
    # some previous-step position
    t = 10
    new = np.setdiff1d(s[t], s[t - 1])
    prev = np.sort(s[t - 1])
    idx = np.searchsorted(prev, new)
    near = np.minimum(np.abs(new - prev[np.clip(idx, 0, prev.size - 1)]),
                      np.abs(new - prev[np.clip(idx - 1, 0, prev.size - 1)]))
    assert (near <= w.local_window).mean() >= 0.69


def test_shared_layers_copy_the_anchor():
    w = configs.TIGHT_PREFETCH.with_(n_requests=2, steps=6)
    s = traces.generate(w)
    for l in range(8):
        assert np.array_equal(s[:, :, l], s[:, :, w.anchors[l]])
    assert not np.array_equal(s[:, :, 0], s[:, :, 4])


def test_quest_pages_structure():
    w = configs.QUEST_PAGES.with_(n_requests=1, steps=8)
    s = traces.stream(w, 0, 0)
    P = w.page_tokens
    for t in range(w.steps):
        pages = s[t].reshape(-1, P)
        assert (pages == pages[:, :1] + np.arange(P)).all()
        assert (pages[:, 0] % P == 0).all()
        assert pages[:4, 0].tolist() == [(2044 + i) * P for i in range(4)]
        assert np.unique(pages[:, 0]).size == w.k // P
