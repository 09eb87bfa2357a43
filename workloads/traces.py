"""Seeded synthetic selection traces (the top-k positions an indexer emits).

A trace is an int32 array ``sel[T][R][N_l][k]``: for decode step t, request r
and sparse layer l, the k distinct logical positions selected at that step,
in the order the indexer hands them over.  This module draws positions only;
it contains nothing of the resolve method.

Random streams: one numpy PCG64 generator per (request, layer), spawned from
``SeedSequence(workload.seed)`` in row-major (r, l) order.  Layers that share
an anchor's selection (``layer_anchor``) copy the anchor's trace and never
draw from their own stream.

Processes (parameters in :mod:`workloads.configs`):

``retain``   step 0: k positions uniform without replacement over [0, L).
             Step t > 0: keep ``floor(retain * k)`` positions chosen uniformly
             without replacement from step t-1's selection; draw the remaining
             n_new positions as ``floor(local_frac * n_new)`` "local" ones
             (a kept position chosen uniformly, plus an offset uniform on
             [-local_window, +local_window]) followed by uniform ones over
             [0, L).  A candidate that is out of range or already selected is
             redrawn.  The k positions are then shuffled.
``uniform``  every step: k positions uniform without replacement over [0, L).
``quest``    the context is cut into pages of ``page_tokens`` tokens.  Each
             page has a score, initially N(0, 1), that drifts by
             N(0, score_drift^2) at every step after the first.  The last
             ``always_last_pages`` pages are always selected; the others are
             ranked by score (descending, stable) and ``k / page_tokens -
             always_last_pages`` distinct ones are drawn with probability
             proportional to rank^-zipf_s (rank 1 = best; inverse-CDF draws
             from uniform doubles), redrawing repeats.
             Pages are emitted last-pages first, then in draw order, each
             expanded to its tokens in ascending order.
"""
from __future__ import annotations

import numpy as np

from .configs import Workload


def _streams(w: Workload):
    ss = np.random.SeedSequence(w.seed)
    children = ss.spawn(w.n_requests * w.n_layers)
    return [np.random.Generator(np.random.PCG64(c)) for c in children]


def _draw_new(rng, n, sampler, mask, L):
    """Draw n distinct positions not yet in ``mask`` (which is updated).

    Candidates come in batches from ``sampler(size)``; they are accepted in
    draw order, skipping out-of-range ones, ones already selected and repeats
    within the batch.
    """
    out = []
    need = n
    while need > 0:
        cand = np.asarray(sampler(2 * need + 16), dtype=np.int64)
        ok = (cand >= 0) & (cand < L)
        cand = cand[ok]
        cand = cand[~mask[cand]]
        if cand.size:
            _, first = np.unique(cand, return_index=True)
            cand = cand[np.sort(first)][:need]
            mask[cand] = True
            out.append(cand)
            need -= cand.size
    if not out:
        return np.zeros(0, np.int64)
    return np.concatenate(out)


def _retain_stream(w: Workload, rng) -> np.ndarray:
    L, k, T = w.n_positions, w.k, w.steps
    out = np.empty((T, k), np.int32)
    n_keep = int(np.floor(w.retain * k))
    n_new = k - n_keep
    n_local = int(np.floor(w.local_frac * n_new))
    n_unif = n_new - n_local
    mask = np.zeros(L, bool)
    prev = None
    for t in range(T):
        if t == 0:
            sel = rng.choice(L, size=k, replace=False).astype(np.int64)
        else:
            keep = rng.choice(prev, size=n_keep, replace=False).astype(np.int64)
            mask[:] = False
            mask[keep] = True
            parts = [keep]
            if n_local:
                win = w.local_window

                def local(size, keep=keep):
                    a = keep[rng.integers(0, keep.size, size)]
                    return a + rng.integers(-win, win + 1, size)

                parts.append(_draw_new(rng, n_local, local, mask, L))
            if n_unif:
                parts.append(_draw_new(
                    rng, n_unif, lambda size: rng.integers(0, L, size), mask, L))
            sel = np.concatenate(parts)
        sel = rng.permutation(sel)
        out[t] = sel
        prev = sel
    return out


def _uniform_stream(w: Workload, rng) -> np.ndarray:
    out = np.empty((w.steps, w.k), np.int32)
    for t in range(w.steps):
        out[t] = rng.permutation(rng.choice(w.n_positions, size=w.k, replace=False))
    return out


def _quest_stream(w: Workload, rng) -> np.ndarray:
    P = w.page_tokens
    n_pages = w.n_positions // P
    n_last = w.always_last_pages
    n_rank = n_pages - n_last
    n_draw = w.k // P - n_last
    weights = np.arange(1, n_rank + 1, dtype=np.float64) ** (-w.zipf_s)
    cdf = np.cumsum(weights / weights.sum())
    cdf[-1] = 1.0
    last = np.arange(n_pages - n_last, n_pages, dtype=np.int64)
    tok = np.arange(P, dtype=np.int64)
    score = rng.standard_normal(n_pages)
    out = np.empty((w.steps, w.k), np.int32)
    for t in range(w.steps):
        if t > 0:
            score = score + rng.normal(0.0, w.score_drift, n_pages)
        by_rank = np.argsort(-score[:n_rank], kind="stable")
        chosen = np.zeros(n_rank, bool)
        drawn = []
        need = n_draw
        while need > 0:
            # inverse-CDF draw of ranks (0-based) with P(j) ~ (j + 1)^-s
            ranks = np.searchsorted(cdf, rng.random(2 * need + 8), side="right")
            ranks = np.minimum(ranks, n_rank - 1)
            ranks = ranks[~chosen[ranks]]
            if ranks.size:
                _, first = np.unique(ranks, return_index=True)
                ranks = ranks[np.sort(first)][:need]
                chosen[ranks] = True
                drawn.append(ranks)
                need -= ranks.size
        pages = np.concatenate([last, by_rank[np.concatenate(drawn)]])
        out[t] = (pages[:, None] * P + tok[None, :]).reshape(-1)
    return out


_PROCESS = {"retain": _retain_stream, "uniform": _uniform_stream,
            "quest": _quest_stream}


def stream(w: Workload, r: int, l: int) -> np.ndarray:
    """Selections ``[T][k]`` of one (request, layer), following its anchor."""
    a = w.anchors[l]
    rng = _streams(w)[r * w.n_layers + a]
    return _PROCESS[w.process](w, rng)


def generate(w: Workload, requests=None) -> np.ndarray:
    """Full trace ``sel[T][R'][N_l][k]`` (int32) for the listed requests."""
    if requests is None:
        requests = range(w.n_requests)
    requests = list(requests)
    rngs = _streams(w)
    out = np.empty((w.steps, len(requests), w.n_layers, w.k), np.int32)
    fn = _PROCESS[w.process]
    for i, r in enumerate(requests):
        done = {}
        for l in range(w.n_layers):
            a = w.anchors[l]
            if a not in done:
                done[a] = fn(w, rngs[r * w.n_layers + a])
            out[:, i, l, :] = done[a]
    return out
