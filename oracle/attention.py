"""Float64 sparse attention over selected KV records -- test infrastructure.

Used for the exactness claim: because only the placement of KV records
changes, attention over the records gathered through the published slots
must equal attention over the same positions read from the host pool
("Inference Systems Infrastructure Notes (6): HiSparse", section 5 "Why It
Is Exact"; Pith review abstract, "model outputs are unchanged").

Record layouts (this package's reading of the workloads' record shapes):
  * 64-element fp16 records (one head): K = V = the record;
  * 576-element bf16 MLA records: K = all 576 elements, V = the first 512
    (the latent part, as in MLA decoding);
  * 2048-element bf16 Quest-style token records: 8 heads of 128, K in
    elements [0, 1024) and V in [1024, 2048), head-major; in general
    `heads` key blocks of 128 followed by `heads` value blocks.

Scores are q . K / sqrt(d_k) in selection order, a max-subtracted softmax,
then the probability-weighted sum of V; all in float64.
"""
from __future__ import annotations

import numpy as np


def _values(rec: np.ndarray, fmt: int) -> np.ndarray:
    u16 = np.ascontiguousarray(rec).view(np.uint16)
    if fmt == 0:
        return u16.view(np.float16).astype(np.float64)
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def split_kv_heads(rec: np.ndarray, fmt: int, heads: int, d: int = 128):
    """(K[h][n][d], V[h][n][d]) from records [n][W] made of `heads` key
    blocks of d elements, head after head, followed by `heads` value blocks
    (the 2048-element Quest token records are heads = 8, d = 128)."""
    x = _values(rec, fmt)              # [n][E]
    n, E = x.shape
    if E != 2 * heads * d:
        raise ValueError(f"{E}-element records do not hold {heads} heads of {d}")
    k = x[:, :heads * d].reshape(n, heads, d).transpose(1, 0, 2)
    v = x[:, heads * d:].reshape(n, heads, d).transpose(1, 0, 2)
    return k, v


def split_kv(rec: np.ndarray, fmt: int):
    """(K[h][n][d], V[h][n][dv]) from records [n][W]."""
    x = _values(rec, fmt)              # [n][E]
    n, E = x.shape
    if E == 64:
        return x[None], x[None]
    if E == 576:
        return x[None], x[None, :, :512]
    if E == 2048:
        return split_kv_heads(rec, fmt, 8)
    raise ValueError(f"no attention layout for {E}-element records")


def query_dims(E: int):
    """(heads, d_k) of the query for E-element records."""
    return {64: (1, 64), 576: (1, 576), 2048: (8, 128)}[E]


def sparse_attention(rec: np.ndarray, fmt: int, q: np.ndarray, heads: int | None = None,
                     scale: float | None = None) -> np.ndarray:
    """Attention output [h][dv] of query q[h][d_k] over records rec[n][W]:
    the layout of `split_kv`, or with `heads` given, of `split_kv_heads`.
    Scores are scaled by 1/sqrt(d_k) unless `scale` is given."""
    K, V = split_kv(rec, fmt) if heads is None else split_kv_heads(rec, fmt, heads)
    h, n, d = K.shape
    q = np.asarray(q, np.float64).reshape(h, d)
    out = np.empty((h, V.shape[2]), np.float64)
    c = 1.0 / np.sqrt(d) if scale is None else float(scale)
    for j in range(h):
        s = (K[j] @ q[j]) * c
        s = np.exp(s - s.max())
        p = s / s.sum()
        out[j] = p @ V[j]
    return out
