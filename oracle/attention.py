"""Exact attention over the sink + window key set (oracle side), float64.

LongLive summary page (yunpan.plus), 方法 §3 高效长推理: with short-window
attention plus the frame sink, a query chunk attends to the sink tokens
concatenated with the keys/values of the recent window; nothing else is
approximated, so the oracle is the plain definition

    o_i = sum_j softmax_j(tau * q_i . k_j) v_j,   j over the visible tokens,

computed per head with a max-subtracted softmax.  Inside the visible set there
is no mask (tokens of a chunk are generated jointly; causality is at chunk
granularity).  A library matmul serves as the dot-product step.
"""

from __future__ import annotations

import numpy as np

from .cache_model import CacheModel


def attention_probs(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """Softmax probabilities P [H][Tq][L] for q [Tq][H][D], k [L][H][D]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    s = np.einsum("qhd,khd->hqk", q, k) * float(scale)
    s -= s.max(axis=2, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=2, keepdims=True)
    return p


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """O [Tq][H][D] = softmax(tau q k^T) v per head (no mask)."""
    out = np.empty(np.shape(q), dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    for h in range(np.shape(q)[1]):
        p = attention_probs(np.asarray(q)[:, h:h + 1, :], np.asarray(k)[:, h:h + 1, :], scale)[0]
        out[:, h, :] = p @ v[:, h, :]
    return out


def sinkwin_attention(cache: CacheModel, q: np.ndarray, scale: float) -> np.ndarray:
    """Attention of query rows q [Tq][H][D] against the cache's visible set."""
    k, v = cache.visible_kv()
    return attention(q, k, v, scale)


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                   rows, heads=None) -> np.ndarray:
    """Attention output for selected query rows only: returns [len(rows)][H'][D]."""
    rows = np.asarray(rows)
    heads = range(np.shape(q)[1]) if heads is None else heads
    qs = np.asarray(q)[rows]
    out = np.empty((len(rows), len(heads), np.shape(q)[2]), dtype=np.float64)
    for i, h in enumerate(heads):
        p = attention_probs(qs[:, h:h + 1, :], np.asarray(k)[:, h:h + 1, :], scale)[0]
        out[:, i, :] = p @ np.asarray(v, dtype=np.float64)[:, h, :]
    return out
