"""KV recache at a prompt switch (oracle side), float64.

LongLive summary page (yunpan.plus), 方法 §1 KV 重缓存: at the prompt-switch
boundary the KV cache is recomputed from the frames already generated, paired
with the new prompt, which clears the old prompt's residue and keeps the
visual and motion cues; generation then continues on the refreshed cache.
The LONGLIVE news page (paooo.com), LONGLIVE的技术原理, restates it.

The per-layer tail of that recompute is restated here: given the hidden states
of the cached tokens,

    [K | V] = Hid @ W_kv                       (plain GEMM, a library matmul)
    K       = RoPE3D(RMSNorm(K) * gamma)       (V unchanged)

and K, V go back into the regions of the listed chunks.

Readings (the pages give no formula for either):
* RMSNorm spans the whole H*D-wide K row (all heads), eps = 1e-6, no bias:
  y = x / sqrt(mean(x^2) + eps) * gamma.
* 3D RoPE: token t of a chunk c sits at frame f = c*chunk_frames + t // tpf,
  row h = (t % tpf) // grid_w, column w = t % grid_w.  The D/2 rotation pairs
  are split into bands [frame | h | w] of (P - 2*(P//3), P//3, P//3) pairs,
  P = D/2 (22/21/21 at D = 128).  In a band of b dims, pair j turns by
  pos * theta^(-2j/b); pairs are adjacent elements (x[2i], x[2i+1]).
  PARITY OF THE BAND SPLIT AND THETA IS PINNED TO THIS READING ONLY.
"""

from __future__ import annotations

import numpy as np


def project(hidden: np.ndarray, w_kv: np.ndarray):
    """[K | V] = hidden @ w_kv; returns K, V each [T][H*D] float64."""
    kv = np.asarray(hidden, dtype=np.float64) @ np.asarray(w_kv, dtype=np.float64)
    hd = kv.shape[1] // 2
    return kv[:, :hd], kv[:, hd:]


def rmsnorm(x: np.ndarray, gamma=None, eps: float = 1e-6) -> np.ndarray:
    """Row-wise RMSNorm over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    y = x / r
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64)
    return y


def rope_bands(head_dim: int):
    """Rotation pairs per axis (frame, h, w)."""
    p = head_dim // 2
    hw = p // 3
    return (p - 2 * hw, hw, hw)


def token_positions(chunk_id: int, chunk_tokens: int, tokens_per_frame: int,
                    chunk_frames: int, grid_w: int, frame0: int | None = None):
    """(frame, h, w) integer positions of the tokens of one chunk, each [Tc].
    frame0: frame position of the chunk's first frame (default chunk_id *
    chunk_frames; a multi-shot cache shifts it, see cache_model)."""
    t = np.arange(chunk_tokens)
    f0 = chunk_id * chunk_frames if frame0 is None else frame0
    f = f0 + t // tokens_per_frame
    p = t % tokens_per_frame
    return f, p // grid_w, p % grid_w


def rope3d(x: np.ndarray, pos_f, pos_h, pos_w, theta: float = 10000.0) -> np.ndarray:
    """Rotate x [T][H][D] by the 3D RoPE of per-token positions (each [T])."""
    x = np.asarray(x, dtype=np.float64)
    T, H, D = x.shape
    out = x.copy()
    bands = rope_bands(D)
    pair0 = 0
    for npairs, pos in zip(bands, (pos_f, pos_h, pos_w)):
        b = 2 * npairs
        for j in range(npairs):
            omega = theta ** (-2.0 * j / b)
            ang = np.asarray(pos, dtype=np.float64) * omega
            c = np.cos(ang)[:, None]
            s = np.sin(ang)[:, None]
            i0 = 2 * (pair0 + j)
            a = x[:, :, i0]
            bb = x[:, :, i0 + 1]
            out[:, :, i0] = a * c - bb * s
            out[:, :, i0 + 1] = a * s + bb * c
        pair0 += npairs
    return out


def recache(hidden, w_kv, gamma, chunk_ids, heads: int, head_dim: int,
            tokens_per_frame: int, chunk_frames: int, grid_w: int,
            eps: float = 1e-6, theta: float = 10000.0, frame0=None):
    """K, V [n*Tc][H][D] float64 for hidden rows of the chunks in ``chunk_ids``
    (logical order, sink first).  frame0: per chunk, the frame position of its
    first frame (default chunk_id * chunk_frames)."""
    k, v = project(hidden, w_kv)
    k = rmsnorm(k, gamma, eps)
    T = k.shape[0]
    n = len(chunk_ids)
    Tc = T // n
    assert Tc * n == T
    k = k.reshape(T, heads, head_dim)
    v = v.reshape(T, heads, head_dim)
    pf, ph, pw = [], [], []
    for i, c in enumerate(chunk_ids):
        f, h, w = token_positions(c, Tc, tokens_per_frame, chunk_frames, grid_w,
                                  None if frame0 is None else frame0[i])
        pf.append(f), ph.append(h), pw.append(w)
    k = rope3d(k, np.concatenate(pf), np.concatenate(ph), np.concatenate(pw), theta)
    return k, v


def project_chunk(hidden, w_qkv, gamma_q, gamma_k, chunk_id: int, heads: int, head_dim: int,
                  tokens_per_frame: int, chunk_frames: int, grid_w: int,
                  eps: float = 1e-6, theta: float = 10000.0, frame0: int | None = None):
    """Q, K, V [Tc][H][D] float64 of ONE new chunk, as the layer produces them
    before they are attended to and appended.

    LongLive summary page, 方法 (causal frame-level autoregression): each new
    chunk's tokens are projected to queries, keys and values; the keys and
    values join the cache every later chunk reads (§3 高效长推理, 帧汇聚点).
    The same readings as ``recache`` hold (norm over the whole H*D row, then
    3D RoPE at the chunk's absolute positions), applied to Q with its own gain:

        [Q | K | V] = hidden @ w_qkv          (w_qkv [H*D][3*H*D], Q columns first)
        Q = RoPE3D(RMSNorm(Q) * gamma_q),  K = RoPE3D(RMSNorm(K) * gamma_k)
    """
    x = np.asarray(hidden, dtype=np.float64) @ np.asarray(w_qkv, dtype=np.float64)
    hd = heads * head_dim
    Tc = x.shape[0]
    f, h, w = token_positions(chunk_id, Tc, tokens_per_frame, chunk_frames, grid_w, frame0)
    q = rope3d(rmsnorm(x[:, :hd], gamma_q, eps).reshape(Tc, heads, head_dim), f, h, w, theta)
    k = rope3d(rmsnorm(x[:, hd:2 * hd], gamma_k, eps).reshape(Tc, heads, head_dim), f, h, w, theta)
    v = x[:, 2 * hd:].reshape(Tc, heads, head_dim)
    return q, k, v
