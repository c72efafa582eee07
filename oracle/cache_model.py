"""Logical model of one layer's sink + short-window KV cache (oracle side).

Restates LongLive summary page (yunpan.plus), 方法 §3 高效长推理:
* 帧汇聚点 (frame sink): the video's first frame chunk is pinned as global sink
  tokens that stay in the KV cache for good and are concatenated with the keys
  and values of every attention layer;
* 短窗口注意力 (short-window attention): attention is limited to a fixed window of
  recent frames, so the per-layer cache size depends on the window only.
The LONGLIVE news page (paooo.com), LONGLIVE的技术原理, states the same pair.

Readings (the pages leave them open):
* region 0 holds the sink chunk (chunk 0); chunk c >= 1 lives in ring slot
  (c-1) mod W, i.e. region 1 + (c-1) mod W, rows [region*Tc, (region+1)*Tc);
* the window's W slots include the chunk currently being generated, so the
  visible set of chunk c is {0} U {max(1, c-W+1) .. c};
* chunks arrive in order: the next chunk is the one after the last appended
  (whether or not that one is still cached), and it needs an empty slot, so the
  caller evicts the oldest window chunk first; re-appending the last chunk while
  it is cached overwrites it (one call per denoise step); the sink is never
  evicted.

Multi-shot sink (LongLive 2.0 inference blog, blog.hotdry.top, "序列并行与注意力
汇聚的协同设计": inference.multi_shot_sink resets the sink at each shot boundary,
inference.multi_shot_rope_offset shifts the RoPE positions).  Readings:
* the first chunk b of a new shot becomes the sink (region 0) and the previous
  sink leaves the cache; the window keeps the previous shot's recent chunks, and
  later chunks fill the ring by the same slot rule (b's own slot stays unused);
* token positions: chunk c's first frame sits at frame0(c) = c * chunk_frames +
  shot(c) * rope_offset_frames, shot(c) = the number of shot boundaries (new
  shots starting at a chunk > 0) at or before c; rope_offset_frames = 0 keeps
  positions absolute.
"""

from __future__ import annotations

import numpy as np


class CacheStateError(Exception):
    """The call is not valid in the cache's current state."""


def region_of_chunk(c: int, window_chunks: int) -> int:
    return 0 if c == 0 else 1 + (c - 1) % window_chunks


def visible_chunks_of_step(c: int, window_chunks: int) -> list[int]:
    """Chunks a query chunk c attends to, in logical order (sink first)."""
    if c == 0:
        return [0]
    return [0] + list(range(max(1, c - window_chunks + 1), c + 1))


class CacheModel:
    """Dict-of-chunks model with the physical layout the library must produce."""

    def __init__(self, heads: int, head_dim: int, chunk_tokens: int, window_chunks: int,
                 chunk_frames: int = 1, rope_offset_frames: int = 0):
        self.H, self.D, self.Tc, self.W = heads, head_dim, chunk_tokens, window_chunks
        self.chunk_frames, self.rope_offset = chunk_frames, rope_offset_frames
        self.chunk_of_region = [-1] * (1 + window_chunks)
        self.last = -1  # highest chunk appended so far
        self.shot = 0   # shot boundaries so far
        self.k: dict[int, np.ndarray] = {}
        self.v: dict[int, np.ndarray] = {}
        self.frame0: dict[int, int] = {}  # first-frame RoPE position of each cached chunk

    def region_of(self, c: int) -> int:
        """Region 0 for the sink (chunk 0, or a shot's first chunk), else the ring slot."""
        return 0 if c == 0 or c == self.chunk_of_region[0] else region_of_chunk(c, self.W)

    # -- state queries ------------------------------------------------------
    def present_chunks(self) -> list[int]:
        """Chunks in the cache in logical order: sink first, then oldest -> newest."""
        win = sorted(c for c in self.chunk_of_region[1:] if c >= 0)
        sink = self.chunk_of_region[0]
        return ([sink] if sink >= 0 else []) + win

    def window_chunks(self) -> list[int]:
        return sorted(c for c in self.chunk_of_region[1:] if c >= 0)

    def frame0_of_region(self) -> list[int]:
        return [self.frame0[c] if c >= 0 else -1 for c in self.chunk_of_region]

    def newest(self) -> int:
        p = self.present_chunks()
        return p[-1] if p else -1

    def kv_length(self) -> int:
        return len(self.present_chunks()) * self.Tc

    # -- state transitions --------------------------------------------------
    def _store(self, c, r, k, v, fresh):
        self.chunk_of_region[r] = c
        self.last = c
        if fresh:
            self.frame0[c] = c * self.chunk_frames + self.shot * self.rope_offset
        self.k[c] = np.array(k, dtype=np.float64, copy=True)
        self.v[c] = np.array(v, dtype=np.float64, copy=True)

    def append(self, c: int, k: np.ndarray, v: np.ndarray) -> None:
        if c < 0:
            raise ValueError("negative chunk index")
        if k.shape != (self.Tc, self.H, self.D) or v.shape != k.shape:
            raise ValueError("chunk shape mismatch")
        r = self.region_of(c)
        if c == self.last + 1:
            if self.chunk_of_region[r] != -1:
                raise CacheStateError("slot still holds an older chunk: evict it first")
        elif not (c == self.last and self.chunk_of_region[r] == c):
            raise CacheStateError("only the next chunk, or the last one while cached, may be appended")
        self._store(c, r, k, v, fresh=(c != self.last or self.chunk_of_region[r] != c))

    def append_shot(self, c: int, k: np.ndarray, v: np.ndarray) -> None:
        """Chunk c opens a new shot: it becomes the sink, the old sink leaves."""
        if k.shape != (self.Tc, self.H, self.D) or v.shape != k.shape:
            raise ValueError("chunk shape mismatch")
        if c == self.last + 1:
            old = self.chunk_of_region[0]
            if old >= 0:
                del self.k[old], self.v[old], self.frame0[old]
            if c > 0:
                self.shot += 1
            self.chunk_of_region[0] = -1
            self._store(c, 0, k, v, fresh=True)
        elif c == self.last and self.chunk_of_region[0] == c:
            self._store(c, 0, k, v, fresh=False)
        else:
            raise CacheStateError("a new shot starts at the next chunk (or overwrites its own sink)")

    def evict(self, c: int) -> None:
        if c == 0 or c == self.chunk_of_region[0]:
            raise CacheStateError("the sink chunk is never evicted")
        win = self.window_chunks()
        if c not in win:
            raise CacheStateError("chunk is not in the window")
        if c != win[0]:
            raise CacheStateError("only the oldest window chunk may be evicted")
        self.chunk_of_region[region_of_chunk(c, self.W)] = -1
        del self.k[c], self.v[c], self.frame0[c]

    def recache(self, chunk_ids: list[int], k_new: np.ndarray, v_new: np.ndarray) -> None:
        """Overwrite the K/V of every present chunk (chunk_ids in logical order)."""
        if list(chunk_ids) != self.present_chunks():
            raise CacheStateError("recache must list exactly the cached chunks, sink first")
        for i, c in enumerate(chunk_ids):
            sl = slice(i * self.Tc, (i + 1) * self.Tc)
            self.k[c] = np.array(k_new[sl], dtype=np.float64, copy=True)
            self.v[c] = np.array(v_new[sl], dtype=np.float64, copy=True)

    # -- views ---------------------------------------------------------------
    def visible_kv(self):
        """Visible K and V concatenated in logical order, [L][H][D]."""
        cs = self.present_chunks()
        if self.chunk_of_region[0] < 0:
            raise CacheStateError("attention needs the sink chunk")
        return (np.concatenate([self.k[c] for c in cs], axis=0),
                np.concatenate([self.v[c] for c in cs], axis=0))

    def physical(self, fill=np.nan):
        """Expected physical cache K, V [(1+W)*Tc][H][D]; empty regions hold ``fill``."""
        rows = (1 + self.W) * self.Tc
        K = np.full((rows, self.H, self.D), fill, dtype=np.float64)
        V = np.full_like(K, fill)
        for r, c in enumerate(self.chunk_of_region):
            if c >= 0:
                K[r * self.Tc:(r + 1) * self.Tc] = self.k[c]
                V[r * self.Tc:(r + 1) * self.Tc] = self.v[c]
        return K, V
