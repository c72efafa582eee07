"""Seeded synthetic tensors with the shapes and value distributions of the
LongLive-1.3B self-attention layer and of the small parity case.

Every draw comes from ``numpy.random.default_rng(SeedSequence([...]))`` keyed by
(config, layer, chunk, tensor id), is drawn in float32 and rounded ONCE to
bfloat16 (round-to-nearest-even, done by torch's dtype conversion).  The
bfloat16 tensor is what the CUDA library reads; its exact float64 image is what
the oracle reads.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

# tensor ids inside a seed tuple
_TID_Q, _TID_K, _TID_V, _TID_OUTLIER_K, _TID_OUTLIER_V = 0, 1, 2, 3, 4
_TID_HIDDEN, _TID_WKV, _TID_WQKV, _TID_GAIN = 10, 11, 12, 13


@dataclass(frozen=True)
class Shapes:
    """Per-layer cache geometry.

    heads, head_dim      attention heads H and their width D
    tokens_per_frame     latent tokens of one frame (grid_h * grid_w)
    chunk_frames         frames per generated chunk; the sink is exactly one chunk
    window_chunks        W: ring slots of the short window (the current chunk included)
    grid_h, grid_w       patch grid of one latent frame (3D RoPE positions)
    """

    heads: int
    head_dim: int
    tokens_per_frame: int
    chunk_frames: int
    window_chunks: int
    grid_h: int
    grid_w: int

    @property
    def chunk_tokens(self) -> int:
        return self.tokens_per_frame * self.chunk_frames

    @property
    def cache_rows(self) -> int:
        return (1 + self.window_chunks) * self.chunk_tokens

    @property
    def model_dim(self) -> int:
        return self.heads * self.head_dim


# small parity case: 1 head, D=64, 16 tokens/frame (4x4 grid), 2-frame chunks, W=2
TINY = Shapes(heads=1, head_dim=64, tokens_per_frame=16, chunk_frames=2,
              window_chunks=2, grid_h=4, grid_w=4)
# LongLive-1.3B-shaped layer: 12 heads x 128, 30x52 patches, 3-frame chunks, W=3
LAYER_1P3B = Shapes(heads=12, head_dim=128, tokens_per_frame=1560, chunk_frames=3,
                    window_chunks=3, grid_h=30, grid_w=52)


def seed_rng(*parts: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(p) for p in parts]))


def _to_bf16(a32: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)


def gaussian_bf16(shape, std: float, *seed_parts: int) -> torch.Tensor:
    """N(0, std^2) drawn in float32, rounded once to bfloat16 (CPU tensor)."""
    g = seed_rng(*seed_parts)
    a = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return _to_bf16(a)


def gaussian_outliers_bf16(shape, frac: float, factor: float, *seed_parts: int) -> torch.Tensor:
    """N(0,1) with a seeded Bernoulli(frac) subset multiplied by ``factor``."""
    g = seed_rng(*seed_parts)
    a = g.standard_normal(size=shape, dtype=np.float32)
    mask = g.random(size=shape) < frac
    a[mask] *= np.float32(factor)
    return _to_bf16(a)


def chunk_qkv(sh: Shapes, cfg: int, layer: int, chunk: int, dist: str = "rms1",
              q_rows: int | None = None):
    """Q, K, V of one chunk, each a bf16 CPU tensor [rows][H][D].

    dist:
      "rms1"     Q, K, V elementwise N(0,1) (rows of RMS 1; logits of std ~ sqrt(D)*tau)
      "literal"  Q, K elementwise N(0,1)/sqrt(D) (row L2 ~ 1), V N(0,1)
      "outliers" Q N(0,1); K, V N(0,1) with 1% of entries x8
    """
    rows = sh.chunk_tokens if q_rows is None else q_rows
    shp_q = (rows, sh.heads, sh.head_dim)
    shp = (sh.chunk_tokens, sh.heads, sh.head_dim)
    if dist == "rms1":
        q = gaussian_bf16(shp_q, 1.0, cfg, layer, chunk, _TID_Q)
        k = gaussian_bf16(shp, 1.0, cfg, layer, chunk, _TID_K)
        v = gaussian_bf16(shp, 1.0, cfg, layer, chunk, _TID_V)
    elif dist == "literal":
        s = 1.0 / np.sqrt(sh.head_dim)
        q = gaussian_bf16(shp_q, s, cfg, layer, chunk, _TID_Q)
        k = gaussian_bf16(shp, s, cfg, layer, chunk, _TID_K)
        v = gaussian_bf16(shp, 1.0, cfg, layer, chunk, _TID_V)
    elif dist == "outliers":
        q = gaussian_bf16(shp_q, 1.0, cfg, layer, chunk, _TID_Q)
        k = gaussian_outliers_bf16(shp, 0.01, 8.0, cfg, layer, chunk, _TID_OUTLIER_K)
        v = gaussian_outliers_bf16(shp, 0.01, 8.0, cfg, layer, chunk, _TID_OUTLIER_V)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return q, k, v


def device_seed(*parts: int) -> int:
    """63-bit seed for torch's device generator, derived from a seed tuple."""
    w = np.random.SeedSequence([int(p) for p in parts]).generate_state(2, np.uint32)
    return (int(w[0]) << 31) ^ int(w[1])


def chunk_qkv_device(sh: Shapes, cfg: int, layer: int, chunk: int, device="cuda"):
    """Q, K, V of one chunk drawn on the GPU, bf16 [Tc][H][D] each, with the
    single-layer distribution: Q, K elementwise N(0,1)/sqrt(D), V N(0,1).

    Each tensor comes from torch's counter-based device generator seeded by
    (config, layer, chunk, tensor id), drawn in float32 and rounded once to
    bfloat16, so re-drawing the same key reproduces it bit for bit: a test can
    rebuild any past chunk for the oracle instead of keeping it.  Used where
    the stream is too long to draw on the host (hundreds of chunks x layers).
    """
    shp = (sh.chunk_tokens, sh.heads, sh.head_dim)
    s = float(np.float32(1.0 / np.sqrt(sh.head_dim)))
    out = []
    for tid, std in ((_TID_Q, s), (_TID_K, s), (_TID_V, 1.0)):
        g = torch.Generator(device=device)
        g.manual_seed(device_seed(cfg, layer, chunk, tid))
        a = torch.randn(shp, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            a.mul_(std)
        out.append(a.to(torch.bfloat16))
    return tuple(out)


def recache_inputs(sh: Shapes, cfg: int, n_chunks: int, w_std: float = 0.02):
    """Hidden states [n*Tc][H*D] ~ N(0,1), K|V weight [H*D][2*H*D] ~ N(0, w_std^2),
    RMSNorm gain (all ones, float32)."""
    rows = n_chunks * sh.chunk_tokens
    hid = gaussian_bf16((rows, sh.model_dim), 1.0, cfg, 0, n_chunks, _TID_HIDDEN)
    wkv = gaussian_bf16((sh.model_dim, 2 * sh.model_dim), w_std, cfg, 0, 0, _TID_WKV)
    gamma = torch.ones(sh.model_dim, dtype=torch.float32)
    return hid, wkv, gamma


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 image of a bfloat16 (or float32) CPU tensor."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def project_inputs(sh: Shapes, cfg: int, chunk: int, w_std: float = 0.02):
    """One chunk's hidden states [Tc][H*D] ~ N(0,1) and the Q|K|V weight
    [H*D][3*H*D] ~ N(0, w_std^2) (the same weight for every chunk of a cfg)."""
    hid = gaussian_bf16((sh.chunk_tokens, sh.model_dim), 1.0, cfg, 1, chunk, _TID_HIDDEN)
    w = gaussian_bf16((sh.model_dim, 3 * sh.model_dim), w_std, cfg, 1, 0, _TID_WQKV)
    return hid, w


def gains(sh: Shapes, cfg: int):
    """RMSNorm gains for Q and K, float32 [H*D] each, uniform in [0.5, 1.5]."""
    g = seed_rng(cfg, 1, 0, _TID_GAIN)
    gq = g.uniform(0.5, 1.5, sh.model_dim).astype(np.float32)
    gk = g.uniform(0.5, 1.5, sh.model_dim).astype(np.float32)
    return torch.from_numpy(gq), torch.from_numpy(gk)
