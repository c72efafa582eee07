"""Torch-facing wrapper of the C ABI: device buffers come from PyTorch, every
step of the path runs in the library's kernels.  Methods only marshal pointers,
sizes and the current CUDA stream, then raise ``KvcError`` on a bad status.
"""

from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import KVC_BF16, KVC_FP4, KvcCache, check, lib


def _cuda_device(device) -> torch.device:
    d = torch.device(device)
    if d.type != "cuda":
        raise ValueError(f"expected a CUDA device, got {d}")
    return torch.device("cuda", torch.cuda.current_device() if d.index is None else d.index)


def _stream(device: torch.device, stream=None) -> ctypes.c_void_p:
    """The given stream (which must belong to `device`), else `device`'s current one."""
    s = torch.cuda.current_stream(device) if stream is None else stream
    if s.device != device:
        raise ValueError(f"stream on {s.device}, tensors on {device}")
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _require(t: torch.Tensor, dtype, shape, name: str, device: torch.device):
    if (t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous()
            or t.device != device):
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


class KVCache:
    """One layer's sink + short-window cache (bf16 or FP4) on a CUDA device.

    Region 0 holds the sink chunk; chunk c >= 1 lives in ring slot (c-1) % W.
    """

    def __init__(self, heads: int, head_dim: int, tokens_per_frame: int, chunk_frames: int,
                 window_chunks: int, dtype: str = "bf16", device="cuda", scrub_on_evict=False,
                 attn_workspace: bool = True, stage=False, rope_offset_frames: int = 0):
        """stage: False (none), True (the largest any call needs, kvc_cache_bytes(c, 8)), a
        size in bytes, or a contiguous CUDA tensor on the cache's device to use as the
        buffer (several caches whose calls are stream-ordered may share one) -- the
        staging buffer kvc_recache on an FP4 cache and kvc_project_append use, and
        that sinkwin_attn on an FP4 cache decodes K/V into when it holds them.
        rope_offset_frames: the multi-shot RoPE offset."""
        self.c = KvcCache()
        c = self.c
        c.heads, c.head_dim = heads, head_dim
        c.tokens_per_frame, c.chunk_frames = tokens_per_frame, chunk_frames
        c.window_chunks = window_chunks
        c.dtype = {"bf16": KVC_BF16, "fp4": KVC_FP4}[dtype]
        c.scrub_on_evict = 1 if scrub_on_evict else 0
        c.rope_offset_frames = int(rope_offset_frames)
        self.dtype = dtype
        self.device = _cuda_device(device)
        self.H, self.D = heads, head_dim
        self.Tc = tokens_per_frame * chunk_frames
        self.W = window_chunks
        self.S = (1 + window_chunks) * self.Tc
        L = lib()
        nbytes = [L.kvc_cache_bytes(ctypes.byref(c), i) for i in range(9)]
        if nbytes[0] == 0:
            raise ValueError("invalid cache geometry")
        if dtype == "bf16":
            self.k = torch.zeros((self.S, heads, head_dim), dtype=torch.bfloat16, device=self.device)
            self.v = torch.zeros_like(self.k)
            self.k_scale = self.v_scale = self.k_gscale = self.v_gscale = None
        else:
            self.k = torch.zeros((self.S, heads, head_dim // 2), dtype=torch.uint8, device=self.device)
            self.v = torch.zeros_like(self.k)
            self.k_scale = torch.zeros((self.S, heads, head_dim // 16), dtype=torch.uint8,
                                       device=self.device)
            self.v_scale = torch.zeros_like(self.k_scale)
            self.k_gscale = torch.zeros(1 + window_chunks, dtype=torch.float32, device=self.device)
            self.v_gscale = torch.zeros_like(self.k_gscale)
        self.ws = torch.zeros(_abi.KVC_WS_WORDS, dtype=torch.int32, device=self.device)
        # attention workspace: lets sinkwin_attn spread the work evenly over all SMs
        self.attn_ws = (torch.zeros(nbytes[7], dtype=torch.uint8, device=self.device)
                        if attn_workspace and nbytes[7] > 0 else None)
        c.attn_ws = 0 if self.attn_ws is None else self.attn_ws.data_ptr()
        c.attn_ws_bytes = 0 if self.attn_ws is None else nbytes[7]
        if isinstance(stage, torch.Tensor):
            if not stage.is_cuda or not stage.is_contiguous() or stage.device != self.device:
                raise ValueError("stage: expected a contiguous CUDA tensor on the cache's device")
            self.stage = stage
            sb = stage.numel() * stage.element_size()
        else:
            sb = nbytes[8] if stage is True else int(stage or 0)
            self.stage = torch.empty(sb, dtype=torch.uint8, device=self.device) if sb > 0 else None
        c.stage = 0 if self.stage is None else self.stage.data_ptr()
        c.stage_bytes = sb
        for name, t, nb in (("k", self.k, nbytes[0]), ("v", self.v, nbytes[1]),
                            ("k_scale", self.k_scale, nbytes[2]), ("v_scale", self.v_scale, nbytes[3]),
                            ("k_gscale", self.k_gscale, nbytes[4]), ("v_gscale", self.v_gscale, nbytes[5]),
                            ("dev_ws", self.ws, nbytes[6])):
            got = 0 if t is None else t.numel() * t.element_size()
            if got != nb:
                raise RuntimeError(f"{name}: {got} bytes allocated, library wants {nb}")
            setattr(c, name, 0 if t is None else t.data_ptr())
        check(L.kvc_init(ctypes.byref(c)), "kvc_init")

    # -- state --------------------------------------------------------------
    @property
    def chunk_of_region(self) -> list[int]:
        return [int(self.c.chunk_of_region[i]) for i in range(1 + self.W)]

    @property
    def frame0_of_region(self) -> list[int]:
        return [int(self.c.frame0_of_region[i]) for i in range(1 + self.W)]

    @property
    def shot(self) -> int:
        return int(self.c.shot)

    # -- calls ---------------------------------------------------------------
    # Every call runs with the cache's device current and on that device's stream:
    # the library launches on the current device, with the pointers it is given.
    def append(self, k: torch.Tensor, v: torch.Tensor, chunk_idx: int, stream=None) -> None:
        shp = (self.Tc, self.H, self.D)
        _require(k, torch.bfloat16, shp, "k", self.device)
        _require(v, torch.bfloat16, shp, "v", self.device)
        with torch.cuda.device(self.device):
            check(lib().kvc_append(ctypes.byref(self.c), _ptr(k), _ptr(v), int(chunk_idx),
                                   _stream(self.device, stream)), "kvc_append")

    def append_shot(self, k: torch.Tensor, v: torch.Tensor, chunk_idx: int, stream=None) -> None:
        """Append chunk_idx as the first chunk of a new shot (it becomes the sink)."""
        shp = (self.Tc, self.H, self.D)
        _require(k, torch.bfloat16, shp, "k", self.device)
        _require(v, torch.bfloat16, shp, "v", self.device)
        with torch.cuda.device(self.device):
            check(lib().kvc_append_shot(ctypes.byref(self.c), _ptr(k), _ptr(v), int(chunk_idx),
                                        _stream(self.device, stream)), "kvc_append_shot")

    def project_append(self, hidden: torch.Tensor, w_qkv: torch.Tensor, gamma_q, gamma_k,
                       chunk_idx: int, grid_h: int, grid_w: int, eps: float = 1e-6,
                       theta: float = 10000.0, new_shot: bool = False, q_out=None,
                       stream=None) -> torch.Tensor:
        """[Q|K|V] = hidden @ w_qkv with Q/K RMSNorm + 3D RoPE; K, V appended as
        chunk_idx; returns Q [Tc][H][D] bf16."""
        HD = self.H * self.D
        _require(hidden, torch.bfloat16, (self.Tc, HD), "hidden", self.device)
        _require(w_qkv, torch.bfloat16, (HD, 3 * HD), "w_qkv", self.device)
        for name, g in (("gamma_q", gamma_q), ("gamma_k", gamma_k)):
            if g is not None:
                _require(g, torch.float32, (HD,), name, self.device)
        if q_out is None:
            q_out = torch.empty((self.Tc, self.H, self.D), dtype=torch.bfloat16, device=self.device)
        _require(q_out, torch.bfloat16, (self.Tc, self.H, self.D), "q_out", self.device)
        with torch.cuda.device(self.device):
            check(lib().kvc_project_append(ctypes.byref(self.c), _ptr(hidden), _ptr(w_qkv),
                                           _ptr(gamma_q), _ptr(gamma_k), float(eps), int(chunk_idx),
                                           1 if new_shot else 0, int(grid_h), int(grid_w),
                                           float(theta), _ptr(q_out), _stream(self.device, stream)),
                  "kvc_project_append")
        return q_out

    def evict(self, chunk_idx: int, stream=None) -> None:
        with torch.cuda.device(self.device):
            check(lib().kvc_evict(ctypes.byref(self.c), int(chunk_idx), _stream(self.device, stream)),
                  "kvc_evict")

    def attn(self, q: torch.Tensor, softmax_scale: float, out: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
        tq = q.shape[0]
        _require(q, torch.bfloat16, (tq, self.H, self.D), "q", self.device)
        if out is None:
            out = torch.empty_like(q)
        _require(out, torch.bfloat16, (tq, self.H, self.D), "out", self.device)
        with torch.cuda.device(self.device):
            check(lib().sinkwin_attn(ctypes.byref(self.c), _ptr(q), _ptr(out), int(tq),
                                     float(softmax_scale), _stream(self.device, stream)), "sinkwin_attn")
        return out

    def recache(self, hidden: torch.Tensor, w_kv: torch.Tensor, gamma: torch.Tensor | None,
                chunk_ids, grid_h: int, grid_w: int, eps: float = 1e-6, theta: float = 10000.0,
                stream=None) -> None:
        n = len(chunk_ids)
        HD = self.H * self.D
        _require(hidden, torch.bfloat16, (n * self.Tc, HD), "hidden", self.device)
        _require(w_kv, torch.bfloat16, (HD, 2 * HD), "w_kv", self.device)
        if gamma is not None:
            _require(gamma, torch.float32, (HD,), "gamma", self.device)
        ids = (ctypes.c_int64 * n)(*[int(x) for x in chunk_ids])
        with torch.cuda.device(self.device):
            check(lib().kvc_recache(ctypes.byref(self.c), _ptr(hidden), _ptr(w_kv), _ptr(gamma),
                                    float(eps), ids, n, int(grid_h), int(grid_w), float(theta),
                                    _stream(self.device, stream)), "kvc_recache")

    def last_device_error(self, stream=None) -> int:
        with torch.cuda.device(self.device):
            return int(lib().kvc_last_device_error(ctypes.byref(self.c), _stream(self.device, stream)))


def quant_fp4(x: torch.Tensor, stream=None):
    """FP4-encode a bf16 tensor (numel % 16 == 0): returns (codes u8 [n/2],
    scales u8 [n/16], gscale f32 [1])."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA bf16 tensor")
    dev = _cuda_device(x.device)
    n = x.numel()
    codes = torch.empty(n // 2, dtype=torch.uint8, device=x.device)
    scales = torch.empty(n // 16, dtype=torch.uint8, device=x.device)
    g = torch.empty(1, dtype=torch.float32, device=x.device)
    ws = torch.empty(_abi.KVC_QUANT_WS_WORDS, dtype=torch.int32, device=x.device)
    with torch.cuda.device(dev):
        check(lib().kvc_quant_fp4(_ptr(x), int(n), _ptr(codes), _ptr(scales), _ptr(g), _ptr(ws),
                                  _stream(dev, stream)), "kvc_quant_fp4")
    return codes, scales, g


def gemm_fp4_ws_bytes(M: int, N: int, K: int) -> int:
    """Workspace bytes of gemm_fp4's two-phase path (f16 copies of A and B)."""
    return (M + N) * K * 2


def gemm_fp4(a, b, M: int, N: int, K: int, out=None, ws=None, dev_err=None,
             stream=None) -> torch.Tensor:
    """W4A4 projection deq(A) deq(B)^T -> bf16 [M][N].  `a` and `b` are
    (codes, scales, gscale) triples as quant_fp4 returns them: A's encode the
    [M][K] activations, B's an [N][K] weight (one row per output feature);
    codes u8 rows*K/2, scales u8 rows*K/16, gscale f32 [1], any contiguous
    shape.  N % 32 == 0 and K % 256 == 0.  ws: None (one fused kernel) or a
    CUDA tensor of at least gemm_fp4_ws_bytes(M, N, K) bytes (decode once,
    then an f16 GEMM).  dev_err: optional int32 CUDA tensor whose first word
    records a kernel timeout."""
    (ac, as_, ag), (bc, bs, bg) = a, b
    for t, name, n in ((ac, "a codes", M * K // 2), (as_, "a scales", M * K // 16),
                       (bc, "b codes", N * K // 2), (bs, "b scales", N * K // 16)):
        if (t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous()
                or t.numel() != n):
            raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor of {n} bytes")
    for t, name in ((ag, "a gscale"), (bg, "b gscale")):
        if t.dtype != torch.float32 or not t.is_cuda or t.numel() != 1:
            raise ValueError(f"{name} must be a CUDA float32 tensor of one element")
    if dev_err is not None and (dev_err.dtype != torch.int32 or not dev_err.is_cuda):
        raise ValueError("dev_err must be a CUDA int32 tensor")
    ws_bytes = 0
    if ws is not None:
        if not ws.is_cuda or not ws.is_contiguous() or ws.device != ac.device:
            raise ValueError("ws must be a contiguous CUDA tensor on the operands' device")
        ws_bytes = ws.numel() * ws.element_size()
    dev = _cuda_device(ac.device)
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=ac.device)
    _require(out, torch.bfloat16, (M, N), "out", ac.device)
    with torch.cuda.device(dev):
        check(lib().kvc_gemm_fp4(_ptr(ac), _ptr(as_), _ptr(ag), _ptr(bc), _ptr(bs), _ptr(bg),
                                 int(M), int(N), int(K), _ptr(out), _ptr(ws), int(ws_bytes),
                                 _ptr(dev_err), _stream(dev, stream)), "kvc_gemm_fp4")
    return out
