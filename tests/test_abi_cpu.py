"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/kvc.h declares, agrees on the struct layout, sizes buffers by the closed
form, and rejects invalid calls before any launch without changing state."""

import ctypes
import os
import re

import pytest

from sink_short_window_sinkwin_b300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    txt = open(os.path.join(ROOT, "include", "kvc.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", txt, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


@pytest.fixture(scope="module")
def lib():
    return _abi.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "sinkwin_attn" in names and "kvc_recache" in names and "kvc_quant_fp4" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in _abi.SIGNATURES, f"binding lacks {n}"
    assert set(_abi.SIGNATURES) == set(names)


def test_struct_layout(lib):
    assert lib.kvc_sizeof_cache() == ctypes.sizeof(_abi.KvcCache)


def _cache(dtype=_abi.KVC_BF16, H=12, D=128, tpf=1560, cf=3, W=3):
    c = _abi.KvcCache()
    c.heads, c.head_dim, c.tokens_per_frame, c.chunk_frames, c.window_chunks = H, D, tpf, cf, W
    c.dtype = dtype
    # fake, never dereferenced device addresses (16-byte aligned)
    c.k, c.v, c.dev_ws = 0x10000000, 0x20000000, 0x30000000
    if dtype == _abi.KVC_FP4:
        c.k_scale, c.v_scale, c.k_gscale, c.v_gscale = 0x40000000, 0x50000000, 0x60000000, 0x70000000
    return c


def test_buffer_sizes_closed_form(lib):
    c = _cache()
    S = 4 * 4680
    assert lib.kvc_cache_bytes(ctypes.byref(c), 0) == S * 12 * 128 * 2 == 57507840
    assert lib.kvc_cache_bytes(ctypes.byref(c), 2) == 0
    assert lib.kvc_cache_bytes(ctypes.byref(c), 6) == _abi.KVC_WS_WORDS * 4
    f = _cache(_abi.KVC_FP4)
    assert lib.kvc_cache_bytes(ctypes.byref(f), 0) == S * 12 * 64
    assert lib.kvc_cache_bytes(ctypes.byref(f), 3) == S * 12 * 8
    assert lib.kvc_cache_bytes(ctypes.byref(f), 4) == 4 * 4
    bad = _cache(D=24)
    assert lib.kvc_cache_bytes(ctypes.byref(bad), 0) == 0


def test_init_validation(lib):
    c = _cache()
    assert lib.kvc_init(ctypes.byref(c)) == _abi.KVC_OK
    assert list(c.chunk_of_region) == [-1] * 17
    assert c.init_magic == _abi.KVC_INIT_MAGIC
    for field, val in (("head_dim", 20), ("window_chunks", 0), ("window_chunks", 17), ("dtype", 7)):
        b = _cache()
        setattr(b, field, val)
        assert lib.kvc_init(ctypes.byref(b)) == _abi.KVC_EINVAL
    b = _cache()
    b.k = 0x10000008  # misaligned
    assert lib.kvc_init(ctypes.byref(b)) == _abi.KVC_EINVAL
    f = _cache(_abi.KVC_FP4)
    f.k_scale = 0
    assert lib.kvc_init(ctypes.byref(f)) == _abi.KVC_EINVAL


def test_geometry_products_cannot_overflow(lib):
    """Geometries whose row count or element count would overflow 64-bit
    arithmetic (int32 fields near 2^31) are rejected, not wrapped."""
    big = 2 ** 31 - 1
    for kw in (dict(tpf=big, cf=big), dict(tpf=big, cf=2), dict(H=big), dict(H=big, tpf=big, cf=big)):
        b = _cache(**kw)
        assert lib.kvc_cache_bytes(ctypes.byref(b), 0) == 0, kw
        assert lib.kvc_init(ctypes.byref(b)) == _abi.KVC_EINVAL, kw


def test_rejections_change_nothing(lib):
    c = _cache(H=1, D=64, tpf=16, cf=2, W=2)
    assert lib.kvc_init(ctypes.byref(c)) == _abi.KVC_OK
    before = list(c.chunk_of_region)
    s = None
    k = v = ctypes.c_void_p(0x80000000)
    assert lib.kvc_append(ctypes.byref(c), k, v, 1, s) == _abi.KVC_ESTATE  # sink first
    assert lib.kvc_append(ctypes.byref(c), k, v, -1, s) == _abi.KVC_EINVAL
    assert lib.kvc_append(ctypes.byref(c), None, v, 0, s) == _abi.KVC_EINVAL
    assert lib.kvc_append(ctypes.byref(c), ctypes.c_void_p(0x80000004), v, 0, s) == _abi.KVC_EINVAL
    assert lib.kvc_evict(ctypes.byref(c), 0, s) == _abi.KVC_ESTATE  # the sink
    assert lib.kvc_evict(ctypes.byref(c), 3, s) == _abi.KVC_ESTATE  # absent
    q = ctypes.c_void_p(0x90000000)
    assert lib.sinkwin_attn(ctypes.byref(c), q, q, 32, 0.125, s) == _abi.KVC_ESTATE  # no sink
    assert lib.sinkwin_attn(ctypes.byref(c), q, q, -1, 0.125, s) == _abi.KVC_EINVAL
    assert lib.sinkwin_attn(ctypes.byref(c), q, q, 0, 0.125, s) == _abi.KVC_OK  # empty: no-op
    assert lib.sinkwin_attn(ctypes.byref(c), q, q, 8, float("nan"), s) == _abi.KVC_EINVAL
    assert lib.sinkwin_attn(ctypes.byref(c), q, q, 8, -0.125, s) == _abi.KVC_EINVAL
    ids = (ctypes.c_int64 * 1)(0)
    assert lib.kvc_recache(ctypes.byref(c), q, q, None, 1e-6, ids, 1, 4, 4, 1e4, s) == _abi.KVC_ESTATE
    assert lib.kvc_recache(ctypes.byref(c), q, q, None, 1e-6, ids, 1, 3, 4, 1e4, s) == _abi.KVC_EINVAL
    assert list(c.chunk_of_region) == before
    # a valid append reaches the launch; without a GPU it fails as a CUDA error
    # and leaves the slot map untouched
    st = lib.kvc_append(ctypes.byref(c), k, v, 0, s)
    if st != _abi.KVC_OK:
        assert st == _abi.KVC_ECUDA
        assert list(c.chunk_of_region) == before
    d = _cache(H=1, D=96, tpf=16, cf=2, W=2)
    assert lib.kvc_init(ctypes.byref(d)) == _abi.KVC_OK
    d.chunk_of_region[0] = 0
    assert lib.sinkwin_attn(ctypes.byref(d), q, q, 8, 0.125, s) == _abi.KVC_EUNSUPPORTED


def test_quant_and_watchdog_validation(lib):
    x = ctypes.c_void_p(0x10000000)
    assert lib.kvc_quant_fp4(x, 15, x, x, x, x, None) == _abi.KVC_EINVAL
    assert lib.kvc_quant_fp4(x, 0, x, x, x, x, None) == _abi.KVC_EINVAL
    assert lib.kvc_quant_fp4(None, 32, x, x, x, x, None) == _abi.KVC_EINVAL
    # W4A4 projection: pointers, alignment and sizes are checked before any
    # launch; M = 0 returns at once
    g = ctypes.c_void_p(0x10000004)
    ok = (x, x, g, x, x, g)
    assert lib.kvc_gemm_fp4(*ok, 0, 256, 256, x, None, 0, None, None) == _abi.KVC_OK
    assert lib.kvc_gemm_fp4(None, None, None, None, None, None, 0, 256, 256, None, None, 0,
                            None, None) == _abi.KVC_OK
    assert lib.kvc_gemm_fp4(None, x, g, x, x, g, 4, 256, 256, x, None, 0, None, None) == _abi.KVC_EINVAL
    assert lib.kvc_gemm_fp4(*ok, 4, 256, 256, None, None, 0, None, None) == _abi.KVC_EINVAL
    assert lib.kvc_gemm_fp4(*ok, -1, 256, 256, x, None, 0, None, None) == _abi.KVC_EINVAL
    assert lib.kvc_gemm_fp4(*ok, 4, 0, 256, x, None, 0, None, None) == _abi.KVC_EINVAL
    assert lib.kvc_gemm_fp4(*ok, 4, 256, 256, ctypes.c_void_p(0x10000008), None, 0, None,
                            None) == _abi.KVC_EINVAL                   # out not 16-byte aligned
    assert lib.kvc_gemm_fp4(x, x, ctypes.c_void_p(0x10000002), x, x, g, 4, 256, 256, x, None, 0,
                            None, None) == _abi.KVC_EINVAL             # gscale not 4-byte aligned
    need = (4 + 256) * 256 * 2
    assert lib.kvc_gemm_fp4(*ok, 4, 256, 256, x, x, need - 1, None,
                            None) == _abi.KVC_EINVAL                   # workspace too small
    assert lib.kvc_gemm_fp4(*ok, 4, 256, 256, x, ctypes.c_void_p(0x10000008), need, None,
                            None) == _abi.KVC_EINVAL                   # workspace misaligned
    assert lib.kvc_gemm_fp4(*ok, 4, 100, 256, x, None, 0, None, None) == _abi.KVC_EUNSUPPORTED
    assert lib.kvc_gemm_fp4(*ok, 4, 256, 128, x, None, 0, None, None) == _abi.KVC_EUNSUPPORTED
    assert lib.kvc_watchdog_selftest(None, 10, None) == _abi.KVC_EINVAL
    assert lib.kvc_watchdog_selftest(x, 0, None) == _abi.KVC_EINVAL
    assert lib.kvc_status_string(_abi.KVC_ESTATE).decode().startswith("invalid in")


def test_binding_rejects_tensors_off_the_cache_device():
    """The binding checks dtype, shape, contiguity and device before any call:
    a host tensor, a tensor on another GPU or a strided view never reaches the
    library (its kernels would be handed a foreign pointer)."""
    import torch
    from sink_short_window_sinkwin_b300 import cache as cb
    dev = torch.device("cuda", 0)
    good = torch.empty(2, 3, dtype=torch.bfloat16, device="meta")
    with pytest.raises(ValueError, match="on cuda:0"):
        cb._require(torch.zeros(2, 3, dtype=torch.bfloat16), torch.bfloat16, (2, 3), "x", dev)
    with pytest.raises(ValueError):
        cb._require(good, torch.float32, (2, 3), "x", dev)
    with pytest.raises(ValueError):
        cb._require(torch.zeros(3, 2, dtype=torch.bfloat16).t(), torch.bfloat16, (2, 3), "x", dev)
    with pytest.raises(ValueError, match="CUDA device"):
        cb._cuda_device("cpu")
    assert cb._cuda_device("cuda:1") == torch.device("cuda", 1)
