"""GPU parity of the prompt-switch KV recache (projection GEMM + RMSNorm + 3D
RoPE written into the cache), then attention over the rebuilt cache."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import recache as orc
from oracle.cache_model import CacheModel
from synth import LAYER_1P3B, TINY, Shapes, chunk_qkv, recache_inputs, bf16_to_f64
from tests.gpu_helpers import ATOL_BF16, RELL2_BF16, SAMPLE_ROWS_4680, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_short_window_sinkwin_b300 as swl
    return swl


def _fill(swl, sh: Shapes, upto: int):
    """Cache + oracle model holding the chunks present after streaming 0..upto
    (zero K/V: the recache overwrites them)."""
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.window_chunks)
    model = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, sh.window_chunks)
    z = torch.zeros((sh.chunk_tokens, sh.heads, sh.head_dim), dtype=torch.bfloat16, device="cuda")
    zn = np.zeros((sh.chunk_tokens, sh.heads, sh.head_dim))
    for c in range(upto + 1):
        if c > sh.window_chunks:
            cache.evict(c - sh.window_chunks)
            model.evict(c - sh.window_chunks)
        cache.append(z, z, c)
        model.append(c, zn, zn)
    return cache, model


def _recache_both(swl, sh, cache, model, cfg, gamma_rand=False):
    ids = model.present_chunks()
    hid, wkv, gamma = recache_inputs(sh, cfg, len(ids))
    if gamma_rand:
        g = np.random.default_rng(cfg).uniform(0.5, 1.5, sh.model_dim).astype(np.float32)
        gamma = torch.from_numpy(g)
    cache.recache(hid.cuda(), wkv.cuda(), gamma.cuda(), ids, sh.grid_h, sh.grid_w)
    k, v = orc.recache(bf16_to_f64(hid), bf16_to_f64(wkv), gamma.double().numpy(), ids,
                       sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.grid_w)
    model.recache(ids, k, v)
    torch.cuda.synchronize()
    return ids


def _compare_cache(cache, model, sh, rows=None, what=""):
    Kp, Vp = model.physical(fill=0.0)
    gk, gv = to64(cache.k), to64(cache.v)
    for r, ch in enumerate(model.chunk_of_region):
        if ch < 0:
            continue
        base = r * sh.chunk_tokens
        sel = np.arange(sh.chunk_tokens) if rows is None else np.asarray(rows)
        assert_close(gk[base + sel], Kp[base + sel], ATOL_BF16, RELL2_BF16, f"{what} K region {r}")
        assert_close(gv[base + sel], Vp[base + sel], ATOL_BF16, RELL2_BF16, f"{what} V region {r}")


def test_recache_tiny_then_attention(swl):
    sh = TINY
    cache, model = _fill(swl, sh, 4)  # present: 0, 3, 4
    assert model.present_chunks() == [0, 3, 4]
    _recache_both(swl, sh, cache, model, 4, gamma_rand=True)
    _compare_cache(cache, model, sh, what="tiny")
    q = chunk_qkv(sh, 4, 0, 5, "rms1")[0]
    out = cache.attn(q.cuda(), 0.125)
    torch.cuda.synchronize()
    assert_close(to64(out), oatt.sinkwin_attention(model, bf16_to_f64(q), 0.125),
                 ATOL_BF16, RELL2_BF16, "tiny attention after recache")


def test_recache_two_column_tiles_noncontiguous_positions(swl):
    """H*D = 512: the K row spans two 256-wide GEMM tiles, so the RMSNorm needs
    the whole parked fp32 row; 180-token chunks make row tiles straddle chunks,
    and chunks {0, 97, 98, 99} put frame positions far apart (294..299 next to
    0..2)."""
    sh = Shapes(4, 128, 60, 3, 3, 6, 10)
    cache, model = _fill(swl, sh, 99)
    assert model.present_chunks() == [0, 97, 98, 99]
    _recache_both(swl, sh, cache, model, 44)
    _compare_cache(cache, model, sh, what="two tiles")


@pytest.mark.parametrize("heads,head_dim", [(1, 128), (2, 128), (6, 128)])
def test_recache_tile_widths(swl, heads, head_dim):
    """H*D = 128, 256, 768: GEMM column tiles 128 or 256 wide (one, one and three
    of them).  Three 120-token chunks are 360 rows, so the last of the three
    row tiles ends inside the tile (rows past the end load as zeros and store
    nothing)."""
    sh = Shapes(heads, head_dim, 40, 3, 2, 4, 10)
    cache, model = _fill(swl, sh, 2)
    assert model.present_chunks() == [0, 1, 2]
    _recache_both(swl, sh, cache, model, 7, gamma_rand=True)
    _compare_cache(cache, model, sh, what=f"H*D={heads * head_dim}")


def test_recache_layer_full_size_then_attention(swl):
    """Prompt switch before chunk 4: chunks {0,1,2,3} = 12 frames, 18720 x 1536
    hidden states, then one 4680-query attention step over the rebuilt cache."""
    sh = LAYER_1P3B
    cache, model = _fill(swl, sh, 3)
    _recache_both(swl, sh, cache, model, 4)
    rows = [0, 1, 51, 52, 127, 128, 1559, 1560, 3000, 4607, 4608, 4679]
    _compare_cache(cache, model, sh, rows=rows, what="layer")
    q = chunk_qkv(sh, 4, 0, 4, "rms1")[0]
    scale = 1.0 / math.sqrt(sh.head_dim)
    out = cache.attn(q.cuda(), scale)
    torch.cuda.synchronize()
    kk, vv = model.visible_kv()
    want = oatt.attention_rows(bf16_to_f64(q), kk, vv, scale, SAMPLE_ROWS_4680)
    print(assert_close(to64(out)[SAMPLE_ROWS_4680], want, ATOL_BF16, RELL2_BF16,
                       "attention after layer recache"))
    assert cache.last_device_error() == swl.KVC_OK


def test_recache_equals_appended_projections(swl):
    """Recache => append consistency on the GPU: stream chunks 0..6 whose K/V
    are the oracle's per-chunk projections (project_chunk: norm + 3D RoPE at
    each chunk's own positions), rounded to bf16 and appended; then recache
    the present chunks {0, 4, 5, 6} from the same hidden states with the K|V
    columns of the same weight.  Both the appended cache and the recached one
    match the oracle model within the bf16 tolerance (H*D = 512: the K row
    spans two GEMM tiles; 180-token chunks straddle row tiles)."""
    sh = Shapes(4, 128, 60, 3, 3, 6, 10)
    HD, Tc = sh.model_dim, sh.chunk_tokens
    rng = np.random.default_rng(61)
    w_qkv = torch.from_numpy((rng.standard_normal((HD, 3 * HD)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    gk = torch.from_numpy(rng.uniform(0.5, 1.5, HD).astype(np.float32))
    w64 = bf16_to_f64(w_qkv)
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.window_chunks)
    model = CacheModel(sh.heads, sh.head_dim, Tc, sh.window_chunks)
    hid = {}
    for c in range(7):
        hid[c] = torch.from_numpy(rng.standard_normal((Tc, HD)).astype(np.float32)).to(torch.bfloat16)
        if c > sh.window_chunks:
            cache.evict(c - sh.window_chunks)
            model.evict(c - sh.window_chunks)
        _, k, v = orc.project_chunk(bf16_to_f64(hid[c]), w64, None, gk.double().numpy(), c,
                                    sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                                    sh.grid_w)
        cache.append(torch.from_numpy(k).to(torch.bfloat16).cuda(),
                     torch.from_numpy(v).to(torch.bfloat16).cuda(), c)
        model.append(c, k, v)
    ids = model.present_chunks()
    assert ids == [0, 4, 5, 6]
    torch.cuda.synchronize()
    _compare_cache(cache, model, sh, what="appended")
    hcat = torch.cat([hid[c] for c in ids]).cuda()
    cache.recache(hcat, w_qkv[:, HD:].contiguous().cuda(), gk.cuda(), ids, sh.grid_h, sh.grid_w)
    torch.cuda.synchronize()
    _compare_cache(cache, model, sh, what="recached")
    assert cache.last_device_error() == swl.KVC_OK


def test_recache_rejections(swl):
    sh = TINY
    cache, model = _fill(swl, sh, 2)
    hid, wkv, gamma = recache_inputs(sh, 0, 3)
    with pytest.raises(swl.KvcError) as e:
        cache.recache(hid.cuda(), wkv.cuda(), None, [0, 2, 1], sh.grid_h, sh.grid_w)
    assert e.value.status == swl.KVC_ESTATE
    # gamma must be 16-byte aligned (read as float4): a view one float in is refused
    g_off = torch.ones(sh.heads * sh.head_dim + 1, dtype=torch.float32, device="cuda")[1:]
    with pytest.raises(swl.KvcError) as e:
        cache.recache(hid.cuda(), wkv.cuda(), g_off, [0, 1, 2], sh.grid_h, sh.grid_w)
    assert e.value.status == swl.KVC_EINVAL
    f = swl.KVCache(1, 64, 16, 2, 2, dtype="fp4")
    z = torch.zeros((32, 1, 64), dtype=torch.bfloat16, device="cuda")
    f.append(z, z, 0)
    with pytest.raises(swl.KvcError) as e:
        f.recache(hid[:32].cuda(), wkv.cuda(), None, [0], 4, 4)
    assert e.value.status == swl.KVC_EUNSUPPORTED
