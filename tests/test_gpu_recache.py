"""GPU parity of the prompt-switch KV recache (projection GEMM + RMSNorm + 3D
RoPE written into the cache), then attention over the rebuilt cache."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import fp4 as ofp4
from oracle import recache as orc
from oracle.cache_model import CacheModel
from synth import LAYER_1P3B, TINY, Shapes, chunk_qkv, recache_inputs, bf16_to_f64
from tests.gpu_helpers import (ATOL_BF16, ATOL_FP4, RELL2_BF16, SAMPLE_ROWS_4680, assert_close,
                               to64)

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
    """H*D = 512: one CTA holds the whole K row (fused launch, a cluster of
    one); 180-token chunks make row tiles straddle chunks, and chunks
    {0, 97, 98, 99} put frame positions far apart (294..299 next to 0..2)."""
    sh = Shapes(4, 128, 60, 3, 3, 6, 10)
    cache, model = _fill(swl, sh, 99)
    assert model.present_chunks() == [0, 97, 98, 99]
    _recache_both(swl, sh, cache, model, 44)
    _compare_cache(cache, model, sh, what="two tiles")


@pytest.mark.parametrize("heads,head_dim", [(8, 128), (8, 64), (16, 64), (16, 128), (16, 32)])
def test_recache_fused_cluster_widths(swl, heads, head_dim):
    """The fused launch at H*D = 1024, 512, 1024 and 2048: clusters of 2, 1, 2
    and 4 CTAs exchange per-row partial sums of squares; head widths 128 and
    64 change how the 32-column chunks map to rotation pairs and heads.  Head
    width 32 (H*D = 512) takes the three-launch path.
    Four 120-token chunks (480 rows) end the last row tile inside the tile,
    and chunks {0, 4, 5, 6} make the frame positions jump."""
    sh = Shapes(heads, head_dim, 40, 3, 3, 4, 10)
    cache, model = _fill(swl, sh, 6)
    assert model.present_chunks() == [0, 4, 5, 6]
    _recache_both(swl, sh, cache, model, 17, gamma_rand=True)
    _compare_cache(cache, model, sh, what=f"fused H*D={heads * head_dim} D={head_dim}")


@pytest.mark.parametrize("shape", [(8, 128, 64, 2, 3, 2, 32), (4, 128, 200, 1, 3, 2, 100),
                                   (4, 128, 60, 3, 3, 6, 10)])
def test_recache_fused_rotation_paths(swl, shape):
    """The fused launch's rotation and store paths: a 2 x 32 grid (every warp's
    32 rows share one grid row and at most two frames: per-warp frame/row
    tables, column table, 8-row bulk stores); a 2 x 100 grid (the column table
    would exceed its space: per-row column rotations); 180-token chunks (not a
    multiple of 8 rows: lane stores) with a 6 x 10 grid (up to four grid rows
    per warp: per-row frame/row rotations)."""
    sh = Shapes(*shape)
    cache, model = _fill(swl, sh, 5)
    _recache_both(swl, sh, cache, model, 23, gamma_rand=True)
    _compare_cache(cache, model, sh, what=f"fused rotation paths {shape}")


def test_recache_side_launch_four_cta_clusters(swl):
    """H*D = 2048: clusters of 4 CTAs (33 fit on 148 SMs), so the 16 SMs left
    take the V items of the last row tiles in the cluster-free launch; 4 chunks
    of 1280 rows (40 row tiles) make that split non-empty.  Sampled rows of
    every region, both launches' row tiles among them."""
    sh = Shapes(16, 128, 640, 2, 3, 10, 64)
    cache, model = _fill(swl, sh, 3)
    assert model.present_chunks() == [0, 1, 2, 3]
    _recache_both(swl, sh, cache, model, 29, gamma_rand=True)
    rows = [0, 1, 127, 128, 640, 1023, 1024, 1151, 1152, 1279]
    _compare_cache(cache, model, sh, rows=rows, what="H*D=2048 side launch")
    assert cache.last_device_error() == swl.KVC_OK


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


def test_recache_layer_graph_capture_matches_eager(swl):
    """At the LongLive-1.3B shape the recache is two launches on two streams
    (3-CTA clusters, and the SMs no cluster fits taking some V items), forked
    from and joined back to the caller's stream with events.  Captured into a
    CUDA graph and replayed onto a scrubbed cache, it must write exactly what
    the eager call wrote."""
    sh = LAYER_1P3B
    cache, model = _fill(swl, sh, 3)
    ids = model.present_chunks()
    hid, wkv, gamma = recache_inputs(sh, 5, len(ids))
    hid, wkv, gamma = hid.cuda(), wkv.cuda(), gamma.cuda()
    cache.recache(hid, wkv, gamma, ids, sh.grid_h, sh.grid_w)
    torch.cuda.synchronize()
    k0, v0 = cache.k.clone(), cache.v.clone()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        cache.recache(hid, wkv, gamma, ids, sh.grid_h, sh.grid_w)
    cache.k.fill_(float("nan"))
    cache.v.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(cache.k.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(cache.v.view(torch.int16), v0.view(torch.int16))
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
    # an FP4 cache recaches through the staging buffer: without one (or with one
    # too small for the listed chunks) the call is refused
    f = swl.KVCache(1, 64, 16, 2, 2, dtype="fp4")
    z = torch.zeros((32, 1, 64), dtype=torch.bfloat16, device="cuda")
    f.append(z, z, 0)
    with pytest.raises(swl.KvcError) as e:
        f.recache(hid[:32].cuda(), wkv.cuda(), None, [0], 4, 4)
    assert e.value.status == swl.KVC_EINVAL
    f2 = swl.KVCache(1, 64, 16, 2, 2, dtype="fp4", stage=32 * 64 * 4 - 16)
    f2.append(z, z, 0)
    with pytest.raises(swl.KvcError) as e:
        f2.recache(hid[:32].cuda(), wkv.cuda(), None, [0], 4, 4)
    assert e.value.status == swl.KVC_EINVAL


# ---------------------------------------------------------------------------
# recache into an FP4 cache
# ---------------------------------------------------------------------------
def _fill_fp4(swl, sh: Shapes, upto: int):
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.window_chunks,
                        dtype="fp4", stage=True)
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


def _check_fp4_recache(swl, sh, upto, cfg, rows=None, what="", q_rows=None):
    """Recache an FP4 cache, then check (1) every region's codes, block scales
    and tensor scale are bit-exactly the oracle's encode of the bf16 K/V the
    kernels left in the staging buffer (one tensor per region); (2) the decoded
    cache lies within the FP4 reconstruction bound (one E2M1 step at the block's
    scale) plus the bf16 tolerance of the oracle's float64 recache; (3) attention
    over the cache matches the oracle run on the oracle's own quantised recache
    (its float64 K/V rounded to bf16, then encoded per region)."""
    cache, model = _fill_fp4(swl, sh, upto)
    ids = model.present_chunks()
    hid, wkv, gamma = recache_inputs(sh, cfg, len(ids))
    cache.recache(hid.cuda(), wkv.cuda(), gamma.cuda(), ids, sh.grid_h, sh.grid_w)
    torch.cuda.synchronize()
    k64, v64 = orc.recache(bf16_to_f64(hid), bf16_to_f64(wkv), gamma.double().numpy(), ids,
                           sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.grid_w)
    Tc, n = sh.chunk_tokens, len(ids)
    hd = sh.model_dim
    st = cache.stage[: 2 * n * Tc * hd * 2].view(torch.bfloat16).view(2, n * Tc, sh.heads, sh.head_dim)
    st_k, st_v = st[0].float().cpu().numpy(), st[1].float().cpu().numpy()
    for i, c in enumerate(ids):
        r = cache.chunk_of_region.index(c)
        sl_r = slice(r * Tc, (r + 1) * Tc)
        sl_i = slice(i * Tc, (i + 1) * Tc)
        sel = np.arange(Tc) if rows is None else np.asarray(rows)
        for tname, stage_x, cb, sb, gb, ref in (
                ("K", st_k, cache.k, cache.k_scale, cache.k_gscale, k64),
                ("V", st_v, cache.v, cache.v_scale, cache.v_gscale, v64)):
            codes, scales, g = ofp4.quantize(stage_x[sl_i])
            assert np.array_equal(cb[sl_r].cpu().numpy(), codes), f"{what} {tname} codes, chunk {c}"
            assert np.array_equal(sb[sl_r].cpu().numpy(), scales), f"{what} {tname} scales, chunk {c}"
            assert gb[r].item() == float(g), f"{what} {tname} tensor scale, chunk {c}"
            xh = ofp4.dequantize(cb[sl_r].cpu().numpy(), sb[sl_r].cpu().numpy(), gb[r].item())
            unit = np.repeat(ofp4.E4M3_ALL[sb[sl_r].cpu().numpy()], 16, axis=-1) * gb[r].item()
            err = np.abs(xh - ref[sl_i])[sel] - unit[sel]
            assert err.max() <= ATOL_BF16, f"{what} {tname} chunk {c}: beyond the FP4 bound by {err.max():.3e}"
    # attention over the recached FP4 cache vs the oracle run on its own
    # quantised recache: float64 K/V rounded to bf16, encoded per region
    kk = np.concatenate([ofp4.dequantize(*ofp4.quantize(_bf16_round(k64[i * Tc:(i + 1) * Tc])))
                         for i in range(n)])
    vv = np.concatenate([ofp4.dequantize(*ofp4.quantize(_bf16_round(v64[i * Tc:(i + 1) * Tc])))
                         for i in range(n)])
    q = chunk_qkv(sh, cfg, 0, 99, "rms1", q_rows=q_rows)[0]
    scale = 1.0 / math.sqrt(sh.head_dim)
    out = cache.attn(q.cuda(), scale)
    torch.cuda.synchronize()
    qr = SAMPLE_ROWS_4680 if q.shape[0] == 4680 else list(range(q.shape[0]))
    want = oatt.attention_rows(bf16_to_f64(q), kk, vv, scale, qr)
    print(assert_close(to64(out)[qr], want, ATOL_FP4, None, f"{what} attention after FP4 recache",
                       plus_output_rounding=True))
    assert cache.last_device_error() == swl.KVC_OK


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 (round to nearest even, through float32) -> float32 values."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_recache_fp4_tiny(swl):
    _check_fp4_recache(swl, TINY, 4, 31, what="tiny")


def test_recache_fp4_noncontiguous_positions(swl):
    """H*D = 512 (two GEMM column tiles), 180-token chunks straddling row tiles,
    chunks {0, 97, 98, 99}: far-apart frame positions."""
    _check_fp4_recache(swl, Shapes(4, 128, 60, 3, 3, 6, 10), 99, 32, what="512-wide", q_rows=300)


def test_recache_fp4_layer_full_size(swl):
    """LongLive-1.3B layer: chunks {0, 1, 2, 3} = 18720 x 1536 hidden states
    recached into an FP4 cache, then one 4680-query attention step.  The
    encode checks cover sampled rows of every region (all of its codes are
    compared bit for bit)."""
    _check_fp4_recache(swl, LAYER_1P3B, 3, 33, rows=[0, 1, 51, 52, 1559, 1560, 3000, 4679],
                       what="layer", q_rows=4680)
