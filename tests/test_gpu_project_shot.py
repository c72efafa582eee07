"""GPU parity of the per-chunk projection that appends its own keys and values
(kvc_project_append) and of the multi-shot sink (kvc_append_shot with the
per-shot RoPE offset), through the C ABI, against the float64 oracle."""

import math
import random

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import fp4 as ofp4
from oracle import recache as orc
from oracle.cache_model import CacheModel, CacheStateError
from synth import LAYER_1P3B, TINY, Shapes, bf16_to_f64, chunk_qkv, gains, project_inputs
from tests.gpu_helpers import ATOL_BF16, ATOL_FP4, RELL2_BF16, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_short_window_sinkwin_b300 as swl
    return swl


def _oracle_chunk(sh, hid, w, gq, gk, c, frame0=None):
    return orc.project_chunk(bf16_to_f64(hid), bf16_to_f64(w), gq.double().numpy(),
                             gk.double().numpy(), c, sh.heads, sh.head_dim, sh.tokens_per_frame,
                             sh.chunk_frames, sh.grid_w, frame0=frame0)


def _stage_kv(cache, sh):
    """bf16 K and V the projection left in the staging buffer of an FP4 cache."""
    f32b = sh.chunk_tokens * sh.model_dim * 4
    kv = cache.stage[2 * f32b: 3 * f32b].view(torch.bfloat16).view(2, sh.chunk_tokens, sh.heads,
                                                                   sh.head_dim)
    return kv[0].float().cpu().numpy(), kv[1].float().cpu().numpy()


def _project_stream(swl, sh, cfg, steps, dtype, rows=None, shots=(), rope_offset=0, check_every=True):
    """Chunks 0..steps-1 through kvc_project_append (chunks in `shots` open a
    new shot), checking Q, the appended K/V (bf16: against the oracle's float64
    projection; FP4: codes bit-exact against the oracle's encode of the bf16
    K/V the kernels staged, decoded values within the FP4 bound) and the slot
    map, frame positions and shot count against the oracle model."""
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.window_chunks,
                        dtype=dtype, stage=True, rope_offset_frames=rope_offset)
    model = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, sh.window_chunks,
                       chunk_frames=sh.chunk_frames, rope_offset_frames=rope_offset)
    gq, gk = gains(sh, cfg)
    W, Tc = sh.window_chunks, sh.chunk_tokens
    sel = np.arange(Tc) if rows is None else np.asarray(rows)
    for c in range(steps):
        hid, w = project_inputs(sh, cfg, c)
        if (c - W) in model.window_chunks():
            cache.evict(c - W)
            model.evict(c - W)
        shot = c in shots
        f0 = c * sh.chunk_frames + (model.shot + (1 if shot and c > 0 else 0)) * rope_offset
        q = cache.project_append(hid.cuda(), w.cuda(), gq.cuda(), gk.cuda(), c, sh.grid_h, sh.grid_w,
                                 new_shot=shot)
        torch.cuda.synchronize()
        oq, ok, ov = _oracle_chunk(sh, hid, w, gq, gk, c, frame0=f0)
        if dtype == "bf16":
            (model.append_shot if shot else model.append)(c, ok, ov)
        else:
            sk, sv = _stage_kv(cache, sh)
            ek, ev = ofp4.quantize(sk), ofp4.quantize(sv)
            (model.append_shot if shot else model.append)(c, ofp4.dequantize(*ek), ofp4.dequantize(*ev))
        assert cache.chunk_of_region == model.chunk_of_region, c
        assert cache.frame0_of_region == model.frame0_of_region(), c
        assert cache.shot == model.shot
        if check_every or c == steps - 1:
            assert_close(to64(q)[sel], oq[sel], ATOL_BF16, RELL2_BF16, f"{dtype} Q of chunk {c}")
            r = model.chunk_of_region.index(c)
            sl = slice(r * Tc, (r + 1) * Tc)
            if dtype == "bf16":
                assert_close(to64(cache.k[sl])[sel], ok[sel], ATOL_BF16, RELL2_BF16, f"K of chunk {c}")
                assert_close(to64(cache.v[sl])[sel], ov[sel], ATOL_BF16, RELL2_BF16, f"V of chunk {c}")
            else:
                for tname, (codes, scales, g), cb, sb, gb, ref in (
                        ("K", ek, cache.k, cache.k_scale, cache.k_gscale, ok),
                        ("V", ev, cache.v, cache.v_scale, cache.v_gscale, ov)):
                    assert np.array_equal(cb[sl].cpu().numpy(), codes), f"{tname} codes of chunk {c}"
                    assert np.array_equal(sb[sl].cpu().numpy(), scales), f"{tname} scales of chunk {c}"
                    assert gb[r].item() == float(g), f"{tname} tensor scale of chunk {c}"
                    xh = ofp4.dequantize(codes, scales, g)
                    unit = np.repeat(ofp4.E4M3_ALL[scales], 16, axis=-1) * float(g)
                    assert (np.abs(xh - ref) - unit)[sel].max() <= ATOL_BF16, f"{tname} FP4 bound, chunk {c}"
        yield c, q, cache, model


@pytest.mark.parametrize("dtype", ["bf16", "fp4"])
def test_project_append_tiny_stream_then_attention(swl, dtype):
    """Six chunks projected and appended (evictions from chunk 3 on), the
    returned Q attending to the cache: against the oracle on the same bf16
    Q/K/V (or the same decoded FP4 K/V)."""
    sh = TINY
    scale = 1.0 / math.sqrt(sh.head_dim)
    for c, q, cache, model in _project_stream(swl, sh, 41, 6, dtype):
        out = cache.attn(q, scale)
        torch.cuda.synchronize()
        if dtype == "bf16":
            kk = np.concatenate([to64(cache.k[model.chunk_of_region.index(x) * sh.chunk_tokens:
                                               (model.chunk_of_region.index(x) + 1) * sh.chunk_tokens])
                                 for x in model.present_chunks()])
            vv = np.concatenate([to64(cache.v[model.chunk_of_region.index(x) * sh.chunk_tokens:
                                               (model.chunk_of_region.index(x) + 1) * sh.chunk_tokens])
                                 for x in model.present_chunks()])
            want = oatt.attention(to64(q), kk, vv, scale)
            assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, f"attention, step {c}")
        else:
            want = oatt.sinkwin_attention(model, to64(q), scale)
            assert_close(to64(out), want, ATOL_FP4, None, f"fp4 attention, step {c}",
                         plus_output_rounding=True)
    assert cache.last_device_error() == swl.KVC_OK


@pytest.mark.parametrize("H,D,tpf,cf,W", [(4, 128, 60, 3, 3), (6, 128, 40, 3, 2), (2, 64, 50, 1, 2)])
def test_project_append_shapes(swl, H, D, tpf, cf, W):
    """H*D = 512, 768, 128: the [Q|K|V] GEMM spans 6, 9 and 3 column tiles;
    ragged row tiles (180, 120 and 50-token chunks)."""
    sh = Shapes(H, D, tpf, cf, W, 1, tpf)
    for dtype in ("bf16", "fp4"):
        for _ in _project_stream(swl, sh, 42, W + 2, dtype):
            pass


def test_project_append_layer_full_size(swl):
    """LongLive-1.3B layer: 4680 x 1536 hidden states through the 1536 x 4608
    Q|K|V weight, chunks 0..4 (eviction at chunk 4); sampled rows of every
    chunk's Q, K and V against the oracle."""
    rows = [0, 1, 51, 52, 127, 128, 1559, 1560, 3000, 4607, 4608, 4679]
    for c, q, cache, model in _project_stream(swl, LAYER_1P3B, 43, 5, "bf16", rows=rows):
        pass
    assert cache.last_device_error() == swl.KVC_OK


def test_project_append_layer_full_size_fp4(swl):
    rows = [0, 52, 1560, 4679]
    for c, q, cache, model in _project_stream(swl, LAYER_1P3B, 44, 2, "fp4", rows=rows):
        pass
    assert cache.last_device_error() == swl.KVC_OK


def test_project_append_rejections(swl):
    sh = TINY
    hid, w = project_inputs(sh, 45, 0)
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.window_chunks)
    with pytest.raises(swl.KvcError) as e:  # no staging buffer
        cache.project_append(hid.cuda(), w.cuda(), None, None, 0, sh.grid_h, sh.grid_w)
    assert e.value.status == swl.KVC_EINVAL
    small = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                        sh.window_chunks, stage=sh.chunk_tokens * sh.model_dim * 8 - 16)
    with pytest.raises(swl.KvcError) as e:  # staging too small
        small.project_append(hid.cuda(), w.cuda(), None, None, 0, sh.grid_h, sh.grid_w)
    assert e.value.status == swl.KVC_EINVAL
    ok = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                     sh.window_chunks, stage=sh.chunk_tokens * sh.model_dim * 8)
    with pytest.raises(swl.KvcError) as e:  # chunk 1 before the sink
        ok.project_append(hid.cuda(), w.cuda(), None, None, 1, sh.grid_h, sh.grid_w)
    assert e.value.status == swl.KVC_ESTATE
    ok.project_append(hid.cuda(), w.cuda(), None, None, 0, sh.grid_h, sh.grid_w)
    assert ok.chunk_of_region[0] == 0 and ok.frame0_of_region[0] == 0


# ---------------------------------------------------------------------------
# multi-shot sink
# ---------------------------------------------------------------------------
def test_multi_shot_projection_stream_then_recache(swl):
    """Shots opening at chunks 0, 4 and 7 with a RoPE offset of 9 frames:
    every chunk is projected at its shifted positions and appended (the new
    shot's first chunk as the sink); after the stream, a recache from the
    present chunks' hidden states rebuilds the cache at the positions the
    cache recorded, against the oracle's recache with the model's frame0."""
    sh = Shapes(2, 128, 40, 2, 2, 4, 10)
    scale = 1.0 / math.sqrt(sh.head_dim)
    for c, q, cache, model in _project_stream(swl, sh, 46, 9, "bf16", shots={0, 4, 7},
                                              rope_offset=9):
        out = cache.attn(q, scale)
        torch.cuda.synchronize()
        kk, vv = model.visible_kv()
        assert_close(to64(out), oatt.attention(to64(q), kk, vv, scale), ATOL_BF16, RELL2_BF16,
                     f"shot stream attention, step {c}")
    assert model.present_chunks() == [7, 8] and cache.shot == 2
    ids = model.present_chunks()
    hid = torch.cat([project_inputs(sh, 46, x)[0] for x in ids])
    w = project_inputs(sh, 46, 0)[1]
    gk = gains(sh, 46)[1]
    cache.recache(hid.cuda(), w[:, sh.model_dim:].contiguous().cuda(), gk.cuda(), ids, sh.grid_h,
                  sh.grid_w)
    torch.cuda.synchronize()
    k, v = orc.recache(bf16_to_f64(hid), bf16_to_f64(w[:, sh.model_dim:]), gk.double().numpy(), ids,
                       sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.grid_w,
                       frame0=[model.frame0[x] for x in ids])
    Tc = sh.chunk_tokens
    for i, x in enumerate(ids):
        r = cache.chunk_of_region.index(x)
        assert_close(to64(cache.k[r * Tc:(r + 1) * Tc]), k[i * Tc:(i + 1) * Tc], ATOL_BF16, RELL2_BF16,
                     f"recached K of chunk {x}")
        assert_close(to64(cache.v[r * Tc:(r + 1) * Tc]), v[i * Tc:(i + 1) * Tc], ATOL_BF16, RELL2_BF16,
                     f"recached V of chunk {x}")
    assert cache.last_device_error() == swl.KVC_OK


@pytest.mark.parametrize("dtype", ["bf16", "fp4"])
def test_multi_shot_append_attention(swl, dtype):
    """kvc_append_shot with given K/V: shots at chunks 0 and 5, W = 2; after
    the boundary the old sink no longer counts (bit-identical output when its
    rows are overwritten), and attention matches the oracle at every step."""
    sh = Shapes(2, 64, 50, 2, 2, 5, 10)
    scale = 1.0 / math.sqrt(sh.head_dim)
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, sh.window_chunks,
                        dtype=dtype)
    model = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, sh.window_chunks, sh.chunk_frames)
    for c in range(9):
        q, k, v = chunk_qkv(sh, 47, 0, c, "rms1" if dtype == "bf16" else "outliers")
        if (c - sh.window_chunks) in model.window_chunks():
            cache.evict(c - sh.window_chunks)
            model.evict(c - sh.window_chunks)
        (cache.append_shot if c in (0, 5) else cache.append)(k.cuda(), v.cuda(), c)
        if dtype == "bf16":
            kk, vv = bf16_to_f64(k), bf16_to_f64(v)
        else:
            kk = ofp4.dequantize(*ofp4.quantize(k.float().numpy()))
            vv = ofp4.dequantize(*ofp4.quantize(v.float().numpy()))
        (model.append_shot if c in (0, 5) else model.append)(c, kk, vv)
        assert cache.chunk_of_region == model.chunk_of_region
        out = cache.attn(q.cuda(), scale)
        torch.cuda.synchronize()
        want = oatt.sinkwin_attention(model, bf16_to_f64(q), scale)
        if dtype == "bf16":
            assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, f"step {c}")
        else:
            assert_close(to64(out), want, ATOL_FP4, None, f"fp4 step {c}", plus_output_rounding=True)
    assert cache.chunk_of_region == [5, 7, 8]
    assert cache.last_device_error() == swl.KVC_OK


def test_multi_shot_state_machine_matches_oracle(swl):
    """Random call sequences with new shots mixed in: the library and the
    oracle model accept and reject the same calls and end in the same slot map,
    frame positions and shot count."""
    sh = Shapes(1, 64, 8, 2, 3, 2, 4)
    rnd = random.Random(9)
    z = torch.zeros((sh.chunk_tokens, 1, 64), dtype=torch.bfloat16, device="cuda")
    zn = np.zeros((sh.chunk_tokens, 1, 64))
    for trial in range(20):
        cache = swl.KVCache(1, 64, 8, 2, 3, rope_offset_frames=5)
        model = CacheModel(1, 64, sh.chunk_tokens, 3, chunk_frames=2, rope_offset_frames=5)
        for _ in range(40):
            op = rnd.choice(["app_next", "app_same", "shot_next", "shot_same", "shot_any",
                             "evict_old", "evict_any"])
            nw = model.last
            if op in ("app_next", "shot_next"):
                args = (op[0], nw + 1)
            elif op in ("app_same", "shot_same"):
                args = (op[0], max(nw, 0))
            elif op == "shot_any":
                args = ("s", rnd.randint(0, nw + 3))
            elif op == "evict_old":
                win = model.window_chunks()
                args = ("e", win[0] if win else 0)
            else:
                args = ("e", rnd.randint(0, nw + 2))
            kind, x = args
            try:
                {"a": lambda: model.append(x, zn, zn), "s": lambda: model.append_shot(x, zn, zn),
                 "e": lambda: model.evict(x)}[kind]()
                want = swl.KVC_OK
            except CacheStateError:
                want = swl.KVC_ESTATE
            try:
                {"a": lambda: cache.append(z, z, x), "s": lambda: cache.append_shot(z, z, x),
                 "e": lambda: cache.evict(x)}[kind]()
                got = swl.KVC_OK
            except swl.KvcError as e:
                got = e.status
            assert got == want, (trial, args)
            assert cache.chunk_of_region == model.chunk_of_region, (trial, args)
            assert cache.frame0_of_region == model.frame0_of_region(), (trial, args)
            assert cache.shot == model.shot
