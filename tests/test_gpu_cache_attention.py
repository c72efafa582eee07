"""GPU parity: cache append / evict / layout and bf16 sink+window attention,
CUDA path (through the C ABI) against the float64 oracle on the same inputs."""

import math
import os
import random
import time

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle.cache_model import CacheModel, CacheStateError
from synth import LAYER_1P3B, TINY, Shapes, chunk_qkv, chunk_qkv_device, bf16_to_f64
from tests.gpu_helpers import (ATOL_BF16, RELL2_BF16, SAMPLE_ROWS_4680, assert_close, to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_short_window_sinkwin_b300 as swl
    return swl


def _stream(swl, sh: Shapes, cfg: int, steps, dist="rms1", dtype="bf16", scrub=False,
            check_every=True):
    """Run chunks 0..steps-1 through GPU cache + oracle model; yields per step."""
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                        sh.window_chunks, dtype=dtype, scrub_on_evict=scrub)
    model = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, sh.window_chunks)
    W = sh.window_chunks
    for c in range(steps):
        q, k, v = chunk_qkv(sh, cfg, 0, c, dist)
        if c > W:
            cache.evict(c - W)
            model.evict(c - W)
        cache.append(k.cuda(), v.cuda(), c)
        model.append(c, bf16_to_f64(k), bf16_to_f64(v))
        assert cache.chunk_of_region == model.chunk_of_region
        yield c, q, cache, model


def test_tiny_stream_layout_and_attention(swl):
    sh = TINY
    scale = 1.0 / math.sqrt(sh.head_dim)
    for c, q, cache, model in _stream(swl, sh, 0, 6, "rms1"):
        Kp, Vp = model.physical()
        got_k, got_v = to64(cache.k), to64(cache.v)
        for r, ch in enumerate(model.chunk_of_region):
            if ch >= 0:
                sl = slice(r * sh.chunk_tokens, (r + 1) * sh.chunk_tokens)
                assert np.array_equal(got_k[sl], Kp[sl]) and np.array_equal(got_v[sl], Vp[sl])
        out = cache.attn(q.cuda(), scale)
        torch.cuda.synchronize()
        want = oatt.sinkwin_attention(model, bf16_to_f64(q), scale)
        assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, f"tiny step {c}")
    assert cache.last_device_error() == swl.KVC_OK


@pytest.mark.parametrize("dist", ["literal", "rms1"])
def test_layer_attention_full_size(swl, dist):
    """LongLive-1.3B layer, 12 x 128, chunk 4680, KV 18720; sampled query rows
    across every tile kind (first, interior, slot 1, last partial)."""
    sh = LAYER_1P3B
    scale = 1.0 / math.sqrt(sh.head_dim)
    *_, (c, q, cache, model) = list(_stream(swl, sh, 1, 4, dist))
    assert model.kv_length() == 18720
    out = cache.attn(q.cuda(), scale)
    torch.cuda.synchronize()
    kk, vv = model.visible_kv()
    want = oatt.attention_rows(bf16_to_f64(q), kk, vv, scale, SAMPLE_ROWS_4680)
    got = to64(out)[SAMPLE_ROWS_4680]
    print(assert_close(got, want, ATOL_BF16, RELL2_BF16, f"layer {dist}"))
    assert cache.last_device_error() == swl.KVC_OK


def test_layer_warmup_and_wrap(swl):
    """KV lengths 4680, 9360, 14040 during warm-up and the ring after wrap-around
    (step 5: regions hold chunks 0, 4, 5, 3)."""
    sh = LAYER_1P3B
    scale = 1.0 / math.sqrt(sh.head_dim)
    rows = [0, 130, 2500, 4679]
    for c, q, cache, model in _stream(swl, sh, 1, 6, "rms1"):
        if c in (0, 1, 2, 5):
            out = cache.attn(q.cuda(), scale)
            torch.cuda.synchronize()
            kk, vv = model.visible_kv()
            want = oatt.attention_rows(bf16_to_f64(q), kk, vv, scale, rows)
            assert_close(to64(out)[rows], want, ATOL_BF16, RELL2_BF16, f"step {c}")
    assert model.chunk_of_region == [0, 4, 5, 3]


@pytest.mark.parametrize("H,D,tpf,cf,W,tq", [
    (2, 128, 100, 1, 3, 100),     # Tc = 100: every KV tile ragged
    (3, 64, 50, 3, 2, 300),       # tq != Tc, slot 1 partly live
    (1, 128, 16, 8, 2, 1),        # one query row
    (2, 64, 129, 1, 4, 257),      # 129-row chunks, tq = 2*128 + 1
    (1, 128, 200, 2, 1, 400),     # W = 1: sink + the current chunk only
])
def test_small_shapes_full_compare(swl, H, D, tpf, cf, W, tq):
    sh = Shapes(H, D, tpf, cf, W, 1, tpf)
    scale = 0.9 / math.sqrt(D)
    for c, q, cache, model in _stream(swl, sh, 7, W + 3, "rms1"):
        qq = chunk_qkv(sh, 8, 0, c, "rms1", q_rows=tq)[0]
        out = cache.attn(qq.cuda(), scale)
        torch.cuda.synchronize()
        want = oatt.sinkwin_attention(model, bf16_to_f64(qq), scale)
        assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, f"{(H, D, tpf, cf, W, tq)} step {c}")


@pytest.mark.parametrize("workspace", [True, False])
def test_many_items_full_compare(swl, workspace):
    """12 heads x 4680 queries = 228 items on at most 148 CTAs: with the
    workspace, shares are step-balanced and most items are computed in two
    pieces by neighbouring CTAs and merged; without it each CTA takes whole
    items.  Short 100-token chunks keep the full oracle compare cheap."""
    sh = Shapes(12, 128, 100, 1, 2, 10, 10)
    scale = 1.0 / math.sqrt(128)
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                        sh.window_chunks, attn_workspace=workspace)
    model = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, sh.window_chunks)
    for c in range(4):
        _, k, v = chunk_qkv(sh, 12, 0, c, "rms1")
        if c > sh.window_chunks:
            cache.evict(c - sh.window_chunks)
            model.evict(c - sh.window_chunks)
        cache.append(k.cuda(), v.cuda(), c)
        model.append(c, bf16_to_f64(k), bf16_to_f64(v))
        if c in (0, 3):  # one segment of 1 tile; then two segments (hole-free ring wrap)
            qq = chunk_qkv(sh, 13, 0, c, "rms1", q_rows=4680)[0]
            out = cache.attn(qq.cuda(), scale)
            torch.cuda.synchronize()
            want = oatt.sinkwin_attention(model, bf16_to_f64(qq), scale)
            assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, f"228 items, step {c}")
    assert cache.last_device_error() == swl.KVC_OK


def _planted_stream(swl, H, D, tpf, cf, W, where, seed, workspace=True):
    """bf16 cache of 1 + W chunks whose keys are 0.3 N(0,1) except planted
    rows 10u (u a unit vector); queries are 10u + 0.3 N(0,1).  A planted key's
    logit lies about 12.7 (log2 units) above the others', beyond the 2^8 by
    which the kernel lets its held row maximum go stale, so a tile that brings
    the first planted keys of a piece forces the O rescale in TMEM.
    where: "late_tile" plants keys only in the last tile of the newest chunk
    (every earlier tile has set the held maximum low); "mid_chunk" plants them
    in the second half of chunk 1 only."""
    Tc = tpf * cf
    rng = np.random.default_rng(seed)
    u = rng.standard_normal(D)
    u /= np.linalg.norm(u)
    cache = swl.KVCache(H, D, tpf, cf, W, attn_workspace=workspace)
    model = CacheModel(H, D, Tc, W)
    for c in range(1 + W):
        k = rng.standard_normal((Tc, H, D)) * 0.3
        v = rng.standard_normal((Tc, H, D))
        if where == "late_tile" and c == W:
            k[Tc - 64:] = 10 * u
        elif where == "mid_chunk" and c == 1:
            k[Tc // 2:] = 10 * u
        kb = torch.from_numpy(k.astype(np.float32)).to(torch.bfloat16)
        vb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
        cache.append(kb.cuda(), vb.cuda(), c)
        model.append(c, bf16_to_f64(kb), bf16_to_f64(vb))
    return cache, model, u, rng


@pytest.mark.parametrize("where", ["late_tile", "mid_chunk"])
def test_bf16_max_jump_rescales_o(swl, where):
    """bf16 twin of the FP4 max-jump test: two heads, 256-token chunks (two
    key tiles each), 130 queries, whole items visited from their first tile,
    so the planted tile comes after tiles that set a low held maximum and the
    kernel must rescale O (alpha = 2^-12 or so) before adding that tile."""
    H, D = 2, 128
    cache, model, u, rng = _planted_stream(swl, H, D, 128, 2, 2, where, 51)
    q = 10 * u + 0.3 * rng.standard_normal((130, H, D))
    qb = torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    out = cache.attn(qb.cuda(), scale)
    torch.cuda.synchronize()
    want = oatt.sinkwin_attention(model, bf16_to_f64(qb), scale)
    print(assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, f"bf16 max jump ({where})"))
    assert cache.last_device_error() == swl.KVC_OK


def test_bf16_max_jump_split_items(swl):
    """12 heads x 4680 queries = 228 items on 148 CTAs (step-balanced shares):
    pieces with and without the planted keys hold maxima about 12 (log2 units)
    apart, so both the in-TMEM rescale and the merge of two pieces with very
    different maxima run."""
    H, D = 12, 128
    cache, model, u, rng = _planted_stream(swl, H, D, 100, 1, 2, "mid_chunk", 52)
    q = 10 * u + 0.3 * rng.standard_normal((4680, H, D))
    qb = torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    out = cache.attn(qb.cuda(), scale)
    torch.cuda.synchronize()
    want = oatt.sinkwin_attention(model, bf16_to_f64(qb), scale)
    print(assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, "bf16 max jump, split items"))
    assert cache.last_device_error() == swl.KVC_OK


def test_layer_attention_full_size_full_compare(swl):
    """LongLive-1.3B layer at full size (4680 queries x 18720 keys x 12 heads,
    RMS-1 rows so the softmax is far from uniform): every one of the
    4680 x 12 x 128 outputs against the float64 oracle, which runs on all host
    cores (oracle.pool)."""
    from oracle.pool import attention_rows_parallel
    sh = LAYER_1P3B
    scale = 1.0 / math.sqrt(sh.head_dim)
    *_, (c, q, cache, model) = list(_stream(swl, sh, 1, 4, "rms1"))
    out = cache.attn(q.cuda(), scale)
    torch.cuda.synchronize()
    got = to64(out)
    kk, vv = model.visible_kv()
    t0 = time.perf_counter()
    want = attention_rows_parallel(bf16_to_f64(q), kk, vv, scale)
    print(f"oracle: {time.perf_counter() - t0:.1f} s on {os.cpu_count()} CPUs")
    print(assert_close(got, want, ATOL_BF16, RELL2_BF16, "layer full compare"))
    assert cache.last_device_error() == swl.KVC_OK


@pytest.mark.parametrize("tq", [1, 100, 128, 129, 256, 300, 700])
@pytest.mark.parametrize("dtype", ["bf16", "fp4"])
def test_split_kv_short_query_chunks(swl, tq, dtype):
    """Short query chunks against the full LongLive-1.3B cache (12 heads,
    18720 keys): 12-36 items on up to 148 CTAs, so every item is spread over
    several CTAs' shares (split-KV) and merged by the CTA that started it.
    Every output against the oracle."""
    sh = LAYER_1P3B
    scale = 1.0 / math.sqrt(sh.head_dim)
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                        sh.window_chunks, dtype=dtype)
    kk, vv = [], []
    for c in range(1 + sh.window_chunks):
        _, k, v = chunk_qkv(sh, 61, 0, c, "rms1" if dtype == "bf16" else "outliers")
        cache.append(k.cuda(), v.cuda(), c)
        if dtype == "bf16":
            kk.append(bf16_to_f64(k)), vv.append(bf16_to_f64(v))
        else:
            from oracle import fp4 as ofp4
            kk.append(ofp4.dequantize(*ofp4.quantize(k.float().numpy())))
            vv.append(ofp4.dequantize(*ofp4.quantize(v.float().numpy())))
    kk, vv = np.concatenate(kk), np.concatenate(vv)
    q = chunk_qkv(sh, 62, 0, tq, "rms1", q_rows=tq)[0]
    out = cache.attn(q.cuda(), scale)
    torch.cuda.synchronize()
    want = oatt.attention(bf16_to_f64(q), kk, vv, scale)
    if dtype == "bf16":
        assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, f"split-KV tq={tq}")
    else:
        assert_close(to64(out), want, 5e-2, None, f"fp4 split-KV tq={tq}", plus_output_rounding=True)
    assert cache.last_device_error() == swl.KVC_OK


def test_split_kv_planted_max_and_no_workspace(swl):
    """tq = 130 on the 12-head cache with keys planted in one late tile: the
    pieces of an item hold maxima ~12 (log2 units) apart.  The same call
    without a workspace (whole items, 12 CTAs) gives the same answer."""
    H, D = 12, 128
    cache, model, u, rng = _planted_stream(swl, H, D, 1560, 3, 3, "late_tile", 63)
    cache2 = swl.KVCache(H, D, 1560, 3, 3, attn_workspace=False)
    for c in range(4):
        r = cache.chunk_of_region.index(c)
        sl = slice(r * 4680, (r + 1) * 4680)
        cache2.append(cache.k[sl].contiguous(), cache.v[sl].contiguous(), c)
    q = 10 * u + 0.3 * rng.standard_normal((130, H, D))
    qb = torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16).cuda()
    scale = 1.0 / math.sqrt(D)
    out, out2 = cache.attn(qb, scale), cache2.attn(qb, scale)
    torch.cuda.synchronize()
    want = oatt.sinkwin_attention(model, to64(qb), scale)
    assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, "split-KV planted")
    assert_close(to64(out2), want, ATOL_BF16, RELL2_BF16, "whole items planted")
    assert cache.last_device_error() == swl.KVC_OK and cache2.last_device_error() == swl.KVC_OK


def test_holes_scrub_and_zero_queries(swl):
    """Evict without append leaves a hole (two KV segments); the scrubbed slot
    holds NaN and must never reach the output."""
    sh = Shapes(2, 128, 100, 1, 3, 10, 10)
    scale = 1.0 / math.sqrt(128)
    gen = _stream(swl, sh, 9, 5, "rms1", scrub=True)
    for c, q, cache, model in gen:
        pass
    cache.evict(2)
    model.evict(2)
    assert cache.chunk_of_region == [0, 4, -1, 3]
    torch.cuda.synchronize()
    assert torch.isnan(cache.k[200:300].float()).all() and torch.isnan(cache.v[200:300].float()).all()
    qq = chunk_qkv(sh, 9, 1, 99, "rms1", q_rows=130)[0]
    out = cache.attn(qq.cuda(), scale)
    torch.cuda.synchronize()
    want = oatt.sinkwin_attention(model, bf16_to_f64(qq), scale)
    assert_close(to64(out), want, ATOL_BF16, RELL2_BF16, "hole")
    # Q = 0 -> mean of the visible V (closed form)
    z = torch.zeros((7, 2, 128), dtype=torch.bfloat16, device="cuda")
    out0 = cache.attn(z, scale)
    torch.cuda.synchronize()
    _, vv = model.visible_kv()
    assert_close(to64(out0), np.broadcast_to(vv.mean(axis=0), (7, 2, 128)), ATOL_BF16, None, "q=0")
    # tq = 0 is a no-op
    cache.attn(torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda"), scale)


def test_evicted_data_does_not_influence_output(swl):
    """Overwrite an evicted slot's rows with garbage: the output is bit-identical."""
    sh = Shapes(2, 128, 100, 1, 3, 10, 10)
    scale = 1.0 / math.sqrt(128)
    for c, q, cache, model in _stream(swl, sh, 11, 5, "rms1"):
        pass
    cache.evict(2)
    qq = chunk_qkv(sh, 11, 1, 5, "rms1", q_rows=100)[0].cuda()
    a = cache.attn(qq, scale).clone()
    cache.k[200:300].normal_()
    cache.v[200:300].fill_(float("inf"))
    b = cache.attn(qq, scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_append_copy_is_exact_full_size(swl):
    sh = LAYER_1P3B
    for c, q, cache, model in _stream(swl, sh, 1, 4, "literal"):
        pass
    torch.cuda.synchronize()
    for c in range(4):
        _, k, v = chunk_qkv(sh, 1, 0, c, "literal")
        sl = slice(c * sh.chunk_tokens, (c + 1) * sh.chunk_tokens)
        assert torch.equal(cache.k[sl].cpu(), k) and torch.equal(cache.v[sl].cpu(), v)


def test_rolling_stream_30_layers_320_chunks(swl):
    """Rolling stream: 30 independent layer caches x 320 chunks (960 latent
    frames), each step evict(c - W) + append(c) + attention, the sink pinned;
    Q/K/V are drawn per (layer, chunk) on the device.  Every step checks the
    slot map against the oracle model.  Sampled (layer, chunk) steps -- the
    warm-up, the first eviction, mid-stream, the last chunk -- check sampled
    query rows against the float64 oracle over the visible chunks re-drawn
    from their seeds.  At the end every layer holds exactly chunks 0, 317, 318
    and 319, bit for bit.  Prints the steady-state (c >= 4) latent frames/s
    per layer, from CUDA events around each layer's evict + append + attention."""
    sh = LAYER_1P3B
    cfg, n_layers, n_chunks, W = 2, 30, 320, sh.window_chunks
    scale = 1.0 / math.sqrt(sh.head_dim)
    rows = [0, 127, 128, 1560, 3119, 4095, 4608, 4679]
    checks = {(0, 0), (1, 1), (2, 2), (3, 3), (4, 4), (29, 5), (17, 100), (5, 201), (0, 319), (29, 319)}
    caches = [swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames, W)
              for _ in range(n_layers)]
    slot_maps = [CacheModel(1, 1, 1, W) for _ in range(n_layers)]  # slot rule only
    z1 = np.zeros((1, 1, 1))
    steady = []
    checked_s = 0.0  # host time spent on the sampled oracle checks (excluded from the wall time)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for c in range(n_chunks):
        for li in range(n_layers):
            q, k, v = chunk_qkv_device(sh, cfg, li, c)
            cache, model = caches[li], slot_maps[li]
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            if c > W:
                cache.evict(c - W)
                model.evict(c - W)
            cache.append(k, v, c)
            model.append(c, z1, z1)
            out = cache.attn(q, scale)
            t1.record()
            assert cache.chunk_of_region == model.chunk_of_region, (li, c)
            if c >= 4:
                steady.append((t0, t1))
            if (li, c) in checks:
                t_chk = time.perf_counter()
                got = to64(out[rows])
                vis = model.present_chunks()
                kv = [chunk_qkv_device(sh, cfg, li, x)[1:] for x in vis]
                kk = np.concatenate([to64(a) for a, _ in kv])
                vv = np.concatenate([to64(b) for _, b in kv])
                want = oatt.attention_rows(to64(q), kk, vv, scale, rows)
                assert_close(got, want, ATOL_BF16, RELL2_BF16, f"layer {li} chunk {c}")
                checked_s += time.perf_counter() - t_chk
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall - checked_s
    for li, cache in enumerate(caches):
        assert cache.chunk_of_region == [0, 319, 317, 318]  # slot (c - 1) mod 3
        for x in (0, 317, 318, 319):
            _, k, v = chunk_qkv_device(sh, cfg, li, x)
            r = cache.chunk_of_region.index(x)
            sl = slice(r * sh.chunk_tokens, (r + 1) * sh.chunk_tokens)
            assert torch.equal(cache.k[sl], k) and torch.equal(cache.v[sl], v), (li, x)
        assert cache.last_device_error() == swl.KVC_OK
    ms = float(np.mean([a.elapsed_time(b) for a, b in steady]))
    print(f"rolling stream: {ms:.4f} ms per layer-step, "
          f"{sh.chunk_frames / ms * 1e3:.1f} latent frames/s per layer (steady state); "
          f"whole stream {wall:.2f} s wall including input generation "
          f"({n_chunks * sh.chunk_frames} latent frames x {n_layers} layers)")


def test_state_machine_matches_oracle(swl):
    """Random call sequences: the library and the oracle model accept and reject
    the same calls and end in the same slot map."""
    sh = Shapes(1, 64, 8, 2, 3, 2, 4)
    rnd = random.Random(5)
    z = torch.zeros((sh.chunk_tokens, 1, 64), dtype=torch.bfloat16, device="cuda")
    zn = np.zeros((sh.chunk_tokens, 1, 64))
    for trial in range(20):
        cache = swl.KVCache(1, 64, 8, 2, 3)
        model = CacheModel(1, 64, sh.chunk_tokens, 3)
        for _ in range(40):
            op = rnd.choice(["app_next", "app_same", "app_any", "evict_old", "evict_any"])
            nw = model.newest()
            if op == "app_next":
                args = ("a", nw + 1)
            elif op == "app_same":
                args = ("a", max(nw, 0))
            elif op == "app_any":
                args = ("a", rnd.randint(0, nw + 3))
            elif op == "evict_old":
                win = [x for x in model.present_chunks() if x != 0]
                args = ("e", win[0] if win else 0)
            else:
                args = ("e", rnd.randint(0, nw + 2))
            try:
                (model.append(args[1], zn, zn) if args[0] == "a" else model.evict(args[1]))
                want = swl.KVC_OK
            except CacheStateError:
                want = swl.KVC_ESTATE
            try:
                (cache.append(z, z, args[1]) if args[0] == "a" else cache.evict(args[1]))
                got = swl.KVC_OK
            except swl.KvcError as e:
                got = e.status
            assert got == want, (trial, args)
            assert cache.chunk_of_region == model.chunk_of_region


def test_watchdog_reports_timeout(swl):
    cache = swl.KVCache(1, 64, 16, 2, 2)
    from sink_short_window_sinkwin_b300._abi import lib
    import ctypes
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib().kvc_watchdog_selftest(ctypes.c_void_p(cache.ws.data_ptr()), 2000, st) == 0
    assert cache.last_device_error() == swl.KVC_ETIMEOUT
    assert cache.last_device_error() == swl.KVC_OK  # read-and-clear
