"""GPU parity of the FP4 KV path: codes, scales and tensor scales bit-exact
against the oracle encoder; attention over an FP4 cache against the oracle run
on the same dequantised K/V."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import fp4 as ofp4
from oracle.cache_model import CacheModel
from synth import LAYER_1P3B, TINY, Shapes, chunk_qkv, bf16_to_f64
from tests.gpu_helpers import ATOL_FP4, SAMPLE_ROWS_4680, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_short_window_sinkwin_b300 as swl
    return swl


def _f32(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float32).numpy()


def _check_quant(swl, x_bf16: torch.Tensor, what: str):
    codes, scales, g = swl.quant_fp4(x_bf16.cuda().contiguous())
    torch.cuda.synchronize()
    wc, ws, wg = ofp4.quantize(_f32(x_bf16).reshape(-1, 16))
    assert np.array_equal(codes.cpu().numpy(), wc.reshape(-1)), f"{what}: codes differ"
    assert np.array_equal(scales.cpu().numpy(), ws.reshape(-1)), f"{what}: scales differ"
    assert g.cpu().numpy()[0].view(np.uint32) == np.float32(wg).view(np.uint32), f"{what}: g differs"


def test_quant_bitexact_layer_chunk(swl):
    sh = LAYER_1P3B
    _, k, v = chunk_qkv(sh, 3, 0, 0, "outliers")
    _check_quant(swl, k, "K chunk")
    _check_quant(swl, v, "V chunk")


def test_quant_bitexact_edge_values(swl):
    rng = np.random.default_rng(4)
    blocks = []
    blocks.append(np.zeros(16, np.float32))                       # all-zero block
    blocks.append(np.full(16, -0.0, np.float32))                  # -0 only
    b = np.zeros(16, np.float32); b[0] = 6.0; b[1:8] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    b[8:] = -b[:8]
    blocks.append(b)                                              # E2M1 ties at s = 1
    blocks.append(np.full(16, 3e-6, np.float32))                  # tiny: subnormal scales
    blocks.append(rng.standard_normal(16).astype(np.float32) * 1e-3)
    blocks.append(np.linspace(-448 * 6, 448 * 6, 16, dtype=np.float32))  # holds the amax
    for _ in range(200):
        blocks.append((rng.standard_normal(16) * np.exp(rng.uniform(-12, 4))).astype(np.float32))
    x = torch.from_numpy(np.concatenate(blocks)).to(torch.bfloat16)
    _check_quant(swl, x, "edge blocks")
    _check_quant(swl, torch.zeros(64, dtype=torch.bfloat16), "all zero")
    # fewer 16-byte vectors than the amax pass has CTAs: one, two and 17 blocks
    for nb in (1, 2, 17):
        _check_quant(swl, x[: 16 * nb].clone(), f"{nb} block(s)")
    # many blocks: every CTA of both passes active, a grid-stride remainder
    y = torch.from_numpy(rng.standard_normal(16 * 300001).astype(np.float32)).to(torch.bfloat16)
    _check_quant(swl, y, "ragged size")


def _near_midpoint_maxima(amax_t: float, n_ulp: int = 8):
    """bf16 block maxima b <= amax_t whose scale quotient fl32(fl32(b/6)/g),
    g = fl32(amax_t/2688), lies within n_ulp float32 ulps of a rounding midpoint
    between two E4M3 values (so a quotient off by an ulp could round to the
    other code)."""
    f32 = np.float32
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)  # positive finite bf16
    b = (bits << 16).view(np.float32)
    b = b[b <= f32(amax_t)]
    g = f32(f32(amax_t) / ofp4.G_DIVISOR)
    q = (b / f32(6.0)).astype(f32) / g
    qb = q.view(np.uint32)
    lo = np.maximum(qb.astype(np.int64) - n_ulp, 0).astype(np.uint32).view(np.float32)
    hi = (qb + n_ulp).view(np.float32)
    near = ofp4.e4m3_rne_satfinite(lo) != ofp4.e4m3_rne_satfinite(hi)
    return b[near]


def test_quant_bitexact_near_scale_midpoints(swl):
    """Blocks whose scale quotient sits within a few ulps of an E4M3 rounding
    midpoint, for tensor maxima over many magnitudes: the encoder's fast
    scale path must defer to the exact quotient there, codes and scales
    bit-exact against the oracle."""
    rng = np.random.default_rng(9)
    for amax_t in (1.0, 3.734375, 1.0e-3, 8.5e5, 2.0 ** -100, 2.0 ** -120, 448.0 * 6.0, 0.15625):
        amax_t = float(torch.tensor(amax_t).to(torch.bfloat16).float())
        maxima = _near_midpoint_maxima(amax_t)
        # g = amax_t / 2688 is a normal float except for the smallest tensor,
        # where 1/g overflows and every block takes the exact quotient
        assert len(maxima) > 0 or amax_t < 2.0 ** -115, amax_t
        spread = amax_t * np.exp2(-rng.uniform(0, 40, 64))
        maxima = np.concatenate([maxima, spread.astype(np.float32)])
        blocks = np.zeros((len(maxima) + 1, 16), np.float32)
        blocks[:-1, 0] = maxima
        blocks[:-1, 1:] = maxima[:, None] * rng.uniform(-1, 1, (len(maxima), 15)).astype(np.float32)
        blocks[-1, 0] = amax_t  # the tensor maximum
        x = torch.from_numpy(blocks.reshape(-1)).to(torch.bfloat16)
        _check_quant(swl, x, f"near-midpoint blocks, tensor amax {amax_t:g} ({len(maxima)} blocks)")


# FP4 attention runs two ways: K/V decoded inside the kernel (no staging
# buffer) or decoded beforehand into the staging buffer and loaded by TMA
PRE = pytest.mark.parametrize("stage", [False, True], ids=["in_kernel", "predecoded"])


def _fp4_stream(swl, sh, cfg, steps, dist, stage=False):
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                        sh.window_chunks, dtype="fp4", stage=stage)
    model = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, sh.window_chunks)
    W, Tc = sh.window_chunks, sh.chunk_tokens
    enc = {}
    for c in range(steps):
        q, k, v = chunk_qkv(sh, cfg, 0, c, dist)
        if c > W:
            cache.evict(c - W)
            model.evict(c - W)
        cache.append(k.cuda(), v.cuda(), c)
        ek = ofp4.quantize(_f32(k))
        ev = ofp4.quantize(_f32(v))
        enc[c] = (ek, ev)
        model.append(c, ofp4.dequantize(*ek), ofp4.dequantize(*ev))
        assert cache.chunk_of_region == model.chunk_of_region
        torch.cuda.synchronize()
        r = model.chunk_of_region.index(c)
        sl = slice(r * Tc, (r + 1) * Tc)
        for (codes, scales, g), cb, sb, gb in ((ek, cache.k, cache.k_scale, cache.k_gscale),
                                              (ev, cache.v, cache.v_scale, cache.v_gscale)):
            assert np.array_equal(cb[sl].cpu().numpy(), codes), f"codes of chunk {c}"
            assert np.array_equal(sb[sl].cpu().numpy(), scales), f"scales of chunk {c}"
            assert gb[r].item() == float(g), f"gscale of chunk {c}"
        yield c, q, cache, model


@PRE
def test_fp4_tiny_stream(swl, stage):
    sh = TINY
    scale = 1.0 / math.sqrt(sh.head_dim)
    for c, q, cache, model in _fp4_stream(swl, sh, 0, 6, "outliers", stage):
        out = cache.attn(q.cuda(), scale)
        torch.cuda.synchronize()
        want = oatt.sinkwin_attention(model, bf16_to_f64(q), scale)
        assert_close(to64(out), want, ATOL_FP4, None, f"fp4 tiny step {c}",
                 plus_output_rounding=True)


@PRE
@pytest.mark.parametrize("H,D,tpf,cf,W,tq", [(2, 128, 100, 1, 3, 130), (3, 64, 50, 3, 2, 300)])
def test_fp4_small_shapes(swl, H, D, tpf, cf, W, tq, stage):
    sh = Shapes(H, D, tpf, cf, W, 1, tpf)
    scale = 1.0 / math.sqrt(D)
    for c, q, cache, model in _fp4_stream(swl, sh, 5, W + 2, "outliers", stage):
        qq = chunk_qkv(sh, 6, 0, c, "rms1", q_rows=tq)[0]
        out = cache.attn(qq.cuda(), scale)
        torch.cuda.synchronize()
        want = oatt.sinkwin_attention(model, bf16_to_f64(qq), scale)
        assert_close(to64(out), want, ATOL_FP4, None, f"fp4 {(H, D, tpf, cf, W, tq)} step {c}",
                 plus_output_rounding=True)


@PRE
@pytest.mark.parametrize("where", ["every_tile", "late_tile"])
def test_fp4_max_jump_within_tile(swl, where, stage):
    """Keys 64..127 of a 128-key tile whose logits lie more than 2^8 (log2
    units) above those of keys 0..63 and of the tiles before: the softmax must
    move its held reference maximum (and rescale O) before forming that tile's
    P.  256-token chunks = two tiles each; queries 10u + noise, planted keys
    10u (u a unit vector).  every_tile: the jump comes on each piece's first
    tile; late_tile: only the last tile of chunk 2 has it, after other tiles
    set the reference."""
    H, D, Tc, W = 2, 128, 256, 2
    rng = np.random.default_rng(31)
    u = rng.standard_normal(D)
    u /= np.linalg.norm(u)
    cache = swl.KVCache(H, D, 128, 2, W, dtype="fp4", stage=stage)
    model = CacheModel(H, D, Tc, W)
    for c in range(1 + W):
        k = rng.standard_normal((Tc, H, D)) * 0.3
        v = rng.standard_normal((Tc, H, D))
        if where == "every_tile":
            k[64:128] = 10 * u
            k[192:256] = 10 * u
        elif c == W:
            k[192:256] = 10 * u
        kb = torch.from_numpy(k.astype(np.float32)).to(torch.bfloat16)
        vb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
        cache.append(kb.cuda(), vb.cuda(), c)
        model.append(c, ofp4.dequantize(*ofp4.quantize(_f32(kb))), ofp4.dequantize(*ofp4.quantize(_f32(vb))))
    q = 10 * u + 0.3 * rng.standard_normal((130, H, D))
    qb = torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    out = cache.attn(qb.cuda(), scale)
    torch.cuda.synchronize()
    want = oatt.sinkwin_attention(model, bf16_to_f64(qb), scale)
    assert_close(to64(out), want, ATOL_FP4, None, f"fp4 max jump ({where})", plus_output_rounding=True)
    assert cache.last_device_error() == swl.KVC_OK


@PRE
@pytest.mark.parametrize("vmag", [2.0 ** -14, 2.0 ** 26])
def test_fp4_v_magnitude_extremes(swl, vmag, stage):
    """P is stored as f16 times the V tensor scale g_V (up to 2^8 under a held
    running max).  V of magnitude 2^-14 (g_V ~ 1e-7: f16 subnormal products) or
    2^26 (g_V ~ 1e5: beyond the f16 range) must give the oracle's output scaled
    by the same factor; the three regions' V differ by 2^-3 per chunk, so the
    regions' g_V differ too.  Compared after dividing by the magnitude (a power
    of two, exact)."""
    H, D, W = 2, 128, 2
    rng = np.random.default_rng(41)
    cache = swl.KVCache(H, D, 128, 1, W, dtype="fp4", stage=stage)
    model = CacheModel(H, D, 128, W)
    for c in range(1 + W):
        k = rng.standard_normal((128, H, D))
        v = rng.standard_normal((128, H, D)) * (vmag * 2.0 ** (-3 * c))
        kb = torch.from_numpy(k.astype(np.float32)).to(torch.bfloat16)
        vb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
        cache.append(kb.cuda(), vb.cuda(), c)
        model.append(c, ofp4.dequantize(*ofp4.quantize(_f32(kb))), ofp4.dequantize(*ofp4.quantize(_f32(vb))))
    q = rng.standard_normal((200, H, D))
    qb = torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    out = cache.attn(qb.cuda(), scale)
    torch.cuda.synchronize()
    want = oatt.sinkwin_attention(model, bf16_to_f64(qb), scale)
    assert_close(to64(out) / vmag, want / vmag, ATOL_FP4, None, f"fp4 |V| ~ {vmag:g}",
                 plus_output_rounding=True)
    assert cache.last_device_error() == swl.KVC_OK


@PRE
def test_fp4_layer_full_size(swl, stage):
    sh = LAYER_1P3B
    scale = 1.0 / math.sqrt(sh.head_dim)
    *_, (c, q, cache, model) = list(_fp4_stream(swl, sh, 3, 4, "outliers", stage))
    out = cache.attn(q.cuda(), scale)
    torch.cuda.synchronize()
    kk, vv = model.visible_kv()
    want = oatt.attention_rows(bf16_to_f64(q), kk, vv, scale, SAMPLE_ROWS_4680)
    print(assert_close(to64(out)[SAMPLE_ROWS_4680], want, ATOL_FP4, None, "fp4 layer",
                 plus_output_rounding=True))
    assert cache.last_device_error() == swl.KVC_OK


@PRE
def test_fp4_many_items_full_compare(swl, stage):
    """FP4 cache, 228 items on 148 CTAs (step-balanced shares, merged pieces),
    one segment per region, full compare of all 4680 x 12 rows."""
    sh = Shapes(12, 128, 100, 1, 2, 10, 10)
    scale = 1.0 / math.sqrt(128)
    for c, q, cache, model in _fp4_stream(swl, sh, 14, 4, "outliers", stage):
        if c in (0, 3):
            qq = chunk_qkv(sh, 15, 0, c, "rms1", q_rows=4680)[0]
            out = cache.attn(qq.cuda(), scale)
            torch.cuda.synchronize()
            want = oatt.sinkwin_attention(model, bf16_to_f64(qq), scale)
            assert_close(to64(out), want, ATOL_FP4, None, f"fp4 228 items step {c}",
                 plus_output_rounding=True)
    assert cache.last_device_error() == swl.KVC_OK


@PRE
def test_fp4_scrub_unaligned_regions(swl, stage):
    """H=3, D=64, 150-token chunks: a slot's scales span 1800 bytes, so slot
    boundaries are not 16-byte aligned.  The scrub on evict writes exactly the
    freed slot (codes 0, scales 0x7F), nothing around it, and attention over the
    remaining chunks still matches the oracle."""
    sh = Shapes(3, 64, 50, 3, 2, 1, 50)
    Tc = sh.chunk_tokens
    cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                        sh.window_chunks, dtype="fp4", scrub_on_evict=True, stage=stage)
    model = CacheModel(sh.heads, sh.head_dim, Tc, sh.window_chunks)
    for c in range(3):
        _, k, v = chunk_qkv(sh, 21, 0, c, "outliers")
        cache.append(k.cuda(), v.cuda(), c)
        model.append(c, ofp4.dequantize(*ofp4.quantize(_f32(k))), ofp4.dequantize(*ofp4.quantize(_f32(v))))
    torch.cuda.synchronize()
    before = [t.clone() for t in (cache.k, cache.v, cache.k_scale, cache.v_scale)]
    cache.evict(1)
    model.evict(1)
    torch.cuda.synchronize()
    r = 1  # region of chunk 1
    sl = slice(r * Tc, (r + 1) * Tc)
    for t, b, fillv in ((cache.k, before[0], 0), (cache.v, before[1], 0),
                        (cache.k_scale, before[2], 0x7F), (cache.v_scale, before[3], 0x7F)):
        assert bool((t[sl] == fillv).all()), "freed slot not scrubbed"
        assert torch.equal(t[:r * Tc], b[:r * Tc]) and torch.equal(t[(r + 1) * Tc:], b[(r + 1) * Tc:]), \
            "scrub wrote outside the freed slot"
    q = chunk_qkv(sh, 22, 0, 3, "rms1", q_rows=70)[0]
    out = cache.attn(q.cuda(), 1.0 / math.sqrt(64))
    torch.cuda.synchronize()
    want = oatt.sinkwin_attention(model, bf16_to_f64(q), 1.0 / math.sqrt(64))
    assert_close(to64(out), want, ATOL_FP4, None, "fp4 after unaligned scrub", plus_output_rounding=True)
    assert cache.last_device_error() == swl.KVC_OK


def test_fp4_caches_sharing_one_staging_buffer(swl):
    """Two FP4 caches (different contents) handed the same staging tensor: the
    decode-once path overwrites it on every call, so calls alternating
    between the caches must each see only their own K/V."""
    sh = Shapes(2, 128, 100, 1, 2, 10, 10)
    scale = 1.0 / math.sqrt(128)
    probe = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                        sh.window_chunks, dtype="fp4", stage=True)
    shared = probe.stage
    caches, models = [], []
    for cfg in (51, 52):
        cache = swl.KVCache(sh.heads, sh.head_dim, sh.tokens_per_frame, sh.chunk_frames,
                            sh.window_chunks, dtype="fp4", stage=shared)
        model = CacheModel(sh.heads, sh.head_dim, sh.chunk_tokens, sh.window_chunks)
        for c in range(1 + sh.window_chunks):
            _, k, v = chunk_qkv(sh, cfg, 0, c, "outliers")
            cache.append(k.cuda(), v.cuda(), c)
            model.append(c, ofp4.dequantize(*ofp4.quantize(_f32(k))), ofp4.dequantize(*ofp4.quantize(_f32(v))))
        caches.append(cache)
        models.append(model)
    for rep in range(2):
        for i in (0, 1):
            q = chunk_qkv(sh, 53 + i, 0, rep, "rms1", q_rows=300)[0]
            out = caches[i].attn(q.cuda(), scale)
            torch.cuda.synchronize()
            want = oatt.sinkwin_attention(models[i], bf16_to_f64(q), scale)
            assert_close(to64(out), want, ATOL_FP4, None, f"shared stage, cache {i}, round {rep}",
                         plus_output_rounding=True)
    for cache in caches:
        assert cache.last_device_error() == swl.KVC_OK
