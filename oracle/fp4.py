"""FP4 KV store encode / decode (oracle side).

LongLive 2.0 inference blog (blog.hotdry.top), "NVFP4 量化与 KV Cache 压缩的工程
实现": with inference.kv_quant the KV cache is stored as FP4 and read through a
fused dequantisation extension; the data-pipeline blog, "三、NVFP4 量化", says the
same.  The pages name the format only as FP4/NVFP4.  The FP4 KV workload fixes
it as: E2M1 codes in 16-element blocks, one E4M3 scale per block, one fp32
per-tensor scale.  E4M3 and E2M1 follow the OCP 8-bit / 4-bit float
definitions (E4M3: 4 exponent bits, bias 7, 3 mantissa bits, subnormals, no
infinity, 0x7F/0xFF NaN, largest finite 448; E2M1 magnitudes
{0, .5, 1, 1.5, 2, 3, 4, 6}).

Encode, in IEEE fp32 with this exact operation order (readings, the pages give
none; the CUDA side follows the same order so codes match bit for bit):
  1. amax = max |x| over the tensor;  g = fl32(amax / 2688)   (2688 = 6 * 448)
     if g == 0 every scale and code is 0 and the stored g is 0.
  2. per block b of 16: s_f = fl32(fl32(amax_b / 6) / g);  s = E4M3_rne_satfinite(s_f)
  3. inv = fl32(1 / fl32(s*g)).  If s == 0, fl32(s*g) == 0 or inv overflows
     to infinity (s*g below about 2^-128: only for tensors whose largest
     magnitude is below about 2^-115), the block is stored as zeros: scale
     byte 0 and codes 0x0 (a reading: the rule has no finite t there);
     else t = fl32(|x| * inv);
          code = signbit(x) << 3 | E2M1_rne_satfinite(t)
  4. element 2i in the low nibble, 2i+1 in the high nibble of a byte.
Decode: x_hat = e2m1(code) * s * g, exact in float64.

Both roundings are written from their definition: the nearest representable
value, found in the table of all values; an exact tie goes to the even code.
"""

from __future__ import annotations

import numpy as np

F4_BLOCK = 16
E4M3_MAX = 448.0
G_DIVISOR = np.float32(2688.0)  # 6 * 448


def e4m3_value(code: int) -> float:
    """Exact value of an OCP E4M3 byte (NaN for 0x7F / 0xFF)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e2m1_value(code: int) -> float:
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * 0.5 * m
    return s * (1.0 + 0.5 * m) * 2.0 ** (e - 1)


# positive finite values in code order (codes 0x00..0x7E / 0..7 are increasing)
E4M3_POS = np.array([e4m3_value(c) for c in range(0x7F)], dtype=np.float64)
E2M1_POS = np.array([e2m1_value(c) for c in range(8)], dtype=np.float64)
E4M3_ALL = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_ALL = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def _round_to_table(x: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Nearest entry of an increasing table (ties to the even index), saturating
    at the last entry.  x >= 0, finite."""
    x = np.asarray(x, dtype=np.float64)
    hi = np.searchsorted(table, x, side="left")
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    d_lo = x - table[lo]
    d_hi = table[hi] - x
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(x >= table[-1], len(table) - 1, idx)
    idx = np.where(x <= 0.0, 0, idx)
    return idx.astype(np.uint8)


def e4m3_rne_satfinite(x) -> np.ndarray:
    """E4M3 code of non-negative finite x: round to nearest, ties to even, clamp to 448."""
    return _round_to_table(x, E4M3_POS)


def e2m1_rne_satfinite(t) -> np.ndarray:
    """3-bit E2M1 magnitude code of non-negative finite t (ties to even, clamp to 6)."""
    return _round_to_table(t, E2M1_POS)


def quantize(x) -> tuple[np.ndarray, np.ndarray, np.float32]:
    """Encode a tensor whose last axis is a multiple of 16.

    Returns (codes uint8 [..., D/2], scales uint8 E4M3 [..., D/16], g float32).
    """
    x = np.asarray(x, dtype=np.float32)
    if x.shape[-1] % F4_BLOCK:
        raise ValueError("last axis must be a multiple of 16")
    lead = x.shape[:-1]
    D = x.shape[-1]
    blocks = x.reshape(-1, F4_BLOCK)
    nb = blocks.shape[0]
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    g = np.float32(amax / G_DIVISOR)
    if g == np.float32(0.0):
        return (np.zeros(lead + (D // 2,), np.uint8), np.zeros(lead + (D // 16,), np.uint8),
                np.float32(0.0))
    amax_b = np.max(np.abs(blocks), axis=1).astype(np.float32)
    s_f = (amax_b / np.float32(6.0)) / g
    s_code = e4m3_rne_satfinite(s_f)
    s_val = E4M3_POS[s_code].astype(np.float32)
    sg = s_val * g
    with np.errstate(divide="ignore", over="ignore"):
        inv = np.float32(1.0) / np.where(sg == np.float32(0.0), np.float32(1.0), sg)
    dead = (s_code == 0) | (sg == np.float32(0.0)) | ~np.isfinite(inv)
    inv = np.where(dead, np.float32(1.0), inv).astype(np.float32)
    t = np.abs(blocks) * inv[:, None]
    mag = e2m1_rne_satfinite(t)
    code = (np.signbit(blocks).astype(np.uint8) << 3) | mag
    code[dead] = 0
    s_code = np.where(dead, np.uint8(0), s_code).astype(np.uint8)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return (packed.reshape(lead + (D // 2,)), s_code.reshape(lead + (D // 16,)), g)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., D/2] -> 4-bit codes [..., D] (low nibble first)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequantize(packed: np.ndarray, scales: np.ndarray, g) -> np.ndarray:
    """x_hat = e2m1(code) * s * g, exact in float64, shape [..., D]."""
    codes = unpack_codes(packed)
    D = codes.shape[-1]
    vals = E2M1_ALL[codes]
    s = E4M3_ALL[np.asarray(scales, dtype=np.uint8)]
    s = np.repeat(s, F4_BLOCK, axis=-1)
    assert s.shape[-1] == D
    return vals * s * float(np.float32(g))


def gemm_dequantized(a_codes, a_scales, a_g, b_codes, b_scales, b_g) -> np.ndarray:
    """W4A4 projection: dequantize(A) @ dequantize(B), exact products summed in
    float64.

    LongLive 2.0 inference blog (blog.hotdry.top), "NVFP4 量化与 KV Cache 压缩的
    工程实现": NVFP4 (W4A4) inference keeps both weights and activations in 4-bit
    floating point; the NVIDIA infrastructure blog (bittide page), §6, lists
    W4A4 execution in the LongLive 2.0 system.  A (activations) is [M][K] and
    B (the weight, one row per output feature) is [N][K]; each is an FP4
    tensor of this module's format, its 16-element blocks along K, one fp32
    tensor scale.  The result is [M][N] = deq(A) deq(B)^T."""
    return dequantize(a_codes, a_scales, a_g) @ dequantize(b_codes, b_scales, b_g).T
