"""Pins for the FP4 oracle (E2M1 codes, E4M3 block scales, fp32 tensor scale).

The pins do not reuse the oracle's table search: E4M3 rounding is checked
against an exact rational rounding written from the exponent/mantissa
definition, E2M1 and E4M3 against hand-written golden tables, and the whole
encoder against exhaustive decode -> re-encode round trips and blocks built
from exactly representable values.
"""

import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp4


def _load_golden(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            a, b, c = line.split()[:3]
            rows.append((a, b, c))
    return rows


def test_e2m1_golden(golden_dir):
    for t, code, val in _load_golden(os.path.join(golden_dir, "e2m1_rne.txt")):
        got = int(fp4.e2m1_rne_satfinite(np.float32(float(t))))
        assert got == int(code), (t, got, code)
        assert fp4.e2m1_value(got) == float(val)


def test_e4m3_golden(golden_dir):
    for x, code, val in _load_golden(os.path.join(golden_dir, "e4m3_rne.txt")):
        got = int(fp4.e4m3_rne_satfinite(np.float32(float(x))))
        assert got == int(code, 16), (x, hex(got), code)
        assert fp4.e4m3_value(got) == float(val)


def _e4m3_round_rational(x: Fraction) -> Fraction:
    """E4M3 RNE-satfinite by exponent/quantum arithmetic on exact rationals."""
    if x <= 0:
        return Fraction(0)
    if x >= 448:
        return Fraction(448)
    e = -6
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    quantum = Fraction(2) ** (e - 3)           # 3 mantissa bits; e >= -6 covers subnormals
    m = x / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return min(Fraction(448), fl * quantum)


def test_e4m3_against_rational_rounding():
    vals = [Fraction(v) for v in fp4.E4M3_POS]
    pts = set()
    for a, b in zip(vals[:-1], vals[1:]):
        mid = (a + b) / 2
        for p in (a, b, mid):
            pts.add(float(p))
        f = np.float32(float(mid))
        pts.add(float(np.nextafter(f, np.float32(0))))
        pts.add(float(np.nextafter(f, np.float32(1e9))))
    rng = np.random.default_rng(7)
    pts.update(float(np.float32(x)) for x in np.exp(rng.uniform(np.log(1e-4), np.log(600), 4000)))
    pts.update([0.0, 1e-12, 500.0, 448.0, 449.0, 1e6])
    xs = np.array(sorted(pts), dtype=np.float32)
    codes = fp4.e4m3_rne_satfinite(xs)
    for x, c in zip(xs, codes):
        want = _e4m3_round_rational(Fraction(float(x)))
        assert Fraction(fp4.E4M3_POS[c]) == want, (float(x), int(c), float(want))


def test_e4m3_e2m1_value_tables():
    # closed forms of the format definitions
    assert fp4.e4m3_value(0x7E) == 448.0
    assert np.isnan(fp4.e4m3_value(0x7F)) and np.isnan(fp4.e4m3_value(0xFF))
    assert fp4.e4m3_value(0x01) == 2.0 ** -9
    assert fp4.e4m3_value(0x08) == 2.0 ** -6
    assert fp4.e4m3_value(0xB8) == -1.0
    assert list(fp4.E2M1_POS) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert fp4.e2m1_value(0xF) == -6.0 and fp4.e2m1_value(0x8) == 0.0
    assert np.all(np.diff(fp4.E4M3_POS) > 0)


@pytest.mark.parametrize("g", [np.float32(1.0), np.float32(2.0 ** -7),
                               np.float32(0.0371), np.float32(3.3e-3)])
def test_exhaustive_decode_reencode(g):
    """Every code x every positive finite E4M3 scale: decode then re-encode with
    the same scale and tensor scale gives back the code."""
    s_codes = np.arange(1, 0x7F, dtype=np.uint8)
    codes = np.arange(16, dtype=np.uint8)
    s_val = fp4.E4M3_POS[s_codes].astype(np.float32)
    x = (fp4.E2M1_ALL[codes][None, :] * s_val[:, None].astype(np.float64)
         * float(g)).astype(np.float32)
    sg = s_val * g
    inv = np.float32(1.0) / sg
    t = np.abs(x) * inv[:, None]
    mag = fp4.e2m1_rne_satfinite(t)
    back = (np.signbit(x).astype(np.uint8) << 3) | mag
    # +-0 both decode to 0; the encoder keeps the sign bit of the input
    assert np.array_equal(back, np.broadcast_to(codes, back.shape))


def test_exact_blocks_reproduce_scales_and_codes():
    """Build a tensor whose amax is 2688*g0 (g0 a power of two) and whose
    blocks are E2M1 values times an E4M3 scale times g0: encode is exact."""
    rng = np.random.default_rng(3)
    g0 = np.float32(2.0 ** -5)
    nblk = 300
    s_codes = rng.integers(1, 0x7F, size=nblk).astype(np.uint8)
    s_codes[0] = 0x7E  # the block holding the tensor amax: scale 448
    codes = rng.integers(0, 16, size=(nblk, 16)).astype(np.uint8)
    codes[:, 0] = 7  # every block reaches |6| so amax_b = 6*s*g0
    codes[0, 0] = 7
    vals = fp4.E2M1_ALL[codes] * fp4.E4M3_POS[s_codes][:, None] * float(g0)
    x = vals.astype(np.float32)
    assert np.array_equal(x.astype(np.float64), vals)  # exactly representable
    packed, scales, g = fp4.quantize(x.reshape(nblk, 16))
    assert g == g0
    assert np.array_equal(scales.reshape(-1), s_codes)
    want = codes  # -0 (code 0x8) is encoded from float -0.0 with its sign bit
    got = fp4.unpack_codes(packed).reshape(nblk, 16)
    assert np.array_equal(got, want)
    assert np.array_equal(fp4.dequantize(packed, scales, g).reshape(nblk, 16), vals)


def test_zero_tensor_and_zero_blocks():
    x = np.zeros((4, 32), np.float32)
    p, s, g = fp4.quantize(x)
    assert g == 0 and not p.any() and not s.any()
    x[1, 3] = -2.0
    x[2, 17] = -0.0
    p, s, g = fp4.quantize(x)
    assert g == np.float32(2.0) / np.float32(2688.0)
    c = fp4.unpack_codes(p)
    assert c[1, 3] == 0x8 | 7  # -6 * s * g with s = 448: the block max maps to code 6
    assert not s[0].any() and not c[0].any()  # all-zero blocks
    assert not c[2].any()                      # block of -0 only: scale 0 -> codes 0x0


def test_sign_of_values_rounding_to_zero():
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 6.0
    x[0, 1] = -0.1  # t = 0.1 -> rounds to 0; the sign bit stays
    p, s, g = fp4.quantize(x)
    c = fp4.unpack_codes(p)[0]
    assert c[0] == 7 and c[1] == 0x8


def test_reconstruction_error_bound():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 4, 128)).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 8
    p, s, g = fp4.quantize(x)
    xh = fp4.dequantize(p, s, g)
    sv = np.repeat(fp4.E4M3_ALL[s], 16, axis=-1) * float(g)
    # below the top of the E2M1 grid the error is at most half a grid step (1 unit
    # at the top, between 4 and 6); the scale choice keeps |x|/(s*g) <= ~6.2
    err = np.abs(xh - x.astype(np.float64))
    assert np.all(err <= sv * 1.0 + 1e-30)
    assert np.all(np.abs(x) / sv <= 6.0 * (1 + 2 ** -3) + 1e-6)
    rel = np.linalg.norm(xh - x) / np.linalg.norm(x)
    assert rel < 0.12


def test_tiny_tensor_blocks_without_finite_reciprocal():
    """A tensor whose largest magnitude is 2^-120: g = 2^-120 / 2688 is an fp32
    subnormal, and blocks whose s*g has no finite fp32 reciprocal are stored
    as zeros.  Every block still decodes within the error bound (a zero
    element never decodes to a nonzero value), and the zeroed blocks are only
    blocks whose values are all below 2^-124."""
    rng = np.random.default_rng(5)
    amax = np.float32(2.0 ** -120)
    mags = amax * np.exp2(-rng.uniform(0, 14, (256, 1))).astype(np.float32)
    x = (mags * rng.uniform(-1, 1, (256, 16))).astype(np.float32)
    x[rng.random(x.shape) < 0.2] = 0.0
    x[0, 0] = amax
    p, s, g = fp4.quantize(x)
    assert 0 < g < np.finfo(np.float32).tiny
    xh = fp4.dequantize(p, s, g)
    c = fp4.unpack_codes(p)
    zeroed = s[:, 0] == 0
    assert zeroed.any() and (~zeroed).any()
    assert not c[zeroed].any()
    assert np.all(np.abs(x[zeroed]) < 2.0 ** -124)
    sv = fp4.E4M3_ALL[s[:, 0]] * float(g)
    live = ~zeroed
    err = np.abs(xh - x.astype(np.float64))
    assert np.all(err[live] <= sv[live][:, None] * 1.0)
    assert np.all(xh[x == 0] == 0)


def test_gemm_dequantized_against_loops():
    """The W4A4 projection against a triple loop written from the format's
    value tables (code -> E2M1 value, scale byte -> E4M3 value, times g)."""
    rng = np.random.default_rng(17)
    M, K, N = 5, 32, 48
    a = (rng.standard_normal((M, K)) * rng.uniform(0.1, 3.0, (M, 1))).astype(np.float32)
    b = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    ac, as_, ag = fp4.quantize(a)
    bc, bs, bg = fp4.quantize(b)
    got = fp4.gemm_dequantized(ac, as_, ag, bc, bs, bg)

    def value(codes, scales, g, r, c):
        byte = int(codes[r, c // 2])
        code = byte & 0xF if c % 2 == 0 else byte >> 4
        return fp4.e2m1_value(code) * fp4.e4m3_value(int(scales[r, c // 16])) * float(g)

    want = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            want[i, j] = sum(value(ac, as_, ag, i, k) * value(bc, bs, bg, j, k) for k in range(K))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)


def test_gemm_dequantized_exact_on_representable_inputs():
    """Inputs already on the FP4 grid come back unchanged, so the projection
    equals the plain product of the inputs.  Each tensor's maximum is 2688
    times a power of two (the tensor scale g is then a power of two) and each
    block is E2M1 values times a block factor f whose f / g is an E4M3 value
    (3.5 * 2^7 = 448, or a power of two)."""
    rng = np.random.default_rng(3)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

    def on_grid(rows, cols, top):
        x = rng.choice(grid, (rows, cols)) * rng.choice([-1, 1], (rows, cols))
        x[:, ::16] = 6.0                       # every block maximum is 6 * f
        f = 2.0 ** rng.integers(-2, 2, (rows, cols // 16))
        f[0, 0] = top                          # the tensor maximum 6 * top
        return x * np.repeat(f, 16, axis=1)

    M, K, N = 4, 32, 32
    a = on_grid(M, K, 1.75)                    # amax 10.5 = 2688 / 2^8
    b = on_grid(N, K, 3.5)                     # amax 21 = 2688 / 2^7
    ac, as_, ag = fp4.quantize(a.astype(np.float32))
    bc, bs, bg = fp4.quantize(b.astype(np.float32))
    assert float(ag) == 2.0 ** -8
    assert float(bg) == 2.0 ** -7
    assert np.array_equal(fp4.dequantize(ac, as_, ag), a)
    assert np.array_equal(fp4.dequantize(bc, bs, bg), b)
    assert np.array_equal(fp4.gemm_dequantized(ac, as_, ag, bc, bs, bg), a @ b.T)
