"""GPU parity of the W4A4 projection (kvc_gemm_fp4) against the oracle's
deq(A) deq(B)^T in float64, on operands the oracle encoder wrote.

Tolerance, from the arithmetic: every decoded element and every product of
two is exact (at most 6 significant bits each), so the kernel's only errors
are the fp32 accumulation over K terms, at most K * 2^-23 * S relative to the
sum S of |products| even with truncating adds (taken twice over), and the
final rounding to bf16, at most 2^-8 of the value."""

import numpy as np
import pytest
import torch

from oracle import fp4 as ofp4
from synth import LAYER_1P3B, gaussian_bf16, gaussian_outliers_bf16, project_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_short_window_sinkwin_b300 as swl
    return swl


def _encode(x: np.ndarray):
    """Oracle-encoded FP4 operand: numpy (codes [rows][K/2], scales, g) and
    the same on the GPU."""
    c, s, g = ofp4.quantize(np.ascontiguousarray(x, dtype=np.float32))
    dev = (torch.from_numpy(np.ascontiguousarray(c)).cuda(),
           torch.from_numpy(np.ascontiguousarray(s)).cuda(),
           torch.tensor([float(g)], dtype=torch.float32).cuda())
    return (c, s, g), dev


def _check(got: np.ndarray, a, b, rows=None, what=""):
    """Compare the kernel's rows `rows` (all when None) with the oracle."""
    ac, as_, ag = a
    bc, bs, bg = b
    if rows is not None:
        ac, as_ = ac[rows], as_[rows]
        got = got[rows]
    want = ofp4.gemm_dequantized(ac, as_, ag, bc, bs, bg)
    s_abs = np.abs(ofp4.dequantize(ac, as_, ag)) @ np.abs(ofp4.dequantize(bc, bs, bg)).T
    K = as_.shape[1] * 16
    tol = 2.0 ** -8 * np.abs(want) + 2 * K * 2.0 ** -23 * s_abs + 1e-38
    err = np.abs(got - want)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside the bound; worst "
                           f"{float((err / tol).max()):.3g}x at {np.unravel_index(np.argmax(err / tol), err.shape)}")
    return want


def _run(swl, a_dev, b_dev, M, N, K, two_phase=False):
    """The kernel's output as float64; two_phase: through a workspace
    (decode once, then the f16 GEMM) filled with garbage first."""
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    if two_phase:
        ws = torch.full((swl.gemm_fp4_ws_bytes(M, N, K),), 0xFF, dtype=torch.uint8, device="cuda")
    swl.gemm_fp4(a_dev, b_dev, M, N, K, out=out, ws=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "a kernel wait ran out"
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K", [
    (1, 192, 256),        # one row, one tile
    (128, 192, 256),      # exactly one tile
    (300, 384, 512),      # ragged last row tile, 2 column tiles, 2 raw stages
    (129, 768, 1024),     # one row past a tile, 4 column tiles, 4 raw stages
    (200, 32, 256),       # one 32-column chunk of a column tile
    (250, 544, 512),      # ragged last column tile (544 = 2 x 192 + 160)
    (1000, 1536, 768),    # 8 x 8 tiles, ragged row tail
    (2500, 4096, 256),    # 20 x 22 tiles (the last ragged): several per CTA
])
@pytest.mark.parametrize("two_phase", [False, True], ids=["fused", "two_phase"])
def test_gemm_fp4_small_shapes(swl, M, N, K, two_phase):
    x = gaussian_bf16((M, K), 1.0, 91, M, N, K).float().numpy()
    w = gaussian_outliers_bf16((N, K), 0.01, 8.0, 92, M, N, K).float().numpy() * 0.02
    a, a_dev = _encode(x)
    b, b_dev = _encode(w)
    got = _run(swl, a_dev, b_dev, M, N, K, two_phase)
    _check(got, a, b, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("two_phase", [False, True], ids=["fused", "two_phase"])
def test_gemm_fp4_exact_on_grid(swl, two_phase):
    """Operands already on the FP4 grid: E2M1 values, every block maximum 6,
    and row 0's first block times 1.75 (maximum 10.5 = 2688 / 2^8, so the
    tensor scale is 2^-8 and every block scale, 256 or 448, is exact).  Every
    product is then a multiple of 2^-6 and every partial sum below 2^17, so
    fp32 accumulation is exact in any order and the bf16 output must equal
    the oracle's value rounded once to bf16."""
    rng = np.random.default_rng(5)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    M, N, K = 200, 512, 512

    def on_grid(rows):
        x = rng.choice(grid, (rows, K)) * rng.choice([-1, 1], (rows, K))
        x[:, ::16] = 6.0
        x[0, :16] *= 1.75
        return x

    x, w = on_grid(M), on_grid(N)
    a, a_dev = _encode(x)
    b, b_dev = _encode(w)
    assert float(a[2]) == 2.0 ** -8 and float(b[2]) == 2.0 ** -8
    assert np.array_equal(ofp4.dequantize(*a), x) and np.array_equal(ofp4.dequantize(*b), w)
    got = _run(swl, a_dev, b_dev, M, N, K, two_phase)
    want = x @ w.T
    assert np.all(np.abs(x) @ np.abs(w).T < 2.0 ** 17)
    assert np.array_equal(want.astype(np.float32).astype(np.float64), want)
    want_bf16 = torch.from_numpy(want.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, want_bf16)


@pytest.mark.parametrize("two_phase", [False, True], ids=["fused", "two_phase"])
def test_gemm_fp4_layer_projection_full_size(swl, two_phase):
    """One LongLive-1.3B chunk's Q|K|V projection (4680 tokens x 1536 ->
    4608) in W4A4, every column of 66 sampled rows (every 73rd and the last)."""
    sh = LAYER_1P3B
    hid, w = project_inputs(sh, 1, 0)
    M, K = hid.shape
    N = w.shape[1]
    a, a_dev = _encode(hid.float().numpy())
    b, b_dev = _encode(np.ascontiguousarray(w.float().numpy().T))
    got = _run(swl, a_dev, b_dev, M, N, K, two_phase)
    assert np.isfinite(got).all()
    rows = np.unique(np.concatenate([np.arange(0, M, 73), [M - 1]]))
    _check(got, a, b, rows=rows, what="layer Q|K|V projection")


def test_gemm_fp4_zero_and_empty(swl):
    """All-zero operands (tensor scale 0, every code and scale 0) give zeros;
    M = 0 launches nothing and leaves the output alone."""
    M, N, K = 130, 256, 256
    a, a_dev = _encode(np.zeros((M, K), np.float32))
    b, b_dev = _encode(gaussian_bf16((N, K), 1.0, 93).float().numpy())
    for two_phase in (False, True):
        got = _run(swl, a_dev, b_dev, M, N, K, two_phase)
        assert np.array_equal(got, np.zeros((M, N)))
    out = torch.empty(0, N, dtype=torch.bfloat16, device="cuda")
    e = (a_dev[0][:0], a_dev[1][:0], a_dev[2])
    swl.gemm_fp4(e, b_dev, 0, N, K, out=out)
    torch.cuda.synchronize()


@pytest.mark.parametrize("two_phase", [False, True], ids=["fused", "two_phase"])
def test_gemm_fp4_magnitude_extremes(swl, two_phase):
    """Block maxima from 2^-30 to 2^12 within one tensor (block scales over
    E4M3's whole range, subnormal ones included) and a weight at the format's
    top (decoded values up to 2688 before the tensor scale)."""
    rng = np.random.default_rng(8)
    M, N, K = 256, 256, 512
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.repeat(2.0 ** rng.uniform(-30, 12, (M, K // 16)), 16, axis=1).astype(np.float32)
    w = rng.standard_normal((N, K)).astype(np.float32) * 1e4
    a, a_dev = _encode(x)
    b, b_dev = _encode(w)
    got = _run(swl, a_dev, b_dev, M, N, K, two_phase)
    _check(got, a, b, what="extremes")


def test_gemm_fp4_rejects_unsupported(swl):
    a, a_dev = _encode(np.ones((4, 256), np.float32))
    b, b_dev = _encode(np.ones((112, 256), np.float32))
    with pytest.raises(swl.KvcError):
        swl.gemm_fp4(a_dev, b_dev, 4, 112, 256)  # N % 32 != 0
    b, b_dev = _encode(np.ones((128, 256), np.float32))
    short = torch.empty(swl.gemm_fp4_ws_bytes(4, 128, 256) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(swl.KvcError):
        swl.gemm_fp4(a_dev, b_dev, 4, 128, 256, ws=short)  # workspace too small
