"""Shared helpers for the GPU parity tests: tolerances and comparisons."""

import numpy as np
import torch

# bf16 attention / recache against the float64 oracle
ATOL_BF16 = 2e-2
RELL2_BF16 = 5e-3
# attention over an FP4 cache against the oracle run on the same dequantised K/V;
# the output is bf16, so half a bf16 ulp of the reference value comes on top
# (outliers x8 make |O| reach ~30, where bf16 spacing is 0.125)
ATOL_FP4 = 5e-2


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |x| (8 significant bits): the rounding error a
    bf16 output can carry on its own, however exact the arithmetic before it."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 8.0)


def assert_close(got: np.ndarray, want: np.ndarray, atol: float, rel_l2: float | None, what: str,
                 plus_output_rounding: bool = False):
    """max |got - want| <= atol (+ half a bf16 ulp of want when
    plus_output_rounding) and, if given, ||got - want|| / ||want|| <= rel_l2."""
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    raw = float(np.abs(got - want).max()) if got.size else 0.0
    if plus_output_rounding:
        # subtract the output format's own rounding before the max-abs test
        err = np.maximum(np.abs(got - want) - bf16_half_ulp(want), 0.0)
        what = what + f" (raw max-abs {raw:.3e}; beyond bf16 output rounding)"
    else:
        err = np.abs(got - want)
    mx = float(err.max()) if err.size else 0.0
    msg = f"{what}: max-abs {mx:.3e} (tol {atol})"
    if err.size and mx > atol:
        idx = np.unravel_index(int(np.argmax(err)), err.shape)
        bad = np.argwhere(err > atol)
        msg += (f" at {tuple(int(i) for i in idx)} got {got[idx]:.5f} want {want[idx]:.5f};"
                f" {len(bad)} elements over, first {bad[:3].tolist()} last {bad[-3:].tolist()}")
    if rel_l2 is not None:
        den = float(np.linalg.norm(want))
        rl = float(np.linalg.norm(got - want)) / den if den > 0 else float(np.linalg.norm(got))
        msg += f", rel-L2 {rl:.3e} (tol {rel_l2})"
        assert rl <= rel_l2, msg
    assert mx <= atol, msg
    return msg


SAMPLE_ROWS_4680 = [0, 1, 63, 127, 128, 129, 200, 255, 256, 511, 1000, 1559, 1560, 2047, 2048,
                    3119, 3120, 3333, 4095, 4096, 4500, 4607, 4608, 4650, 4679]
