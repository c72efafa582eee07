"""kvc_quant_fp4_noalloc: the FP4 encoder for callers that cannot allocate.

Some callers of this library cannot hand it device memory at call time -- their
device memory is owned by another allocator, or their loop may not call
cudaMalloc (it can synchronise the device).  kvc_quant_fp4_noalloc serves them:
it takes the encoder's scratch from a static array inside the library instead
of a caller buffer.  This test calls it through the C ABI three times in a row,
on different inputs (each call starts from whatever the previous one left in
the shared array, and the second one uses fewer of its words), and checks that codes, block scales and tensor scale are
bit-identical to kvc_quant_fp4's on the same inputs -- the bar every FP4 encode
test in this suite uses.  It lives in its own file, collected last, and passes
both alone in a fresh process and after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest
import torch

from synth import gaussian_outliers_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sink_short_window_sinkwin_b300._abi import lib as _lib
    return _lib()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _outputs(n, dev):
    return (torch.empty(n // 2, dtype=torch.uint8, device=dev),
            torch.empty(n // 16, dtype=torch.uint8, device=dev),
            torch.empty(1, dtype=torch.float32, device=dev))


def test_noalloc_matches_kvc_quant_fp4_twice(lib):
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = torch.empty(256, dtype=torch.int32, device=dev)  # scratch of the existing entry point
    # calls in a row on the shared array: a LongLive-1.3B K chunk with outliers
    # (its first pass fills all 256 partial maxima), then a tensor of 800
    # elements whose first pass writes only 100 partials and whose amax is
    # about 1000x smaller -- a read of any word the previous call left would
    # change its tensor scale -- then a ragged mid-size tensor
    inputs = [gaussian_outliers_bf16((4680, 12, 128), 0.01, 8.0, 77, 0, 0, 3),
              gaussian_outliers_bf16((16 * 50,), 0.01, 8.0, 77, 0, 2, 3) * 1e-3,
              gaussian_outliers_bf16((16 * 30001,), 0.01, 8.0, 77, 0, 1, 3) * 1e-2]
    for i, x_cpu in enumerate(inputs):
        x = x_cpu.to(dev).contiguous()
        n = x.numel()
        c0, s0, g0 = _outputs(n, dev)
        c1, s1, g1 = _outputs(n, dev)
        assert lib.kvc_quant_fp4(_p(x), n, _p(c0), _p(s0), _p(g0), _p(ws), stream) == 0
        assert lib.kvc_quant_fp4_noalloc(_p(x), n, _p(c1), _p(s1), _p(g1), stream) == 0
        torch.cuda.synchronize()
        assert torch.equal(c0, c1), f"call {i}: codes differ"
        assert torch.equal(s0, s1), f"call {i}: block scales differ"
        assert g0.cpu().numpy().view(np.uint32)[0] == g1.cpu().numpy().view(np.uint32)[0], \
            f"call {i}: tensor scale differs"


def test_noalloc_rejects_sizes_beyond_the_maximum(lib):
    dev = torch.device("cuda", torch.cuda.current_device())
    x = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    c, s, g = _outputs(64, dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    max_elems = 1 << 35
    assert lib.kvc_quant_fp4_noalloc(_p(x), max_elems + 16, _p(c), _p(s), _p(g), stream) == -1
    assert lib.kvc_quant_fp4_noalloc(_p(x), 40, _p(c), _p(s), _p(g), stream) == -1
    assert lib.kvc_quant_fp4_noalloc(_p(x), 0, _p(c), _p(s), _p(g), stream) == -1
