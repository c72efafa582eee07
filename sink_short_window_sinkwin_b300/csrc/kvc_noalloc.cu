// FP4 encode without caller-provided scratch (kvc_quant_fp4_noalloc).
//
// kvc_quant_fp4 needs KVC_QUANT_WS_WORDS int32 of device scratch for the
// per-CTA magnitude maxima of its first pass, and takes that scratch from the
// caller.  Some callers cannot hand out device memory at call time: a host
// program whose device memory is entirely owned by another allocator, or a
// latency-critical loop in which a cudaMalloc (which may synchronise the
// device) is not allowed.  For them this entry point keeps the scratch in a
// file-scope __device__ array that every GPU loading the library holds until
// the process exits, and allocates nothing.
//
// The array is a host-side stand-in in host code, not a device address: its
// device address is looked up with cudaGetSymbolAddress, with the caller's
// device current, on every call (a host-side lookup; the first one on a device
// may load the library's device code there, so make the first call before any
// stream capture) and then passed to the kernels.  Looking it up each time
// keeps the address right after a cudaDeviceReset re-creates the device's
// context and reloads the module.
#include <cuda_runtime.h>

#include "internal.h"
#include "kvc.h"

namespace kvc {
namespace {

static_assert(kQuantPartials <= KVC_NOALLOC_SCRATCH_WORDS, "scratch too small for one encode");

// one magnitude maximum per CTA of the encoder's first pass
__device__ __align__(256) int32_t g_quant_scratch[KVC_NOALLOC_SCRATCH_WORDS];

// Device address of g_quant_scratch on the current device.
int32_t* scratch_on_current_device(int32_t* status) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_quant_scratch) != cudaSuccess || !p) {
    *status = KVC_ECUDA;
    return nullptr;
  }
  *status = KVC_OK;
  return static_cast<int32_t*>(p);
}

}  // namespace
}  // namespace kvc

using namespace kvc;

extern "C" int32_t kvc_quant_fp4_noalloc(const void* x, int64_t n, uint8_t* codes, uint8_t* scales,
                                         float* gscale, kvc_stream_t stream) {
  if (!x || !codes || !scales || !gscale) return KVC_EINVAL;
  if (n < 16 || n % 16 != 0 || n > KVC_NOALLOC_MAX_ELEMS) return KVC_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(codes) & 7u) ||
      (reinterpret_cast<uintptr_t>(gscale) & 3u))
    return KVC_EINVAL;
  int32_t st = KVC_OK;
  int32_t* scratch = scratch_on_current_device(&st);
  if (st != KVC_OK) return st;
  // The first pass writes every one of its kQuantPartials words before the
  // second pass reads them, so nothing has to be cleared between calls.
  QuantJob job{x, codes, scales, gscale};
  return launch_quant_fp4(&job, 1, n, scratch, kQuantPartials, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? KVC_OK
             : KVC_ECUDA;
}
