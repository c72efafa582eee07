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
// device address is looked up once per device with cudaGetSymbolAddress (with
// that device current) and then passed to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "kvc.h"

namespace kvc {
namespace {

static_assert(kQuantPartials <= KVC_NOALLOC_SCRATCH_WORDS, "scratch too small for one encode");

// one magnitude maximum per CTA of the encoder's first pass
__device__ __align__(256) int32_t g_quant_scratch[KVC_NOALLOC_SCRATCH_WORDS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_quant_scratch on the current device (looked up once).
int32_t scratch_on_current_device(int32_t* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return *status = KVC_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return *status = KVC_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_quant_scratch) != cudaSuccess || !p) return *status = KVC_ECUDA;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *status = KVC_OK;
  return dev;
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
  const int dev = scratch_on_current_device(&st);
  if (st != KVC_OK) return st;
  // The first pass writes every one of its kQuantPartials words before the
  // second pass reads them, so nothing has to be cleared between calls.
  QuantJob job{x, codes, scales, gscale};
  return launch_quant_fp4(&job, 1, n, g_scratch_ptr[dev], reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? KVC_OK
             : KVC_ECUDA;
}
