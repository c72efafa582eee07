// FP4 -> f16 decode pass: contiguous runs of FP4 (E2M1 codes, E4M3 scale per
// 16 elements) written out as f16, one launch for several runs ("jobs").
// Used by the FP4 attention with a staging buffer (the visible regions' K and
// V, V with its tensor scale over the attention's V shift folded in) and by
// the two-phase W4A4 projection (A and B).  Format: LongLive 2.0 inference
// blog (blog.hotdry.top), "NVFP4 量化与 KV Cache 压缩的工程实现".
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecUnroll = 4;

struct Fp4DecodeJobs {
  Fp4DecodeJob j[kMaxDecodeJobs];
  const float* gscale;
  int32_t nregions;
  int32_t regions[1 + KVC_MAX_WINDOW];
};

// 1 / G: G the power of two with the largest listed tensor scale in [G/2, G)
// (1 when that scale is 0 or not below 1e36), the rule of the attention's V shift
__device__ __forceinline__ float inv_v_shift_of(const Fp4DecodeJobs& jj) {
  float gmax = 0.0f;
  for (int i = 0; i < jj.nregions; ++i) gmax = fmaxf(gmax, __ldg(jj.gscale + jj.regions[i]));
  if (gmax > 0.0f && gmax < 1.0e36f) {
    const int e = max(-125, ((int)((__float_as_uint(gmax) >> 23) & 0xFFu)) - 126);  // gmax < 2^e
    return __uint_as_float((uint32_t)(127 - e) << 23);
  }
  return 1.0f;
}

// blockIdx.y = job.  Rows are contiguous, so group i (8 elements) of a job has
// its 4 code bytes at 4 i, its scale byte at i / 2 and its 16 bytes of f16 at
// 16 i: a warp's loads and stores are contiguous.  Each thread takes
// kDecUnroll groups a pass, its loads issued before any use.  The f16 value is
// e2m1(code) * e4m3(scale), exact; the tensor scale is applied by the consumer.
__global__ void __launch_bounds__(kDecThreads) fp4_to_f16_kernel(const __grid_constant__ Fp4DecodeJobs jobs) {
  pdl_launch_dependents();  // a dependent launched with PDL may set up meanwhile
  const Fp4DecodeJob& jb = jobs.j[blockIdx.y];
  const int64_t n = jb.groups;
  // tensor scale over G (jobs with a region): one fp32 rounding of the exact
  // e2m1 * s times this factor, then one rounding to f16
  const bool scaled = jb.g_region >= 0;
  const float f = scaled ? __ldg(jobs.gscale + jb.g_region) * inv_v_shift_of(jobs) : 1.0f;
  const int64_t stride = (int64_t)gridDim.x * kDecThreads;
  for (int64_t base = (int64_t)blockIdx.x * kDecThreads + threadIdx.x; base < n;
       base += stride * kDecUnroll) {
    uint32_t w[kDecUnroll], sc[kDecUnroll];
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int64_t i = base + u * stride;
      w[u] = 0;
      sc[u] = 0;
      if (i < n) {
        w[u] = __ldg(reinterpret_cast<const uint32_t*>(jb.codes) + i);
        sc[u] = __ldg(jb.scales + (i >> 1));
      }
    }
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int64_t i = base + u * stride;
      if (i >= n) break;
      const uint32_t sp = e4m3x2_to_f16x2(sc[u]);  // low half: the scale
      const __half2 s2 = __low2half2(*reinterpret_cast<const __half2*>(&sp));
      uint32_t h4[4];
      e2m1x8_to_f16x8(w[u], h4);
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2 hv = __hmul2(*reinterpret_cast<const __half2*>(&h4[k]), s2);  // exact
        if (scaled) {
          const float2 fv = __half22float2(hv);
          o[k] = pack_f16x2(fv.x * f, fv.y * f);
        } else {
          o[k] = *reinterpret_cast<const uint32_t*>(&hv);
        }
      }
      reinterpret_cast<uint4*>(jb.out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_fp4_to_f16(const Fp4DecodeJob* jobs, int njobs, cudaStream_t st, const float* gscale,
                              const int32_t* regions, int nregions) {
  if (njobs < 1 || njobs > kMaxDecodeJobs || nregions < 0 || nregions > 1 + KVC_MAX_WINDOW)
    return cudaErrorInvalidValue;
  Fp4DecodeJobs jj{};
  jj.gscale = gscale;
  jj.nregions = nregions;
  for (int i = 0; i < nregions; ++i) jj.regions[i] = regions[i];
  for (int i = 0; i < njobs; ++i)
    if (jobs[i].g_region >= 0 && !gscale) return cudaErrorInvalidValue;
  int64_t most = 0;
  for (int i = 0; i < njobs; ++i) {
    jj.j[i] = jobs[i];
    most = jobs[i].groups > most ? jobs[i].groups : most;
  }
  if (most == 0) return cudaSuccess;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static int sm_count[64] = {};
  if (!sm_count[dev] && cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  // about eight blocks per SM in all, shared by the jobs
  const int64_t need = (most + kDecThreads * kDecUnroll - 1) / (kDecThreads * kDecUnroll);
  int64_t cap = (int64_t)sm_count[dev] * 8 / njobs;
  if (cap < 1) cap = 1;
  const int gx = (int)(need < cap ? need : cap);
  fp4_to_f16_kernel<<<dim3(gx, njobs, 1), kDecThreads, 0, st>>>(jj);
  return cudaGetLastError();
}

}  // namespace kvc
