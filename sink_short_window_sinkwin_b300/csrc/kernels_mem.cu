// HBM-bound kernels: cache append (vectorised copy), evict scrub (fill) and the
// FP4 KV encoder (tensor amax, E4M3 block scales, E2M1 codes).
//
// FP4 KV store: LongLive 2.0 inference blog (blog.hotdry.top), "NVFP4 量化与
// KV Cache 压缩的工程实现" -- inference.kv_quant keeps the cache in FP4.  The
// encode below is the fixed-order fp32 rule stated in kvc.h (kvc_quant_fp4).
#include <cuda_bf16.h>

#include "internal.h"

namespace kvc {
namespace {

constexpr int kMemThreads = 256;
constexpr int kUnroll = 4;

// 128-bit read-only load that does not allocate in L1
__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// blockIdx.y picks the tensor; every thread moves kUnroll 16-byte vectors per
// trip with all loads issued before the stores.
__global__ void __launch_bounds__(kMemThreads) copy2_kernel(uint4* __restrict__ d0,
                                                            const uint4* __restrict__ s0,
                                                            uint4* __restrict__ d1,
                                                            const uint4* __restrict__ s1,
                                                            size_t n16) {
  const uint4* s = blockIdx.y ? s1 : s0;
  uint4* d = blockIdx.y ? d1 : d0;
  const size_t stride = (size_t)gridDim.x * kMemThreads;
  size_t i = (size_t)blockIdx.x * kMemThreads + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) r[u] = ld_nc_v4(s + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[i + u * stride] = r[u];
  }
  for (; i < n16; i += stride) d[i] = ld_nc_v4(s + i);
}

__global__ void __launch_bounds__(kMemThreads) fill2_kernel(uint4* __restrict__ d0,
                                                            uint4* __restrict__ d1, size_t n16,
                                                            uint32_t word) {
  uint4* d = blockIdx.y ? d1 : d0;
  const uint4 w = make_uint4(word, word, word, word);
  const size_t stride = (size_t)gridDim.x * kMemThreads;
  for (size_t i = (size_t)blockIdx.x * kMemThreads + threadIdx.x; i < n16; i += stride) d[i] = w;
}

int mem_grid(size_t n16) {
  // enough CTAs for ~kUnroll vectors per thread, capped at 8 waves of 148 SMs
  size_t want = (n16 + (size_t)kMemThreads * kUnroll - 1) / ((size_t)kMemThreads * kUnroll);
  if (want < 1) want = 1;
  if (want > 148 * 8) want = 148 * 8;
  return (int)want;
}

// ---------------------------------------------------------------------------
// FP4 encode
// ---------------------------------------------------------------------------
struct QuantJobs {
  QuantJob j[2];
};

// max |x| over bf16 bits: clearing the sign bit leaves bit patterns whose
// unsigned order is the order of the magnitudes (finite inputs)
__device__ __forceinline__ uint32_t absmax_bf16x8(uint4 v, uint32_t acc2) {
  acc2 = __vmaxu2(acc2, v.x & 0x7FFF7FFFu);
  acc2 = __vmaxu2(acc2, v.y & 0x7FFF7FFFu);
  acc2 = __vmaxu2(acc2, v.z & 0x7FFF7FFFu);
  acc2 = __vmaxu2(acc2, v.w & 0x7FFF7FFFu);
  return acc2;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
  v = __reduce_max_sync(0xffffffffu, v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
    v = __reduce_max_sync(0xffffffffu, v);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  v = red[0];
  __syncthreads();
  return v;
}

// Pass 1: every CTA writes the magnitude maximum of its grid-stride share as
// bf16 bits into its own scratch word (no atomics, no zeroing needed).
__global__ void __launch_bounds__(kMemThreads) amax_kernel(QuantJobs jobs, int64_t n,
                                                           int32_t* __restrict__ ws) {
  __shared__ uint32_t red[32];
  // select, not index: a dynamic index would copy the parameter struct to local memory
  const uint4* x = reinterpret_cast<const uint4*>(blockIdx.y ? jobs.j[1].x : jobs.j[0].x);
  const int64_t n8 = n >> 3;
  uint32_t acc2 = 0;
  const int64_t stride = (int64_t)gridDim.x * kMemThreads;
  int64_t i = (int64_t)blockIdx.x * kMemThreads + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 r0 = ld_nc_v4(x + i), r1 = ld_nc_v4(x + i + stride), r2 = ld_nc_v4(x + i + 2 * stride),
          r3 = ld_nc_v4(x + i + 3 * stride);
    acc2 = absmax_bf16x8(r0, acc2);
    acc2 = absmax_bf16x8(r1, acc2);
    acc2 = absmax_bf16x8(r2, acc2);
    acc2 = absmax_bf16x8(r3, acc2);
  }
  for (; i < n8; i += stride) acc2 = absmax_bf16x8(ld_nc_v4(x + i), acc2);
  uint32_t m = max(acc2 & 0xFFFFu, acc2 >> 16);
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) ws[blockIdx.y * kQuantPartials + blockIdx.x] = (int32_t)m;
}

// E4M3 code of x >= 0, round to nearest even, saturating at 448 (the
// hardware conversion; OCP E4M3: bias 7, subnormal quantum 2^-9)
__device__ __forceinline__ uint32_t e4m3_rne_satfinite(float x) {
  uint16_t e;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(e) : "f"(0.0f), "f"(x));
  return (uint32_t)e & 0xFFu;  // the second operand lands in the low byte
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  if (e == 0) return (float)m * 0.001953125f;             // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) * 2^(e-7)
}

// Two E2M1 codes (sign | magnitude, round to nearest even, saturating at 6):
// lo in the low nibble.  The sign of a value that rounds to 0 is kept.
__device__ __forceinline__ uint32_t e2m1x2_rne_satfinite(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Pass 2: tensor scale from the partial maxima, then one thread per 16-element
// block: its E4M3 scale byte and 8 bytes of packed E2M1 codes.
__global__ void __launch_bounds__(kMemThreads) quant_kernel(QuantJobs jobs, int64_t n,
                                                            const int32_t* __restrict__ ws) {
  __shared__ uint32_t red[32];
  const QuantJob job = blockIdx.y ? jobs.j[1] : jobs.j[0];
  uint32_t m = 0;
  for (int i = threadIdx.x; i < kQuantPartials; i += kMemThreads)
    m = max(m, (uint32_t)ws[blockIdx.y * kQuantPartials + i]);
  m = block_max_u32(m, red);
  const float amax = __uint_as_float(m << 16);
  const float g = __fdiv_rn(amax, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *job.gscale = g;

  const uint4* x = reinterpret_cast<const uint4*>(job.x);
  uint2* codes = reinterpret_cast<uint2*>(job.codes);
  const int64_t nblk = n >> 4;
  const int64_t stride = (int64_t)gridDim.x * kMemThreads;
  for (int64_t b = (int64_t)blockIdx.x * kMemThreads + threadIdx.x; b < nblk; b += stride) {
    const uint4 v0 = ld_nc_v4(x + 2 * b), v1 = ld_nc_v4(x + 2 * b + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t acc2 = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc2 = __vmaxu2(acc2, w[k] & 0x7FFF7FFFu);
    const float amax_b = __uint_as_float(max(acc2 & 0xFFFFu, acc2 >> 16) << 16);
    uint32_t s = 0, lo = 0, hi = 0;
    if (g != 0.0f) {
      s = e4m3_rne_satfinite(__fdiv_rn(__fdiv_rn(amax_b, 6.0f), g));
      const float sg = __fmul_rn(e4m3_value(s), g);
      if (s != 0 && sg != 0.0f) {
        const float inv = __frcp_rn(sg);
        // |x| * inv and x * inv round to the same magnitude; the sign rides along
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t byte =
              e2m1x2_rne_satfinite(__fmul_rn(bf16_lo(w[k]), inv), __fmul_rn(bf16_hi(w[k]), inv));
          if (k < 4) lo |= byte << (8 * k);
          else hi |= byte << (8 * (k - 4));
        }
      } else {
        s = 0;
      }
    }
    codes[b] = make_uint2(lo, hi);
    job.scales[b] = (uint8_t)s;
  }
}

}  // namespace

cudaError_t launch_copy2(void* dst0, const void* src0, void* dst1, const void* src1, size_t bytes,
                         cudaStream_t st) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  dim3 grid(mem_grid(n16), dst1 ? 2 : 1);
  copy2_kernel<<<grid, kMemThreads, 0, st>>>(
      static_cast<uint4*>(dst0), static_cast<const uint4*>(src0), static_cast<uint4*>(dst1),
      static_cast<const uint4*>(src1), n16);
  return cudaGetLastError();
}

cudaError_t launch_fill2_u16(void* d0, void* d1, size_t bytes, uint16_t pattern, cudaStream_t st) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  dim3 grid(mem_grid(n16), d1 ? 2 : 1);
  fill2_kernel<<<grid, kMemThreads, 0, st>>>(static_cast<uint4*>(d0), static_cast<uint4*>(d1), n16,
                                             (uint32_t)pattern * 0x00010001u);
  return cudaGetLastError();
}

cudaError_t launch_fill2_u8(void* d0, void* d1, size_t bytes, uint8_t pattern, cudaStream_t st) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  dim3 grid(mem_grid(n16), d1 ? 2 : 1);
  fill2_kernel<<<grid, kMemThreads, 0, st>>>(static_cast<uint4*>(d0), static_cast<uint4*>(d1), n16,
                                             (uint32_t)pattern * 0x01010101u);
  return cudaGetLastError();
}

cudaError_t launch_quant_fp4(const QuantJob* jobs, int njobs, int64_t n, int32_t* ws,
                             cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  QuantJobs qj{};
  for (int i = 0; i < njobs; ++i) qj.j[i] = jobs[i];
  amax_kernel<<<dim3(kQuantPartials, njobs), kMemThreads, 0, st>>>(qj, n, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nblk = n >> 4;
  int64_t want = (nblk + kMemThreads - 1) / kMemThreads;
  if (want > 148 * 8) want = 148 * 8;
  if (want < 1) want = 1;
  quant_kernel<<<dim3((unsigned)want, njobs), kMemThreads, 0, st>>>(qj, n, ws);
  return cudaGetLastError();
}

}  // namespace kvc
