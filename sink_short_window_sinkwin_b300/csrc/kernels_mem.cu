// HBM-bound kernels: cache append (vectorised copy), evict scrub (fill) and the
// FP4 KV encoder (tensor amax, E4M3 block scales, E2M1 codes).
//
// FP4 KV store: LongLive 2.0 inference blog (blog.hotdry.top), "NVFP4 量化与
// KV Cache 压缩的工程实现" -- inference.kv_quant keeps the cache in FP4.  The
// encode below is the fixed-order fp32 rule stated in kvc.h (kvc_quant_fp4).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

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

// Up to four byte ranges, each filled with a repeated byte pattern (given as a
// 32-bit word); blockIdx.y picks the range (selected, not indexed, so the
// parameters stay in constant space).  The 16-byte-aligned body is written
// with vector stores, the head and tail bytes by the first CTA of the range.
struct FillJobs {
  uint8_t* d[4];
  size_t bytes[4];
  uint32_t word[4];
};
__global__ void __launch_bounds__(kMemThreads) fill_kernel(FillJobs f) {
  const int y = blockIdx.y;
  uint8_t* d = y == 0 ? f.d[0] : y == 1 ? f.d[1] : y == 2 ? f.d[2] : f.d[3];
  const size_t n = y == 0 ? f.bytes[0] : y == 1 ? f.bytes[1] : y == 2 ? f.bytes[2] : f.bytes[3];
  const uint32_t word = y == 0 ? f.word[0] : y == 1 ? f.word[1] : y == 2 ? f.word[2] : f.word[3];
  const uintptr_t p0 = reinterpret_cast<uintptr_t>(d), p1 = p0 + n;
  uintptr_t a = (p0 + 15) & ~uintptr_t(15), e = p1 & ~uintptr_t(15);
  if (a > e) a = e = p1;  // shorter than one aligned vector: all head bytes
  uint4* body = reinterpret_cast<uint4*>(a);
  const size_t n16 = (e - a) / 16;
  const uint4 w = make_uint4(word, word, word, word);
  const size_t stride = (size_t)gridDim.x * kMemThreads;
  for (size_t i = (size_t)blockIdx.x * kMemThreads + threadIdx.x; i < n16; i += stride) body[i] = w;
  if (blockIdx.x == 0 && threadIdx.x < 32) {  // at most 15 head and 15 tail bytes
    const uintptr_t h = p0 + threadIdx.x, t = e + threadIdx.x;
    if (h < a) *reinterpret_cast<uint8_t*>(h) = (uint8_t)(word >> (8 * (h & 3)));
    if (t < p1) *reinterpret_cast<uint8_t*>(t) = (uint8_t)(word >> (8 * (t & 3)));
  }
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

// Per-tensor table over the 127 finite positive E4M3 codes s:
// {fl32(e4m3(s) * g), fl32(1 / that)}, built once per CTA and tensor so the
// per-block reciprocal of the encode rule becomes a lookup.
struct ScaleTab {
  float2 e[128];
};
__device__ __forceinline__ void build_scale_tab(ScaleTab& t, float g, int tid, int nthreads) {
  for (int s = tid; s < 128; s += nthreads) {
    const float sg = __fmul_rn(e4m3_value((uint32_t)s), g);
    t.e[s] = make_float2(sg, sg != 0.0f ? __frcp_rn(sg) : 0.0f);
  }
}

// fl32(a / 6) for a bf16 value a >= 0 without a division: the rounded product
// corrected by one FMA residual step; checked exhaustively against the
// correctly rounded quotient for every bf16 value.
__device__ __forceinline__ float div6_bf16(float a) {
  const float r = 0.16666667163372039794921875f;  // fl32(1/6)
  const float q = __fmul_rn(a, r);
  const float e = __fmaf_rn(-q, 6.0f, a);
  return __fmaf_rn(e, r, q);
}

// One 16-element block (8 words of bf16 pairs) under tensor scale g: its E4M3
// scale byte and 8 bytes of packed E2M1 codes, in the fixed fp32 order of the
// encode rule.
__device__ __forceinline__ void encode_block(const uint32_t (&w)[8], float g, const ScaleTab& tab,
                                             uint32_t& s, uint32_t& lo, uint32_t& hi) {
  uint32_t acc2 = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) acc2 = __vmaxu2(acc2, w[k] & 0x7FFF7FFFu);
  const float amax_b = __uint_as_float(max(acc2 & 0xFFFFu, acc2 >> 16) << 16);
  s = 0;
  lo = 0;
  hi = 0;
  if (g == 0.0f) return;
  s = e4m3_rne_satfinite(__fdiv_rn(div6_bf16(amax_b), g));
  const float2 sgi = tab.e[s];  // {s * g, 1 / (s * g)}
  if (s == 0 || sgi.x == 0.0f) {
    s = 0;
    return;
  }
  const float inv = sgi.y;
  // |x| * inv and x * inv round to the same magnitude; the sign rides along
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t byte =
        e2m1x2_rne_satfinite(__fmul_rn(bf16_lo(w[k]), inv), __fmul_rn(bf16_hi(w[k]), inv));
    if (k < 4) lo |= byte << (8 * k);
    else hi |= byte << (8 * (k - 4));
  }
}

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
  __shared__ ScaleTab tab;
  build_scale_tab(tab, g, threadIdx.x, kMemThreads);
  __syncthreads();

  const uint4* x = reinterpret_cast<const uint4*>(job.x);
  uint2* codes = reinterpret_cast<uint2*>(job.codes);
  const int64_t nblk = n >> 4;
  const int64_t stride = (int64_t)gridDim.x * kMemThreads;
  for (int64_t b = (int64_t)blockIdx.x * kMemThreads + threadIdx.x; b < nblk; b += stride) {
    const uint4 v0 = ld_nc_v4(x + 2 * b), v1 = ld_nc_v4(x + 2 * b + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t s, lo, hi;
    encode_block(w, g, tab, s, lo, hi);
    codes[b] = make_uint2(lo, hi);
    job.scales[b] = (uint8_t)s;
  }
}

// ---------------------------------------------------------------------------
// FP4 encode in one pass over HBM (cooperative; used by the FP4 append)
// ---------------------------------------------------------------------------
// Every CTA (one per SM) parks its contiguous share of the 16-element blocks
// of both tensors in shared memory with one or two bulk copies, takes the
// partial magnitude maxima, meets the other CTAs at a grid barrier (bounded
// wait on an arrival counter in the cache's device workspace), derives the
// tensor scales from all partials, and encodes its blocks from shared memory.
// The input is read from HBM once.  The last CTA to leave resets the
// counters, so each launch starts from zero (the workspace is zero-filled at
// kvc_init and kvc_last_device_error clears the counters after an error).
constexpr int kFusedThreads = 1024;
constexpr int kFusedMaxBlocks = 6912;  // 216 KiB of parked blocks per CTA
constexpr int kCntArrive = KVC_WS_WORDS - 2;
constexpr int kCntDepart = KVC_WS_WORDS - 1;

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ int32_t ld_acquire_gpu_s32(const int32_t* a) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

__global__ void __launch_bounds__(kFusedThreads, 1)
    quant_fused_kernel(QuantJobs jobs, int njobs, int64_t nb, int32_t* __restrict__ dev_ws) {
  extern __shared__ uint4 park[];  // [blocks][2]
  __shared__ uint64_t bar;
  __shared__ uint32_t red[32];
  __shared__ float gsh[2];
  __shared__ ScaleTab tabs[2];
  __shared__ int32_t abort_flag;
  const int G = gridDim.x, g = blockIdx.x, tid = threadIdx.x;
  int32_t* part = dev_ws + 1;  // [2][G] partial maxima (bf16 magnitude bits)
  const int64_t T = nb * njobs;
  const int64_t b0 = (int64_t)g * T / G, b1 = (int64_t)(g + 1) * T / G;
  const int cnt = (int)(b1 - b0);
  const int j0 = (int)(b0 / nb);
  const int c0 = (int)min((int64_t)cnt, (int64_t)(j0 + 1) * nb - b0);  // blocks of job j0
  const QuantJob ja = j0 ? jobs.j[1] : jobs.j[0];
  const QuantJob jb = jobs.j[1];
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Watchdog wd{&abort_flag, dev_ws};
  if (tid == 0 && cnt > 0) {
    mbar_expect_tx(&bar, (uint32_t)cnt * 32u);
    bulk_g2s(park, static_cast<const uint8_t*>(ja.x) + (b0 - (int64_t)j0 * nb) * 32, (uint32_t)c0 * 32u, &bar);
    if (cnt > c0) bulk_g2s(park + 2 * c0, jb.x, (uint32_t)(cnt - c0) * 32u, &bar);
  }
  // block-uniform (a __syncthreads below depends on it)
  const bool landed = __syncthreads_and(cnt == 0 || mbar_wait(&bar, 0, wd)) != 0;
  // partial maxima of the (at most two) tensors this share touches
  uint32_t a0 = 0, a1 = 0;
  if (landed) {
    for (int i = tid; i < cnt; i += kFusedThreads) {
      const int f = (i >> 2) & 1;  // bank-group order, as in the encode loop
      const uint32_t m = absmax_bf16x8(park[2 * i + 1 - f], absmax_bf16x8(park[2 * i + f], 0u));
      if (i < c0) a0 = __vmaxu2(a0, m);
      else a1 = __vmaxu2(a1, m);
    }
  }
  const uint32_t m0 = block_max_u32(max(a0 & 0xFFFFu, a0 >> 16), red);
  const uint32_t m1 = block_max_u32(max(a1 & 0xFFFFu, a1 >> 16), red);
  if (tid == 0) {
    part[g] = (int32_t)(j0 == 0 ? m0 : 0u);
    part[G + g] = (int32_t)(j0 == 0 ? m1 : m0);
    __threadfence();
    atomicAdd(dev_ws + kCntArrive, 1);
    // grid barrier: every CTA of this cooperative launch is resident
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu_s32(dev_ws + kCntArrive) < G) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        abort_flag = 1;
        atomicCAS(dev_ws, DEVERR_NONE, DEVERR_TIMEOUT);
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (!abort_flag && landed) {
    // tensor scale of each tensor from all G partial maxima (warp j: tensor j)
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < njobs) {
      uint32_t m = 0;
      for (int i = lane; i < G; i += 32) m = max(m, (uint32_t)part[warp * G + i]);
      m = __reduce_max_sync(0xffffffffu, m);
      if (lane == 0) gsh[warp] = __fdiv_rn(__uint_as_float(m << 16), 2688.0f);
    }
    __syncthreads();
    if (g == 0 && tid < njobs) *(tid ? jobs.j[1].gscale : jobs.j[0].gscale) = gsh[tid];
    for (int j = 0; j < njobs; ++j) build_scale_tab(tabs[j], gsh[j], tid, kFusedThreads);
    __syncthreads();
    for (int i = tid; i < cnt; i += kFusedThreads) {
      const bool first = i < c0;
      const int j = first ? j0 : j0 + 1;
      const QuantJob& jo = first ? ja : jb;
      const int64_t lb = b0 + i - (int64_t)j * nb;  // block within its tensor
      // the two 16-byte halves are read in an order that keeps the 8 lanes of
      // a quarter-warp on 8 different bank groups
      const int f = (i >> 2) & 1;
      const uint4 va = park[2 * i + f], vb = park[2 * i + 1 - f];
      const uint4 v0 = f ? vb : va, v1 = f ? va : vb;
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t sc, lo, hi;
      encode_block(w, gsh[j], tabs[j], sc, lo, hi);
      reinterpret_cast<uint2*>(jo.codes)[lb] = make_uint2(lo, hi);
      jo.scales[lb] = (uint8_t)sc;
    }
  } else if (tid == 0 && cnt > 0 && !landed) {
    mbar_drain(&bar, 0);  // the bulk copies land before the CTA exits
  }
  // leave; the last CTA out resets the counters for the next launch
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(dev_ws + kCntDepart, 1) == G - 1) {
      atomicExch(dev_ws + kCntArrive, 0);
      atomicExch(dev_ws + kCntDepart, 0);
    }
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

cudaError_t launch_fill(void* const* dst, const size_t* bytes, const uint32_t* words, int n,
                        cudaStream_t st) {
  if (n < 1 || n > 4) return cudaErrorInvalidValue;
  FillJobs f{};
  size_t most = 0;
  for (int i = 0; i < n; ++i) {
    f.d[i] = static_cast<uint8_t*>(dst[i]);
    f.bytes[i] = bytes[i];
    f.word[i] = words[i];
    most = bytes[i] > most ? bytes[i] : most;
  }
  if (most == 0) return cudaSuccess;
  fill_kernel<<<dim3(mem_grid(most / 16 + 1), n), kMemThreads, 0, st>>>(f);
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

cudaError_t launch_quant_fp4_fused(const QuantJob* jobs, int njobs, int64_t n, int32_t* dev_ws,
                                   int nsm, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t nb = n >> 4;
  const int64_t T = nb * njobs;
  const int G = nsm;
  if (njobs < 1 || njobs > 2 || G < 1 || 1 + 2 * G >= kCntArrive) return cudaErrorNotSupported;
  const int64_t per = (T + G - 1) / G;
  if (per > kFusedMaxBlocks || T < G) return cudaErrorNotSupported;
  for (int i = 0; i < njobs; ++i)
    if ((reinterpret_cast<uintptr_t>(jobs[i].x) & 15u) || (reinterpret_cast<uintptr_t>(jobs[i].codes) & 7u))
      return cudaErrorNotSupported;
  QuantJobs qj{};
  for (int i = 0; i < njobs; ++i) qj.j[i] = jobs[i];
  const size_t smem = (size_t)per * 32;
  static bool smem_set[64] = {};
  cudaError_t e = set_smem_once(quant_fused_kernel, (size_t)kFusedMaxBlocks * 32, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(G, 1, 1);
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_fused_kernel, qj, njobs, nb, dev_ws);
}

}  // namespace kvc
