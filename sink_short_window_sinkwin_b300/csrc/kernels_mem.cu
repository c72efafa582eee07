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
constexpr int kFillThreads = 512;

// 128-bit read-only load that does not allocate in L1
__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// blockIdx.y picks the tensor; every thread moves up to kUnroll 16-byte vectors
// per trip with all loads issued before the stores.
__global__ void __launch_bounds__(kMemThreads) copy2_kernel(uint4* __restrict__ d0,
                                                            const uint4* __restrict__ s0,
                                                            uint4* __restrict__ d1,
                                                            const uint4* __restrict__ s1,
                                                            size_t n16) {
  const uint4* s = blockIdx.y ? s1 : s0;
  uint4* d = blockIdx.y ? d1 : d0;
  const size_t stride = (size_t)gridDim.x * kMemThreads;
  // bounds-predicated loads, so the ragged last trip also has all of its loads
  // in flight at once
  for (size_t i = (size_t)blockIdx.x * kMemThreads + threadIdx.x; i < n16; i += kUnroll * stride) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (i + u * stride < n16) r[u] = ld_nc_v4(s + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (i + u * stride < n16) d[i + u * stride] = r[u];
  }
}

// Up to four byte ranges, each filled with a repeated byte pattern (given as a
// 32-bit word).  The 16-byte-aligned bodies of the ranges form one index
// space of vectors (range r holds vectors [s[r], s[r+1])), so one grid-stride
// loop sized to a single wave covers all of them; the range of a vector is
// picked by comparisons and selects (the parameters stay in constant space).
// The at most 15 head and 15 tail bytes of range r are written by warp r of
// the first CTA.
struct FillJobs {
  uint4* body[4];
  uint8_t* head[4];  // [head, body) and [tail, end) are the unaligned bytes
  uint8_t* tail[4];
  uint8_t* end[4];
  uint64_t s[5];  // vector prefix sums of the bodies
  uint32_t word[4];
};
template <typename T>
__device__ __forceinline__ T pick4(int r, T a, T b, T c, T d) {
  return r == 0 ? a : r == 1 ? b : r == 2 ? c : d;
}
__global__ void __launch_bounds__(kFillThreads) fill_kernel(FillJobs f) {
  const uint64_t total = f.s[4];
  const uint64_t stride = (uint64_t)gridDim.x * kFillThreads;
  for (uint64_t i = (uint64_t)blockIdx.x * kFillThreads + threadIdx.x; i < total; i += stride) {
    const int r = (int)(i >= f.s[1]) + (int)(i >= f.s[2]) + (int)(i >= f.s[3]);
    uint4* d = pick4(r, f.body[0], f.body[1], f.body[2], f.body[3]);
    const uint32_t w = pick4(r, f.word[0], f.word[1], f.word[2], f.word[3]);
    d[i - pick4(r, f.s[0], f.s[1], f.s[2], f.s[3])] = make_uint4(w, w, w, w);
  }
  const int r = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && r < 4) {
    const uint32_t w = pick4(r, f.word[0], f.word[1], f.word[2], f.word[3]);
    uint8_t* h = pick4(r, f.head[0], f.head[1], f.head[2], f.head[3]) + lane;
    uint8_t* t = pick4(r, f.tail[0], f.tail[1], f.tail[2], f.tail[3]) + lane;
    if (h < reinterpret_cast<uint8_t*>(pick4(r, f.body[0], f.body[1], f.body[2], f.body[3])))
      *h = (uint8_t)(w >> (8 * (reinterpret_cast<uintptr_t>(h) & 3)));
    if (t < pick4(r, f.end[0], f.end[1], f.end[2], f.end[3]))
      *t = (uint8_t)(w >> (8 * (reinterpret_cast<uintptr_t>(t) & 3)));
  }
}

// CTAs per tensor of a copy: about kUnroll vectors per thread, and at most one
// wave of 8 CTAs per SM over all `ny` tensors
int mem_grid(size_t n16, int ny) {
  size_t want = (n16 + (size_t)kMemThreads * kUnroll - 1) / ((size_t)kMemThreads * kUnroll);
  const size_t wave = (size_t)attn_sm_count() * 8 / (size_t)ny;
  if (want > wave) want = wave;
  if (want < 1) want = 1;
  return (int)want;
}

// ---------------------------------------------------------------------------
// FP4 encode
// ---------------------------------------------------------------------------
struct QuantJobs {
  QuantJob j[kMaxQuantJobs];
};

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
    const float r = sg != 0.0f ? __frcp_rn(sg) : 0.0f;
    // no finite reciprocal (s * g below ~2^-128): the block is stored as zeros
    t.e[s] = r < 3.0e38f ? make_float2(sg, r) : make_float2(0.0f, 0.0f);
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

// Eight E2M1 codes (four RNE-satfinite pair conversions) packed into one word,
// element 0 in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8_rne_satfinite(float a0, float a1, float a2, float a3,
                                                         float a4, float a5, float a6, float a7) {
  uint32_t r;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7));
  return r;
}

// max(|a|, |b|) per bf16 lane (the sign bit of the result is the XOR of the
// operands' signs, which the callers mask off)
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16 magnitude bits of the largest |x| over a 16-element block (finite x)
__device__ __forceinline__ uint32_t block_amax_bits(const uint32_t (&w)[8]) {
  const uint32_t m = bf16x2_max_abs(bf16x2_max_abs(bf16x2_max_abs(w[0], w[1]), bf16x2_max_abs(w[2], w[3])),
                                    bf16x2_max_abs(bf16x2_max_abs(w[4], w[5]), bf16x2_max_abs(w[6], w[7]))) &
                     0x7FFF7FFFu;
  return max(m & 0xFFFFu, m >> 16);
}

// E4M3 code of fl32(a / g) (a >= 0 finite, g > 0), round to nearest even,
// saturating -- without a division on the common path.  q = fl32(a * ginv)
// (ginv = fl32(1 / g)) corrected by one FMA residual step is within an ulp or
// two of the correctly rounded quotient, so whenever the E4M3 rounding of
// q - 2 ulp and of q + 2 ulp agree (every case but quotients within a few ulps
// of a rounding midpoint between two E4M3 values), that code is the code of
// the correctly rounded quotient as well; otherwise the quotient is computed
// exactly.
__device__ __forceinline__ uint32_t e4m3_scale_code(float a, float g, float ginv) {
  if (!(ginv < 3.0e38f)) return e4m3_rne_satfinite(__fdiv_rn(a, g));  // g below 2^-127
  const float q0 = __fmul_rn(a, ginv);
  const float q = __fmaf_rn(__fmaf_rn(-q0, g, a), ginv, q0);
  const uint32_t qb = __float_as_uint(q);
  const float lo = qb >= 2u ? __uint_as_float(qb - 2u) : 0.0f;
  const float hi = __uint_as_float(qb + 2u);  // q < 2^127: no overflow into inf
  uint16_t pair;  // E4M3 codes of hi (high byte) and lo (low byte)
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi), "f"(lo));
  if ((pair >> 8) == (pair & 0xFFu)) return pair & 0xFFu;
  return e4m3_rne_satfinite(__fdiv_rn(a, g));  // near a rounding midpoint
}

// One 16-element block (8 words of bf16 pairs, block amax given as bf16
// magnitude bits) under tensor scale g: its E4M3 scale byte and 8 bytes of
// packed E2M1 codes, in the fixed fp32 order of the encode rule.
__device__ __forceinline__ void encode_block_amax(const uint32_t (&w)[8], uint32_t amax_bits, float g,
                                                  float ginv, const ScaleTab& tab, uint32_t& s,
                                                  uint32_t& lo, uint32_t& hi) {
  s = 0;
  lo = 0;
  hi = 0;
  if (g == 0.0f) return;
  s = e4m3_scale_code(div6_bf16(__uint_as_float(amax_bits << 16)), g, ginv);
  const float2 sgi = tab.e[s];  // {s * g, 1 / (s * g)}
  if (s == 0 || sgi.x == 0.0f) {
    s = 0;
    return;
  }
  const uint64_t inv2 = f32x2(sgi.y, sgi.y);
  // |x| * inv and x * inv round to the same magnitude; the sign rides along.
  // Both elements of a word are scaled by one packed (per-lane IEEE) multiply.
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float y[8];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      f32x2_split(fmul2(f32x2(bf16_lo(w[4 * h + k]), bf16_hi(w[4 * h + k])), inv2), y[2 * k], y[2 * k + 1]);
    (h ? hi : lo) = e2m1x8_rne_satfinite(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
  }
}

__device__ __forceinline__ void encode_block(const uint32_t (&w)[8], float g, float ginv,
                                             const ScaleTab& tab, uint32_t& s, uint32_t& lo, uint32_t& hi) {
  encode_block_amax(w, block_amax_bits(w), g, ginv, tab, s, lo, hi);
}

// ---------------------------------------------------------------------------
// FP4 encode in two passes; the second runs as a programmatic dependent launch
// ---------------------------------------------------------------------------
// The encode pass re-reads the input the amax pass just streamed; a K/V chunk
// (2 x 14.4 MB for the LongLive-1.3B layer shape) fits the 126 MB L2.
__device__ __forceinline__ uint32_t absmax_acc(uint32_t acc, uint4 v) {
  return bf16x2_max_abs(acc, bf16x2_max_abs(bf16x2_max_abs(v.x, v.y), bf16x2_max_abs(v.z, v.w)));
}

// Pass 1: CTA (x, j) takes a contiguous range of tensor j's 16-byte vectors and
// writes the range's magnitude maximum (bf16 bits) to ws[j * stride + x]
// (no atomics, nothing to zero).  Two CTAs per SM, six loads in flight per
// thread on every trip.
constexpr int kAmaxThreads = 1024;
constexpr int kAmaxUnroll = 6;
__global__ void __launch_bounds__(kAmaxThreads, 2) amax_kernel(const __grid_constant__ QuantJobs jobs,
                                                               int64_t n, int32_t* __restrict__ ws,
                                                               int stride) {
  pdl_launch_dependents();  // the encode pass may take the SM slots this grid frees
  __shared__ uint32_t red[32];
  // (a __grid_constant__ parameter is indexed in place, not copied)
  const uint4* x = reinterpret_cast<const uint4*>(jobs.j[blockIdx.y].x);
  const int64_t n8 = n >> 3, G = gridDim.x;
  const int64_t v1 = ((int64_t)blockIdx.x + 1) * n8 / G;
  uint32_t acc = 0;
  // every trip issues all of its (bounds-predicated) loads before using any,
  // the ragged last trip included
  for (int64_t i = (int64_t)blockIdx.x * n8 / G + threadIdx.x; i < v1; i += kAmaxUnroll * kAmaxThreads) {
    uint4 r[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u)
      r[u] = i + u * kAmaxThreads < v1 ? ld_nc_v4(x + i + u * kAmaxThreads) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) acc = absmax_acc(acc, r[u]);
  }
  acc &= 0x7FFF7FFFu;
  const uint32_t m = block_max_u32(max(acc & 0xFFFFu, acc >> 16), red);
  if (threadIdx.x == 0) ws[blockIdx.y * stride + blockIdx.x] = (int32_t)m;
}

// Pass 2: CTA (x, j) encodes a contiguous range of tensor j's 16-element
// blocks: blocks i and i + kEncThreads of the range per thread and trip, the
// next pair's loads in flight while the current pair is encoded (two register
// sets used in turn).  The first pair is read before waiting on the amax pass
// (it is input, not written by that pass); the tensor scale then comes from
// that pass's `parts` partial maxima.
constexpr int kEncThreads = 512;
struct BlockPair {
  uint4 v[4];
};
__device__ __forceinline__ void load_pair(const uint4* x, int i, int cnt, BlockPair& r) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int b = i + h * kEncThreads;
    if (b < cnt) {
      r.v[2 * h] = ld_nc_v4(x + 2 * b);
      r.v[2 * h + 1] = ld_nc_v4(x + 2 * b + 1);
    }
  }
}
__device__ __forceinline__ void encode_pair(const BlockPair& r, int i, int cnt, float g, float ginv,
                                            const ScaleTab& tab, uint2* codes, uint8_t* scales) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int b = i + h * kEncThreads;
    if (b < cnt) {
      const uint32_t w[8] = {r.v[2 * h].x,     r.v[2 * h].y,     r.v[2 * h].z,     r.v[2 * h].w,
                             r.v[2 * h + 1].x, r.v[2 * h + 1].y, r.v[2 * h + 1].z, r.v[2 * h + 1].w};
      uint32_t sc, lo, hi;
      encode_block(w, g, ginv, tab, sc, lo, hi);
      codes[b] = make_uint2(lo, hi);
      scales[b] = (uint8_t)sc;
    }
  }
}
__global__ void __launch_bounds__(kEncThreads, 2) quant_kernel(const __grid_constant__ QuantJobs jobs,
                                                               int64_t n, const int32_t* __restrict__ ws,
                                                               int stride, int parts) {
  __shared__ float gsh;
  __shared__ ScaleTab tab;
  const QuantJob& job = jobs.j[blockIdx.y];
  const int tid = threadIdx.x;
  const int64_t nb = n >> 4, G = gridDim.x;
  const int64_t b0 = (int64_t)blockIdx.x * nb / G;
  const int cnt = (int)(((int64_t)blockIdx.x + 1) * nb / G - b0);  // blocks of this CTA
  const uint4* x = reinterpret_cast<const uint4*>(job.x) + 2 * b0;
  uint2* codes = reinterpret_cast<uint2*>(job.codes) + b0;
  uint8_t* scales = job.scales + b0;
  BlockPair A, B;
  int i = tid;
  load_pair(x, i, cnt, A);
  pdl_wait();  // the amax pass's partial maxima are complete and visible
  if (tid < 32) {  // one warp, all of its loads in flight at once
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < kQuantPartials / 32; ++u) {
      const int k = tid + 32 * u;
      if (k < parts) m = max(m, (uint32_t)__ldcg(ws + blockIdx.y * stride + k));
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if (tid == 0) gsh = __fdiv_rn(__uint_as_float(m << 16), 2688.0f);
  }
  __syncthreads();
  const float g = gsh;
  const float ginv = g != 0.0f ? __frcp_rn(g) : 0.0f;
  if (blockIdx.x == 0 && tid == 0) *job.gscale = g;
  build_scale_tab(tab, g, tid, kEncThreads);
  __syncthreads();
  while (i < cnt) {
    load_pair(x, i + 2 * kEncThreads, cnt, B);
    encode_pair(A, i, cnt, g, ginv, tab, codes, scales);
    i += 2 * kEncThreads;
    if (i >= cnt) break;
    load_pair(x, i + 2 * kEncThreads, cnt, A);
    encode_pair(B, i, cnt, g, ginv, tab, codes, scales);
    i += 2 * kEncThreads;
  }
}

}  // namespace

cudaError_t launch_copy2(void* dst0, const void* src0, void* dst1, const void* src1, size_t bytes,
                         cudaStream_t st) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  dim3 grid(mem_grid(n16, dst1 ? 2 : 1), dst1 ? 2 : 1);
  copy2_kernel<<<grid, kMemThreads, 0, st>>>(
      static_cast<uint4*>(dst0), static_cast<const uint4*>(src0), static_cast<uint4*>(dst1),
      static_cast<const uint4*>(src1), n16);
  return cudaGetLastError();
}

cudaError_t launch_fill(void* const* dst, const size_t* bytes, const uint32_t* words, int n,
                        cudaStream_t st) {
  if (n < 1 || n > 4) return cudaErrorInvalidValue;
  size_t any = 0;
  for (int r = 0; r < n; ++r) any |= bytes[r];
  if (any == 0) return cudaSuccess;
  FillJobs f{};
  for (int r = 0; r < 4; ++r) {
    // unused ranges: empty, at the first range's start
    const uintptr_t p0 = reinterpret_cast<uintptr_t>(dst[r < n ? r : 0]);
    const uintptr_t p1 = p0 + (r < n ? bytes[r] : 0);
    uintptr_t a = (p0 + 15) & ~uintptr_t(15), e = p1 & ~uintptr_t(15);
    if (a > e) a = e = p1;  // shorter than one aligned vector: all head bytes
    f.head[r] = reinterpret_cast<uint8_t*>(p0);
    f.body[r] = reinterpret_cast<uint4*>(a);
    f.tail[r] = reinterpret_cast<uint8_t*>(e);
    f.end[r] = reinterpret_cast<uint8_t*>(p1);
    f.word[r] = r < n ? words[r] : 0u;
    f.s[r + 1] = f.s[r] + (e - a) / 16;
  }
  const uint64_t total = f.s[4];
  // a single wave: at most 4 CTAs of 512 threads per SM, about 8 vectors a thread
  uint64_t ctas = (total + (uint64_t)kFillThreads * 8 - 1) / ((uint64_t)kFillThreads * 8);
  const uint64_t wave = (uint64_t)attn_sm_count() * 4;
  if (ctas > wave) ctas = wave;
  if (ctas < 1) ctas = 1;
  fill_kernel<<<(unsigned)ctas, kFillThreads, 0, st>>>(f);
  return cudaGetLastError();
}

cudaError_t launch_quant_fp4(const QuantJob* jobs, int njobs, int64_t n, int32_t* ws, int ws_words,
                             cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (njobs < 1 || njobs > kMaxQuantJobs) return cudaErrorInvalidValue;
  const int stride = ws_words / njobs;  // partial-maximum words per tensor
  if (stride < 1) return cudaErrorInvalidValue;
  QuantJobs qj{};
  for (int i = 0; i < njobs; ++i) qj.j[i] = jobs[i];
  const int nsm = attn_sm_count();
  // pass 1: two 1024-thread CTAs per SM over all tensors
  int64_t parts = 2 * (int64_t)nsm / njobs;
  if (parts > kQuantPartials) parts = kQuantPartials;
  if (parts > stride) parts = stride;
  const int64_t n8 = n >> 3;
  if (parts > n8) parts = n8;
  if (parts < 1) parts = 1;
  amax_kernel<<<dim3((unsigned)parts, njobs), kAmaxThreads, 0, st>>>(qj, n, ws, stride);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // pass 2: two 512-thread CTAs per SM over all tensors, as a dependent launch
  int64_t ctas = 2 * (int64_t)nsm / njobs;
  const int64_t nb = n >> 4;
  if (ctas > (nb + kEncThreads - 1) / kEncThreads) ctas = (nb + kEncThreads - 1) / kEncThreads;
  if (ctas < 1) ctas = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)ctas, (unsigned)njobs, 1);
  cfg.blockDim = dim3(kEncThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_kernel, qj, n, static_cast<const int32_t*>(ws), stride, (int)parts);
}


}  // namespace kvc
