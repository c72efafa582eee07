// Launchers shared between the C-ABI layer (kvc_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kvc.h"

namespace kvc {

constexpr int kMaxSeg = 1 + KVC_MAX_WINDOW;

// A run of visible cache rows [row0, row0 + rows).
struct Seg {
  int32_t row0;
  int32_t rows;
};

// ---- bandwidth kernels (kernels_mem.cu) ----
// dst[i] = src[i] for two tensors of `bytes` bytes each (16-byte aligned, bytes % 16 == 0)
cudaError_t launch_copy2(void* dst0, const void* src0, void* dst1, const void* src1, size_t bytes,
                         cudaStream_t st);
// fill n <= 4 byte ranges (any alignment and length) with a repeated byte pattern
// given as a 32-bit word (byte i of a 4-byte-aligned group takes byte i of it), one launch
cudaError_t launch_fill(void* const* dst, const size_t* bytes, const uint32_t* words, int n,
                        cudaStream_t st);

// FP4 encode of up to kMaxQuantJobs tensors of n elements each (n % 16 == 0),
// each its own tensor.  ws: ws_words int32 words of scratch (per-CTA partial
// maxima, ws_words / njobs per tensor, at least one).
constexpr int kQuantPartials = 256;  // partial maxima of one tensor, at most
constexpr int kMaxQuantJobs = 2 * kMaxSeg;
struct QuantJob {
  const void* x;
  uint8_t* codes;
  uint8_t* scales;
  float* gscale;
};
// Two launches: per-CTA partial maxima, then the block encode as a programmatic
// dependent launch (its first loads overlap the end of the first pass).
cudaError_t launch_quant_fp4(const QuantJob* jobs, int njobs, int64_t n, int32_t* ws, int ws_words,
                             cudaStream_t st);

// ---- attention (kernels_attn.cu) ----
struct AttnLaunch {
  const void* q;        // bf16 [tq][H][D]
  void* out;            // bf16 [tq][H][D]
  int32_t tq, H, D;
  int32_t S;            // physical cache rows
  float scale_log2;     // softmax_scale * log2(e)
  int32_t nseg;
  Seg seg[kMaxSeg];
  int32_t* dev_err;
  // bf16 cache
  const void* k;
  const void* v;
  // FP4 cache
  int32_t fp4;
  const uint8_t* k_scale;
  const uint8_t* v_scale;
  const float* k_gscale;
  const float* v_gscale;
  int32_t chunk_tokens;  // rows per region (FP4: region of a row -> its tensor scale)
  // FP4 cache decoded beforehand: f16 [S][H][D] K and V (e2m1 * s, no tensor
  // scale) of every visible region, or null (decoded inside the kernel)
  const void* k16;
  const void* v16;
  // split-item workspace (null: whole items per CTA)
  void* ws;
  size_t ws_bytes;
};
cudaError_t launch_sinkwin_attn(const AttnLaunch& a, cudaStream_t st);
// bytes of the attention workspace for head dim D and `ctas` persistent CTAs
size_t attn_workspace_bytes(int D, int ctas);
// SMs of the current device (0 when there is none)
int attn_sm_count();

// ---- projection GEMMs + norm/RoPE (kernels_recache.cu) ----
struct RecacheLaunch {
  const void* hidden;  // bf16 [n*Tc][H*D]
  const void* w_kv;    // bf16 [H*D][2*H*D]
  const float* gamma;  // fp32 [H*D] or null
  float eps, theta;
  int32_t rows, H, D, Tc, tpf, grid_w;
  int32_t n;
  int64_t frame0[kMaxSeg];  // RoPE frame position of each chunk's first frame
  int32_t region[kMaxSeg];  // destination region of each chunk
  void* k;  // bf16 [regions * Tc][H][D]: the cache, or a staging buffer
  void* v;
  int32_t* dev_err;
};
cudaError_t launch_recache(const RecacheLaunch& r, cudaStream_t st);
// Q, K, V of one chunk: [Q|K|V] = hidden @ w_qkv, Q and K normed + rotated.
struct ProjectLaunch {
  const void* hidden;  // bf16 [Tc][H*D]
  const void* w_qkv;   // bf16 [H*D][3*H*D]
  const float* gamma_q;
  const float* gamma_k;
  float eps, theta;
  int32_t Tc, H, D, tpf, grid_w;
  int64_t frame0;
  float* stage_f32;  // [Tc][2*H*D] fp32 scratch
  void* q_out;       // bf16 [Tc][H*D]
  void* k_dst;       // bf16 [Tc][H*D]
  void* v_dst;       // bf16 [Tc][H*D]
  int32_t* dev_err;
};
cudaError_t launch_project_chunk(const ProjectLaunch& r, cudaStream_t st);
// H*D in {64, 128, 256, 512, 768, 1024, 1536, 2048, 3072} and D even, D/2 <= 128
bool recache_supported(int H, int D);

// Raise a kernel's dynamic shared-memory limit once per device (the setting
// is per function and device; repeating it on every launch costs host time).
// `done` is a per-kernel flag array owned by the caller.
template <typename K>
cudaError_t set_smem_once(K kern, size_t bytes, bool (&done)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// ---- W4A4 projection (FP4 x FP4 -> bf16) ----
struct GemmFp4Launch {
  const uint8_t* a_codes;   // [M][K/2]
  const uint8_t* a_scales;  // [M][K/16]
  const float* a_gscale;    // device [1]
  const uint8_t* b_codes;   // [N][K/2]
  const uint8_t* b_scales;  // [N][K/16]
  const float* b_gscale;    // device [1]
  int64_t M, N, K;          // N % 32 == 0, K % 256 == 0
  void* out;                // bf16 [M][N]
  int32_t* dev_err;         // may be null
  void* ws;                 // null: fused kernel; else gemm_fp4_ws_bytes(M, N, K) bytes
};
cudaError_t launch_gemm_fp4(const GemmFp4Launch& g, cudaStream_t st);
// FP4 -> f16 (e2m1 * e4m3 scale, exact; no tensor scale) of contiguous runs:
// codes [groups * 4] bytes, scales [groups / 2], out [groups * 8] f16; groups
// (of 8 elements) even, all pointers 16-byte aligned.
struct Fp4DecodeJob {
  const uint8_t* codes;
  const uint8_t* scales;
  void* out;
  int64_t groups;
  int32_t g_region;  // -1: no tensor scale; else the output is rounded to f16 after
                     // multiplying by gscale[g_region] / G (see below)
};
constexpr int kMaxDecodeJobs = 2 * (1 + KVC_MAX_WINDOW);
// gscale: device tensor scales (used by jobs with g_region >= 0); G is the
// power of two of the FP4 attention's V shift: from the largest of
// gscale[regions[0..nregions)], as the attention kernel computes it.
cudaError_t launch_fp4_to_f16(const Fp4DecodeJob* jobs, int njobs, cudaStream_t st,
                              const float* gscale = nullptr, const int32_t* regions = nullptr,
                              int nregions = 0);
size_t gemm_fp4_smem_bytes();
int64_t gemm_fp4_ws_bytes(int64_t M, int64_t N, int64_t K);

// ---- diagnostics ----
cudaError_t launch_watchdog_selftest(int32_t* dev_ws, int32_t limit_us, cudaStream_t st);

// driver entry point for tensor-map encoding (resolved once through the runtime)
bool encode_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                         uint32_t box1, uint32_t box2, bool swizzle128);
bool encode_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                         uint64_t stride1_bytes, uint32_t box0, uint32_t box1, bool swizzle128);
// the same with a swizzle of 0, 32, 64 or 128 bytes
bool encode_tmap_2d_bf16_sw(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                            uint64_t stride1_bytes, uint32_t box0, uint32_t box1, int swizzle_bytes);
// 2D tensor of bytes (d0 innermost), swizzle of 0, 32, 64 or 128 bytes; rows
// past d1 read as zero
bool encode_tmap_2d_u8(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                       uint64_t stride1_bytes, uint32_t box0, uint32_t box1, int swizzle_bytes);

}  // namespace kvc
