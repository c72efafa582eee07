// W4A4 projection: C = deq(A) deq(B)^T with both operands in the library's FP4
// format (E2M1 codes, one E4M3 scale per 16 elements along K, one fp32 tensor
// scale), the output bf16.
//
// LongLive 2.0 inference blog (blog.hotdry.top), "NVFP4 量化与 KV Cache 压缩的
// 工程实现": NVFP4 W4A4 inference keeps weights and activations in 4-bit
// floating point (45.7 FPS against 24.8 in bf16 on the blog's figures); the
// NVIDIA infrastructure blog (bittide page), §6, lists W4A4 execution among the
// LongLive 2.0 system's parts.  The pages give no kernel, only the format.
//
// Design.  Every E2M1 value times its E4M3 block scale has at most 6
// significant bits and lies in [2^-10, 2688], so it is exact in f16; every
// product of two such values is exact in fp32.  The kernel therefore decodes
// the operands into f16 shared-memory tiles and multiplies them with the
// kind::f16 tcgen05 MMA, fp32 accumulators in TMEM; the two tensor scales are
// applied once to the accumulator.  The only roundings are the fp32
// accumulation and the final bf16 conversion.
//
// Warp roles (448 threads, one CTA per SM, persistent over 128 x 256 tiles):
//   warps 0-7   decode: raw FP4 stage (K = 256) -> four f16 stages (K = 64)
//   warp 8      TMA: raw codes (128-byte swizzled) and scales of A and B
//   warp 9      MMA issue (one thread): 4 x (128 x 256 x 16) per f16 stage
//   warps 10-13 epilogue: TMEM -> x (g_a g_b) -> bf16 -> global
// Every wait is bounded (the device error word records a timeout).
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int GM = 128;   // rows of A per tile (TMEM lanes)
constexpr int GN = 256;   // rows of B (output columns) per tile
constexpr int GKR = 256;  // K elements per raw stage
constexpr int GKD = 64;   // K elements per decoded f16 stage (128 bytes a row)
constexpr int kRawStages = 2;
constexpr int kDecStages = 2;
constexpr int kDecodeWarps = 8;
constexpr int kTmaWarp = 8, kMmaWarp = 9;  // warps 10-13: epilogue
constexpr int kGThreads = 32 * 14;
constexpr uint32_t kTmemCols = 2 * GN;  // two accumulators
constexpr int kRows = GM + GN;          // operand rows decoded per stage
// (row, half of a decoded stage) tasks per decode thread
constexpr int kTasks = kRows * 2 / (kDecodeWarps * 32);
static_assert(kTasks * kDecodeWarps * 32 == kRows * 2, "decode tasks must divide evenly");
static_assert(GKR / GKD == 4, "a raw stage is four decoded stages");

struct Fp4GemmSmem {
  uint8_t a_codes[kRawStages][GM * GKR / 2];  // [row][128 B], 128-byte swizzled
  uint8_t b_codes[kRawStages][GN * GKR / 2];
  uint8_t a_sc[kRawStages][GM * GKR / 16];  // [row][16 B]
  uint8_t b_sc[kRawStages][GN * GKR / 16];
  uint8_t a_dec[kDecStages][GM * GKD * 2];  // f16 [row][64], 128-byte swizzled (MMA operand)
  uint8_t b_dec[kDecStages][GN * GKD * 2];
  uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  uint64_t dec_full[kDecStages], dec_empty[kDecStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};
constexpr uint32_t kRawBytes = (GM + GN) * (GKR / 2 + GKR / 16);

struct Fp4GemmParams {
  int32_t M, ntn, ntiles, nks;  // rows, column tiles, tiles, raw stages along K
  int64_t ldc;                  // output row stride (elements)
  __nv_bfloat16* c;
  const float* a_g;
  const float* b_g;
  int32_t* dev_err;
};

// Decode 32 elements (16 code bytes, two 16-element blocks) of operand row r
// into chunks 4 half .. 4 half + 3 of its 128-byte row in the f16 tile.
__device__ __forceinline__ void decode32(uint8_t* dec, int r, int half, uint4 codes,
                                         uint32_t scale_pair) {
  const uint32_t sp = e4m3x2_to_f16x2(scale_pair);
  const __half2 s2 = *reinterpret_cast<const __half2*>(&sp);
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const __half2 sc = wi < 2 ? __low2half2(s2) : __high2half2(s2);
    uint32_t h4[4];
    e2m1x8_to_f16x8(w[wi], h4);
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 hv = __hmul2(*reinterpret_cast<const __half2*>(&h4[k]), sc);  // exact
      o[k] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    const int ch = half * 4 + wi;
    *reinterpret_cast<uint4*>(dec + r * 128 + ((ch ^ (r & 7)) << 4)) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmAc, const __grid_constant__ CUtensorMap tmAs,
                    const __grid_constant__ CUtensorMap tmBc, const __grid_constant__ CUtensorMap tmBs,
                    const __grid_constant__ Fp4GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  Fp4GemmSmem& sm =
      *reinterpret_cast<Fp4GemmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, ncta = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(&sm.raw_full[s], 1);
      mbar_init(&sm.raw_empty[s], kDecodeWarps);
    }
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&sm.dec_full[s], kDecodeWarps);
      mbar_init(&sm.dec_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 128);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const Watchdog wd{&sm.abort_flag, p.dev_err};

  if (warp < kDecodeWarps) {
    // ------------------------------------------------------------ decode
    // Thread t owns tasks t + 256 i (i < 3): operand row id % 384 (A rows
    // 0..127, then B rows), half id / 384 of every decoded stage.  A warp's
    // lanes take 32 consecutive rows, so the swizzled loads and stores hit 8
    // distinct 16-byte bank groups per quarter warp.
    const int t = threadIdx.x;
    int row[kTasks], half[kTasks];
#pragma unroll
    for (int i = 0; i < kTasks; ++i) {
      const int id = t + i * kDecodeWarps * 32;
      row[i] = id % kRows;
      half[i] = id / kRows;
    }
    int rs = 0, ds = 0;  // raw / decoded stages passed (ring positions)
    bool ok = true;
    for (int tile = cta; tile < p.ntiles && ok; tile += ncta) {
      for (int ks = 0; ks < p.nks && ok; ++ks, ++rs) {
        const int s = rs % kRawStages;
        if (!mbar_wait(&sm.raw_full[s], (rs / kRawStages) & 1, wd)) {
          ok = false;
          break;
        }
        // the row's 16 scale bytes of this raw stage (one per 16 elements)
        uint4 sc[kTasks];
#pragma unroll
        for (int i = 0; i < kTasks; ++i) {
          const int r = row[i];
          sc[i] = r < GM ? *reinterpret_cast<const uint4*>(&sm.a_sc[s][r * 16])
                         : *reinterpret_cast<const uint4*>(&sm.b_sc[s][(r - GM) * 16]);
        }
#pragma unroll 1
        for (int j = 0; j < GKR / GKD; ++j, ++ds) {
          const int d = ds % kDecStages;
          if (ds >= kDecStages && !mbar_wait(&sm.dec_empty[d], ((ds / kDecStages) - 1) & 1, wd)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int i = 0; i < kTasks; ++i) {
            const int r = row[i];
            const int cidx = j * 2 + half[i];  // 16-byte chunk of the raw row
            const bool is_a = r < GM;
            const int rr = is_a ? r : r - GM;
            const uint8_t* src = is_a ? sm.a_codes[s] : sm.b_codes[s];
            const uint4 codes =
                *reinterpret_cast<const uint4*>(src + rr * 128 + ((cidx ^ (rr & 7)) << 4));
            const uint32_t sw = j == 0 ? sc[i].x : j == 1 ? sc[i].y : j == 2 ? sc[i].z : sc[i].w;
            decode32(is_a ? sm.a_dec[d] : sm.b_dec[d], rr, half[i], codes,
                     sw >> (16 * half[i]));
          }
          fence_proxy_async_smem();  // the f16 tile is read by the tensor cores
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.dec_full[d]);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.raw_empty[s]);  // the raw stage may be refilled
      }
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA
    if (lane == 0) {
      tma_prefetch_desc(&tmAc);
      tma_prefetch_desc(&tmAs);
      tma_prefetch_desc(&tmBc);
      tma_prefetch_desc(&tmBs);
      int issued = 0;
      bool ok = true;
      for (int tile = cta; tile < p.ntiles && ok; tile += ncta) {
        const int m0 = (tile / p.ntn) * GM, n0 = (tile % p.ntn) * GN;
        for (int ks = 0; ks < p.nks; ++ks, ++issued) {
          const int s = issued % kRawStages, u = issued / kRawStages;
          if (issued >= kRawStages && !mbar_wait(&sm.raw_empty[s], (u - 1) & 1, wd)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.raw_full[s], kRawBytes);
          // x coordinates in bytes: ks * 128 and ks * 16, multiples of 16
          tma_load_2d(sm.a_codes[s], &tmAc, &sm.raw_full[s], ks * (GKR / 2), m0);
          tma_load_2d(sm.b_codes[s], &tmBc, &sm.raw_full[s], ks * (GKR / 2), n0);
          tma_load_2d(sm.a_sc[s], &tmAs, &sm.raw_full[s], ks * (GKR / 16), m0);
          tma_load_2d(sm.b_sc[s], &tmBs, &sm.raw_full[s], ks * (GKR / 16), n0);
        }
      }
      if (sm.abort_flag) {  // every copy started here lands before the CTA exits
        for (int s = 0; s < kRawStages; ++s) {
          const int cnt = issued > s ? (issued - s + kRawStages - 1) / kRawStages : 0;
          if (cnt) mbar_drain(&sm.raw_full[s], (cnt - 1) & 1);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(GM, GN, false, false);
      int ds = 0, jt = 0;
      bool ok = true;
      for (int tile = cta; tile < p.ntiles && ok; tile += ncta, ++jt) {
        const int buf = jt & 1;
        if (jt >= 2 && !mbar_wait(&sm.acc_empty[buf], ((jt >> 1) - 1) & 1, wd)) break;
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(buf * GN);
        const int nsteps = p.nks * (GKR / GKD);
        for (int kd = 0; kd < nsteps; ++kd, ++ds) {
          const int d = ds % kDecStages;
          if (!mbar_wait(&sm.dec_full[d], (ds / kDecStages) & 1, wd)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < GKD / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(smem_u32(sm.a_dec[d]) + kk * 32, 0, 1024);
            const uint64_t bd = sdesc_sw128(smem_u32(sm.b_dec[d]) + kk * 32, 0, 1024);
            mma_bf16_ss(acc, ad, bd, idesc, (kd > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&sm.dec_empty[d]);  // the decoders may overwrite the stage
        }
        if (ok) mma_commit(&sm.acc_full[buf]);
      }
      mma_commit(&sm.drain);  // every MMA issued above completes before TMEM is freed
      mbar_drain(&sm.drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;  // TMEM lane quarter: tile rows 32 wq .. 32 wq + 31
    const float gs = __ldg(p.a_g) * __ldg(p.b_g);
    int jt = 0;
    for (int tile = cta; tile < p.ntiles; tile += ncta, ++jt) {
      const int buf = jt & 1;
      const int m0 = (tile / p.ntn) * GM, n0 = (tile % p.ntn) * GN;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.acc_full[buf], (jt >> 1) & 1, wd))) break;
      tc_fence_after();
      const uint32_t trow = tmem + (uint32_t)(buf * GN) + ((uint32_t)(wq * 32) << 16);
      const int grow = m0 + wq * 32 + lane;
      uint4* dst = reinterpret_cast<uint4*>(p.c + (int64_t)grow * p.ldc + n0);
      uint32_t x[32];
#pragma unroll 1
      for (int c = 0; c < GN / 32; ++c) {
        tmem_ld32(trow + c * 32, x);  // warp-collective; only the stores are predicated
        tmem_ld_wait();
        if (grow < p.M) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[c * 4 + e] = make_uint4(
                pack_bf16x2(__uint_as_float(x[8 * e + 0]) * gs, __uint_as_float(x[8 * e + 1]) * gs),
                pack_bf16x2(__uint_as_float(x[8 * e + 2]) * gs, __uint_as_float(x[8 * e + 3]) * gs),
                pack_bf16x2(__uint_as_float(x[8 * e + 4]) * gs, __uint_as_float(x[8 * e + 5]) * gs),
                pack_bf16x2(__uint_as_float(x[8 * e + 6]) * gs, __uint_as_float(x[8 * e + 7]) * gs));
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_empty[buf]);  // the MMA may reuse this accumulator
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t gemm_fp4_smem_bytes() { return sizeof(Fp4GemmSmem) + 1024; }

cudaError_t launch_gemm_fp4(const GemmFp4Launch& g, cudaStream_t st) {
  CUtensorMap tmAc, tmAs, tmBc, tmBs;
  const uint64_t kc = (uint64_t)g.K / 2, ksc = (uint64_t)g.K / 16;
  if (!encode_tmap_2d_u8(&tmAc, g.a_codes, kc, (uint64_t)g.M, kc, GKR / 2, GM, 128) ||
      !encode_tmap_2d_u8(&tmBc, g.b_codes, kc, (uint64_t)g.N, kc, GKR / 2, GN, 128) ||
      !encode_tmap_2d_u8(&tmAs, g.a_scales, ksc, (uint64_t)g.M, ksc, GKR / 16, GM, 0) ||
      !encode_tmap_2d_u8(&tmBs, g.b_scales, ksc, (uint64_t)g.N, ksc, GKR / 16, GN, 0))
    return cudaErrorInvalidValue;
  Fp4GemmParams p{};
  p.M = (int32_t)g.M;
  p.ntn = (int32_t)(g.N / GN);
  const int64_t ntm = (g.M + GM - 1) / GM;
  p.ntiles = (int32_t)(ntm * p.ntn);
  p.nks = (int32_t)(g.K / GKR);
  p.ldc = g.N;
  p.c = reinterpret_cast<__nv_bfloat16*>(g.out);
  p.a_g = g.a_gscale;
  p.b_g = g.b_gscale;
  p.dev_err = g.dev_err;

  const size_t smem = gemm_fp4_smem_bytes();
  static bool smem_done[64] = {};
  cudaError_t e = set_smem_once(gemm_fp4_kernel, smem, smem_done);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int grid = (int)(p.ntiles < nsm ? p.ntiles : nsm);
  gemm_fp4_kernel<<<grid, kGThreads, smem, st>>>(tmAc, tmAs, tmBc, tmBs, p);
  return cudaGetLastError();
}

}  // namespace kvc
