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
// the operands to f16 and multiplies them with the kind::f16 tcgen05 MMA, fp32
// accumulators in TMEM; the two tensor scales are applied once to the
// accumulator.  The only roundings are the fp32 accumulation and the final
// bf16 conversion.
//
// Shared-memory bandwidth is what limits a decode-in-the-loop GEMM: the MMA
// reads its shared-memory operands at a large fraction of it already.  So the
// decoded A tile goes to TMEM (tcgen05.st; the MMA takes A from TMEM) and
// only B's decoded tile is written to and read from shared memory.
//
// Warp roles (576 threads, one CTA per SM, persistent over 128 x 192 tiles):
//   warps 0-11  decode: raw FP4 stage (K = 256) -> four f16 stages (K = 64):
//               A rows into TMEM, B rows into 128-byte swizzled shared memory
//   warp 12     TMA: raw codes (128-byte swizzled) and scales of A and B
//   warp 13     MMA issue (one thread): 4 x (128 x 192 x 16) per f16 stage
//   warps 14-17 epilogue: TMEM -> x (g_a g_b) -> bf16 -> global
// TMEM: two 192-column accumulators (columns 0-383) and two A stages of 32
// columns (384-447).  The epilogue writes bf16 boxes of 32 x 32 through
// shared memory with bulk tensor stores.  Every wait is bounded (the device error word records a
// timeout).
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int GM = 128;   // rows of A per tile (TMEM lanes)
constexpr int GN = 192;   // rows of B (output columns) per tile
constexpr int GKR = 256;  // K elements per raw stage
constexpr int GKD = 64;   // K elements per decoded f16 stage (128 bytes a row)
constexpr int kRawStages = 3;
constexpr int kDecStages = 2;
constexpr int kDecodeWarps = 12;
constexpr int kTmaWarp = 12, kMmaWarp = 13;  // warps 14-17: epilogue
constexpr int kGThreads = 32 * 18;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = GN;             // accumulator b at columns b * GN
constexpr uint32_t kACol0 = 2 * GN;           // A stage d at columns kACol0 + 32 d
static_assert(kACol0 + kDecStages * 32 <= kTmemCols, "TMEM holds both accumulators and the A stages");
// Warp-tasks of one decoded stage: 32 rows x one half (32 elements) each.
// A: 4 row quarters x 2 halves = 8; B: GN / 32 x 2 = 12.  Decode warp w takes
// B task w, and warps 0-7 also A task w, which covers rows 32 (w % 4) .. : the
// TMEM lane quarter warp w may access.  (A's TMEM store costs less than B's
// shared-memory store, so no warp holds two B tasks.)
constexpr int kATasks = 8, kBTasks = 2 * GN / 32;
static_assert(kBTasks == kDecodeWarps && kATasks <= kDecodeWarps, "one B task per decode warp");
static_assert(GKR / GKD == 4, "a raw stage is four decoded stages");

struct Fp4GemmSmem {
  uint8_t a_codes[kRawStages][GM * GKR / 2];  // [row][128 B], 128-byte swizzled
  uint8_t b_codes[kRawStages][GN * GKR / 2];
  uint8_t a_sc[kRawStages][GM * GKR / 16];  // [row][16 B]
  uint8_t b_sc[kRawStages][GN * GKR / 16];
  uint8_t b_dec[kDecStages][GN * GKD * 2];  // f16 [row][64], 128-byte swizzled (MMA operand)
  // epilogue staging: per warp two 32 x 32 bf16 boxes, 64-byte swizzled rows
  uint32_t ostage[4][2][32][16];
  uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  uint64_t dec_full[kDecStages], dec_empty[kDecStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};
constexpr uint32_t kRawBytes = (GM + GN) * (GKR / 2 + GKR / 16);

struct Fp4GemmParams {
  int32_t M, N, ntn, ntiles, nks;  // rows, columns, column tiles, tiles, raw stages along K
  const float* a_g;
  const float* b_g;
  int32_t* dev_err;
};

// 32 elements (16 code bytes = two 16-element blocks, `scale_pair` their two
// E4M3 scales in its low 16 bits) -> 16 f16x2 words in element order
__device__ __forceinline__ void decode32(uint4 codes, uint32_t scale_pair, uint32_t (&o)[16]) {
  const uint32_t sp = e4m3x2_to_f16x2(scale_pair);
  const __half2 s2 = *reinterpret_cast<const __half2*>(&sp);
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const __half2 sc = wi < 2 ? __low2half2(s2) : __high2half2(s2);
    uint32_t h4[4];
    e2m1x8_to_f16x8(w[wi], h4);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 hv = __hmul2(*reinterpret_cast<const __half2*>(&h4[k]), sc);  // exact
      o[wi * 4 + k] = *reinterpret_cast<const uint32_t*>(&hv);
    }
  }
}

// One decode warp-task: which operand, its first row and its half.
struct DecTask {
  bool is_a;
  int row0;  // first of the 32 rows (within the operand's tile)
  int half;  // elements 32 half .. 32 half + 31 of each decoded stage
};
__device__ __forceinline__ DecTask a_task(int u) { return {true, 32 * (u % 4), u / 4}; }
__device__ __forceinline__ DecTask b_task(int v) { return {false, 32 * (v % (GN / 32)), v / (GN / 32)}; }

// Slot of 16-byte piece c (0..3) of staging row r: the layout of a 64-byte
// swizzled box; 8 lanes writing piece c of 8 consecutive rows hit 8 bank groups.
__device__ __forceinline__ int ostage_slot(int r, int c) { return c ^ ((r >> 1) & 3); }

// One warp's 32 accumulator rows of a 128 x GN tile -> x gs -> bf16, stored
// as 32 x 32 boxes through two staging buffers (`nst` counts this warp's boxes
// and picks the buffer).  Row quarters past M are skipped (partial ones are
// clipped by the store), and so are column chunks past N.
__device__ __forceinline__ void store_tile(const CUtensorMap* tmC, uint32_t (*stage)[32][16], uint32_t acc,
                                           int m0, int n0, int M, int N, float gs, int wq, int lane,
                                           int& nst) {
  const uint32_t trow = acc + ((uint32_t)(wq * 32) << 16);
  const int row0 = m0 + wq * 32;
  const bool live = row0 < M;
  const int nch = min(GN, N - n0) / 32;
  uint32_t x[32];
#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    tmem_ld32(trow + c * 32, x);  // warp-collective
    tmem_ld_wait();
    if (!live) continue;
    uint32_t (*stg)[16] = stage[nst & 1];
    if (lane == 0) bulk_wait_read<1>();  // this buffer's previous box has been read
    __syncwarp();
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint4*>(&stg[lane][4 * ostage_slot(lane, e)]) = make_uint4(
          pack_bf16x2(__uint_as_float(x[8 * e + 0]) * gs, __uint_as_float(x[8 * e + 1]) * gs),
          pack_bf16x2(__uint_as_float(x[8 * e + 2]) * gs, __uint_as_float(x[8 * e + 3]) * gs),
          pack_bf16x2(__uint_as_float(x[8 * e + 4]) * gs, __uint_as_float(x[8 * e + 5]) * gs),
          pack_bf16x2(__uint_as_float(x[8 * e + 6]) * gs, __uint_as_float(x[8 * e + 7]) * gs));
    fence_proxy_async_smem();  // the bulk copy reads what the generic stores wrote
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, &stg[0][0], n0 + c * 32, row0);
      bulk_commit();
    }
    ++nst;
  }
}

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmAc, const __grid_constant__ CUtensorMap tmAs,
                    const __grid_constant__ CUtensorMap tmBc, const __grid_constant__ CUtensorMap tmBs,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ Fp4GemmParams p) {
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
    // Lanes take 32 consecutive rows, so the swizzled 16-byte loads and
    // stores of a quarter warp hit 8 distinct bank groups.
    // tk[0] is B task `warp`; warps 0-7 also hold A task `warp` as tk[1]
    const int ntask = warp < kATasks ? 2 : 1;  // warp-uniform
    const DecTask tk[2] = {b_task(warp), a_task(warp < kATasks ? warp : 0)};
    int rs = 0, ds = 0;  // raw / decoded stages passed (ring positions)
    bool ok = true;
    for (int tile = cta; tile < p.ntiles && ok; tile += ncta) {
      for (int ks = 0; ks < p.nks && ok; ++ks, ++rs) {
        const int s = rs % kRawStages;
        if (!mbar_wait(&sm.raw_full[s], (rs / kRawStages) & 1, wd)) {
          ok = false;
          break;
        }
        // each task row's 16 scale bytes of this raw stage (one per 16 elements)
        uint4 sc[2];
        const uint8_t* cbase[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = tk[i].row0 + lane;
          sc[i] = make_uint4(0, 0, 0, 0);
          if (i < ntask)
            sc[i] = *reinterpret_cast<const uint4*>(tk[i].is_a ? &sm.a_sc[s][r * 16] : &sm.b_sc[s][r * 16]);
          cbase[i] = (tk[i].is_a ? sm.a_codes[s] : sm.b_codes[s]) + r * 128;
        }
        const int sw = lane & 7;  // (row & 7): the rows of a task start at multiples of 32
        // 16-byte chunk 2 j + half of the raw row: the next stage's chunk is
        // loaded before this stage's decode, so the load latency overlaps it
        uint4 nxt[2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
          nxt[i] = i < ntask ? *reinterpret_cast<const uint4*>(cbase[i] + ((tk[i].half ^ sw) << 4))
                             : make_uint4(0, 0, 0, 0);
#pragma unroll 1
        for (int j = 0; j < GKR / GKD; ++j, ++ds) {
          const int d = ds % kDecStages;
          uint4 codes[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            codes[i] = nxt[i];
            if (i < ntask && j + 1 < GKR / GKD)
              nxt[i] = *reinterpret_cast<const uint4*>(cbase[i] + (((2 * (j + 1) + tk[i].half) ^ sw) << 4));
          }
          if (ds >= kDecStages && !mbar_wait(&sm.dec_empty[d], ((ds / kDecStages) - 1) & 1, wd)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (i >= ntask) break;
            const uint32_t scw = j == 0 ? sc[i].x : j == 1 ? sc[i].y : j == 2 ? sc[i].z : sc[i].w;
            uint32_t o[16];
            decode32(codes[i], scw >> (16 * tk[i].half), o);
            if (tk[i].is_a) {
              // lane = tile row; columns 16 half .. of the stage's 32 (two f16 a column)
              tmem_st16(tmem + ((uint32_t)tk[i].row0 << 16) + kACol0 + 32 * d + 16 * tk[i].half, o);
            } else {
              uint8_t* dst = sm.b_dec[d] + (tk[i].row0 + lane) * 128;
#pragma unroll
              for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(dst + (((4 * tk[i].half + c) ^ sw) << 4)) =
                    make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            }
          }
          tmem_st_wait();            // the A words are in TMEM
          fence_proxy_async_smem();  // the B tile is read by the tensor cores
          tc_fence_before();
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
          // x coordinates in bytes: ks * 128 and ks * 16, multiples of 16;
          // rows past M or N read as zero
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
        const uint32_t acc = tmem + (uint32_t)buf * kAccCols;
        const int nsteps = p.nks * (GKR / GKD);
        for (int kd = 0; kd < nsteps; ++kd, ++ds) {
          const int d = ds % kDecStages;
          if (!mbar_wait(&sm.dec_full[d], (ds / kDecStages) & 1, wd)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_t = tmem + kACol0 + 32 * d;
#pragma unroll
          for (int kk = 0; kk < GKD / 16; ++kk) {
            const uint64_t bd = sdesc_sw128(smem_u32(sm.b_dec[d]) + kk * 32, 0, 1024);
            mma_bf16_ts(acc, a_t + kk * 8, bd, idesc, (kd > 0 || kk > 0) ? 1u : 0u);
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
    const float gs = __ldg(p.a_g) * __ldg(p.b_g);
    if (lane == 0) tma_prefetch_desc(&tmC);
    int jt = 0, nst = 0;
    for (int tile = cta; tile < p.ntiles; tile += ncta, ++jt) {
      const int buf = jt & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.acc_full[buf], (jt >> 1) & 1, wd))) break;
      tc_fence_after();
      store_tile(&tmC, sm.ostage[warp & 3], tmem + (uint32_t)buf * kAccCols, (tile / p.ntn) * GM,
                 (tile % p.ntn) * GN, p.M, p.N, gs, warp & 3, lane, nst);
      tc_fence_before();
      mbar_arrive(&sm.acc_empty[buf]);  // the MMA may reuse this accumulator
    }
    if (lane == 0) bulk_wait_all();  // every box has left shared memory and landed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Two-phase path (caller workspace): decode A and B once to f16, then a plain
// f16 GEMM fed by TMA.  The decode is done (M + N) K times instead of once per
// tile, which on this GPU is worth the round trip through L2.
// ---------------------------------------------------------------------------
constexpr int kFStages = 5;
constexpr int kFThreads = 32 * 6;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue

struct F16GemmSmem {
  uint8_t a[kFStages][GM * GKD * 2];  // f16 [128][64], 128-byte swizzled (TMA)
  uint8_t b[kFStages][GN * GKD * 2];  // f16 [192][64]
  uint32_t ostage[4][2][32][16];
  uint64_t full[kFStages], empty[kFStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};

__global__ void __launch_bounds__(kFThreads, 1)
    gemm_f16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ Fp4GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  F16GemmSmem& sm =
      *reinterpret_cast<F16GemmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const int nk = p.nks * (GKR / GKD);  // K / 64

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 128);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const Watchdog wd{&sm.abort_flag, p.dev_err};

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      // launched as a programmatic dependent of the decode pass: everything
      // above overlapped its tail; the f16 operands are complete from here on
      // (every other access of this kernel follows these loads)
      pdl_wait();
      int issued = 0;
      bool ok = true;
      for (int tile = cta; tile < p.ntiles && ok; tile += ncta) {
        const int m0 = (tile / p.ntn) * GM, n0 = (tile % p.ntn) * GN;
        for (int kb = 0; kb < nk; ++kb, ++issued) {
          const int s = issued % kFStages, u = issued / kFStages;
          if (issued >= kFStages && !mbar_wait(&sm.empty[s], (u - 1) & 1, wd)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.full[s], (GM + GN) * GKD * 2);
          tma_load_2d(sm.a[s], &tmA, &sm.full[s], kb * GKD, m0);  // rows past M or N read as zero
          tma_load_2d(sm.b[s], &tmB, &sm.full[s], kb * GKD, n0);
        }
      }
      if (sm.abort_flag) {  // every copy started here lands before the CTA exits
        for (int s = 0; s < kFStages; ++s) {
          const int cnt = issued > s ? (issued - s + kFStages - 1) / kFStages : 0;
          if (cnt) mbar_drain(&sm.full[s], (cnt - 1) & 1);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(GM, GN, false, false);
      int used = 0, jt = 0;
      bool ok = true;
      for (int tile = cta; tile < p.ntiles && ok; tile += ncta, ++jt) {
        const int buf = jt & 1;
        if (jt >= 2 && !mbar_wait(&sm.acc_empty[buf], ((jt >> 1) - 1) & 1, wd)) break;
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)buf * kAccCols;
        for (int kb = 0; kb < nk; ++kb, ++used) {
          const int s = used % kFStages;
          if (!mbar_wait(&sm.full[s], (used / kFStages) & 1, wd)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < GKD / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(smem_u32(sm.a[s]) + kk * 32, 0, 1024);
            const uint64_t bd = sdesc_sw128(smem_u32(sm.b[s]) + kk * 32, 0, 1024);
            mma_bf16_ss(acc, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&sm.empty[s]);  // frees the stage for the producer
        }
        if (ok) mma_commit(&sm.acc_full[buf]);
      }
      mma_commit(&sm.drain);  // every MMA issued above completes before TMEM is freed
      mbar_drain(&sm.drain, 0);
    }
  } else {
    const float gs = __ldg(p.a_g) * __ldg(p.b_g);
    if (lane == 0) tma_prefetch_desc(&tmC);
    int jt = 0, nst = 0;
    for (int tile = cta; tile < p.ntiles; tile += ncta, ++jt) {
      const int buf = jt & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.acc_full[buf], (jt >> 1) & 1, wd))) break;
      tc_fence_after();
      store_tile(&tmC, sm.ostage[warp & 3], tmem + (uint32_t)buf * kAccCols, (tile / p.ntn) * GM,
                 (tile % p.ntn) * GN, p.M, p.N, gs, warp & 3, lane, nst);
      tc_fence_before();
      mbar_arrive(&sm.acc_empty[buf]);
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t gemm_fp4_smem_bytes() { return sizeof(Fp4GemmSmem) + 1024; }

int64_t gemm_fp4_ws_bytes(int64_t M, int64_t N, int64_t K) { return (M + N) * K * 2; }

cudaError_t launch_gemm_fp4(const GemmFp4Launch& g, cudaStream_t st) {
  CUtensorMap tmC;
  if (!encode_tmap_2d_bf16_sw(&tmC, g.out, (uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.N * 2, 32, 32, 64))
    return cudaErrorInvalidValue;
  Fp4GemmParams p{};
  p.M = (int32_t)g.M;
  p.N = (int32_t)g.N;
  p.ntn = (int32_t)((g.N + GN - 1) / GN);
  const int64_t ntm = (g.M + GM - 1) / GM;
  p.ntiles = (int32_t)(ntm * p.ntn);
  p.nks = (int32_t)(g.K / GKR);
  p.a_g = g.a_gscale;
  p.b_g = g.b_gscale;
  p.dev_err = g.dev_err;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static int sm_count[64] = {};  // per device, looked up once
  if (!sm_count[dev] && cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  const int nsm = sm_count[dev];
  const int grid = (int)(p.ntiles < nsm ? p.ntiles : nsm);

  if (g.ws) {
    // two phases: FP4 -> f16 into the workspace ([M][K] then [N][K]), f16 GEMM.
    // The tensor maps are typed bf16: TMA moves 2-byte elements either way.
    __half* a16 = reinterpret_cast<__half*>(g.ws);
    __half* b16 = a16 + g.M * g.K;
    const Fp4DecodeJob jobs[2] = {{g.a_codes, g.a_scales, a16, g.M * g.K / 8, -1},
                                  {g.b_codes, g.b_scales, b16, g.N * g.K / 8, -1}};
    cudaError_t e = launch_fp4_to_f16(jobs, 2, st);
    if (e != cudaSuccess) return e;
    CUtensorMap tmA, tmB;
    if (!encode_tmap_2d_bf16_sw(&tmA, a16, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.K * 2, GKD, GM, 128) ||
        !encode_tmap_2d_bf16_sw(&tmB, b16, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.K * 2, GKD, GN, 128))
      return cudaErrorInvalidValue;
    const size_t smem = sizeof(F16GemmSmem) + 1024;
    static bool done16[64] = {};
    e = set_smem_once(gemm_f16_kernel, smem, done16);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_f16_kernel, tmA, tmB, tmC, p);
  }

  CUtensorMap tmAc, tmAs, tmBc, tmBs;
  const uint64_t kc = (uint64_t)g.K / 2, ksc = (uint64_t)g.K / 16;
  if (!encode_tmap_2d_u8(&tmAc, g.a_codes, kc, (uint64_t)g.M, kc, GKR / 2, GM, 128) ||
      !encode_tmap_2d_u8(&tmBc, g.b_codes, kc, (uint64_t)g.N, kc, GKR / 2, GN, 128) ||
      !encode_tmap_2d_u8(&tmAs, g.a_scales, ksc, (uint64_t)g.M, ksc, GKR / 16, GM, 0) ||
      !encode_tmap_2d_u8(&tmBs, g.b_scales, ksc, (uint64_t)g.N, ksc, GKR / 16, GN, 0))
    return cudaErrorInvalidValue;
  const size_t smem = gemm_fp4_smem_bytes();
  static bool smem_done[64] = {};
  cudaError_t e = set_smem_once(gemm_fp4_kernel, smem, smem_done);
  if (e != cudaSuccess) return e;
  gemm_fp4_kernel<<<grid, kGThreads, smem, st>>>(tmAc, tmAs, tmBc, tmBs, tmC, p);
  return cudaGetLastError();
}

}  // namespace kvc
