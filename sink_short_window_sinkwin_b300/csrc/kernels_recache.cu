// Projection GEMMs on tcgen05 with an RMSNorm + 3D RoPE pass: the KV recache at
// a prompt switch, and the per-chunk Q|K|V projection whose K and V go straight
// into the cache.
//
// LongLive summary page (yunpan.plus), 方法 §1 KV 重缓存: at the switch the cache
// is recomputed from the frames already generated paired with the new prompt;
// the recache kernels are the per-layer tail of that recompute (K/V projection,
// key norm, rotary positions, cache write).  The same page's 方法 (causal
// frame-level autoregression) and §3 (帧汇聚点: every layer's cache) describe
// the per-chunk projection whose keys and values join the cache.
//
// RMSNorm spans the whole H*D-wide row, which no single 128 x 256 output tile
// holds, and rounding to bf16 before the norm and again after it would round
// twice.  The recache at H*D = 512 .. 2048 in steps of 512 (D 64 or 128) is the
// fused kernel further down: a thread-block cluster holds a whole row in TMEM
// and exchanges the per-row sums of squares through distributed shared memory.
// Other shapes, and the chunk projection, store the rows to be normalised as
// fp32 ("parked") and a second launch normalises them:
//   recache into a bf16 cache (three stream-ordered launches):
//   1. K GEMM: the unnormalised fp32 K row of token `dest` is parked in the
//      cache's own K and V rows of that token (each row is H*D*2 bytes, so the
//      two together hold exactly H*D fp32 values: columns [0, HD/2) in the K row,
//      [HD/2, HD) in the V row);
//   2. norm + RoPE: one warp per token reads its fp32 row, takes the mean square,
//      applies gamma and the 3D rotation and writes the bf16 K row (one rounding);
//   3. V GEMM: bf16 V straight into the V rows (overwriting the parked halves).
//   chunk projection (two launches): one GEMM over all 3*H*D columns of
//   [Q | K | V] parks Q and K as fp32 in a caller staging buffer and writes V as
//   bf16 to its destination; one norm launch turns the parked Q and K into
//   their bf16 destinations.
// The GEMM: a CTA computes a 128 x BN tile (BN = 256 at H*D = 1536) with 64-wide
// K steps through a 4-stage TMA ring; one thread issues tcgen05.mma into a TMEM
// accumulator; four epilogue warps read it back with tcgen05.ld.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int RM = 128;         // rows per tile
constexpr int RK = 64;          // K per stage (one 128-byte swizzle row of bf16)
constexpr int kRThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kStages = 4;

// Output row gr (of `rows`) is destination row region[gr / Tc] * Tc + gr % Tc.
// Output column j (of this launch's ncol * BN) goes to
//   j <  n_f32: fp32, f32a + d * ld_f32 + j              (j <  f32_split)
//                     f32b + d * ld_f32 + j - f32_split  (j >= f32_split)
//   j >= n_f32: bf16, bf + d * ld_bf + j - n_f32
// (n_f32 and f32_split are multiples of BN, so each tile has one kind.)
struct GemmParams {
  int32_t rows, HD, Tc;  // HD: contraction length (the model width H*D)
  int32_t col0;          // first column of the weight this launch computes
  int32_t ncol;          // column tiles of this launch
  int32_t ntiles;        // row tiles x column tiles
  int32_t region[kMaxSeg];
  int32_t n_f32, f32_split;
  int64_t ld_f32, ld_bf;
  float* f32a;
  float* f32b;
  __nv_bfloat16* bf;
  int32_t* dev_err;
};

// Slot of 16-byte piece c of staged row r: c ^ f(r) with f(r) = 4 (r & 1) +
// (r >> 1) % 4, a permutation of 0..7 over any 8 consecutive rows, and with bit
// 2 different for the two rows of an even/odd pair.  So 8 lanes writing piece c
// of 8 consecutive rows, 8 lanes reading pieces 0..7 of one row, and 4 + 4 lanes
// reading pieces 0..3 of rows 2i and 2i+1 each touch 8 different bank groups.
__device__ __forceinline__ int stage_slot(int r, int c) { return c ^ (((r & 1) << 2) | ((r >> 1) & 3)); }

template <int BN>
struct __align__(1024) GemmSmem {
  __nv_bfloat16 a[kStages][RM * RK];
  __nv_bfloat16 b[kStages][BN / 64][RK * 64];
  uint64_t bar_full[kStages], bar_empty[kStages];
  uint64_t bar_acc_full[2], bar_acc_empty[2];  // two TMEM accumulators
  uint64_t bar_drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  // epilogue staging: per epilogue warp 32 rows x 32 words, 16-byte pieces
  // placed by stage_slot() so that the row-wise writes and the transposed reads
  // are both free of bank conflicts
  uint32_t stage[4][32][32];
};

// Persistent: one CTA per SM.  Tiles are row-major over [row tile][column
// tile], CTA c takes tiles c, c + G, ... (so concurrent CTAs share hidden rows
// and weight columns through L2).  Every CTA loads its own A and B tiles into
// its own shared memory.  Row tiles past the last row load as TMA zero fill and
// store nothing.  The accumulator alternates between two TMEM buffers, so the
// epilogue of one tile overlaps the MMAs of the next.
// Store one warp's 32 rows x BN columns of an accumulator tile (TMEM load of
// the first 32-column chunk already issued into x).  Each chunk goes through
// the warp's staging rows (lane = row) and back out transposed: in store step
// k, lane l writes one 16-byte piece of row k * (32 / pieces) + l / pieces, so
// each store instruction covers whole 128-byte (fp32) or 64-byte (bf16) row
// segments instead of 16 bytes of 32 different rows.
template <int BN, bool kF32>
__device__ __forceinline__ void store_tile(const GemmParams& p, uint32_t (*stg)[32], uint32_t trow,
                                           uint32_t (&x)[32], int row0, int nloc, int64_t my_dest,
                                           int lane) {
#pragma unroll 1
  for (int jj = 0; jj < BN / 32; ++jj) {
    tmem_ld_wait();
    const int col = nloc + jj * 32;  // output column of this launch, a multiple of 32
    __syncwarp();                    // the previous chunk's transposed reads are done
    if constexpr (kF32) {
      // fp32: 32 words per row
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<uint4*>(&stg[lane][4 * stage_slot(lane, e)]) =
            make_uint4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
    } else {
      // bf16: 16 words per row
#pragma unroll
      for (int e = 0; e < 4; ++e)
        *reinterpret_cast<uint4*>(&stg[lane][4 * stage_slot(lane, e)]) =
            make_uint4(pack_bf16x2(__uint_as_float(x[8 * e + 0]), __uint_as_float(x[8 * e + 1])),
                       pack_bf16x2(__uint_as_float(x[8 * e + 2]), __uint_as_float(x[8 * e + 3])),
                       pack_bf16x2(__uint_as_float(x[8 * e + 4]), __uint_as_float(x[8 * e + 5])),
                       pack_bf16x2(__uint_as_float(x[8 * e + 6]), __uint_as_float(x[8 * e + 7])));
    }
    __syncwarp();
    if (jj + 1 < BN / 32) tmem_ld32(trow + (jj + 1) * 32, x);  // x is free again
    constexpr int kChunksPerRow = kF32 ? 8 : 4;  // 16-byte pieces of a row's 32 values
    constexpr int kRowsPerStep = 32 / kChunksPerRow;
    // the chunk's destination base (the row offset is added per row)
    uint4* base;
    int64_t ld;
    if constexpr (kF32) {
      const bool lo = col < p.f32_split;
      base = reinterpret_cast<uint4*>((lo ? p.f32a + col : p.f32b + (col - p.f32_split)));
      ld = p.ld_f32 / 4;  // in uint4
    } else {
      base = reinterpret_cast<uint4*>(p.bf + (col - p.n_f32));
      ld = p.ld_bf / 8;
    }
#pragma unroll
    for (int k = 0; k < 32 / kRowsPerStep; ++k) {
      const int rl = k * kRowsPerStep + lane / kChunksPerRow;  // row within the warp's 32
      const int piece = lane % kChunksPerRow;
      const int64_t dst = __shfl_sync(0xffffffffu, my_dest, rl);
      if (row0 + rl >= p.rows) continue;
      base[dst * ld + piece] = *reinterpret_cast<const uint4*>(&stg[rl][4 * stage_slot(rl, piece)]);
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(kRThreads, 1)
    recache_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ GemmParams p) {
  using Smem = GemmSmem<BN>;
  // two accumulators of BN columns; TMEM is allocated in powers of two >= 32
  constexpr uint32_t kCols = 2 * BN <= 32 ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.HD / RK;
  const int cid = blockIdx.x, ncl = gridDim.x;
  // row tile and first column of tile t
  auto tile_m0 = [&](int t) { return (t / p.ncol) * RM; };
  auto tile_n0 = [&](int t) { return (t % p.ncol) * BN; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.bar_full[s], 1);
      mbar_init(&sm.bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.bar_acc_full[b], 1);
      mbar_init(&sm.bar_acc_empty[b], 128);
    }
    mbar_init(&sm.bar_drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kCols);
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
      int issued = 0;  // K-steps loaded by this CTA (ring position)
      bool ok = true;
      for (int t = cid; t < p.ntiles && ok; t += ncl) {
        const int m0 = tile_m0(t), nloc = tile_n0(t);
        for (int kb = 0; kb < nk; ++kb, ++issued) {
          const int s = issued % kStages, u = issued / kStages;
          if (issued >= kStages && !mbar_wait(&sm.bar_empty[s], (u - 1) & 1, wd)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.bar_full[s], RM * RK * 2 + RK * BN * 2);
          tma_load_2d(&sm.a[s][0], &tmA, &sm.bar_full[s], kb * RK, m0);
#pragma unroll
          for (int nb = 0; nb < BN / 64; ++nb)
            tma_load_2d(&sm.b[s][nb][0], &tmB, &sm.bar_full[s], p.col0 + nloc + nb * 64, kb * RK);
        }
      }
      if (sm.abort_flag) {  // every copy this thread started lands before the CTA exits
        for (int s = 0; s < kStages; ++s) {
          const int cnt = issued > s ? (issued - s + kStages - 1) / kStages : 0;
          if (cnt) mbar_drain(&sm.bar_full[s], (cnt - 1) & 1);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(RM, BN, false, true);
      int used = 0;  // K-steps consumed (ring position)
      int j = 0;     // tiles of this CTA
      bool ok = true;
      for (int t = cid; t < p.ntiles && ok; t += ncl, ++j) {
        const int buf = j & 1;
        if (j >= 2 && !mbar_wait(&sm.bar_acc_empty[buf], ((j >> 1) - 1) & 1, wd)) break;
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(buf * BN);
        for (int kb = 0; kb < nk; ++kb, ++used) {
          const int s = used % kStages, u = used / kStages;
          if (!mbar_wait(&sm.bar_full[s], u & 1, wd)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < RK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(smem_u32(&sm.a[s][0]) + kk * 32, 0, 1024);
            const uint64_t bd = sdesc_sw128(smem_u32(&sm.b[s][0][0]) + kk * 2048, RK * 128, 1024);
            mma_bf16_ss(acc, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&sm.bar_empty[s]);  // frees the stage for the producer
        }
        if (ok) mma_commit(&sm.bar_acc_full[buf]);
      }
      mma_commit(&sm.bar_drain);  // every MMA issued above completes before TMEM is freed
      mbar_drain(&sm.bar_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;  // TMEM lane quarter: rows 32 wq .. 32 wq + 31 of the tile
    int j = 0;
    for (int t = cid; t < p.ntiles; t += ncl, ++j) {
      const int buf = j & 1;
      const int m0 = tile_m0(t), nloc = tile_n0(t);
      const uint32_t trow = tmem + (uint32_t)(buf * BN) + ((uint32_t)(wq * 32) << 16);
      // tcgen05.ld is warp-collective (.sync.aligned): the whole warp loads, and
      // only the stores are predicated on the row being real (the last row tile
      // can end inside a warp)
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.bar_acc_full[buf], (j >> 1) & 1, wd))) break;
      tc_fence_after();
      uint32_t (*stg)[32] = sm.stage[wq];
      // destination row of this lane's tile row (lane = row within the warp's
      // 32); store steps fetch the row they write from its lane
      int64_t my_dest = 0;
      {
        const int gr = m0 + wq * 32 + lane;
        if (gr < p.rows) {
          const int ci = gr / p.Tc;
          my_dest = (int64_t)p.region[ci] * p.Tc + (gr - ci * p.Tc);
        }
      }
      // The TMEM load of chunk jj + 1 is in flight while chunk jj is stored.
      uint32_t x[32];
      tmem_ld32(trow, x);
      if (nloc < p.n_f32)
        store_tile<BN, true>(p, stg, trow, x, m0 + wq * 32, nloc, my_dest, lane);
      else
        store_tile<BN, false>(p, stg, trow, x, m0 + wq * 32, nloc, my_dest, lane);
      tc_fence_before();
      mbar_arrive(&sm.bar_acc_empty[buf]);  // the MMA may reuse this accumulator
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ---------------------------------------------------------------------------
// norm + 3D RoPE: one warp per token row
// ---------------------------------------------------------------------------
// Row gr (of `rows`) of a job lives at destination row d = region[gr / Tc] * Tc
// + gr % Tc; its fp32 source is srca + d * ld_src (floats [0, src_split)) and
// srcb + d * ld_src (the rest), its bf16 output dst + d * ld_dst.  The output
// may overwrite the source (the parked recache rows): every lane reads its
// whole share of the row before any lane writes.
struct NormJob {
  const float* srca;
  const float* srcb;
  int64_t ld_src;  // floats
  int32_t src_split;
  __nv_bfloat16* dst;
  int64_t ld_dst;  // bf16 elements
  const float* gamma;
};
struct NormParams {
  int32_t rows, D, Tc, tpf, grid_w;
  int32_t pf, ph;  // RoPE pairs of the frame and row bands (column band = rest)
  float eps;
  int64_t frame0[kMaxSeg];  // frame position of the first frame of each chunk
  int32_t region[kMaxSeg];
  float omega[128];  // per rotation pair of a head: theta^(-2j/b) of its band
  NormJob job[2];    // blockIdx.y selects the job
};

constexpr int kNormWarps = 8;

// Lane l owns fp32 columns 4*(l + 32*i) .. +3, i < HD/128: 16-byte coalesced
// loads, the row's mean square by a warp reduction, then two rotation pairs per
// float4.
template <int HD>
__global__ void __launch_bounds__(kNormWarps * 32) recache_norm_rope_kernel(const __grid_constant__ NormParams p) {
  constexpr int NV = (HD + 127) / 128;  // float4 per lane (the last one may be partial)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grow = blockIdx.x * kNormWarps + warp;
  if (grow >= p.rows) return;
  // select, not index: a dynamic index would copy the parameter array to local memory
  const NormJob& jb = blockIdx.y ? p.job[1] : p.job[0];
  const int ci = grow / p.Tc;
  const int t = grow - ci * p.Tc;
  const int64_t dest = (int64_t)p.region[ci] * p.Tc + t;
  const float4* arow = reinterpret_cast<const float4*>(jb.srca + dest * jb.ld_src);
  const float4* brow = reinterpret_cast<const float4*>(jb.srcb + dest * jb.ld_src);
  const int split4 = jb.src_split / 4;
  float4 x[NV];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c4 = lane + 32 * i;  // float4 index in the fp32 row
    x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c4 < HD / 4) x[i] = c4 < split4 ? arow[c4] : brow[c4 - split4];
    ss = fmaf(x[i].x, x[i].x, ss);
    ss = fmaf(x[i].y, x[i].y, ss);
    ss = fmaf(x[i].z, x[i].z, ss);
    ss = fmaf(x[i].w, x[i].w, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float rstd = 1.0f / sqrtf(ss / (float)HD + p.eps);
  const int64_t fr = p.frame0[ci] + t / p.tpf;
  const int pp = t % p.tpf;
  const float pos_f = (float)fr, pos_h = (float)(pp / p.grid_w), pos_w = (float)(pp % p.grid_w);
  // the output may overwrite the source: every lane's reads of it come first
  __syncwarp();
  uint2* out = reinterpret_cast<uint2*>(jb.dst + dest * jb.ld_dst);
  // the two rotation pairs of a float4; when D divides 128 they are the same
  // pairs in every head, so their angles are evaluated once per row
  int pr_cached = -1;
  float cs[2] = {1.0f, 1.0f}, sn[2] = {0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c4 = lane + 32 * i;
    if (c4 >= HD / 4) break;
    const int col = 4 * c4;
    const int pr0 = (col % p.D) >> 1;  // pairs pr0, pr0 + 1 (col is a multiple of 4)
    if (pr0 != pr_cached) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int pr = pr0 + e;
        const float pos = pr < p.pf ? pos_f : (pr < p.pf + p.ph ? pos_h : pos_w);
        sincosf(pos * p.omega[pr], &sn[e], &cs[e]);
      }
      pr_cached = pr0;
    }
    const float v4[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
    const float4 g4 = jb.gamma ? __ldg(reinterpret_cast<const float4*>(jb.gamma) + c4) : make_float4(1.f, 1.f, 1.f, 1.f);
    const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
    uint32_t o[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float y0 = v4[2 * e] * rstd * gv[2 * e];
      const float y1 = v4[2 * e + 1] * rstd * gv[2 * e + 1];
      o[e] = pack_bf16x2(y0 * cs[e] - y1 * sn[e], y0 * sn[e] + y1 * cs[e]);
    }
    out[c4] = make_uint2(o[0], o[1]);
  }
}

// ---------------------------------------------------------------------------
// Fused recache: the K and V projections in one launch, RMSNorm + 3D RoPE in
// the K epilogue, nothing parked
// ---------------------------------------------------------------------------
// A cluster of HD / 512 CTAs owns a 128-row output tile: CTA r of the cluster
// computes columns [512 r, 512 r + 512) of it in a 128 x 512 fp32 TMEM
// accumulator (the whole TMEM; two N = 256 MMAs per 16-wide K step).  Work
// items are (row tile, K or V): item i is row tile i / 2, K for even i, and the
// clusters take items in turn, so the K and V items of a row tile run on
// neighbouring clusters at about the same time and share the hidden rows
// through L2.  The SMs that no cluster fits on run a second, cluster-free
// launch of the same kernel that takes the V items of the last row tiles
// (FusedParams::vonly).  K item epilogue: every thread sums the squares of its row over
// its 256 columns and stores that partial into every CTA of the cluster (its
// own included) before a release-arrive on the receiver's exchange barrier;
// with all 2 * HD / 512 partials of its rows in hand (summed in slot order, so
// every CTA of the cluster derives the same scale) a CTA applies
// x * rstd * gamma and the rotation and writes bf16 K, one rounding.  V items
// store bf16 directly.  DRAM sees the hidden rows, the weights and the bf16 K
// and V rows once each.
constexpr int FW = 512;           // output columns per CTA
constexpr int kFASlots = 3;       // A ring: 128 x 64 hidden tile per K step (16 KB)
constexpr int kFBSlots = 4;       // B ring: 64 x 256 weight tile per K step and half (32 KB)
constexpr int kFEpiWarps = 8;     // two per TMEM lane quarter, one per column half
// warp 0 TMA, warp 1 MMA, warps 2-3 idle (warpgroup 0), warps 4-11 epilogue
constexpr int kFThreads = 128 + 32 * kFEpiWarps;
// Register split (setmaxnreg, per thread): the block launches with
// kFLaunch registers a thread (the launch-bounds maximum, which ptxas takes
// when setmaxnreg is present; the launcher checks it); warpgroup 0 lowers to
// kFCtl, the two epilogue warpgroups raise to kFEpi.  The new counts add up to
// exactly the launch's registers (a larger sum would wait forever).
constexpr int kFLaunch = 168, kFCtl = 72, kFEpi = 216;
static_assert(4 * kFCtl + kFEpiWarps * kFEpi == (kFThreads / 32) * kFLaunch, "register split must match the launch");
static_assert(65536 / kFThreads / 8 * 8 == kFLaunch, "launch registers a thread");
static_assert(kFCtl % 8 == 0 && kFEpi % 8 == 0 && kFCtl >= 24 && kFCtl < kFLaunch && kFEpi > kFLaunch &&
                  kFEpi <= 256,
              "setmaxnreg takes multiples of 8 in [24, 256]; .dec only lowers, .inc only raises");
constexpr int kFMaxCluster = 4;   // H*D up to 2048
constexpr int kFhMax = 64;        // frame + row band pairs held in a warp's rotation table
constexpr int kTwMax = 1536;      // grid_w x column band pairs held in the column table

struct FusedParams {
  int32_t rows, HD, Tc, D, tpf, grid_w, pf, ph;
  // Work items.  Cluster launch (vonly == 0): K and V of row tiles
  // [0, rt_split) alternate (item 2 t is K, 2 t + 1 is V of row tile t), then
  // K alone of row tiles [rt_split, row tiles).  Cluster-free launch
  // (vonly == 1, on the SMs no cluster fits): V of row tiles [rt_split, row
  // tiles), one 512-column block per item.
  int32_t nitems, rt_split, vonly;
  float eps;
  int32_t region[kMaxSeg];
  int64_t frame0[kMaxSeg];
  float omega[128];
  const float* gamma;  // [HD] or null (1)
  __nv_bfloat16* k;    // destination rows: region[gr / Tc] * Tc + gr % Tc, stride HD
  __nv_bfloat16* v;
  int32_t* dev_err;
  int32_t w_tab;    // column-band rotations from the per-launch table (else sincosf per row)
  int32_t tma_out;  // output through bulk tensor stores of 8-row boxes (Tc % 8 == 0)
};

struct __align__(1024) FusedSmem {
  __nv_bfloat16 a[kFASlots][RM * RK];
  __nv_bfloat16 b[kFBSlots][4][RK * 64];
  uint32_t stage[kFEpiWarps][32][16];   // bf16 staging: 32 rows x 32 values per warp
  float exch[2][2 * kFMaxCluster][RM];  // [buffer][sender slot][row] partial sums of squares
  float gam[FW];
  float om[128];
  float2 tfh[kFEpiWarps][2][kFhMax];  // per warp: {cos, sin} of the frame and row bands for two positions
  float2 tw[kTwMax];                  // {cos, sin} of the column band: [w][pair]
  uint64_t a_full[kFASlots], a_empty[kFASlots], b_full[kFBSlots], b_empty[kFBSlots];
  uint64_t acc_full, acc_empty, bar_exch[2], bar_drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};

struct FItem {
  int m0;      // first row of the tile
  bool is_k;   // K (normed, rotated) or V
  int cb;      // 512-column block of the projection this CTA computes
};
__device__ __forceinline__ FItem fused_item(const FusedParams& p, int it, int rank) {
  if (p.vonly) {
    const int ncb = p.HD / FW;
    return FItem{(p.rt_split + it / ncb) * RM, false, it % ncb};
  }
  if (it < 2 * p.rt_split) return FItem{(it >> 1) * RM, (it & 1) == 0, rank};
  return FItem{(p.rt_split + (it - 2 * p.rt_split)) * RM, true, rank};
}

// Slot of 16-byte piece c (0..3) of bf16 staging row r (16 words a row).  Writes
// (8 lanes = 8 consecutive rows, one piece each) and transposed reads (8 lanes =
// pieces 0..3 of two rows) each touch 8 different bank groups.
__device__ __forceinline__ int stage16_slot(int r, int c) { return c ^ ((r >> 1) & 3); }

// One warp's 32 rows x 32 bf16 values (w: this lane's row, 16 packed words) to
// base[dest * ld + piece], through the staging rows: each store instruction
// writes 8 whole 64-byte row segments.
__device__ __forceinline__ void stage_store16(uint32_t (*stg)[16], const uint32_t (&w)[16], uint4* base,
                                              int64_t ld, int64_t my_dest, int row0, int rows, int lane) {
  __syncwarp();  // the previous chunk's transposed reads are done
#pragma unroll
  for (int e = 0; e < 4; ++e)
    *reinterpret_cast<uint4*>(&stg[lane][4 * stage16_slot(lane, e)]) =
        make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rl = 8 * k + (lane >> 2), piece = lane & 3;
    const int64_t dst = __shfl_sync(0xffffffffu, my_dest, rl);
    if (row0 + rl < rows) base[dst * ld + piece] = *reinterpret_cast<const uint4*>(&stg[rl][4 * stage16_slot(rl, piece)]);
  }
}

// The same 32 rows x 32 values through bulk tensor stores: the staging rows
// are 64-byte rows in the 64-byte swizzle (piece c of row r at c ^ ((r >> 1) & 3)
// within each 512-byte group, the layout of a SWIZZLE_64B box), and one lane
// sends them as one 32-row box when the warp's rows are consecutive in the
// destination, else as 8-row boxes to the rows d8[g] (each group of 8 rows
// lies in one chunk when the chunk length is a multiple of 8).
__device__ __forceinline__ void stage_store_bulk(uint32_t (*stg)[16], const uint32_t (&w)[16],
                                                 const CUtensorMap* tm32, const CUtensorMap* tm8, int gcol,
                                                 const int (&d8)[4], int ngroups, bool whole, int lane) {
  if (lane == 0) bulk_wait_read_all();  // the previous chunk's boxes have left the staging rows
  __syncwarp();
#pragma unroll
  for (int e = 0; e < 4; ++e)
    *reinterpret_cast<uint4*>(&stg[lane][4 * stage16_slot(lane, e)]) =
        make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
  fence_proxy_async_smem();  // the bulk copy reads what the generic stores wrote
  __syncwarp();
  if (lane == 0) {
    if (whole) {
      tma_store_2d(tm32, &stg[0][0], gcol, d8[0]);
    } else {
#pragma unroll
      for (int g = 0; g < 4; ++g)
        if (g < ngroups) tma_store_2d(tm8, &stg[8 * g][0], gcol, d8[g]);
    }
    bulk_commit();
  }
}

// 32 accumulator values of a row (16 rotation pairs) -> 16 packed bf16 pairs:
// y = x * gamma, then the rotation by {cos, sin} (already scaled by rstd)
__device__ __forceinline__ void rope_pack(const uint32_t (&x)[32], const float* g, const float (&cs)[16],
                                          const float (&sn)[16], uint32_t (&w)[16]) {
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 g4 = *reinterpret_cast<const float4*>(g + 4 * e4);
    const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = 2 * e4 + u;
      const float y0 = __uint_as_float(x[2 * e]) * gv[2 * u];
      const float y1 = __uint_as_float(x[2 * e + 1]) * gv[2 * u + 1];
      w[e] = pack_bf16x2(y0 * cs[e] - y1 * sn[e], y0 * sn[e] + y1 * cs[e]);
    }
  }
}

// {cos, sin} of one angle, for rotations that no table holds
__device__ __noinline__ float2 rot_slow(float angle) {
  float sv, cv;
  sincosf(angle, &sv, &cv);
  return make_float2(cv, sv);
}

__global__ void __launch_bounds__(kFThreads, 1)
    recache_fused_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmK32, const __grid_constant__ CUtensorMap tmV32,
                         const __grid_constant__ FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  FusedSmem& sm = *reinterpret_cast<FusedSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncta = p.HD / FW;  // CTAs of a cluster
  const int rank = (int)cluster_ctarank();
  const int cl = (int)cluster_index_x(), ncl = (int)cluster_count_x();
  const int nk = p.HD / RK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFASlots; ++s) {
      mbar_init(&sm.a_full[s], 1);
      mbar_init(&sm.a_empty[s], 1);
    }
    for (int s = 0; s < kFBSlots; ++s) {
      mbar_init(&sm.b_full[s], 1);
      mbar_init(&sm.b_empty[s], 1);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, 32 * kFEpiWarps);
    for (int b = 0; b < 2; ++b) mbar_init(&sm.bar_exch[b], 32 * kFEpiWarps * ncta);
    mbar_init(&sm.bar_drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < FW; i += kFThreads) sm.gam[i] = p.gamma ? p.gamma[rank * FW + i] : 1.0f;
  for (int i = threadIdx.x; i < 128; i += kFThreads) sm.om[i] = p.omega[i];
  if (p.w_tab) {  // {cos, sin}(w * omega) of the column band, for every grid column w
    const int nfh = p.pf + p.ph, nw = p.D / 2 - nfh;
    for (int i = threadIdx.x; i < p.grid_w * nw; i += kFThreads) {
      const int w = i / nw;
      float sv, cv;
      sincosf((float)w * p.omega[nfh + (i - w * nw)], &sv, &cv);
      sm.tw[i] = make_float2(cv, sv);
    }
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, FW);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const Watchdog wd{&sm.abort_flag, p.dev_err};

  if (warp < 4) {
    setmaxnreg_dec<kFCtl>();
    if (warp == 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        int na = 0, nb = 0;  // A and B ring positions
        bool ok = true;
        for (int it = cl; it < p.nitems && ok; it += ncl) {
          const FItem fi = fused_item(p, it, rank);
          const int m0 = fi.m0;
          const int c0 = (fi.is_k ? 0 : p.HD) + fi.cb * FW;  // first weight column of this CTA
          for (int kb = 0; kb < nk && ok; ++kb) {
            {
              const int s = na % kFASlots, u = na / kFASlots;
              if (na >= kFASlots && !mbar_wait(&sm.a_empty[s], (u - 1) & 1, wd)) {
                ok = false;
                break;
              }
              mbar_expect_tx(&sm.a_full[s], RM * RK * 2);
              tma_load_2d(&sm.a[s][0], &tmA, &sm.a_full[s], kb * RK, m0);
              ++na;
            }
            for (int h = 0; h < 2; ++h) {
              const int s = nb % kFBSlots, u = nb / kFBSlots;
              if (nb >= kFBSlots && !mbar_wait(&sm.b_empty[s], (u - 1) & 1, wd)) {
                ok = false;
                break;
              }
              mbar_expect_tx(&sm.b_full[s], RK * 256 * 2);
  #pragma unroll
              for (int q = 0; q < 4; ++q)
                tma_load_2d(&sm.b[s][q][0], &tmB, &sm.b_full[s], c0 + h * 256 + q * 64, kb * RK);
              ++nb;
            }
          }
        }
        if (sm.abort_flag) {  // every copy this thread started lands before the CTA exits
          for (int s = 0; s < kFASlots; ++s) {
            const int cnt = na > s ? (na - s + kFASlots - 1) / kFASlots : 0;
            if (cnt) mbar_drain(&sm.a_full[s], (cnt - 1) & 1);
          }
          for (int s = 0; s < kFBSlots; ++s) {
            const int cnt = nb > s ? (nb - s + kFBSlots - 1) / kFBSlots : 0;
            if (cnt) mbar_drain(&sm.b_full[s], (cnt - 1) & 1);
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(RM, 256, false, true);
        int na = 0, nb = 0, j = 0;
        bool ok = true;
        for (int it = cl; it < p.nitems && ok; it += ncl, ++j) {
          if (j >= 1 && !mbar_wait(&sm.acc_empty, (j - 1) & 1, wd)) break;
          tc_fence_after();
          for (int kb = 0; kb < nk && ok; ++kb) {
            const int sa = na % kFASlots;
            if (!mbar_wait(&sm.a_full[sa], (na / kFASlots) & 1, wd)) {
              ok = false;
              break;
            }
            for (int h = 0; h < 2; ++h) {
              const int sb = nb % kFBSlots;
              if (!mbar_wait(&sm.b_full[sb], (nb / kFBSlots) & 1, wd)) {
                ok = false;
                break;
              }
              tc_fence_after();
  #pragma unroll
              for (int kk = 0; kk < RK / 16; ++kk) {
                const uint64_t ad = sdesc_sw128(smem_u32(&sm.a[sa][0]) + kk * 32, 0, 1024);
                const uint64_t bd = sdesc_sw128(smem_u32(&sm.b[sb][0][0]) + kk * 2048, RK * 128, 1024);
                mma_bf16_ss(tmem + (uint32_t)(h * 256), ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
              }
              mma_commit(&sm.b_empty[sb]);  // frees the B slot for the producer
              ++nb;
            }
            if (!ok) break;
            mma_commit(&sm.a_empty[sa]);
            ++na;
          }
          if (ok) mma_commit(&sm.acc_full);
        }
        mma_commit(&sm.bar_drain);  // every MMA issued above completes before TMEM is freed
        mbar_drain(&sm.bar_drain, 0);
      }
    }
  } else {
    setmaxnreg_inc<kFEpi>();
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 4;         // 0..7
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int half = ew >> 2;        // column half: [256 half, 256 half + 256) of the CTA's 512
    const int rloc = q * 32 + lane;  // row within the tile
    uint32_t (*stg)[16] = sm.stage[ew];
    float2 (*tfh)[kFhMax] = sm.tfh[ew];
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 256);
    const float* gam = sm.gam + half * 256;
    const int nh = 256 / p.D;          // heads in a column half
    const int npc = p.D / 32;          // 32-column chunks (16 rotation pairs) of a head
    const int nfh = p.pf + p.ph;       // pairs of the frame and row bands
    const int nw = p.D / 2 - nfh;      // pairs of the column band
    const int64_t ld = p.HD / 8;       // output row stride in 16-byte pieces
    int j = 0, nkit = 0;
    for (int it = cl; it < p.nitems; it += ncl, ++j) {
      const FItem fi = fused_item(p, it, rank);
      const bool is_k = fi.is_k;
      const int m0 = fi.m0;
      const int gcol0 = fi.cb * FW + half * 256;
      const int gr = m0 + rloc;
      const int row0 = m0 + q * 32;
      int64_t my_dest = 0, fr = 0;
      int hh = 0, ww = 0;
      const bool real = gr < p.rows;
      if (real) {
        const int ci = gr / p.Tc;
        const int t = gr - ci * p.Tc;
        my_dest = (int64_t)p.region[ci] * p.Tc + t;
        const int pp = t % p.tpf;
        fr = p.frame0[ci] + t / p.tpf;
        hh = pp / p.grid_w;
        ww = pp % p.grid_w;
      }
      // destination rows of the warp's four 8-row groups (bulk stores)
      int d8[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) d8[g] = (int)__shfl_sync(0xffffffffu, my_dest, 8 * g);
      const int ngroups = min(4, max(0, (p.rows - row0 + 7) / 8));
      // all 32 rows real and consecutive in the destination: one 32-row box
      const bool whole = ngroups == 4 && d8[1] == d8[0] + 8 && d8[2] == d8[0] + 16 && d8[3] == d8[0] + 24;
      // K: while the MMAs run, the {cos, sin} of the frame and row bands for
      // the (at most two) frames and rows of this warp's 32 rows
      bool fh_tab = false;
      int sf = 0, sh = 0;
      if (is_k) {
        const int64_t f0 = __shfl_sync(0xffffffffu, fr, 0);
        const int h0 = __shfl_sync(0xffffffffu, hh, 0);
        if (!real) {  // rows past the end take the first row's values
          fr = f0;
          hh = h0;
        }
        const int64_t f1 = __shfl_sync(0xffffffffu, fr, 31);
        const int h1 = __shfl_sync(0xffffffffu, hh, 31);
        fh_tab = nfh <= kFhMax && __all_sync(0xffffffffu, (fr == f0 || fr == f1) && (hh == h0 || hh == h1));
        if (fh_tab) {
          for (int i = lane; i < 2 * nfh; i += 32) {
            const int slot = i >= nfh ? 1 : 0, pr = i - slot * nfh;
            const float pos = pr < p.pf ? (float)(slot ? f1 : f0) : (float)(slot ? h1 : h0);
            float sv, cv;
            sincosf(pos * sm.om[pr], &sv, &cv);
            tfh[slot][pr] = make_float2(cv, sv);
          }
          __syncwarp();
          sf = fr == f0 ? 0 : 1;
          sh = hh == h0 ? 0 : 1;
        }
      }
      // tcgen05.ld is warp-collective: the whole warp loads, stores are
      // predicated on the row being real
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.acc_full, j & 1, wd))) break;
      tc_fence_after();
      const CUtensorMap* tmo = is_k ? &tmK : &tmV;
      const CUtensorMap* tmo32 = is_k ? &tmK32 : &tmV32;
      uint4* obase = reinterpret_cast<uint4*>((is_k ? p.k : p.v) + gcol0);
      uint32_t xa[32], xb[32];
      if (is_k) {
        // pass 1: this row's sum of squares over the half's 256 columns, two
        // 32-column TMEM loads in flight per wait
        float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        tmem_ld32(tq, xa);
        tmem_ld32(tq + 32u, xb);
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) s4[e & 3] = fmaf(__uint_as_float(xa[e]), __uint_as_float(xa[e]), s4[e & 3]);
          if (c + 2 < 8) tmem_ld32(tq + (uint32_t)((c + 2) * 32), xa);
#pragma unroll
          for (int e = 0; e < 32; ++e) s4[e & 3] = fmaf(__uint_as_float(xb[e]), __uint_as_float(xb[e]), s4[e & 3]);
          if (c + 2 < 8) tmem_ld32(tq + (uint32_t)((c + 3) * 32), xb);
        }
        const float ss = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        // the partial goes into slot 2 rank + half of every CTA of the cluster
        const int buf = nkit & 1;
        const uint32_t la = smem_u32(&sm.exch[buf][2 * rank + half][rloc]);
        const uint32_t lb = smem_u32(&sm.bar_exch[buf]);
        for (int r = 0; r < ncta; ++r) {
          st_cluster_f32(mapa_shared(la, (uint32_t)r), ss);
          mbar_arrive_remote(mapa_shared(lb, (uint32_t)r));
        }
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&sm.bar_exch[buf], (nkit >> 1) & 1, wd))) break;
        ++nkit;
        float tot = 0.0f;
        for (int s2 = 0; s2 < 2 * ncta; ++s2) tot += sm.exch[buf][s2][rloc];
        const float rstd = 1.0f / sqrtf(tot / (float)p.HD + p.eps);
        // pass 2: x * gamma, rotated, rstd riding on cos and sin
        const int nch = npc * nh;
        tmem_ld32(tq, xa);
        tmem_ld32(tq + (uint32_t)p.D, xb);
        // {cos, sin} * rstd of the 16 rotation pairs of pair chunk pc
        auto rotations = [&](int pc, float (&cs)[16], float (&sn)[16]) {
          if (fh_tab && p.w_tab) {  // every rotation from a table (warp-uniform)
            const float2* tf = tfh[sf];
            const float2* th = tfh[sh];
            const float2* tw = sm.tw + ww * nw - nfh;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int pr = pc * 16 + e;
              const float2 t = pr < p.pf ? tf[pr] : (pr < nfh ? th[pr] : tw[pr]);
              cs[e] = t.x * rstd;
              sn[e] = t.y * rstd;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int pr = pc * 16 + e;
              float2 t;
              if (pr < nfh)
                t = fh_tab ? tfh[pr < p.pf ? sf : sh][pr]
                           : rot_slow((pr < p.pf ? (float)fr : (float)hh) * sm.om[pr]);
              else
                t = p.w_tab ? sm.tw[ww * nw + (pr - nfh)] : rot_slow((float)ww * sm.om[pr]);
              cs[e] = t.x * rstd;
              sn[e] = t.y * rstd;
            }
          }
        };
        // chunk i at column (i % nh) * D + (i / nh) * 32: the nh chunks of a
        // pair chunk (the same 16 rotations in every head) in turn, two per
        // TMEM wait, so each pair chunk's rotations are looked up once
        float cs[16], sn[16];
#pragma unroll 1
        for (int i = 0; i < nch; i += 2) {
          const int pc = i / nh;
          if (i % nh == 0) rotations(pc, cs, sn);
          const int cola = (i % nh) * p.D + pc * 32;
          const int colb = cola + p.D;  // chunk i + 1: the next head, same pair chunk
          const int i2 = i + 2;
          const uint32_t c2 = (uint32_t)((i2 % nh) * p.D + (i2 / nh) * 32);  // next pair's first column
          uint32_t wa[16], wb[16];
          tmem_ld_wait();
          rope_pack(xa, gam + cola, cs, sn, wa);
          if (i2 < nch) tmem_ld32(tq + c2, xa);
          rope_pack(xb, gam + colb, cs, sn, wb);
          if (i2 < nch) tmem_ld32(tq + c2 + (uint32_t)p.D, xb);
          if (p.tma_out) {
            stage_store_bulk(stg, wa, tmo32, tmo, gcol0 + cola, d8, ngroups, whole, lane);
            stage_store_bulk(stg, wb, tmo32, tmo, gcol0 + colb, d8, ngroups, whole, lane);
          } else {
            stage_store16(stg, wa, obase + cola / 8, ld, my_dest, row0, p.rows, lane);
            stage_store16(stg, wb, obase + colb / 8, ld, my_dest, row0, p.rows, lane);
          }
        }
      } else {
        tmem_ld32(tq, xa);
        tmem_ld32(tq + 32u, xb);
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          tmem_ld_wait();
          uint32_t wa[16], wb[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            wa[e] = pack_bf16x2(__uint_as_float(xa[2 * e]), __uint_as_float(xa[2 * e + 1]));
            wb[e] = pack_bf16x2(__uint_as_float(xb[2 * e]), __uint_as_float(xb[2 * e + 1]));
          }
          if (c + 2 < 8) {
            tmem_ld32(tq + (uint32_t)((c + 2) * 32), xa);
            tmem_ld32(tq + (uint32_t)((c + 3) * 32), xb);
          }
          if (p.tma_out) {
            stage_store_bulk(stg, wa, tmo32, tmo, gcol0 + c * 32, d8, ngroups, whole, lane);
            stage_store_bulk(stg, wb, tmo32, tmo, gcol0 + c * 32 + 32, d8, ngroups, whole, lane);
          } else {
            stage_store16(stg, wa, obase + c * 4, ld, my_dest, row0, p.rows, lane);
            stage_store16(stg, wb, obase + c * 4 + 4, ld, my_dest, row0, p.rows, lane);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_empty);  // the MMA may overwrite the accumulator
    }
    if (lane == 0) bulk_wait_all();  // this warp's bulk stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, FW);
  }
  cluster_sync_all();  // no CTA leaves while a peer may still store into its shared memory
}

// One CTA per SM (persistent), never more CTAs than tiles.  ncol: column tiles
// of this launch (its width / BN).
template <int BN>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, GemmParams p, cudaStream_t st) {
  const size_t smem = sizeof(GemmSmem<BN>) + 1024;
  auto kern = recache_gemm_kernel<BN>;
  static bool smem_set[64] = {};  // one per instantiation of this launcher
  cudaError_t e = set_smem_once(kern, smem, smem_set);
  if (e != cudaSuccess) return e;
  const int nsm = attn_sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  p.ntiles = ((p.rows + RM - 1) / RM) * p.ncol;
  int grid = nsm < p.ntiles ? nsm : p.ntiles;
  if (grid < 1) grid = 1;
  kern<<<grid, kRThreads, smem, st>>>(ta, tb, p);
  return cudaGetLastError();
}

// RoPE geometry shared by both paths.
void fill_rope(float* omega, int32_t& pf_out, int32_t& ph_out, int D, float theta) {
  const int P = D / 2, hw = P / 3, pf = P - 2 * hw;
  pf_out = pf;
  ph_out = hw;
  for (int i = 0; i < P; ++i) {
    int j, b;
    if (i < pf) {
      j = i;
      b = 2 * pf;
    } else if (i < pf + hw) {
      j = i - pf;
      b = 2 * hw;
    } else {
      j = i - pf - hw;
      b = 2 * hw;
    }
    omega[i] = (float)std::pow((double)theta, -2.0 * j / b);
  }
}
void fill_rope(NormParams& q, int D, float theta) { fill_rope(q.omega, q.pf, q.ph, D, theta); }

// Clusters of `ncta` fused-recache CTAs resident at once on the current
// device (queried once per device and cluster size; 0 when the query fails).
int fused_max_clusters(int ncta, size_t smem) {
  static int cache[64][kFMaxCluster + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev][ncta] > 0) return cache[dev][ncta];
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)ncta, 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, recache_fused_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cache[dev][ncta] = n;
  return n;
}

// A second stream and two events per host thread and device, created on first
// use and kept (host objects only; no device memory): the fused recache's
// cluster-free launch runs on it, forked from and joined back to the caller's
// stream with the events (this also holds under stream capture).
cudaError_t side_stream(cudaStream_t* s, cudaEvent_t* fork, cudaEvent_t* join) {
  struct Side {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
  };
  thread_local Side sides[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  Side& d = sides[dev];
  if (!d.s) {
    Side n;
    cudaError_t e = cudaStreamCreateWithFlags(&n.s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      if (n.join) cudaEventDestroy(n.join);
      if (n.fork) cudaEventDestroy(n.fork);
      if (n.s) cudaStreamDestroy(n.s);
      return e;
    }
    d = n;
  }
  *s = d.s;
  *fork = d.fork;
  *join = d.join;
  return cudaSuccess;
}

// H*D a multiple of 512 (at most 4 x 512) and D in {64, 128}: one
// fused launch (K and V items, the norm in the K epilogue).
bool recache_fusable(int H, int D) {
  const int HD = H * D;
  return HD % FW == 0 && HD / FW <= kFMaxCluster && D % 64 == 0 && 128 % D == 0;
}

cudaError_t launch_recache_fused(const RecacheLaunch& r, cudaStream_t st) {
  if (r.rows <= 0) return cudaSuccess;
  const int HD = r.H * r.D;
  CUtensorMap ta{}, tb{};
  if (!encode_tmap_2d_bf16(&ta, r.hidden, HD, r.rows, (uint64_t)HD * 2, RK, RM, true))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d_bf16(&tb, r.w_kv, 2 * HD, HD, (uint64_t)HD * 4, 64, RK, true))
    return cudaErrorInvalidValue;
  FusedParams p{};
  p.rows = r.rows;
  p.HD = HD;
  p.Tc = r.Tc;
  p.D = r.D;
  p.tpf = r.tpf;
  p.grid_w = r.grid_w;
  p.eps = r.eps;
  fill_rope(p.omega, p.pf, p.ph, r.D, r.theta);
  for (int i = 0; i < r.n; ++i) {
    p.region[i] = r.region[i];
    p.frame0[i] = r.frame0[i];
  }
  p.gamma = r.gamma;
  p.k = static_cast<__nv_bfloat16*>(r.k);
  p.v = static_cast<__nv_bfloat16*>(r.v);
  p.dev_err = r.dev_err;
  p.w_tab = r.grid_w * (r.D / 2 - p.pf - p.ph) <= kTwMax;
  // bulk stores of 8-row boxes: every 8-row group of a tile lies in one chunk
  p.tma_out = r.Tc % 8 == 0;
  CUtensorMap tk{}, tv{}, tk32{}, tv32{};
  if (p.tma_out) {
    int32_t nreg = 0;
    for (int i = 0; i < r.n; ++i) nreg = r.region[i] + 1 > nreg ? r.region[i] + 1 : nreg;
    const uint64_t drows = (uint64_t)nreg * (uint64_t)r.Tc;  // destination rows the launch may write
    if (!encode_tmap_2d_bf16_sw(&tk, r.k, HD, drows, (uint64_t)HD * 2, 32, 8, 64) ||
        !encode_tmap_2d_bf16_sw(&tv, r.v, HD, drows, (uint64_t)HD * 2, 32, 8, 64) ||
        !encode_tmap_2d_bf16_sw(&tk32, r.k, HD, drows, (uint64_t)HD * 2, 32, 32, 64) ||
        !encode_tmap_2d_bf16_sw(&tv32, r.v, HD, drows, (uint64_t)HD * 2, 32, 32, 64))
      return cudaErrorInvalidValue;
  }
  const size_t smem = sizeof(FusedSmem) + 1024;
  static bool smem_set[64] = {};
  cudaError_t e = set_smem_once(recache_fused_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  {
    // the setmaxnreg split hands out exactly the registers the block launches
    // with: refuse to launch if the compiled kernel's count differs (an
    // increase that the launch cannot cover would wait forever)
    static int regs_ok[64] = {};  // per device: 0 unknown, 1 ok, -1 mismatch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (regs_ok[dev] == 0) {
      cudaFuncAttributes fa{};
      e = cudaFuncGetAttributes(&fa, recache_fused_kernel);
      if (e != cudaSuccess) return e;
      regs_ok[dev] = fa.numRegs == kFLaunch ? 1 : -1;
    }
    if (regs_ok[dev] < 0) return cudaErrorInvalidConfiguration;
  }
  const int ncta = HD / FW, nrt = (r.rows + RM - 1) / RM;
  const int ncl = fused_max_clusters(ncta, smem);
  if (ncl <= 0) return cudaErrorInvalidConfiguration;
  // SMs that no cluster fits on (13 of 148 for 3-CTA clusters) take the V
  // items of the last x row tiles in a second, cluster-free launch beside the
  // first: x balances the two by the measured item costs (a K item, with its
  // norm and rotation epilogue, takes about 1.35 times a V item)
  const int nsm = attn_sm_count();
  const int nfree = nsm - ncl * ncta;
  int x = 0;
  if (nfree > 0) {
    constexpr double kCostK = 1.35, kCostV = 1.0;
    double best = (nrt * kCostK + nrt * kCostV) / ncl;
    for (int xx = 1; xx <= nrt; ++xx) {
      const double ta = (nrt * kCostK + (nrt - xx) * kCostV) / ncl;
      const double tb = (double)((xx * ncta + nfree - 1) / nfree) * kCostV;
      const double t = ta > tb ? ta : tb;
      if (t < best - 1e-9) {
        best = t;
        x = xx;
      }
    }
  }
  p.vonly = 0;
  p.rt_split = nrt - x;
  p.nitems = nrt + p.rt_split;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  if (x > 0) {
    // the side launch starts with the main one: both wait for the work already
    // in `st`, and `st` waits for the side launch before anything after it
    e = side_stream(&side, &ev_fork, &ev_join);
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(ev_fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ev_fork, 0);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(ncta * (ncl < p.nitems ? ncl : p.nitems)), 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, recache_fused_kernel, ta, tb, tk, tv, tk32, tv32, p);
  if (e != cudaSuccess || x == 0) return e;
  FusedParams pv = p;
  pv.vonly = 1;
  pv.nitems = x * ncta;
  cfg.gridDim = dim3((unsigned)(nfree < pv.nitems ? nfree : pv.nitems), 1, 1);
  cfg.stream = side;
  attr[0].val.clusterDim.x = 1;
  e = cudaLaunchKernelEx(&cfg, recache_fused_kernel, ta, tb, tk, tv, tk32, tv32, pv);
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(ev_join, side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_join, 0);
  return e;
}

template <int HD>
cudaError_t launch_norm(const NormParams& q, int njobs, cudaStream_t st) {
  recache_norm_rope_kernel<HD><<<dim3((q.rows + kNormWarps - 1) / kNormWarps, njobs), kNormWarps * 32, 0, st>>>(q);
  return cudaGetLastError();
}

template <int BN, int HD>
cudaError_t launch_recache_t(const RecacheLaunch& r, cudaStream_t st) {
  CUtensorMap ta{}, tb{};
  if (!encode_tmap_2d_bf16(&ta, r.hidden, HD, r.rows, (uint64_t)HD * 2, RK, RM, true))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d_bf16(&tb, r.w_kv, 2 * HD, HD, (uint64_t)HD * 4, 64, RK, true))
    return cudaErrorInvalidValue;
  __nv_bfloat16* k = static_cast<__nv_bfloat16*>(r.k);
  __nv_bfloat16* v = static_cast<__nv_bfloat16*>(r.v);
  GemmParams g{};
  g.rows = r.rows;
  g.HD = HD;
  g.Tc = r.Tc;
  g.ncol = HD / BN;
  for (int i = 0; i < r.n; ++i) g.region[i] = r.region[i];
  g.dev_err = r.dev_err;

  NormParams q{};
  q.rows = r.rows;
  q.D = r.D;
  q.Tc = r.Tc;
  q.tpf = r.tpf;
  q.grid_w = r.grid_w;
  q.eps = r.eps;
  fill_rope(q, r.D, r.theta);
  for (int i = 0; i < r.n; ++i) {
    q.frame0[i] = r.frame0[i];
    q.region[i] = r.region[i];
  }
  // the fp32 K row of a token is parked across its K row (first half) and V row
  q.job[0] = NormJob{reinterpret_cast<const float*>(k), reinterpret_cast<const float*>(v), HD / 2,
                     HD / 2, k, HD, r.gamma};

  // 1. K GEMM, parked
  g.col0 = 0;
  g.n_f32 = HD;
  g.f32_split = HD / 2;
  g.f32a = reinterpret_cast<float*>(k);
  g.f32b = reinterpret_cast<float*>(v);
  g.ld_f32 = HD / 2;
  cudaError_t e = launch_gemm<BN>(ta, tb, g, st);
  if (e != cudaSuccess) return e;
  // 2. norm + RoPE in place
  e = launch_norm<HD>(q, 1, st);
  if (e != cudaSuccess) return e;
  // 3. V GEMM, bf16 over the parked halves
  g.col0 = HD;
  g.n_f32 = 0;
  g.bf = v;
  g.ld_bf = HD;
  return launch_gemm<BN>(ta, tb, g, st);
}

template <int BN, int HD>
cudaError_t launch_project_t(const ProjectLaunch& r, cudaStream_t st) {
  CUtensorMap ta{}, tb{};
  if (!encode_tmap_2d_bf16(&ta, r.hidden, HD, r.Tc, (uint64_t)HD * 2, RK, RM, true))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d_bf16(&tb, r.w_qkv, 3 * HD, HD, (uint64_t)HD * 6, 64, RK, true))
    return cudaErrorInvalidValue;
  // one GEMM over [Q | K | V]: Q and K parked as fp32 rows [Tc][2 HD] in the
  // staging buffer, V as bf16 at its destination
  GemmParams g{};
  g.rows = r.Tc;
  g.HD = HD;
  g.Tc = r.Tc;  // one chunk: destination row = output row
  g.ncol = 3 * HD / BN;
  g.region[0] = 0;
  g.dev_err = r.dev_err;
  g.col0 = 0;
  g.n_f32 = 2 * HD;
  g.f32_split = 2 * HD;
  g.f32a = g.f32b = r.stage_f32;
  g.ld_f32 = 2 * HD;
  g.bf = static_cast<__nv_bfloat16*>(r.v_dst);
  g.ld_bf = HD;
  cudaError_t e = launch_gemm<BN>(ta, tb, g, st);
  if (e != cudaSuccess) return e;
  NormParams q{};
  q.rows = r.Tc;
  q.D = r.D;
  q.Tc = r.Tc;
  q.tpf = r.tpf;
  q.grid_w = r.grid_w;
  q.eps = r.eps;
  fill_rope(q, r.D, r.theta);
  q.frame0[0] = r.frame0;
  q.region[0] = 0;
  q.job[0] = NormJob{r.stage_f32, r.stage_f32, 2 * HD, HD, static_cast<__nv_bfloat16*>(r.q_out), HD,
                     r.gamma_q};
  q.job[1] = NormJob{r.stage_f32 + HD, r.stage_f32 + HD, 2 * HD, HD,
                     static_cast<__nv_bfloat16*>(r.k_dst), HD, r.gamma_k};
  return launch_norm<HD>(q, 2, st);
}

}  // namespace

bool recache_supported(int H, int D) {
  const int HD = H * D;
  if (D % 2 != 0 || D / 2 > 128) return false;
  switch (HD) {
    case 64: case 128: case 256: case 512: case 768: case 1024: case 1536: case 2048: case 3072:
      return true;
    default:
      return false;
  }
}

cudaError_t launch_recache(const RecacheLaunch& r, cudaStream_t st) {
  if (recache_fusable(r.H, r.D)) return launch_recache_fused(r, st);
  switch (r.H * r.D) {
    case 64: return launch_recache_t<64, 64>(r, st);
    case 128: return launch_recache_t<128, 128>(r, st);
    case 256: return launch_recache_t<256, 256>(r, st);
    case 512: return launch_recache_t<256, 512>(r, st);
    case 768: return launch_recache_t<256, 768>(r, st);
    case 1024: return launch_recache_t<256, 1024>(r, st);
    case 1536: return launch_recache_t<256, 1536>(r, st);
    case 2048: return launch_recache_t<256, 2048>(r, st);
    case 3072: return launch_recache_t<256, 3072>(r, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_project_chunk(const ProjectLaunch& r, cudaStream_t st) {
  switch (r.H * r.D) {
    case 64: return launch_project_t<64, 64>(r, st);
    case 128: return launch_project_t<128, 128>(r, st);
    case 256: return launch_project_t<256, 256>(r, st);
    case 512: return launch_project_t<256, 512>(r, st);
    case 768: return launch_project_t<256, 768>(r, st);
    case 1024: return launch_project_t<256, 1024>(r, st);
    case 1536: return launch_project_t<192, 1536>(r, st);  // 4608 = 24 x 192: whole waves at 4680 rows
    case 2048: return launch_project_t<256, 2048>(r, st);
    case 3072: return launch_project_t<256, 3072>(r, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvc
