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
// twice.  So the GEMM stores the rows to be normalised as fp32 ("parked"), and
// a second launch normalises them:
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
void fill_rope(NormParams& q, int D, float theta) {
  const int P = D / 2, hw = P / 3, pf = P - 2 * hw;
  q.pf = pf;
  q.ph = hw;
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
    q.omega[i] = (float)std::pow((double)theta, -2.0 * j / b);
  }
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
