// KV recache at a prompt switch: [K | V] = Hid @ W_kv on tcgen05, then
// K <- RoPE3D(RMSNorm(K) * gamma), written into the cache.
//
// LongLive summary page (yunpan.plus), 方法 §1 KV 重缓存: at the switch the cache
// is recomputed from the frames already generated paired with the new prompt;
// these kernels are the per-layer tail of that recompute (K/V projection, key
// norm, rotary positions, cache write).
//
// RMSNorm spans the whole H*D-wide K row, which no single 128 x 256 output tile
// holds, and rounding K to bf16 before the norm and again after it would round
// twice.  So the work runs as three stream-ordered launches with no cross-CTA
// waits at all:
//   1. K GEMM: the unnormalised fp32 K row of token `dest` is parked in the
//      cache's own K and V rows of that token (each row is H*D*2 bytes, so the
//      two together hold exactly H*D fp32 values: columns [0, HD/2) in the K row,
//      [HD/2, HD) in the V row);
//   2. norm + RoPE: one warp per token reads its fp32 row, takes the mean square,
//      applies gamma and the 3D rotation and writes the bf16 K row (one rounding);
//   3. V GEMM: bf16 V straight into the V rows (overwriting the parked halves).
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

struct GemmParams {
  int32_t rows, HD, Tc;
  int32_t col0;    // first output column of this launch in [K | V]: 0 (K) or HD (V)
  int32_t ncol;    // column tiles (HD / BN)
  int32_t ntiles;  // row tiles x column tiles
  int32_t region[kMaxSeg];
  __nv_bfloat16* k;
  __nv_bfloat16* v;
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
// kKf32: K launch (fp32 rows parked in the K|V rows); else the V launch (bf16).
template <int BN, bool kKf32>
__global__ void __launch_bounds__(kRThreads, 1)
    recache_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ GemmParams p) {
  using Smem = GemmSmem<BN>;
  constexpr uint32_t kCols = 2 * BN < 32 ? 32 : 2 * BN;
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
      // Each 32-column chunk goes through the warp's staging rows (lane = row)
      // and back out transposed: in store step k, lane l writes one 16-byte
      // piece of row k * (32 / pieces) + l / pieces, so each store instruction
      // covers whole 128-byte (fp32) or 64-byte (bf16) row segments instead of
      // 16 bytes of 32 different rows.
      uint32_t (*stg)[32] = sm.stage[wq];
      // cache row of this lane's tile row (lane = row within the warp's 32);
      // store steps fetch the row they write from its lane
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
#pragma unroll 1
      for (int jj = 0; jj < BN / 32; ++jj) {
        tmem_ld_wait();
        const int col = nloc + jj * 32;  // column within the half, a multiple of 32
        __syncwarp();                    // the previous chunk's transposed reads are done
        if constexpr (kKf32) {
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
        constexpr int kChunksPerRow = kKf32 ? 8 : 4;  // 16-byte pieces of a row's 32 values
        constexpr int kRowsPerStep = 32 / kChunksPerRow;
#pragma unroll
        for (int k = 0; k < 32 / kRowsPerStep; ++k) {
          const int rl = k * kRowsPerStep + lane / kChunksPerRow;  // row within the warp's 32
          const int piece = lane % kChunksPerRow;
          const int64_t dst = __shfl_sync(0xffffffffu, my_dest, rl);
          if (m0 + wq * 32 + rl >= p.rows) continue;
          const uint4 v = *reinterpret_cast<const uint4*>(&stg[rl][4 * stage_slot(rl, piece)]);
          if constexpr (kKf32) {
            const int half = p.HD / 2;
            float* row = reinterpret_cast<float*>(col < half ? p.k + dst * p.HD : p.v + dst * p.HD);
            reinterpret_cast<uint4*>(row + (col < half ? col : col - half))[piece] = v;
          } else {
            reinterpret_cast<uint4*>(p.v + dst * p.HD + col)[piece] = v;
          }
        }
      }
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
struct NormParams {
  int32_t rows, D, Tc, tpf, chunk_frames, grid_w;
  int32_t pf, ph;  // RoPE pairs of the frame and row bands (column band = rest)
  float eps;
  int64_t chunk_id[kMaxSeg];
  int32_t region[kMaxSeg];
  float omega[128];  // per rotation pair of a head: theta^(-2j/b) of its band
  const float* gamma;
  __nv_bfloat16* k;
  const __nv_bfloat16* v;
};

constexpr int kNormWarps = 8;

// Lane l owns fp32 columns 4*(l + 32*i) .. +3, i < HD/128: 16-byte coalesced
// loads from the parked halves, the row's mean square by a warp reduction,
// then two rotation pairs per float4.
template <int HD>
__global__ void __launch_bounds__(kNormWarps * 32) recache_norm_rope_kernel(const __grid_constant__ NormParams p) {
  constexpr int NV = (HD + 127) / 128;  // float4 per lane (the last one may be partial)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grow = blockIdx.x * kNormWarps + warp;
  if (grow >= p.rows) return;
  const int ci = grow / p.Tc;
  const int t = grow - ci * p.Tc;
  const int64_t dest = (int64_t)p.region[ci] * p.Tc + t;
  const float4* krow = reinterpret_cast<const float4*>(p.k + dest * HD);
  const float4* vrow = reinterpret_cast<const float4*>(p.v + dest * HD);
  float4 x[NV];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c4 = lane + 32 * i;  // float4 index in the fp32 row
    x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c4 < HD / 4) x[i] = c4 < HD / 8 ? krow[c4] : vrow[c4 - HD / 8];
    ss = fmaf(x[i].x, x[i].x, ss);
    ss = fmaf(x[i].y, x[i].y, ss);
    ss = fmaf(x[i].z, x[i].z, ss);
    ss = fmaf(x[i].w, x[i].w, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float rstd = 1.0f / sqrtf(ss / (float)HD + p.eps);
  const int64_t fr = p.chunk_id[ci] * p.chunk_frames + t / p.tpf;
  const int pp = t % p.tpf;
  const float pos_f = (float)fr, pos_h = (float)(pp / p.grid_w), pos_w = (float)(pp % p.grid_w);
  // the K row is overwritten in place: every lane's reads of it come first
  __syncwarp();
  uint2* out = reinterpret_cast<uint2*>(p.k + dest * HD);
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
    const float4 g4 = p.gamma ? __ldg(reinterpret_cast<const float4*>(p.gamma) + c4) : make_float4(1.f, 1.f, 1.f, 1.f);
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

// One CTA per SM (persistent), never more CTAs than tiles.
template <int BN, bool kKf32>
cudaError_t launch_gemm(int rows, const CUtensorMap& ta, const CUtensorMap& tb, GemmParams p,
                        cudaStream_t st) {
  const size_t smem = sizeof(GemmSmem<BN>) + 1024;
  auto kern = recache_gemm_kernel<BN, kKf32>;
  static bool smem_set[64] = {};  // one per instantiation of this launcher
  cudaError_t e = set_smem_once(kern, smem, smem_set);
  if (e != cudaSuccess) return e;
  const int nsm = attn_sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  p.ncol = p.HD / BN;
  p.ntiles = ((rows + RM - 1) / RM) * p.ncol;
  int grid = nsm < p.ntiles ? nsm : p.ntiles;
  if (grid < 1) grid = 1;
  kern<<<grid, kRThreads, smem, st>>>(ta, tb, p);
  return cudaGetLastError();
}

template <int BN, int HD>
cudaError_t launch_recache_t(const RecacheLaunch& r, cudaStream_t st) {
  CUtensorMap ta{}, tb{};
  if (!encode_tmap_2d_bf16(&ta, r.hidden, HD, r.rows, (uint64_t)HD * 2, RK, RM, true))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d_bf16(&tb, r.w_kv, 2 * HD, HD, (uint64_t)HD * 4, 64, RK, true))
    return cudaErrorInvalidValue;
  GemmParams g{};
  g.rows = r.rows;
  g.HD = HD;
  g.Tc = r.Tc;
  for (int i = 0; i < r.n; ++i) g.region[i] = r.region[i];
  g.k = static_cast<__nv_bfloat16*>(r.k);
  g.v = static_cast<__nv_bfloat16*>(r.v);
  g.dev_err = r.dev_err;

  NormParams q{};
  q.rows = r.rows;
  q.D = r.D;
  q.Tc = r.Tc;
  q.tpf = r.tpf;
  q.chunk_frames = r.chunk_frames;
  q.grid_w = r.grid_w;
  q.eps = r.eps;
  const int P = r.D / 2, hw = P / 3, pf = P - 2 * hw;
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
    q.omega[i] = (float)std::pow((double)r.theta, -2.0 * j / b);
  }
  for (int i = 0; i < r.n; ++i) {
    q.chunk_id[i] = r.chunk_id[i];
    q.region[i] = r.region[i];
  }
  q.gamma = r.gamma;
  q.k = g.k;
  q.v = g.v;

  g.col0 = 0;
  cudaError_t e = launch_gemm<BN, true>(r.rows, ta, tb, g, st);
  if (e != cudaSuccess) return e;
  recache_norm_rope_kernel<HD><<<(r.rows + kNormWarps - 1) / kNormWarps, kNormWarps * 32, 0, st>>>(q);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  g.col0 = HD;
  return launch_gemm<BN, false>(r.rows, ta, tb, g, st);
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

}  // namespace kvc
