// KV recache at a prompt switch: [K | V] = Hid @ W_kv on tcgen05, then
// K <- RoPE3D(RMSNorm(K) * gamma) in the epilogue, written into the cache.
//
// LongLive summary page (yunpan.plus), 方法 §1 KV 重缓存: at the switch the cache
// is recomputed from the frames already generated paired with the new prompt;
// this kernel is the per-layer tail of that recompute (K/V projection, key norm,
// rotary positions, cache write).
//
// Tiling: a CTA computes a 128 x BN tile (BN = 256 at H*D = 1536) with BK = 64
// K-steps through a TMA ring.  The K half of the output is covered by a
// thread-block cluster of H*D/BN CTAs along N: each CTA sums x^2 over its BN
// columns, the partial sums are exchanged through distributed shared memory,
// and every CTA normalises and rotates its own columns.  V tiles run the same
// cluster shape and only cast and store.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int RM = 128;  // rows per tile
constexpr int RK = 64;   // K per stage (one 128-byte swizzle row of bf16)
constexpr int kRThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue

struct RecacheParams {
  int32_t rows, HD, Tc, tpf, chunk_frames, grid_w, D;
  int32_t n;
  int32_t pf, ph;  // RoPE pairs of the frame and row bands (column band = rest)
  float eps;
  int64_t chunk_id[kMaxSeg];
  int32_t region[kMaxSeg];
  float omega[128];  // per rotation pair of a head: theta^(-2j/b) of its band
  const float* gamma;
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  int32_t* dev_err;
};

template <int BN, int STAGES>
struct __align__(1024) RecacheSmem {
  __nv_bfloat16 a[STAGES][RM * RK];
  __nv_bfloat16 b[STAGES][BN / 64][RK * 64];
  uint64_t bar_full[STAGES], bar_empty[STAGES];
  uint64_t bar_acc, bar_drain;
  float ss[RM];  // per-row partial sum of squares (read by the whole cluster)
  uint32_t tmem_base;
  int32_t abort_flag;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nrank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(raddr) : "memory");
  return v;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kRThreads, 1)
    recache_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ RecacheParams p) {
  using Smem = RecacheSmem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;  // output column of [K | V]
  const int m0 = blockIdx.y * RM;
  const int nk = p.HD / RK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.bar_full[s], 1);
      mbar_init(&sm.bar_empty[s], 1);
    }
    mbar_init(&sm.bar_acc, 1);
    mbar_init(&sm.bar_drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, BN < 32 ? 32 : BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const Watchdog wd{&sm.abort_flag, p.dev_err};
  bool acc_ok = false;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % STAGES, u = kb / STAGES;
        if (kb >= STAGES && !mbar_wait(&sm.bar_empty[s], (u - 1) & 1, wd)) break;
        mbar_expect_tx(&sm.bar_full[s], RM * RK * 2 + RK * BN * 2);
        tma_load_2d(&sm.a[s][0], &tmA, &sm.bar_full[s], kb * RK, m0);
        for (int nb = 0; nb < BN / 64; ++nb)
          tma_load_2d(&sm.b[s][nb][0], &tmB, &sm.bar_full[s], n0 + nb * 64, kb * RK);
        issued = kb + 1;
      }
      if (sm.abort_flag) {
        for (int s = 0; s < STAGES; ++s) {
          const int cnt = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
          if (cnt) mbar_drain(&sm.bar_full[s], (cnt - 1) & 1);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(RM, BN, false, true);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % STAGES, u = kb / STAGES;
        if (!mbar_wait(&sm.bar_full[s], u & 1, wd)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < RK / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(smem_u32(&sm.a[s][0]) + kk * 32, 0, 1024);
          const uint64_t bd = sdesc_sw128(smem_u32(&sm.b[s][0][0]) + kk * 2048, RK * 128, 1024);
          mma_bf16_ss(tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&sm.bar_empty[s]);
      }
      if (ok) mma_commit(&sm.bar_acc);
      mma_commit(&sm.bar_drain);
      mbar_drain(&sm.bar_drain, 0);
    }
  } else {
    // epilogue pass 1: wait for the accumulator, row sum of squares
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(wq * 32) << 16);
    if (mbar_wait(&sm.bar_acc, 0, wd)) {
      tc_fence_after();
      acc_ok = true;
      float ss = 0.0f;
      if (n0 < p.HD) {
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
          uint32_t x[32];
          tmem_ld32(trow + j * 32, x);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ss = fmaf(__uint_as_float(x[e]), __uint_as_float(x[e]), ss);
        }
      }
      sm.ss[r] = ss;
    } else {
      sm.ss[r] = 0.0f;
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();  // partial sums of every CTA of the cluster are visible
  tc_fence_after();

  if (warp >= 2) {
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int grow = m0 + r;
    const uint32_t trow = tmem + ((uint32_t)(wq * 32) << 16);
    const bool all_ok = acc_ok && !sm.abort_flag;
    if (all_ok && grow < p.rows) {
      const int ci = grow / p.Tc;
      const int t = grow - ci * p.Tc;
      const int64_t dest = (int64_t)p.region[ci] * p.Tc + t;
      if (n0 < p.HD) {
        float tot = 0.0f;
        const uint32_t nr = cluster_nrank();
        for (uint32_t q = 0; q < nr; ++q) tot += ld_dsmem_f32(&sm.ss[r], q);
        const float rstd = 1.0f / sqrtf(tot / (float)p.HD + p.eps);
        const int64_t fr = p.chunk_id[ci] * p.chunk_frames + t / p.tpf;
        const int pp = t % p.tpf;
        const float pos_f = (float)fr, pos_h = (float)(pp / p.grid_w), pos_w = (float)(pp % p.grid_w);
        __nv_bfloat16* dst = p.k + dest * p.HD + n0;
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
          uint32_t x[32];
          tmem_ld32(trow + j * 32, x);
          tmem_ld_wait();
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = n0 + j * 32 + 2 * e;  // K column of the pair's first element
            const int pr = (col % p.D) >> 1;       // rotation pair within the head
            const float g0 = p.gamma ? p.gamma[col] : 1.0f;
            const float g1 = p.gamma ? p.gamma[col + 1] : 1.0f;
            const float y0 = __uint_as_float(x[2 * e]) * rstd * g0;
            const float y1 = __uint_as_float(x[2 * e + 1]) * rstd * g1;
            const float pos = pr < p.pf ? pos_f : (pr < p.pf + p.ph ? pos_h : pos_w);
            float sn, cs;
            sincosf(pos * p.omega[pr], &sn, &cs);
            o[e] = pack_bf16x2(y0 * cs - y1 * sn, y0 * sn + y1 * cs);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + j * 32);
          d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
          d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
          d4[2] = make_uint4(o[8], o[9], o[10], o[11]);
          d4[3] = make_uint4(o[12], o[13], o[14], o[15]);
        }
      } else {
        __nv_bfloat16* dst = p.v + dest * p.HD + (n0 - p.HD);
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
          uint32_t x[32];
          tmem_ld32(trow + j * 32, x);
          tmem_ld_wait();
          uint4* d4 = reinterpret_cast<uint4*>(dst + j * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(pack_bf16x2(__uint_as_float(x[8 * e + 0]), __uint_as_float(x[8 * e + 1])),
                               pack_bf16x2(__uint_as_float(x[8 * e + 2]), __uint_as_float(x[8 * e + 3])),
                               pack_bf16x2(__uint_as_float(x[8 * e + 4]), __uint_as_float(x[8 * e + 5])),
                               pack_bf16x2(__uint_as_float(x[8 * e + 6]), __uint_as_float(x[8 * e + 7])));
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while a peer may still read its partial sums
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, BN < 32 ? 32 : BN);
  }
}

template <int BN, int STAGES>
cudaError_t launch_recache_t(const RecacheLaunch& r, cudaStream_t st) {
  CUtensorMap ta{}, tb{};
  const int HD = r.H * r.D;
  if (!encode_tmap_2d_bf16(&ta, r.hidden, HD, r.rows, (uint64_t)HD * 2, RK, RM, true))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d_bf16(&tb, r.w_kv, 2 * HD, HD, (uint64_t)HD * 4, 64, RK, true))
    return cudaErrorInvalidValue;
  RecacheParams p{};
  p.rows = r.rows;
  p.HD = HD;
  p.Tc = r.Tc;
  p.tpf = r.tpf;
  p.chunk_frames = r.chunk_frames;
  p.grid_w = r.grid_w;
  p.D = r.D;
  p.n = r.n;
  p.eps = r.eps;
  const int P = r.D / 2, hw = P / 3, pf = P - 2 * hw;
  p.pf = pf;
  p.ph = hw;
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
    p.omega[i] = (float)std::pow((double)r.theta, -2.0 * j / b);
  }
  for (int i = 0; i < r.n; ++i) {
    p.chunk_id[i] = r.chunk_id[i];
    p.region[i] = r.region[i];
  }
  p.gamma = r.gamma;
  p.k = static_cast<__nv_bfloat16*>(r.k);
  p.v = static_cast<__nv_bfloat16*>(r.v);
  p.dev_err = r.dev_err;

  const size_t smem = sizeof(RecacheSmem<BN, STAGES>) + 1024;
  auto kern = recache_kernel<BN, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * HD / BN, (r.rows + RM - 1) / RM, 1);
  cfg.blockDim = dim3(kRThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = HD / BN;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, p);
}

}  // namespace

cudaError_t launch_recache(const RecacheLaunch& r, cudaStream_t st) {
  const int HD = r.H * r.D;
  if (HD % 256 == 0 && HD / 256 <= 8) return launch_recache_t<256, 4>(r, st);
  if (HD % 128 == 0 && HD / 128 <= 8) return launch_recache_t<128, 4>(r, st);
  if (HD % 64 == 0 && HD / 64 <= 8) return launch_recache_t<64, 4>(r, st);
  return cudaErrorInvalidValue;
}

}  // namespace kvc
