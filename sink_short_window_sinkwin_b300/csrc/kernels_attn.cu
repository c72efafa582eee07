// Sink + short-window chunk attention on tcgen05 tensor cores.
//
// LongLive summary page (yunpan.plus), 方法 §3 高效长推理: each new chunk's
// queries attend to the frame-sink tokens (first chunk, kept for good) joined
// with a short window of recent chunks; the cost is bounded by the window.
// Here: O = softmax(tau Q K^T) V per head over the visible cache rows, exact up
// to floating-point rounding (bf16 operands, fp32 accumulation and softmax).
//
// Work: an "item" is one head x two 128-row query tiles ("slots") that share
// every K/V tile; a "step" is one item x one 128-key K/V tile.  The kernel is
// persistent: G CTAs (at most one per SM) each take an equal contiguous share
// of all items' steps, so the last wave is as full as the first.  With fewer
// items than SMs (a short query chunk), G still covers every SM and an item is
// spread over several shares (split-KV).  An item cut by share boundaries is
// computed in pieces by neighbouring CTAs: every CTA g' > g whose share starts
// inside the item writes its piece's unnormalised O and (max, sum) rows to its
// workspace slot and raises a flag; CTA g (whose share ends inside the item, and
// which reaches that piece last) waits for those flags -- bounded waits, in a
// cooperative launch -- and merges the pieces.  Without a workspace the shares
// are whole items.
//
// Warp roles (320 threads; 512 with an FP4 cache):
//   warps 0-3  softmax of slot 0 (thread i owns query row i: TMEM lane i)
//   warps 4-7  softmax of slot 1
//   warp  8    TMA producer: Q per piece, then K/V tiles through a 2-stage ring
//   warp  9    TMEM allocator + single-thread tcgen05.mma issuer
//   FP4 cache only: warps 10-11 idle; warps 12-15 dequantise K/V tiles into
//   the smem ring.  512 threads launch at 128 registers each; the warpgroups
//   then split the register file with setmaxnreg: softmax 160 (the whole S row
//   of a thread in registers, one pass), decode 104, TMA/MMA 72 -- per SM
//   sub-partition 2 x 168 + 104 + 72 = 512, the launch's own share.
// TMEM (512 columns): S0 [0,128) O0 [128,256) S1 [256,384) O1 [384,512);
// P (bf16; f16 for FP4) overwrites the first 64 columns of S and feeds the
// P*V MMA from TMEM.  The running max only moves when it grows by more than
// 2^8 (log2 domain), so O is rescaled in TMEM rarely.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int BM = 128;  // query rows per slot
constexpr int BN = 128;  // keys per K/V tile
constexpr int kStages = 2;
constexpr int kSoftmaxWarps = 8;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDequantWarp0 = 12;  // FP4: warps 12-15 (warpgroup 3)
// FP4 warpgroup register split (setmaxnreg), per thread.  The block launches
// with kLaunch registers a thread (the launch-bounds maximum, which ptxas takes
// when setmaxnreg is present; the launcher checks it), and the new counts of
// all warps must add up to exactly that budget:
//   16 warps at 128: softmax 8 x 168 + TMA/MMA/idle 4 x 72 + decode 4 x 104 = 16 x 128
// and per SM sub-partition (one warp of each warpgroup) at most 512.  The bf16
// kernel (10 warps, no split) runs at the 168 its launch allows.
template <bool kFp4>
struct RegSplit;
template <>
struct RegSplit<false> {
  static constexpr int kThreads = 320;
};
template <>
struct RegSplit<true> {
  static constexpr int kThreads = 512, kLaunch = 128, kSoftmax = 168, kCtl = 72, kDecode = 104;
};
constexpr bool fp4_split_ok() {
  using R = RegSplit<true>;
  return 8 * R::kSoftmax + 4 * R::kCtl + 4 * R::kDecode == (R::kThreads / 32) * R::kLaunch &&
         2 * R::kSoftmax + R::kCtl + R::kDecode <= 512 &&
         // setmaxnreg takes multiples of 8 in [24, 256]; .inc may only raise a
         // warp's count and .dec only lower it (else: an illegal instruction)
         R::kSoftmax % 8 == 0 && R::kCtl % 8 == 0 && R::kDecode % 8 == 0 &&
         R::kSoftmax > R::kLaunch && R::kSoftmax <= 256 && R::kCtl < R::kLaunch && R::kCtl >= 24 &&
         R::kDecode < R::kLaunch && R::kDecode >= 24 && 65536 / R::kThreads / 8 * 8 == R::kLaunch;
}
static_assert(fp4_split_ok(), "register split");
template <bool kFp4>
constexpr int attn_threads() { return RegSplit<kFp4>::kThreads; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMinShareSteps = 8;          // K/V tiles per share at least (split-KV)

struct AttnParams {
  int32_t tq, H, D, S, nt;  // nt: K/V tiles of one item (over all segments)
  int32_t nseg;
  Seg seg[kMaxSeg];
  int32_t seg_t0[kMaxSeg];  // first tile of each segment
  float scale_log2;
  __nv_bfloat16* out;
  int32_t* dev_err;
  // schedule
  int32_t n_pairs;  // items per head
  int32_t NI;       // items
  int32_t G;        // CTAs
  int32_t split;    // 1: step-balanced shares with merges; 0: whole items
  int64_t NS;       // NI * nt
  float* ws_o;      // [G][2*BM][D]     unnormalised O of a share's first piece
  float2* ws_ml;    // [G][2*BM]        its (running max, running sum)
  unsigned long long* ws_flag;  // [G]  == epoch once slot g is written
  unsigned long long epoch;
  // FP4 cache
  const uint8_t* kc;
  const uint8_t* vc;
  const uint8_t* ks;
  const uint8_t* vs;
  const float* kg;
  const float* vg;
  int32_t Tc;
  int32_t seg_region[kMaxSeg];  // region of each segment (an FP4 segment lies in one)
};

template <int D>
struct __align__(1024) AttnSmem {
  static constexpr int DB = D / 64;  // 128-byte swizzle blocks along the head dim
  __nv_bfloat16 q[2][DB][BM * 64];
  __nv_bfloat16 k[kStages][DB][BN * 64];
  __nv_bfloat16 v[kStages][DB][BN * 64];
  uint64_t bar_q, bar_qempty;
  uint64_t bar_qcvt;       // FP4: Q rows converted to f16 (128 decode threads)
  uint64_t bar_qread;      // FP4: every softmax thread holds its row's Q scale
  float qinv[2][BM];       // FP4: per query row, 1 / its power-of-two f16 scale
  uint64_t bar_kfull[kStages], bar_kempty[kStages];
  uint64_t bar_vfull[kStages], bar_vempty[kStages];
  uint64_t bar_s[2], bar_p[2], bar_o[2], bar_ofree[2];
  uint64_t bar_part;  // all 256 partial rows of the share's first piece are written
  uint64_t bar_drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};

// FP4 cache: the decode warps' own prefetch ring of raw rows (codes and block
// scales), filled by per-thread cp.async copies.  Items alternate K and V of
// consecutive tiles and take slots 0, 1, 2, 0, ...; thread r owns row r of
// each slot.  A row's 16-byte code chunks are XOR-swizzled so that the eight
// threads of a quarter-warp read eight different bank groups.
template <int D>
struct __align__(16) RawRing {
  static constexpr int kSlots = 3;
  static constexpr int kNch = D / 32;                   // 16-byte code chunks of a row
  static constexpr int kShift = D == 128 ? 1 : 2;       // log2(rows per 128-byte line)
  uint8_t codes[kSlots][BN * (D / 2)];
  uint8_t scales[kSlots][BN * (D / 16)];
  __device__ __forceinline__ static int chunk_off(int r, int q) {
    return r * (D / 2) + ((q ^ ((r >> kShift) & (kNch - 1))) << 4);
  }
};

// K/V tile cursor over the visible segments.
struct KvCursor {
  int seg = 0, off = 0;
  __device__ __forceinline__ void seek(const AttnParams& p, int t) {
    seg = 0;
    while (seg + 1 < p.nseg && p.seg_t0[seg + 1] <= t) ++seg;
    off = (t - p.seg_t0[seg]) * BN;
  }
  __device__ __forceinline__ int row0(const AttnParams& p) const { return p.seg[seg].row0 + off; }
  __device__ __forceinline__ int valid(const AttnParams& p) const {
    return min(BN, p.seg[seg].rows - off);
  }
  __device__ __forceinline__ void next(const AttnParams& p) {  // wraps after the last tile
    off += BN;
    if (off >= p.seg[seg].rows) {
      off = 0;
      if (++seg >= p.nseg) seg = 0;
    }
  }
};

// A piece: item u, logical K/V tiles [t0, t1) of it.  Every role walks the same list.
// Softmax does not see key order, so a piece may visit its item's K/V tiles in
// any order.  Tiles are visited rotated so that at local step tau of every
// share the tile is about tau mod nt: CTAs working on the same head then read
// the same tile at about the same time and share it through L2.  All pieces of
// a split item take the rotation of the piece that ends it (its share starts
// with it), so together they still visit every tile once.
struct Piece {
  int u, t0, t1;
  int rot;  // physical tile of logical tile t is (t + rot) mod nt
};
// First step of share g, and the share holding step s (shares are never empty:
// G <= NS).
__device__ __forceinline__ int64_t share_begin(const AttnParams& p, int g) {
  return p.split ? (int64_t)g * p.NS / p.G : ((int64_t)g * p.NI / p.G) * p.nt;
}
__device__ __forceinline__ int share_of_step(const AttnParams& p, int64_t s) {
  return (int)(((s + 1) * p.G + p.NS - 1) / p.NS) - 1;
}
struct Share {
  int64_t b, s, e;
  __device__ __forceinline__ bool next(const AttnParams& p, Piece& pc) {
    if (s >= e) return false;
    pc.u = (int)(s / p.nt);
    pc.t0 = (int)(s - (int64_t)pc.u * p.nt);
    pc.t1 = (int)min((int64_t)p.nt, pc.t0 + (e - s));
    const int64_t ib = (int64_t)pc.u * p.nt;  // the item's first step
    if (ib >= b && ib + p.nt <= e) {
      pc.rot = (int)((s - b) % p.nt);  // a whole item
    } else {
      // the item's last piece starts the share holding its last step
      const int64_t tb = share_begin(p, share_of_step(p, ib + p.nt - 1));
      const int t0_tail = (int)(tb > ib ? tb - ib : 0);
      pc.rot = (p.nt - t0_tail) % p.nt;
    }
    s += pc.t1 - pc.t0;
    return true;
  }
  // first physical tile of the piece
  __device__ __forceinline__ static int first_tile(const AttnParams& p, const Piece& pc) {
    return (pc.t0 + pc.rot) % p.nt;
  }
};
__device__ __forceinline__ Share share_of(const AttnParams& p, int g) {
  const int64_t b = share_begin(p, g);
  return Share{b, b, g + 1 < p.G ? share_begin(p, g + 1) : (p.split ? p.NS : (int64_t)p.NI * p.nt)};
}

// ---------------------------------------------------------------------------
// FP4 tile dequantisation: thread i writes key row i of a K or V tile in the
// 128-byte-swizzled layout the MMA descriptors expect.
// ---------------------------------------------------------------------------
// One key row of FP4 codes and block scales, held in registers so the loads
// for the next tile can be in flight while this one is decoded.
template <int D>
struct RawRow {
  uint4 c[D / 32];      // 16 code bytes = 32 elements each
  uint32_t s[D / 64];   // 4 E4M3 scale bytes each
};
template <int D>
__device__ __forceinline__ void load_raw(RawRow<D>& raw, const uint8_t* codes, const uint8_t* scales,
                                         int grow, const AttnParams& p, int h) {
  const uint8_t* crow = codes + ((size_t)grow * p.H + h) * (D / 2);
  const uint8_t* srow = scales + ((size_t)grow * p.H + h) * (D / 16);
#pragma unroll
  for (int q = 0; q < D / 32; ++q) raw.c[q] = *reinterpret_cast<const uint4*>(crow + q * 16);
  if constexpr (D == 128) {
    const uint2 s8 = *reinterpret_cast<const uint2*>(srow);
    raw.s[0] = s8.x;
    raw.s[1] = s8.y;
  } else {
    raw.s[0] = *reinterpret_cast<const uint32_t*>(srow);
  }
}

// Exact partial decode e2m1(code) * e4m3(scale): at most 6 significant bits
// and a range of [2^-10, 2688], so the product is exact in f16 and in bf16.
// The fp32 tensor scale of the region is applied by the softmax instead (K: in
// the logit scale, V: folded into P), so no tile value is rounded here.
// Thread r writes key row r in the 128-byte-swizzled layout of the MMA operands.
template <int D, bool kHalfOut>
__device__ __forceinline__ void decode_row(__nv_bfloat16 (*dst)[BN * 64], int r, bool live,
                                           const RawRow<D>& raw) {
  uint8_t* base = reinterpret_cast<uint8_t*>(dst);
  if (!live) {
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const int db = c >> 3, ch = c & 7;
      *reinterpret_cast<uint4*>(base + db * (BN * 128) + r * 128 + ((ch ^ (r & 7)) << 4)) =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }
#pragma unroll
  for (int q16 = 0; q16 < D / 32; ++q16) {  // 16 code bytes = 32 elements = 2 blocks
    const uint32_t w[4] = {raw.c[q16].x, raw.c[q16].y, raw.c[q16].z, raw.c[q16].w};
    // the scales of blocks 2 q16 and 2 q16 + 1 (bytes 2 q16, 2 q16 + 1 of the row's scales)
    const uint32_t spair = e4m3x2_to_f16x2(raw.s[q16 >> 1] >> (16 * (q16 & 1)));
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // one 16-element block -> two 16-byte chunks
      const __half2 sp = *reinterpret_cast<const __half2*>(&spair);
      const __half2 s2 = half ? __high2half2(sp) : __low2half2(sp);
      uint32_t outw[8];
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {
        uint32_t h4[4];
        e2m1x8_to_f16x8(w[half * 2 + wi], h4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __half2 hv = __hmul2(*reinterpret_cast<const __half2*>(&h4[k]), s2);  // exact
          if constexpr (kHalfOut) {
            outw[wi * 4 + k] = *reinterpret_cast<const uint32_t*>(&hv);
          } else {
            const float2 fv = __half22float2(hv);
            outw[wi * 4 + k] = pack_bf16x2(fv.x, fv.y);  // exact
          }
        }
      }
      const int e0 = q16 * 32 + half * 16;  // first element of this block
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int c = (e0 >> 3) + part;  // 16-byte chunk index along D
        const int db = c >> 3, ch = c & 7;
        *reinterpret_cast<uint4*>(base + db * (BN * 128) + r * 128 + ((ch ^ (r & 7)) << 4)) =
            make_uint4(outw[part * 4 + 0], outw[part * 4 + 1], outw[part * 4 + 2],
                       outw[part * 4 + 3]);
      }
    }
  }
}

// FP4 cache: query row r of a Q tile (bf16, 128-byte swizzled) turned into
// f16 in place, times 2^k with k chosen so the row's largest magnitude lies in
// [2^14, 2^15): exact for every value that stays in the f16 normal range (a
// bf16 value has 8 significant bits), which covers all but values below
// 2^-28 of the row maximum.  Writes 2^-k (the factor the row's logits need).
template <int D>
__device__ __forceinline__ void convert_q_row(__nv_bfloat16 (*tile)[BM * 64], int r, float* inv_out) {
  uint8_t* base = reinterpret_cast<uint8_t*>(tile);
  auto at = [&](int c) -> uint4* {
    return reinterpret_cast<uint4*>(base + (c >> 3) * (BM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  };
  uint32_t mx = 0;  // largest |bf16| bit pattern of the row (monotone in the magnitude)
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 v = *at(c);
    const uint32_t w[4] = {v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu, v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu};
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = max(mx, max(w[e] & 0xFFFFu, w[e] >> 16));
  }
  int k = 0;  // zero, infinite or NaN rows keep scale 1
  if (mx != 0 && mx < 0x7F80u) {
    const int ex = (int)(mx >> 7) - 127;  // exponent field of the bf16 maximum, unbiased
    k = min(126, max(-126, 14 - ex));
  }
  const float scale = __uint_as_float((uint32_t)(127 + k) << 23);
  *inv_out = __uint_as_float((uint32_t)(127 - k) << 23);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    uint4* a = at(c);
    const uint4 v = *a;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_f16x2(__uint_as_float(w[e] << 16) * scale, __uint_as_float(w[e] & 0xFFFF0000u) * scale);
    *a = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu_u64(unsigned long long* a, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}

// kPre (FP4 caches only): K and V were decoded to f16 by a pass before the
// launch (K' = e2m1 * s exactly; V' = e2m1 * s * g_V / G rounded once to f16,
// G the V shift below).  The kernel then has the bf16 kernel's shape (no
// decode warps, no register split): the TMA producer loads f16 K/V tiles, and
// each softmax thread converts its own query row to f16 at the start of a
// piece, keeping the row's scale in a register.  Otherwise the arithmetic is
// the FP4 path's (f16 operands, K's tensor scale in the logit scale, G
// multiplied back in the normalisation); P is stored as plain f16.
template <int D, bool kFp4, bool kPre = false>
__global__ void __launch_bounds__(attn_threads<kFp4 && !kPre>(), 1)
    sinkwin_attn_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ AttnParams p) {
  using Smem = AttnSmem<D>;
  constexpr int DB = Smem::DB;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x;
  static_assert(kFp4 || !kPre, "pre-decoded tiles exist only for FP4 caches");
  constexpr bool kTmaKV = !kFp4 || kPre;  // K/V tiles arrive by TMA
  const uint32_t kvfull_count = kTmaKV ? 1u : 128u;

  if (threadIdx.x == 0) {
    mbar_init(&sm.bar_q, 1);
    mbar_init(&sm.bar_qcvt, kPre ? 2 * BM : BN);  // converted by the softmax / decode threads
    mbar_init(&sm.bar_qread, 2 * BM);
    mbar_init(&sm.bar_qempty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.bar_kfull[s], kvfull_count);
      mbar_init(&sm.bar_vfull[s], kvfull_count);
      mbar_init(&sm.bar_kempty[s], 1);
      mbar_init(&sm.bar_vempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.bar_s[s], 1);
      mbar_init(&sm.bar_o[s], 1);
      mbar_init(&sm.bar_p[s], BM);
      mbar_init(&sm.bar_ofree[s], BM);
    }
    mbar_init(&sm.bar_part, 2 * BM);
    mbar_init(&sm.bar_drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    if (kTmaKV) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const Watchdog wd{&sm.abort_flag, p.dev_err};

  if (warp >= kTmaWarp && warp < kTmaWarp + 4) {
    // warpgroup 2: TMA producer, MMA issuer (FP4: two idle warps)
    if constexpr (kFp4 && !kPre) setmaxnreg_dec<RegSplit<true>::kCtl>();
    if (warp == kTmaWarp) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        Share sh = share_of(p, g);
        Piece pc;
        uint32_t it = 0;  // K/V tiles of this CTA so far (ring position)
        int npc = 0, nk = 0, nv = 0;
        bool ok = true;
        while (ok && sh.next(p, pc)) {
          const int h = pc.u / p.n_pairs;
          const int m0 = (pc.u % p.n_pairs) * (2 * BM);
          const bool act1 = m0 + BM < p.tq;
          if (npc > 0 && !mbar_wait(&sm.bar_qempty, (npc - 1) & 1, wd)) break;
          // FP4: the next Q (and its row scales) only once the softmax threads
          // hold the previous piece's scales
          if (kFp4 && !kPre && npc > 0 && !mbar_wait(&sm.bar_qread, (npc - 1) & 1, wd)) break;
          mbar_expect_tx(&sm.bar_q, (act1 ? 2u : 1u) * DB * BM * 64 * 2);
          for (int s = 0; s < (act1 ? 2 : 1); ++s)
            for (int db = 0; db < DB; ++db)
              tma_load_3d(&sm.q[s][db][0], &tmQ, &sm.bar_q, db * 64, h, m0 + s * BM);
          ++npc;
          if (kTmaKV) {
            KvCursor cur;
            cur.seek(p, Share::first_tile(p, pc));
            const uint32_t tbytes = DB * BN * 64 * 2;
            for (int t = pc.t0; t < pc.t1; ++t, ++it) {
              const int st = it & 1, n = it >> 1;
              if (it >= kStages && !mbar_wait(&sm.bar_kempty[st], (n - 1) & 1, wd)) {
                ok = false;
                break;
              }
              mbar_expect_tx(&sm.bar_kfull[st], tbytes);
              for (int db = 0; db < DB; ++db)
                tma_load_3d(&sm.k[st][db][0], &tmK, &sm.bar_kfull[st], db * 64, h, cur.row0(p));
              ++nk;
              if (it >= kStages && !mbar_wait(&sm.bar_vempty[st], (n - 1) & 1, wd)) {
                ok = false;
                break;
              }
              mbar_expect_tx(&sm.bar_vfull[st], tbytes);
              for (int db = 0; db < DB; ++db)
                tma_load_3d(&sm.v[st][db][0], &tmV, &sm.bar_vfull[st], db * 64, h, cur.row0(p));
              ++nv;
              cur.next(p);
            }
          }
        }
        // teardown after an abort: every copy this thread started must land
        // before the CTA exits (the consumers waited for the rest)
        if (sm.abort_flag) {
          for (int st = 0; st < kStages; ++st) {
            const int ck = nk > st ? (nk - st + 1) / 2 : 0;  // uses of stage st
            const int cv = nv > st ? (nv - st + 1) / 2 : 0;
            if (ck) mbar_drain(&sm.bar_kfull[st], (ck - 1) & 1);
            if (cv) mbar_drain(&sm.bar_vfull[st], (cv - 1) & 1);
          }
          if (npc) mbar_drain(&sm.bar_q, (npc - 1) & 1);
        }
      }
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        // FP4 cache: Q (converted in place) and K' are f16
        constexpr uint32_t idesc_qk =
            kFp4 ? idesc_f16_f32(BM, BN, false, false) : idesc_bf16_f32(BM, BN, false, false);
        // FP4 cache: P (scaled by the V tensor scale) and V' are f16
        constexpr uint32_t idesc_pv =
            kFp4 ? idesc_f16_f32(BM, D, false, true) : idesc_bf16_f32(BM, D, false, true);
        const uint32_t tS[2] = {tmem, tmem + 256};
        const uint32_t tO[2] = {tmem + 128, tmem + 384};
        // Descriptors: one base per operand, plus the slot / stage / k-step
        // byte offset / 16.  FP4 (72-register control warps): added right
        // before each MMA with an opaque add, so the compiler keeps no table
        // of precomputed descriptors alive.
        const uint64_t qdesc = sdesc_sw128(smem_u32(&sm.q[0][0][0]), 0, 1024);
        const uint64_t kdesc = sdesc_sw128(smem_u32(&sm.k[0][0][0]), 0, 1024);
        const uint64_t vdesc = sdesc_sw128(smem_u32(&sm.v[0][0][0]), BN * 64 * 2, 1024);
        constexpr uint32_t kDb16 = BM * 64 * 2 / 16;          // one 64-column block
        constexpr uint32_t kQSlot16 = DB * kDb16;             // one query tile
        constexpr uint32_t kKvStage16 = DB * BN * 64 * 2 / 16;  // one K or V stage
        auto qk = [&](int slot, int st) {
          const uint64_t qa = qdesc + slot * kQSlot16, kb = kdesc + st * kKvStage16;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kDb16 + (kk & 3) * 2;  // + 32 bytes per k-step
            if constexpr (kFp4)
              mma_bf16_ss(tS[slot], add_opaque(qa, off), add_opaque(kb, off), idesc_qk, kk > 0);
            else
              mma_bf16_ss(tS[slot], qa + off, kb + off, idesc_qk, kk > 0);
          }
        };
        auto pv = [&](int slot, int st, bool acc) {
          const uint64_t vb = vdesc + st * kKvStage16;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bd = kFp4 ? add_opaque(vb, kk * (2048 / 16)) : vb + kk * (2048 / 16);
            mma_bf16_ts(tO[slot], tS[slot] + kk * 8, bd, idesc_pv, (acc || kk > 0) ? 1u : 0u);
          }
        };
        Share sh = share_of(p, g);
        Piece pc;
        uint32_t it = 0;
        int npc = 0;
        int np[2] = {0, 0}, nof[2] = {0, 0};
        bool pend[2] = {false, false};  // an epilogue of this slot may still read O
        bool ok = true;
        while (ok && sh.next(p, pc)) {
          const int m0 = (pc.u % p.n_pairs) * (2 * BM);
          const bool act1 = m0 + BM < p.tq;
          const int n = pc.t1 - pc.t0;
          const int st0 = it & 1;
          ok = mbar_wait(kFp4 ? &sm.bar_qcvt : &sm.bar_q, npc & 1, wd) &&
               mbar_wait(&sm.bar_kfull[st0], (it >> 1) & 1, wd);
          if (!ok) break;
          tc_fence_after();
          qk(0, st0);
          mma_commit(&sm.bar_s[0]);
          if (act1) {
            qk(1, st0);
            mma_commit(&sm.bar_s[1]);
          }
          mma_commit(&sm.bar_kempty[st0]);
          if (n == 1) mma_commit(&sm.bar_qempty);
          for (int i = 0; i < n && ok; ++i) {
            const uint32_t ti = it + i;
            const int st = ti & 1, ph = (ti >> 1) & 1;
            const int nst = (ti + 1) & 1, nph = ((ti + 1) >> 1) & 1;
            const bool more = i + 1 < n;
            ok = mbar_wait(&sm.bar_p[0], np[0] & 1, wd) && mbar_wait(&sm.bar_vfull[st], ph, wd);
            ++np[0];
            if (ok && i == 0 && pend[0]) {
              ok = mbar_wait(&sm.bar_ofree[0], nof[0] & 1, wd);
              ++nof[0];
              pend[0] = false;
            }
            if (!ok) break;
            tc_fence_after();
            pv(0, st, i > 0);
            if (more) {
              ok = mbar_wait(&sm.bar_kfull[nst], nph, wd);
              if (!ok) break;
              tc_fence_after();
              qk(0, nst);
              mma_commit(&sm.bar_s[0]);
            } else {
              mma_commit(&sm.bar_o[0]);
            }
            if (act1) {
              ok = mbar_wait(&sm.bar_p[1], np[1] & 1, wd);
              ++np[1];
              if (ok && i == 0 && pend[1]) {
                ok = mbar_wait(&sm.bar_ofree[1], nof[1] & 1, wd);
                ++nof[1];
                pend[1] = false;
              }
              if (!ok) break;
              tc_fence_after();
              pv(1, st, i > 0);
              mma_commit(&sm.bar_vempty[st]);
              if (more) {
                qk(1, nst);
                mma_commit(&sm.bar_s[1]);
              } else {
                mma_commit(&sm.bar_o[1]);
              }
            } else {
              mma_commit(&sm.bar_vempty[st]);
            }
            if (more) mma_commit(&sm.bar_kempty[nst]);
            if (i + 2 == n) mma_commit(&sm.bar_qempty);  // the piece's last QK went out above
          }
          it += n;
          ++npc;
          pend[0] = true;
          if (act1) pend[1] = true;
        }
        // drain: every MMA issued above completes before TMEM is released
        mma_commit(&sm.bar_drain);
        mbar_drain(&sm.bar_drain, 0);
      }
    }
  } else if (kFp4 && !kPre && warp >= kDequantWarp0) {
    if constexpr (kFp4 && !kPre) setmaxnreg_dec<RegSplit<true>::kDecode>();
    // ------------------------------------------------------------ FP4 dequant producer
    const int r = threadIdx.x - kDequantWarp0 * 32;  // key row within the tile
    RawRing<D>& raw = *reinterpret_cast<RawRing<D>*>(reinterpret_cast<uint8_t*>(&sm) + sizeof(Smem));
    Share sh = share_of(p, g);
    Piece pc;
    uint32_t it = 0;
    int npc = 0;
    bool ok = true;
    while (ok && sh.next(p, pc)) {
      const int h = pc.u / p.n_pairs;
      // Q of the piece, once its TMA load landed: thread r turns query row r of
      // each live slot into f16 in place, scaled by a power of two that puts
      // the row's largest magnitude in [2^14, 2^15) (exact: a bf16 value has 8
      // significant bits), and hands 1 / scale to that row's softmax thread
      {
        const int m0 = (pc.u % p.n_pairs) * (2 * BM);
        const int nslot = m0 + BM < p.tq ? 2 : 1;
        if (!mbar_wait(&sm.bar_q, npc & 1, wd)) break;
        for (int sl = 0; sl < nslot; ++sl) convert_q_row<D>(sm.q[sl], r, &sm.qinv[sl][r]);
        fence_proxy_async_smem();
        mbar_arrive(&sm.bar_qcvt);
        ++npc;
      }
      // Items j = 0, 1, ... of the piece are K (even j) and V (odd j) of its
      // tiles in turn; item j's raw row is copied into slot j % 3 three items
      // ahead of its decode, so it has had a tile and a half to land.
      KvCursor cur, icur;  // tile being decoded / tile of the next item to copy
      cur.seek(p, Share::first_tile(p, pc));
      icur = cur;
      const int nitems = 2 * (pc.t1 - pc.t0);
      int issued = 0, islot = 0;
      auto issue = [&]() {
        const bool isv = issued & 1;
        if (r < icur.valid(p)) {
          const size_t row = (size_t)(icur.row0(p) + r) * p.H + h;
          const uint8_t* cs = (isv ? p.vc : p.kc) + row * (D / 2);
          const uint8_t* ss = (isv ? p.vs : p.ks) + row * (D / 16);
#pragma unroll
          for (int q = 0; q < RawRing<D>::kNch; ++q) cp_async_16(raw.codes[islot] + RawRing<D>::chunk_off(r, q), cs + 16 * q);
          if constexpr (D == 128) cp_async_8(raw.scales[islot] + r * 8, ss);
          else cp_async_4(raw.scales[islot] + r * 4, ss);
        }
        cp_async_commit();  // one group per item, empty for a row past the tile's end
        if (isv) icur.next(p);
        ++issued;
        islot = islot == 2 ? 0 : islot + 1;
      };
      for (int k = 0; k < 3 && k < nitems; ++k) issue();
      for (int j = 0; j < nitems; ++j) {
        const bool isv = j & 1;
        const uint32_t ti = it + (j >> 1);
        const int st = ti & 1, n = ti >> 1;
        const int pending = issued - 1 - j;  // items copied after this one
        if (pending >= 2) cp_async_wait<2>();
        else if (pending == 1) cp_async_wait<1>();
        else cp_async_wait<0>();
        uint64_t* empty = isv ? &sm.bar_vempty[st] : &sm.bar_kempty[st];
        if (ti >= kStages && !mbar_wait(empty, (n - 1) & 1, wd)) {
          ok = false;
          break;
        }
        const bool live = r < cur.valid(p);
        RawRow<D> rw;
        if (live) {
          const int sl = j % 3;
#pragma unroll
          for (int q = 0; q < RawRing<D>::kNch; ++q)
            rw.c[q] = *reinterpret_cast<const uint4*>(raw.codes[sl] + RawRing<D>::chunk_off(r, q));
          if constexpr (D == 128) {
            const uint2 s8 = *reinterpret_cast<const uint2*>(raw.scales[sl] + r * 8);
            rw.s[0] = s8.x;
            rw.s[1] = s8.y;
          } else {
            rw.s[0] = *reinterpret_cast<const uint32_t*>(raw.scales[sl] + r * 4);
          }
        }
        decode_row<D, true>(isv ? sm.v[st] : sm.k[st], r, live, rw);
        fence_proxy_async_smem();
        mbar_arrive(isv ? &sm.bar_vfull[st] : &sm.bar_kfull[st]);
        if (isv) cur.next(p);
        if (issued < nitems) issue();  // into the slot just read
      }
      it += pc.t1 - pc.t0;
    }
    cp_async_wait<0>();  // no copy into this CTA's shared memory outlives it
  } else if (warp < kSoftmaxWarps) {
    if constexpr (kFp4 && !kPre) setmaxnreg_inc<RegSplit<true>::kSoftmax>();
    // ------------------------------------------------------------ softmax
    const int slot = warp >> 2;
    const int wq = warp & 3;
    const int row = threadIdx.x & (BM - 1);
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + slot * 256 + lane_off;
    const uint32_t tO = tS + 128;
    const float c = p.scale_log2;
    Share sh = share_of(p, g);
    Piece pc;
    uint32_t it = 0;
    int ns = 0, no = 0;
    [[maybe_unused]] int nq = 0;  // FP4: converted-Q phases waited
    bool ok = true;
    int kv_region = -1;  // FP4: region whose tensor scales are held below
    float kv_kg = 0.0f, kv_vg = 0.0f;
    // FP4: P is stored as f16 times the region's V tensor scale, and P itself
    // reaches 2^8 under a held running max.  Every region's V scale is divided
    // by one power of two G >= the largest visible one, so that product lies
    // in [0, 2^8] whatever the magnitude of V (no f16 overflow for large V, no
    // subnormal P for small V); G returns in the final normalisation (exact).
    [[maybe_unused]] float v_shift = 1.0f, inv_v_shift = 1.0f;
    if constexpr (kFp4) {
      float gmax = 0.0f;
      for (int s2 = 0; s2 < p.nseg; ++s2) gmax = fmaxf(gmax, __ldg(p.vg + p.seg_region[s2]));
      if (gmax > 0.0f && gmax < 1.0e36f) {  // a tensor scale is at most 3.39e38 / 2688
        const int e = max(-125, ((int)((__float_as_uint(gmax) >> 23) & 0xFFu)) - 126);  // gmax < 2^e
        v_shift = __uint_as_float((uint32_t)(127 + e) << 23);
        inv_v_shift = __uint_as_float((uint32_t)(127 - e) << 23);
      }
    }
    while (ok && sh.next(p, pc)) {
      const int h = pc.u / p.n_pairs;
      const int m0 = (pc.u % p.n_pairs) * (2 * BM);
      const bool act1 = m0 + BM < p.tq;
      const int n = pc.t1 - pc.t0;
      const uint32_t it0 = it;
      it += n;
      [[maybe_unused]] float qinv = 1.0f;
      if constexpr (kPre) {
        // this thread's query row of its slot, once the piece's Q landed: to
        // f16 in place with its power-of-two scale (both slots arrive, so the
        // count holds when slot 1 is idle)
        const bool got = mbar_wait(&sm.bar_q, nq & 1, wd);
        ++nq;
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        if (slot == 0 || act1) convert_q_row<D>(sm.q[slot], row, &qinv);
        fence_proxy_async_smem();
        mbar_arrive(&sm.bar_qcvt);
      } else if constexpr (kFp4) {
        // every piece converts Q once (both slots' rows in the same phase)
        const bool got = mbar_wait(&sm.bar_qcvt, nq & 1, wd);
        ++nq;
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        qinv = sm.qinv[slot][row];
        mbar_arrive(&sm.bar_qread);  // the decode warps may overwrite qinv from now on
      }
      if (slot == 1 && !act1) continue;
      float m_ref = -INFINITY, l = 0.0f;
      // Keep a stale running max unless it grew by more than 2^8.  decide()
      // moves the reference and returns the factor for O (1 when unchanged);
      // apply() rescales O in TMEM, warp-collectively, once P is written (the
      // P*V MMA of this tile only starts after this warp's P arrival), so the
      // S row and the O chunk are never live in registers together.
      auto decide = [&](int i, float mx_scaled) -> float {
        const float m_new = fmaxf(m_ref, mx_scaled);
        if (i == 0) {
          m_ref = m_new;
          return 1.0f;
        }
        const bool need = m_new > m_ref + kRescaleThreshold;
        const float alpha = need ? ex2_approx(m_ref - m_new) : 1.0f;
        if (need) m_ref = m_new;
        l *= alpha;
        return alpha;
      };
      auto apply = [&](float alpha) {
        if (!__any_sync(0xffffffffu, alpha != 1.0f)) return;
#pragma unroll 1
        for (int j = 0; j < D / 32; ++j) {
          uint32_t o[32];
          tmem_ld32(tO + j * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + j * 32, o);
        }
      };
      KvCursor cur;
      cur.seek(p, Share::first_tile(p, pc));
      for (int i = 0; i < n; ++i) {
        // warp-uniform exit: the tcgen05.ld/st below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.bar_s[slot], ns & 1, wd))) {
          ok = false;
          break;
        }
        ++ns;
        tc_fence_after();
        const int valid = cur.valid(p);
        if (kTmaKV && slot == 0 && valid < BN) {
          // key rows past the segment end may hold anything (NaN scrub,
          // never-written memory): zero them in the V stage before P*V
          const uint32_t ti = it0 + i;
          const int st = ti & 1;
          if (!__all_sync(0xffffffffu, mbar_wait(&sm.bar_vfull[st], (ti >> 1) & 1, wd))) {
            ok = false;
            break;
          }
          uint8_t* vb = reinterpret_cast<uint8_t*>(&sm.v[st][0][0]);
          for (int idx = row; idx < (BN - valid) * 8 * DB; idx += BM) {
            const int rr = valid + idx / (8 * DB);
            const int rem = idx % (8 * DB);
            *reinterpret_cast<uint4*>(vb + (rem >> 3) * (BN * 128) + rr * 128 + ((rem & 7) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        // one pass: the whole S row lives in registers.  FP4: the tile lies in
        // one region; its K tensor scale joins the logit scale and its V
        // tensor scale multiplies P (stored as f16 for the f16 P*V MMA)
        float cg = c;
        [[maybe_unused]] float gv = 1.0f;
        if constexpr (kFp4) {
          const int region = p.seg_region[cur.seg];
          if (region != kv_region) {  // consecutive tiles mostly share a region
            kv_region = region;
            kv_kg = __ldg(p.kg + region);
            kv_vg = __ldg(p.vg + region) * inv_v_shift;
          }
          cg = c * kv_kg * qinv;
          gv = kv_vg;
        }
        uint32_t sr[BN];
#pragma unroll
        for (int j = 0; j < BN / 32; ++j)
          tmem_ld32(tS + j * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[j * 32]));
        tmem_ld_wait();
        if (valid < BN) {  // ragged tile (warp-uniform): keys past the end do not count
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (j >= valid) sr[j] = __float_as_uint(-INFINITY);
        }
        // row max: four independent 3-input max chains
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < BN; j += 8)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            m4[q] = fmax3(m4[q], __uint_as_float(sr[j + 2 * q]), __uint_as_float(sr[j + 2 * q + 1]));
        const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
        const float alpha = decide(i, mx * cg);
        // p = 2^(s*cg - m): one packed FFMA per pair, packed row sum; pairs
        // (bf16, or f16 times the V tensor scale) written back over the
        // consumed S columns
        const uint64_t c2 = f32x2(cg, cg), n2 = f32x2(-m_ref, -m_ref);
        [[maybe_unused]] const uint64_t g2 = f32x2(gv, gv);
        uint64_t acc2 = f32x2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const uint64_t y2 = ffma2(f32x2(__uint_as_float(sr[j * 64 + 2 * e]),
                                            __uint_as_float(sr[j * 64 + 2 * e + 1])), c2, n2);
            float y0, y1;
            f32x2_split(y2, y0, y1);
            const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
            const uint64_t p2 = f32x2(p0, p1);
            acc2 = fadd2(acc2, p2);
            if constexpr (kPre) {
              pk[e] = pack_f16x2(p0, p1);  // the V tensor scale is in the decoded V
            } else if constexpr (kFp4) {
              float q0, q1;
              f32x2_split(fmul2(p2, g2), q0, q1);
              pk[e] = pack_f16x2(q0, q1);
            } else {
              pk[e] = pack_bf16x2(p0, p1);
            }
          }
          tmem_st32(tS + j * 32, pk);
        }
        float s0, s1;
        f32x2_split(acc2, s0, s1);
        l += s0 + s1;
        apply(alpha);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.bar_p[slot]);
        cur.next(p);
      }
      if (!ok) break;
      // ---- epilogue of the piece: O of its final tile is complete
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.bar_o[slot], no & 1, wd))) {
        ok = false;
        break;
      }
      ++no;
      tc_fence_after();
      const int prow = slot * BM + row;  // row within the item's 256
      const int grow = m0 + prow;
      const bool head = pc.t0 == 0, tail = pc.t1 == p.nt;
      // head && !tail: the item's later pieces are in the workspace slots of
      // shares g+1 .. gt; wait for each, then merge all of them
      int gt = g;
      float mm = m_ref, inv_l = 0.0f;
      if (head && !tail) {
        gt = share_of_step(p, (int64_t)(pc.u + 1) * p.nt - 1);
        bool got = true;
        for (int q = g + 1; q <= gt && got; ++q) {
          const unsigned long long* f = p.ws_flag + q;
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_gpu_u64(f) != p.epoch) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              sm.abort_flag = 1;
              if (p.dev_err) atomicCAS(p.dev_err, DEVERR_NONE, DEVERR_TIMEOUT);
              got = false;
              break;
            }
          }
        }
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        for (int q = g + 1; q <= gt; ++q) mm = fmaxf(mm, p.ws_ml[(size_t)q * 2 * BM + prow].x);
        float lt = l * ex2_approx(m_ref - mm);
        for (int q = g + 1; q <= gt; ++q) {
          const float2 ml = p.ws_ml[(size_t)q * 2 * BM + prow];
          lt += ml.y * ex2_approx(ml.x - mm);
        }
        inv_l = 1.0f / lt;
      } else if (head) {
        inv_l = 1.0f / l;
      }
      const float fa = ex2_approx(m_ref - mm);  // 1 unless merging
      if constexpr (kFp4) inv_l *= v_shift;
      float* wsw = nullptr;  // this piece handed to the CTA that started the item (!head)
      if (!head) {
        wsw = p.ws_o + ((size_t)g * 2 * BM + prow) * D;
        p.ws_ml[(size_t)g * 2 * BM + prow] = make_float2(m_ref, l);
      }
      __nv_bfloat16* dst = p.out + ((size_t)grow * p.H + h) * D;
#pragma unroll 1
      for (int j = 0; j < D / 32; ++j) {
        uint32_t o[32];
        tmem_ld32(tO + j * 32, o);
        tmem_ld_wait();
        if (!head) {  // partial: unnormalised fp32 for the merging CTA
          float4* w4 = reinterpret_cast<float4*>(wsw + j * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w4[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
          continue;
        }
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(o[e]) * fa;
#pragma unroll 1
        for (int q = g + 1; q <= gt; ++q) {
          const float fb = ex2_approx(p.ws_ml[(size_t)q * 2 * BM + prow].x - mm);
          const float4* r4 = reinterpret_cast<const float4*>(p.ws_o + ((size_t)q * 2 * BM + prow) * D + j * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 b = r4[e];
            x[4 * e + 0] = fmaf(b.x, fb, x[4 * e + 0]);
            x[4 * e + 1] = fmaf(b.y, fb, x[4 * e + 1]);
            x[4 * e + 2] = fmaf(b.z, fb, x[4 * e + 2]);
            x[4 * e + 3] = fmaf(b.w, fb, x[4 * e + 3]);
          }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] *= inv_l;
        if (grow < p.tq) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = pack_bf16x2(x[e + 0], x[e + 1]);
            w.y = pack_bf16x2(x[e + 2], x[e + 3]);
            w.z = pack_bf16x2(x[e + 4], x[e + 5]);
            w.w = pack_bf16x2(x[e + 6], x[e + 7]);
            *reinterpret_cast<uint4*>(dst + j * 32 + e) = w;
          }
        }
      }
      if (!head) {
        // publish slot g once every row of both slots is written (a share's
        // first piece is the only one that can end an item it did not start,
        // so bar_part completes at most once per launch: parity 0)
        mbar_arrive(&sm.bar_part);
        if (threadIdx.x == 0) {
          if (!act1) mbar_arrive_count(&sm.bar_part, BM);  // slot 1 has no rows here
          if (mbar_wait(&sm.bar_part, 0, wd)) {
            __threadfence();
            st_release_gpu_u64(p.ws_flag + g, p.epoch);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.bar_ofree[slot]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

template <int D, bool kFp4, bool kPre = false>
cudaError_t launch_attn_t(const AttnLaunch& a, cudaStream_t st) {
  CUtensorMap tq{}, tk{}, tv{};
  const uint64_t rs = (uint64_t)a.H * a.D * 2;  // bytes per token row
  if (!encode_tmap_3d_bf16(&tq, a.q, a.D, a.H, a.tq, (uint64_t)a.D * 2, rs, 64, 1, BM, true))
    return cudaErrorInvalidValue;
  if (!kFp4 || kPre) {
    // bf16 cache, or the f16 tiles of a pre-decoded FP4 cache (2-byte
    // elements either way; the map's type only sizes them)
    const void* kb = kPre ? a.k16 : a.k;
    const void* vb = kPre ? a.v16 : a.v;
    if (!encode_tmap_3d_bf16(&tk, kb, a.D, a.H, a.S, (uint64_t)a.D * 2, rs, 64, 1, BN, true))
      return cudaErrorInvalidValue;
    if (!encode_tmap_3d_bf16(&tv, vb, a.D, a.H, a.S, (uint64_t)a.D * 2, rs, 64, 1, BN, true))
      return cudaErrorInvalidValue;
  } else {
    tk = tq;  // unused
    tv = tq;
  }
  AttnParams p{};
  p.tq = a.tq;
  p.H = a.H;
  p.D = a.D;
  p.S = a.S;
  p.nseg = a.nseg;
  int nt = 0;
  for (int i = 0; i < a.nseg; ++i) {
    p.seg[i] = a.seg[i];
    p.seg_t0[i] = nt;
    nt += (a.seg[i].rows + BN - 1) / BN;
  }
  p.nt = nt;
  p.scale_log2 = a.scale_log2;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.dev_err = a.dev_err;
  p.kc = static_cast<const uint8_t*>(a.k);
  p.vc = static_cast<const uint8_t*>(a.v);
  p.ks = a.k_scale;
  p.vs = a.v_scale;
  p.kg = a.k_gscale;
  p.vg = a.v_gscale;
  p.Tc = a.chunk_tokens;
  for (int i = 0; i < a.nseg; ++i) p.seg_region[i] = p.Tc > 0 ? a.seg[i].row0 / p.Tc : 0;
  // schedule: at most one CTA per SM.  With the workspace, shares are
  // step-balanced and an item may spread over several shares (at least
  // kMinShareSteps K/V tiles each); without it every CTA takes whole items.
  const int nsm = sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  p.n_pairs = (a.tq + 2 * BM - 1) / (2 * BM);
  p.NI = p.n_pairs * a.H;
  p.NS = (int64_t)p.NI * nt;
  const size_t need = attn_workspace_bytes(a.D, nsm);
  const bool have_ws = a.ws != nullptr && a.ws_bytes >= need;
  int64_t G = have_ws ? p.NS / kMinShareSteps : p.NI;
  if (G > nsm) G = nsm;
  if (G > p.NS) G = p.NS;
  if (G < 1) G = 1;
  p.G = (int32_t)G;
  p.split = (have_ws && p.G > 1 && (p.G > p.NI || p.NI % p.G != 0)) ? 1 : 0;
  if (!p.split && p.G > p.NI) p.G = p.NI;
  if (p.split) {
    uint8_t* w = static_cast<uint8_t*>(a.ws);
    p.ws_o = reinterpret_cast<float*>(w);
    p.ws_ml = reinterpret_cast<float2*>(w + (size_t)nsm * 2 * BM * a.D * 4);
    p.ws_flag = reinterpret_cast<unsigned long long*>(w + (size_t)nsm * 2 * BM * (a.D * 4 + 8));
    static std::atomic<unsigned long long> epochs{0};
    p.epoch = epochs.fetch_add(1) + 1;
  }
  // one CTA per SM: a second resident CTA would wait in tcgen05.alloc for the
  // 512 TMEM columns the first one holds
  size_t smem = sizeof(AttnSmem<D>) + (kFp4 && !kPre ? sizeof(RawRing<D>) : 0) + 1024;
  if (smem < 120 * 1024) smem = 120 * 1024;
  auto kern = sinkwin_attn_kernel<D, kFp4, kPre>;
  static bool smem_set[64] = {};  // one per instantiation of this launcher
  cudaError_t e = set_smem_once(kern, smem, smem_set);
  if (e != cudaSuccess) return e;
  if constexpr (kFp4 && !kPre) {
    // the setmaxnreg split hands out exactly the registers the block launches
    // with: refuse to launch if the compiled kernel's count differs (an
    // increase that the launch cannot cover would wait forever)
    static int regs_ok[64] = {};  // per device: 0 unknown, 1 ok, -1 mismatch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (regs_ok[dev] == 0) {
      cudaFuncAttributes fa{};
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      regs_ok[dev] = fa.numRegs == RegSplit<true>::kLaunch ? 1 : -1;
    }
    if (regs_ok[dev] < 0) return cudaErrorInvalidConfiguration;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.G, 1, 1);
  cfg.blockDim = dim3(attn_threads<kFp4 && !kPre>(), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // a merge waits on a neighbouring CTA: all CTAs must be resident together
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.split ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace

size_t attn_workspace_bytes(int D, int ctas) {
  return (size_t)ctas * 2 * BM * ((size_t)D * 4 + 8) + (size_t)ctas * 8;
}

int attn_sm_count() { return sm_count(); }

cudaError_t launch_sinkwin_attn(const AttnLaunch& a, cudaStream_t st) {
  const bool pre = a.fp4 && a.k16 && a.v16;
  if (a.D == 128)
    return !a.fp4 ? launch_attn_t<128, false>(a, st)
                  : (pre ? launch_attn_t<128, true, true>(a, st) : launch_attn_t<128, true>(a, st));
  if (a.D == 64)
    return !a.fp4 ? launch_attn_t<64, false>(a, st)
                  : (pre ? launch_attn_t<64, true, true>(a, st) : launch_attn_t<64, true>(a, st));
  return cudaErrorInvalidValue;
}

}  // namespace kvc
