// C ABI: argument validation, the host-side slot map of the sink + window ring,
// and the kernel launches.  Every entry point validates first, launches second,
// and only then commits the new slot-map state, so an error changes nothing.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "kvc.h"
#include "ptx.cuh"

namespace kvc {

// ---------------------------------------------------------------------------
// tensor maps (cuTensorMapEncodeTiled, resolved through the runtime so the
// library does not link the driver library directly)
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                         uint32_t box1, uint32_t box2, bool swizzle128) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                         uint64_t stride1_bytes, uint32_t box0, uint32_t box1, bool swizzle128) {
  return encode_tmap_2d_bf16_sw(m, base, d0, d1, stride1_bytes, box0, box1, swizzle128 ? 128 : 0);
}

static bool encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0,
                           uint64_t d1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                           int swizzle_bytes) {
  CUtensorMapSwizzle sw;
  switch (swizzle_bytes) {
    case 0: sw = CU_TENSOR_MAP_SWIZZLE_NONE; break;
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return false;
  }
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {stride1_bytes};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_2d_bf16_sw(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                            uint64_t stride1_bytes, uint32_t box0, uint32_t box1, int swizzle_bytes) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, d0, d1, stride1_bytes, box0, box1,
                        swizzle_bytes);
}

bool encode_tmap_2d_u8(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
                       uint64_t stride1_bytes, uint32_t box0, uint32_t box1, int swizzle_bytes) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, d0, d1, stride1_bytes, box0, box1,
                        swizzle_bytes);
}

// ---------------------------------------------------------------------------
// watchdog self-test: one CTA waits for a phase nothing completes
// ---------------------------------------------------------------------------
__global__ void watchdog_selftest_kernel(int32_t* dev_ws, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Watchdog wd{&abort_flag, dev_ws};
    mbar_wait(&bar, 0, wd, limit_ns);  // no arrive ever happens: runs out
  }
}

cudaError_t launch_watchdog_selftest(int32_t* dev_ws, int32_t limit_us, cudaStream_t st) {
  watchdog_selftest_kernel<<<1, 32, 0, st>>>(dev_ws, (uint64_t)limit_us * 1000ull);
  return cudaGetLastError();
}

}  // namespace kvc

using namespace kvc;

namespace {

constexpr int32_t kMaxRows = 1 << 30;
constexpr int32_t kMaxHeads = 1 << 16;

int64_t chunk_tokens(const kvc_cache* c) { return (int64_t)c->tokens_per_frame * c->chunk_frames; }
int64_t cache_rows(const kvc_cache* c) { return (1 + (int64_t)c->window_chunks) * chunk_tokens(c); }

bool geometry_ok(const kvc_cache* c) {
  if (!c) return false;
  if (c->heads < 1 || c->head_dim < 16 || c->head_dim % 16 != 0 || c->head_dim > 256) return false;
  if (c->tokens_per_frame < 1 || c->chunk_frames < 1) return false;
  if (c->window_chunks < 1 || c->window_chunks > KVC_MAX_WINDOW) return false;
  if (c->dtype != KVC_BF16 && c->dtype != KVC_FP4) return false;
  // bound each factor before the products below, so none of them can overflow
  if (c->heads > kMaxHeads || chunk_tokens(c) > kMaxRows) return false;
  const int64_t S = cache_rows(c);
  if (S > kMaxRows) return false;
  if (S * c->heads * (int64_t)c->head_dim > (int64_t(1) << 40)) return false;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ready(const kvc_cache* c) { return c && c->init_magic == KVC_INIT_MAGIC && geometry_ok(c); }

// Region of a chunk: 0 for the sink (chunk 0, or a shot's first chunk once it
// is the sink), else its ring slot.
int32_t region_of(const kvc_cache* c, int64_t chunk) {
  if (chunk == 0 || chunk == c->chunk_of_region[0]) return 0;
  return 1 + (int32_t)((chunk - 1) % c->window_chunks);
}

// RoPE frame position of a chunk's first frame, `shot` boundaries in.
int64_t frame0_of(const kvc_cache* c, int64_t chunk, int32_t shot) {
  return chunk * c->chunk_frames + (int64_t)shot * c->rope_offset_frames;
}

int64_t oldest_window_chunk(const kvc_cache* c) {
  int64_t m = -1;
  for (int r = 1; r <= c->window_chunks; ++r) {
    const int64_t x = c->chunk_of_region[r];
    if (x >= 0 && (m < 0 || x < m)) m = x;
  }
  return m;
}

// present chunks in logical order: sink first, then window chunks ascending
int present_chunks(const kvc_cache* c, int64_t* out) {
  int n = 0;
  if (c->chunk_of_region[0] >= 0) out[n++] = c->chunk_of_region[0];
  int64_t last = -1;
  while (true) {
    int64_t best = -1;
    for (int r = 1; r <= c->window_chunks; ++r) {
      const int64_t x = c->chunk_of_region[r];
      if (x > last && (best < 0 || x < best)) best = x;
    }
    if (best < 0) break;
    out[n++] = best;
    last = best;
  }
  return n;
}

int32_t cuda_status(cudaError_t e) { return e == cudaSuccess ? KVC_OK : KVC_ECUDA; }

size_t row_bytes(const kvc_cache* c, int which) {
  const size_t hd = (size_t)c->heads * c->head_dim;
  switch (which) {
    case 0:
    case 1:
      return c->dtype == KVC_BF16 ? hd * 2 : hd / 2;
    case 2:
    case 3:
      return c->dtype == KVC_FP4 ? hd / 16 : 0;
    default:
      return 0;
  }
}

// bytes of one chunk of fp32 rows of width H*D
size_t chunk_f32_bytes(const kvc_cache* c) {
  return (size_t)chunk_tokens(c) * c->heads * c->head_dim * 4;
}

bool stage_ok(const kvc_cache* c, size_t need) {
  return c->stage && aligned16(c->stage) && c->stage_bytes >= need;
}

// Copy (bf16) or FP4-encode one chunk's K and V into region r.
cudaError_t store_chunk(kvc_cache* c, const void* k, const void* v, int32_t r, cudaStream_t st) {
  const int64_t Tc = chunk_tokens(c);
  const int64_t n = Tc * c->heads * (int64_t)c->head_dim;  // elements per tensor
  if (c->dtype == KVC_BF16) {
    const size_t off = (size_t)r * Tc * row_bytes(c, 0);
    return launch_copy2(static_cast<uint8_t*>(c->k) + off, k, static_cast<uint8_t*>(c->v) + off, v,
                        (size_t)n * 2, st);
  }
  const size_t coff = (size_t)r * Tc * row_bytes(c, 0);
  const size_t soff = (size_t)r * Tc * row_bytes(c, 2);
  QuantJob jobs[2] = {{k, static_cast<uint8_t*>(c->k) + coff, c->k_scale + soff, c->k_gscale + r},
                      {v, static_cast<uint8_t*>(c->v) + coff, c->v_scale + soff, c->v_gscale + r}};
  return launch_quant_fp4(jobs, 2, n, c->dev_ws + 1, KVC_WS_WORDS - 1, st);
}

// State check of an append of chunk_idx (as a new shot's sink when `shot`):
// the region it goes to, or -1 when the call is not valid now.
int32_t append_region(const kvc_cache* c, int64_t chunk_idx, bool shot) {
  if (shot) {
    if (chunk_idx == c->last_chunk + 1) return (chunk_idx > 0 || c->chunk_of_region[0] == -1) ? 0 : -1;
    return (chunk_idx == c->last_chunk && c->chunk_of_region[0] == chunk_idx) ? 0 : -1;
  }
  const int32_t r = region_of(c, chunk_idx);
  const int64_t occ = c->chunk_of_region[r];
  if (chunk_idx == c->last_chunk + 1) return occ == -1 ? r : -1;  // next chunk: needs a free slot
  return (chunk_idx == c->last_chunk && occ == chunk_idx) ? r : -1;  // overwrite while cached
}

// Commit an append's state (after its launches succeeded).
void commit_append(kvc_cache* c, int64_t chunk_idx, int32_t r, bool shot) {
  const bool fresh = c->chunk_of_region[r] != chunk_idx;
  if (shot && fresh && chunk_idx > 0) c->shot += 1;
  if (fresh) c->frame0_of_region[r] = frame0_of(c, chunk_idx, c->shot);
  c->chunk_of_region[r] = chunk_idx;
  c->last_chunk = chunk_idx;
}

}  // namespace

extern "C" {

size_t kvc_sizeof_cache(void) { return sizeof(kvc_cache); }

size_t kvc_cache_bytes(const kvc_cache* c, int32_t which) {
  if (!geometry_ok(c)) return 0;
  const size_t S = (size_t)cache_rows(c);
  switch (which) {
    case 0:
    case 1:
    case 2:
    case 3:
      return S * row_bytes(c, which);
    case 4:
    case 5:
      return c->dtype == KVC_FP4 ? (size_t)(1 + c->window_chunks) * sizeof(float) : 0;
    case 6:
      return (size_t)KVC_WS_WORDS * sizeof(int32_t);
    case 7: {
      const int nsm = attn_sm_count();
      return nsm > 0 ? attn_workspace_bytes(c->head_dim, nsm) : 0;
    }
    case 8: {
      const size_t m = 1 + (size_t)c->window_chunks;
      return chunk_f32_bytes(c) * (m > 3 ? m : 3);
    }
    default:
      return 0;
  }
}

int32_t kvc_init(kvc_cache* c) {
  if (!geometry_ok(c)) return KVC_EINVAL;
  if (!c->k || !c->v || !c->dev_ws || !aligned16(c->k) || !aligned16(c->v) || !aligned16(c->dev_ws))
    return KVC_EINVAL;
  if (c->attn_ws && !aligned16(c->attn_ws)) return KVC_EINVAL;
  if (c->stage && !aligned16(c->stage)) return KVC_EINVAL;
  if (c->dtype == KVC_FP4) {
    if (!c->k_scale || !c->v_scale || !c->k_gscale || !c->v_gscale) return KVC_EINVAL;
    if (!aligned16(c->k_scale) || !aligned16(c->v_scale)) return KVC_EINVAL;
    if ((reinterpret_cast<uintptr_t>(c->k_gscale) & 3u) || (reinterpret_cast<uintptr_t>(c->v_gscale) & 3u))
      return KVC_EINVAL;
  }
  for (int r = 0; r < 1 + KVC_MAX_WINDOW; ++r) {
    c->chunk_of_region[r] = -1;
    c->frame0_of_region[r] = -1;
  }
  c->last_chunk = -1;
  c->shot = 0;
  c->init_magic = KVC_INIT_MAGIC;
  return KVC_OK;
}

static int32_t append_impl(kvc_cache* c, const void* k_chunk, const void* v_chunk, int64_t chunk_idx,
                           kvc_stream_t stream, bool shot) {
  if (!ready(c) || !k_chunk || !v_chunk || !aligned16(k_chunk) || !aligned16(v_chunk) || chunk_idx < 0)
    return KVC_EINVAL;
  const int32_t r = append_region(c, chunk_idx, shot);
  if (r < 0) return KVC_ESTATE;
  if (store_chunk(c, k_chunk, v_chunk, r, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVC_ECUDA;
  commit_append(c, chunk_idx, r, shot);
  return KVC_OK;
}

int32_t kvc_append(kvc_cache* c, const void* k_chunk, const void* v_chunk, int64_t chunk_idx,
                   kvc_stream_t stream) {
  return append_impl(c, k_chunk, v_chunk, chunk_idx, stream, false);
}

int32_t kvc_append_shot(kvc_cache* c, const void* k_chunk, const void* v_chunk, int64_t chunk_idx,
                        kvc_stream_t stream) {
  return append_impl(c, k_chunk, v_chunk, chunk_idx, stream, true);
}

int32_t kvc_evict(kvc_cache* c, int64_t chunk_idx, kvc_stream_t stream) {
  if (!ready(c) || chunk_idx < 0) return KVC_EINVAL;
  if (chunk_idx == 0) return KVC_ESTATE;
  if (oldest_window_chunk(c) != chunk_idx) return KVC_ESTATE;
  const int32_t r = 1 + (int32_t)((chunk_idx - 1) % c->window_chunks);
  if (c->chunk_of_region[r] != chunk_idx) return KVC_ESTATE;
  if (c->scrub_on_evict) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t Tc = chunk_tokens(c);
    cudaError_t e;
    if (c->dtype == KVC_BF16) {
      const size_t off = (size_t)r * Tc * row_bytes(c, 0);
      void* d[2] = {static_cast<uint8_t*>(c->k) + off, static_cast<uint8_t*>(c->v) + off};
      const size_t b[2] = {(size_t)Tc * row_bytes(c, 0), (size_t)Tc * row_bytes(c, 0)};
      const uint32_t w[2] = {0x7FC07FC0u, 0x7FC07FC0u};  // bf16 NaN
      e = launch_fill(d, b, w, 2, st);
    } else {
      const size_t coff = (size_t)r * Tc * row_bytes(c, 0);
      const size_t soff = (size_t)r * Tc * row_bytes(c, 2);
      void* d[4] = {static_cast<uint8_t*>(c->k) + coff, static_cast<uint8_t*>(c->v) + coff,
                    c->k_scale + soff, c->v_scale + soff};
      const size_t cb = (size_t)Tc * row_bytes(c, 0), sb = (size_t)Tc * row_bytes(c, 2);
      const size_t b[4] = {cb, cb, sb, sb};
      const uint32_t w[4] = {0u, 0u, 0x7F7F7F7Fu, 0x7F7F7F7Fu};  // codes 0, scales E4M3 NaN
      e = launch_fill(d, b, w, 4, st);
    }
    if (e != cudaSuccess) return KVC_ECUDA;
  }
  c->chunk_of_region[r] = -1;
  c->frame0_of_region[r] = -1;
  return KVC_OK;
}

int32_t sinkwin_attn(const kvc_cache* c, const void* q, void* out, int32_t tq, float softmax_scale,
                     kvc_stream_t stream) {
  if (!ready(c) || tq < 0) return KVC_EINVAL;
  if (tq == 0) return KVC_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out) || !std::isfinite(softmax_scale) ||
      softmax_scale < 0.0f)
    return KVC_EINVAL;
  if (c->head_dim != 64 && c->head_dim != 128) return KVC_EUNSUPPORTED;
  if (c->chunk_of_region[0] < 0) return KVC_ESTATE;
  AttnLaunch a{};
  a.q = q;
  a.out = out;
  a.tq = tq;
  a.H = c->heads;
  a.D = c->head_dim;
  a.S = (int32_t)cache_rows(c);
  a.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
  const int32_t Tc = (int32_t)chunk_tokens(c);
  a.nseg = 0;
  for (int r = 0; r <= c->window_chunks; ++r) {
    if (c->chunk_of_region[r] < 0) continue;
    const int32_t row0 = r * Tc;
    // bf16: adjacent regions merge into one run of keys.  FP4: one segment per
    // region, so every K/V tile has a single pair of tensor scales.
    if (c->dtype == KVC_BF16 && a.nseg > 0 && a.seg[a.nseg - 1].row0 + a.seg[a.nseg - 1].rows == row0)
      a.seg[a.nseg - 1].rows += Tc;
    else
      a.seg[a.nseg++] = Seg{row0, Tc};
  }
  a.dev_err = c->dev_ws;
  a.k = c->k;
  a.v = c->v;
  a.fp4 = c->dtype == KVC_FP4;
  a.k_scale = c->k_scale;
  a.v_scale = c->v_scale;
  a.k_gscale = c->k_gscale;
  a.v_gscale = c->v_gscale;
  a.chunk_tokens = Tc;
  a.ws = c->attn_ws;
  a.ws_bytes = c->attn_ws ? (size_t)c->attn_ws_bytes : 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // FP4 cache with room in the staging buffer for f16 K and V of every region:
  // decode the visible regions once, then the attention loads f16 tiles by TMA
  // instead of decoding each tile for every query item.  K' = e2m1 * s (exact;
  // its tensor scale joins the logit scale), V' = f16(e2m1 * s * g_V / G) with
  // G the kernel's power-of-two V shift (so P needs no per-element factor)
  const size_t kv16 = (size_t)a.S * a.H * a.D * 2;  // bytes of one f16 K (or V)
  if (a.fp4 && stage_ok(c, 2 * kv16)) {
    uint8_t* k16 = static_cast<uint8_t*>(c->stage);
    uint8_t* v16 = k16 + kv16;
    Fp4DecodeJob jobs[kMaxDecodeJobs];
    int32_t regions[1 + KVC_MAX_WINDOW];
    int nj = 0;
    const size_t row_elems = (size_t)a.H * a.D;
    for (int i = 0; i < a.nseg; ++i) {
      const size_t e0 = (size_t)a.seg[i].row0 * row_elems, ne = (size_t)a.seg[i].rows * row_elems;
      const int32_t region = a.seg[i].row0 / Tc;
      regions[i] = region;
      const uint8_t* kc = static_cast<const uint8_t*>(c->k);
      const uint8_t* vc = static_cast<const uint8_t*>(c->v);
      jobs[nj++] = Fp4DecodeJob{kc + e0 / 2, c->k_scale + e0 / 16, k16 + e0 * 2, (int64_t)(ne / 8), -1};
      jobs[nj++] = Fp4DecodeJob{vc + e0 / 2, c->v_scale + e0 / 16, v16 + e0 * 2, (int64_t)(ne / 8), region};
    }
    const cudaError_t e = launch_fp4_to_f16(jobs, nj, st, c->v_gscale, regions, a.nseg);
    if (e != cudaSuccess) return cuda_status(e);
    a.k16 = k16;
    a.v16 = v16;
  }
  return cuda_status(launch_sinkwin_attn(a, st));
}

int32_t kvc_recache(kvc_cache* c, const void* hidden, const void* w_kv, const float* gamma_k,
                    float eps, const int64_t* chunk_ids, int32_t n, int32_t grid_h, int32_t grid_w,
                    float rope_theta, kvc_stream_t stream) {
  if (!ready(c) || !hidden || !w_kv || !chunk_ids || n < 1 || n > 1 + c->window_chunks)
    return KVC_EINVAL;
  if (!aligned16(hidden) || !aligned16(w_kv) || (gamma_k && !aligned16(gamma_k)))
    return KVC_EINVAL;
  if (grid_h < 1 || grid_w < 1 || (int64_t)grid_h * grid_w != c->tokens_per_frame) return KVC_EINVAL;
  if (!(eps >= 0.0f) || !std::isfinite(eps) || !(rope_theta > 0.0f) || !std::isfinite(rope_theta))
    return KVC_EINVAL;
  if (!recache_supported(c->heads, c->head_dim)) return KVC_EUNSUPPORTED;
  const bool fp4 = c->dtype == KVC_FP4;
  if (fp4 && !stage_ok(c, (size_t)n * chunk_f32_bytes(c))) return KVC_EINVAL;
  int64_t present[1 + KVC_MAX_WINDOW];
  const int np = present_chunks(c, present);
  if (np != n) return KVC_ESTATE;
  for (int i = 0; i < n; ++i)
    if (chunk_ids[i] != present[i]) return KVC_ESTATE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  RecacheLaunch rl{};
  rl.hidden = hidden;
  rl.w_kv = w_kv;
  rl.gamma = gamma_k;
  rl.eps = eps;
  rl.theta = rope_theta;
  rl.Tc = (int32_t)chunk_tokens(c);
  rl.rows = n * rl.Tc;
  rl.H = c->heads;
  rl.D = c->head_dim;
  rl.tpf = c->tokens_per_frame;
  rl.grid_w = grid_w;
  rl.n = n;
  for (int i = 0; i < n; ++i) {
    const int32_t r = region_of(c, chunk_ids[i]);
    rl.frame0[i] = c->frame0_of_region[r];
    // FP4: bf16 K and V of chunk i go to rows [i Tc, (i+1) Tc) of the staging buffer
    rl.region[i] = fp4 ? i : r;
  }
  const size_t hd2 = (size_t)rl.Tc * c->heads * c->head_dim * 2;  // bf16 bytes of one chunk
  rl.k = fp4 ? c->stage : c->k;
  rl.v = fp4 ? static_cast<uint8_t*>(c->stage) + (size_t)n * hd2 : c->v;
  rl.dev_err = c->dev_ws;
  cudaError_t e = launch_recache(rl, st);
  if (e != cudaSuccess || !fp4) return cuda_status(e);
  // every region's K and V encoded as its own tensor, all in one encode (two launches)
  QuantJob jobs[kMaxQuantJobs];
  const int64_t Tc = chunk_tokens(c);
  for (int i = 0; i < n; ++i) {
    const int32_t r = region_of(c, chunk_ids[i]);
    const size_t coff = (size_t)r * Tc * row_bytes(c, 0);
    const size_t soff = (size_t)r * Tc * row_bytes(c, 2);
    jobs[2 * i] = QuantJob{static_cast<const uint8_t*>(rl.k) + (size_t)i * hd2,
                           static_cast<uint8_t*>(c->k) + coff, c->k_scale + soff, c->k_gscale + r};
    jobs[2 * i + 1] = QuantJob{static_cast<const uint8_t*>(rl.v) + (size_t)i * hd2,
                               static_cast<uint8_t*>(c->v) + coff, c->v_scale + soff, c->v_gscale + r};
  }
  e = launch_quant_fp4(jobs, 2 * n, Tc * c->heads * (int64_t)c->head_dim, c->dev_ws + 1, KVC_WS_WORDS - 1, st);
  return e == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

int32_t kvc_project_append(kvc_cache* c, const void* hidden, const void* w_qkv,
                           const float* gamma_q, const float* gamma_k, float eps,
                           int64_t chunk_idx, int32_t new_shot, int32_t grid_h, int32_t grid_w,
                           float rope_theta, void* q_out, kvc_stream_t stream) {
  if (!ready(c) || !hidden || !w_qkv || !q_out || chunk_idx < 0) return KVC_EINVAL;
  if (!aligned16(hidden) || !aligned16(w_qkv) || !aligned16(q_out) ||
      (gamma_q && !aligned16(gamma_q)) || (gamma_k && !aligned16(gamma_k)))
    return KVC_EINVAL;
  if (grid_h < 1 || grid_w < 1 || (int64_t)grid_h * grid_w != c->tokens_per_frame) return KVC_EINVAL;
  if (!(eps >= 0.0f) || !std::isfinite(eps) || !(rope_theta > 0.0f) || !std::isfinite(rope_theta))
    return KVC_EINVAL;
  if (!recache_supported(c->heads, c->head_dim)) return KVC_EUNSUPPORTED;
  const bool fp4 = c->dtype == KVC_FP4;
  const size_t f32b = chunk_f32_bytes(c);  // one chunk of fp32 rows
  if (!stage_ok(c, 2 * f32b + (fp4 ? f32b : 0))) return KVC_EINVAL;
  const bool shot = new_shot != 0;
  const int32_t r = append_region(c, chunk_idx, shot);
  if (r < 0) return KVC_ESTATE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t Tc = chunk_tokens(c);
  ProjectLaunch pl{};
  pl.hidden = hidden;
  pl.w_qkv = w_qkv;
  pl.gamma_q = gamma_q;
  pl.gamma_k = gamma_k;
  pl.eps = eps;
  pl.theta = rope_theta;
  pl.Tc = (int32_t)Tc;
  pl.H = c->heads;
  pl.D = c->head_dim;
  pl.tpf = c->tokens_per_frame;
  pl.grid_w = grid_w;
  // positions: an overwrite keeps the chunk's; a new shot counts one boundary more
  const bool fresh = c->chunk_of_region[r] != chunk_idx;
  pl.frame0 = fresh ? frame0_of(c, chunk_idx, c->shot + ((shot && chunk_idx > 0) ? 1 : 0))
                    : c->frame0_of_region[r];
  pl.stage_f32 = static_cast<float*>(c->stage);
  pl.q_out = q_out;
  if (fp4) {  // bf16 K and V wait in the staging buffer for the FP4 encode
    pl.k_dst = static_cast<uint8_t*>(c->stage) + 2 * f32b;
    pl.v_dst = static_cast<uint8_t*>(c->stage) + 2 * f32b + f32b / 2;
  } else {
    const size_t off = (size_t)r * Tc * row_bytes(c, 0);
    pl.k_dst = static_cast<uint8_t*>(c->k) + off;
    pl.v_dst = static_cast<uint8_t*>(c->v) + off;
  }
  pl.dev_err = c->dev_ws;
  if (launch_project_chunk(pl, st) != cudaSuccess) return KVC_ECUDA;
  if (fp4 && store_chunk(c, pl.k_dst, pl.v_dst, r, st) != cudaSuccess) return KVC_ECUDA;
  commit_append(c, chunk_idx, r, shot);
  return KVC_OK;
}

int32_t kvc_quant_fp4(const void* x, int64_t n, uint8_t* codes, uint8_t* scales, float* gscale,
                      int32_t* ws, kvc_stream_t stream) {
  if (!x || !codes || !scales || !gscale || !ws) return KVC_EINVAL;
  if (n < 16 || n % 16 != 0 || n / 16 > (int64_t(1) << 31)) return KVC_EINVAL;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 7u) ||
      (reinterpret_cast<uintptr_t>(gscale) & 3u) || (reinterpret_cast<uintptr_t>(ws) & 3u))
    return KVC_EINVAL;
  QuantJob job{x, codes, scales, gscale};
  return cuda_status(launch_quant_fp4(&job, 1, n, ws, KVC_QUANT_WS_WORDS, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvc_gemm_fp4(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_gscale,
                     const uint8_t* b_codes, const uint8_t* b_scales, const float* b_gscale,
                     int64_t M, int64_t N, int64_t K, void* out, void* ws, size_t ws_bytes,
                     int32_t* dev_err, kvc_stream_t stream) {
  if (M < 0 || N <= 0 || K <= 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
      K >= (int64_t(1) << 31))
    return KVC_EINVAL;
  if (M == 0) return KVC_OK;  // an empty product: no pointer is read
  if (!a_codes || !a_scales || !a_gscale || !b_codes || !b_scales || !b_gscale || !out)
    return KVC_EINVAL;
  if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(b_codes) || !aligned16(b_scales) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(a_gscale) & 3u) ||
      (reinterpret_cast<uintptr_t>(b_gscale) & 3u) || (reinterpret_cast<uintptr_t>(dev_err) & 3u))
    return KVC_EINVAL;
  if (N % 32 != 0 || K % 256 != 0) return KVC_EUNSUPPORTED;
  if (((M + 127) / 128) * ((N + 191) / 192) >= (int64_t(1) << 31)) return KVC_EUNSUPPORTED;
  if (ws && (!aligned16(ws) || (uint64_t)ws_bytes < (uint64_t)gemm_fp4_ws_bytes(M, N, K)))
    return KVC_EINVAL;
  GemmFp4Launch g{a_codes, a_scales, a_gscale, b_codes, b_scales, b_gscale, M, N, K, out, dev_err, ws};
  return cuda_status(launch_gemm_fp4(g, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvc_last_device_error(const kvc_cache* c, kvc_stream_t stream) {
  if (!c || !c->dev_ws) return KVC_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVC_ECUDA;
  int32_t w = 0;
  if (cudaMemcpy(&w, c->dev_ws, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return KVC_ECUDA;
  if (w != 0) {
    const int32_t z = 0;
    if (cudaMemcpy(c->dev_ws, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return KVC_ECUDA;
    return KVC_ETIMEOUT;
  }
  return KVC_OK;
}

int32_t kvc_watchdog_selftest(int32_t* dev_ws, int32_t limit_us, kvc_stream_t stream) {
  if (!dev_ws || limit_us < 1 || limit_us > 2000000) return KVC_EINVAL;
  return cuda_status(launch_watchdog_selftest(dev_ws, limit_us, reinterpret_cast<cudaStream_t>(stream)));
}

const char* kvc_status_string(int32_t s) {
  switch (s) {
    case KVC_OK:
      return "ok";
    case KVC_EINVAL:
      return "invalid argument";
    case KVC_ESTATE:
      return "invalid in the cache's current state";
    case KVC_ECUDA:
      return "CUDA error";
    case KVC_ETIMEOUT:
      return "device wait timed out";
    case KVC_EUNSUPPORTED:
      return "unsupported";
    default:
      return "unknown status";
  }
}

}  // extern "C"
