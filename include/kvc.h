/*
 * kvc.h -- C ABI of the sink + short-window KV-cache attention library (sm_103a).
 *
 * What it computes.  LongLive's frame-level autoregressive video generator keeps,
 * per self-attention layer, a KV cache made of the first frame chunk pinned as
 * "frame sink" tokens plus a short rolling window of recent chunks; each new
 * chunk's queries attend to [sink | window] (LongLive summary page, yunpan.plus,
 * 方法 §3 高效长推理: 短窗口注意力 and 帧汇聚点; LONGLIVE news page, paooo.com,
 * LONGLIVE的技术原理).  At a prompt switch the cache is rebuilt from the frames
 * already generated (方法 §1 KV 重缓存).  LongLive 2.0 can hold the cache in FP4
 * and dequantise it inside the attention read (LongLive 2.0 inference blog,
 * blog.hotdry.top, "NVFP4 量化与 KV Cache 压缩的工程实现": inference.kv_quant).
 *
 * Layout.  One layer's cache has (1 + W) regions of Tc = chunk_frames *
 * tokens_per_frame rows each.  Region 0 holds the sink (chunk 0, or the first
 * chunk of the current shot after kvc_append_shot); a window chunk c >= 1 lives
 * in region 1 + (c - 1) % W.  Row r of region g is physical row g * Tc + r of
 *     bf16 cache:  k, v            bf16  [S][H][D]          S = (1 + W) * Tc
 *     FP4 cache:   k, v            uint8 [S][H][D/2]        E2M1 codes, element 2i in
 *                                                           the low nibble
 *                  k_scale,v_scale uint8 [S][H][D/16]       E4M3 scale per 16 elements
 *                  k_gscale,...    float [1 + W]            fp32 tensor scale per region
 * Decoded value: e2m1(code) * e4m3(scale) * gscale[region].
 *
 * RoPE positions.  Token t of chunk c sits at frame frame0(c) + t / tokens_per_frame,
 * patch row (t % tokens_per_frame) / grid_w, column t % grid_w, with
 * frame0(c) = c * chunk_frames + shot(c) * rope_offset_frames, shot(c) being the
 * number of shot boundaries (kvc_append_shot of a chunk > 0) at or before c.  Keys
 * handed to kvc_append are expected to carry these positions; kvc_recache and
 * kvc_project_append apply them.
 *
 * Conventions.
 *  - All device memory (cache, inputs, outputs, workspace) is allocated by the
 *    caller; the library allocates nothing and frees nothing.  The kvc_cache
 *    struct is caller-owned host memory.
 *  - Pointers documented as "device" are CUDA device addresses; "host" ones are
 *    ordinary host addresses.  Device buffers must be 16-byte aligned.
 *  - Every call that touches the GPU is asynchronous on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and never synchronises, except
 *    kvc_last_device_error.  Inputs must stay alive until the stream passes them.
 *  - The host-side slot map is updated when the call is made, so the call order
 *    defines the cache state; a caller must not reorder the work across streams.
 *  - Errors are returned as kvc_status values, never by aborting.  A call that
 *    returns an error has changed nothing: neither the slot map nor (apart from
 *    KVC_ECUDA after a launch) any device memory.
 *  - One kvc_cache is used by one host thread at a time.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kvc_stream_t; /* == cudaStream_t */

typedef enum {
  KVC_OK = 0,
  KVC_EINVAL = -1,       /* bad sizes, null pointers, dtype mismatch, misalignment */
  KVC_ESTATE = -2,       /* the call is not valid in the cache's current state */
  KVC_ECUDA = -3,        /* a CUDA launch / runtime error */
  KVC_ETIMEOUT = -4,     /* a kernel's bounded wait ran out (device error word set) */
  KVC_EUNSUPPORTED = -5  /* valid request outside what the kernels implement */
} kvc_status;

typedef enum { KVC_BF16 = 0, KVC_FP4 = 1 } kvc_dtype;

#define KVC_MAX_WINDOW 16 /* ring slots W <= 16 */
#define KVC_WS_WORDS 1024 /* device workspace words (int32) per cache */
#define KVC_QUANT_WS_WORDS 256 /* scratch words kvc_quant_fp4 needs */
#define KVC_INIT_MAGIC 0x4B564331

typedef struct kvc_cache {
  /* ---- geometry: set by the caller before kvc_init ---- */
  int32_t heads;            /* H, 1..65536 */
  int32_t head_dim;         /* D, a multiple of 16 up to 256; attention supports 64 and 128 */
  int32_t tokens_per_frame; /* latent tokens of one frame (1560 = 30 x 52 for LongLive-1.3B) */
  int32_t chunk_frames;     /* frames per chunk; the sink is exactly one chunk.  The cache's
                               rows (1 + W) * tokens_per_frame * chunk_frames are at most
                               2^30, and rows * H * D at most 2^40 (else KVC_EINVAL) */
  int32_t window_chunks;    /* W, 1..KVC_MAX_WINDOW ring slots, the current chunk included */
  int32_t dtype;            /* kvc_dtype */
  /* ---- device buffers: caller-allocated, sizes from kvc_cache_bytes ---- */
  void* k;
  void* v;
  uint8_t* k_scale;  /* FP4 only, else NULL */
  uint8_t* v_scale;  /* FP4 only, else NULL */
  float* k_gscale;   /* FP4 only, [1 + W], else NULL */
  float* v_gscale;   /* FP4 only, [1 + W], else NULL */
  int32_t* dev_ws;   /* KVC_WS_WORDS int32, zero-filled by the caller before kvc_init;
                        word 0 is the device error word, the rest is reduction scratch */
  void* attn_ws;     /* optional attention workspace of kvc_cache_bytes(c, 7) bytes,
                        zero-filled by the caller before first use, or NULL.  With it
                        sinkwin_attn balances work evenly over all SMs (items cut at a
                        CTA boundary are merged through it); without it every CTA
                        takes whole items.  Calls sharing it must be stream-ordered. */
  uint64_t attn_ws_bytes; /* its size in bytes */
  void* stage;       /* optional staging buffer (16-byte aligned) of up to
                        kvc_cache_bytes(c, 8) bytes, or NULL: fp32 rows waiting for
                        their RMSNorm, bf16 K/V waiting for their FP4 encode, and
                        the f16 K/V sinkwin_attn decodes an FP4 cache into.
                        Needed by kvc_recache on an FP4 cache and by kvc_project_append
                        (each states how much it uses).  Contents need no init;
                        calls sharing it must be stream-ordered (caches whose calls
                        are may share one). */
  uint64_t stage_bytes; /* its size in bytes */
  /* ---- options ---- */
  int32_t scrub_on_evict;     /* nonzero: kvc_evict overwrites the freed slot with NaN */
  int32_t rope_offset_frames; /* multi-shot RoPE offset: each shot boundary (kvc_append_shot)
                                 shifts the frame positions of that chunk and every later
                                 one by this many frames (0: positions stay absolute) */
  /* ---- library-maintained state: read-only for the caller ---- */
  int32_t init_magic;
  int32_t shot;                                /* shot boundaries so far */
  int64_t chunk_of_region[1 + KVC_MAX_WINDOW]; /* -1 = empty; region 0 = the sink */
  int64_t frame0_of_region[1 + KVC_MAX_WINDOW]; /* RoPE frame position of the first frame
                                                   of the chunk each region holds; -1 = empty */
  int64_t last_chunk;                          /* highest chunk appended so far, -1 = none */
} kvc_cache;

/* sizeof(kvc_cache) as compiled into the library (lets bindings check the layout). */
size_t kvc_sizeof_cache(void);

/* Bytes of one device buffer of a cache with this geometry.
 * which: 0 k, 1 v, 2 k_scale, 3 v_scale, 4 k_gscale, 5 v_gscale, 6 dev_ws,
 * 7 attn_ws (depends on the SM count of the current device; 0 without one),
 * 8 stage (the most any call uses: Tc * H*D * 4 * max(1 + W, 3)).
 * Returns 0 for a buffer the dtype does not use or for an invalid geometry.
 * Cache = sink + W window slots: LongLive summary page, 方法 §3 高效长推理 (帧汇聚点,
 * 短窗口注意力: the per-layer cache size depends on the window only). */
size_t kvc_cache_bytes(const kvc_cache* c, int32_t which);

/* Validate geometry and buffers, mark every region empty.  No GPU work.
 * KVC_EINVAL on a bad geometry or a missing / misaligned buffer. */
int32_t kvc_init(kvc_cache* c);

/* Append chunk `chunk_idx`: k_chunk, v_chunk are device bf16 [Tc][H][D]
 * (post-norm, post-RoPE keys, as the layer produced them).  The sink is chunk 0;
 * chunk c >= 1 goes to ring slot (c-1) % W.  Allowed: chunk 0 into an empty
 * cache; the last appended chunk again while it is still cached (overwrite, one
 * call per denoise step); chunk last_chunk + 1 once its slot is empty (evict the
 * oldest window chunk first).  Else KVC_ESTATE.  bf16 cache: a 128-bit
 * vectorised copy.  FP4 cache: the chunk's K and V are quantised (tensor amax ->
 * fp32 gscale[region], E4M3 block scales, E2M1 codes; the encode rule is
 * kvc_quant_fp4's).
 * Defined by: LongLive summary page, 方法 §3 (each new chunk's keys/values join
 * the window; the first chunk stays as the frame sink). */
int32_t kvc_append(kvc_cache* c, const void* k_chunk, const void* v_chunk, int64_t chunk_idx,
                   kvc_stream_t stream);

/* Append chunk `chunk_idx` as the first chunk of a new shot: it becomes the
 * sink (region 0) and the previous sink leaves the cache; the window slots keep
 * what they hold (the previous shot's recent chunks still give continuity) and
 * later chunks fill the ring as usual (chunk_idx's own ring slot stays unused).
 * Allowed: chunk last_chunk + 1 (or 0 into an empty cache), or the current sink
 * again when it is the last chunk appended (overwrite); else KVC_ESTATE.  The
 * shot count grows by one for chunk_idx > 0, which shifts RoPE positions by
 * rope_offset_frames from this chunk on.  Arguments and encode as kvc_append.
 * Defined by: LongLive 2.0 inference blog (blog.hotdry.top), "序列并行与注意力汇聚的
 * 协同设计" (inference.multi_shot_sink resets the sink at each shot boundary;
 * inference.multi_shot_rope_offset shifts the RoPE positions). */
int32_t kvc_append_shot(kvc_cache* c, const void* k_chunk, const void* v_chunk, int64_t chunk_idx,
                        kvc_stream_t stream);

/* Evict chunk `chunk_idx`, which must be the oldest window chunk (the sink is
 * never evicted: KVC_ESTATE).  Moves no data: the slot is marked empty.  With
 * scrub_on_evict set, the slot's rows are overwritten with NaN (bf16 0x7FC0;
 * FP4: codes 0, scales 0x7F) so a stale read would show.
 * Defined by: LongLive summary page, 方法 §3 短窗口注意力 (attention covers only a
 * fixed window of recent frames). */
int32_t kvc_evict(kvc_cache* c, int64_t chunk_idx, kvc_stream_t stream);

/* out = softmax(softmax_scale * q K^T) V per head, over the visible keys: the
 * sink region plus every occupied window slot (no mask inside that set; keys are
 * read in physical order, which softmax does not see).  q, out: device bf16
 * [tq][H][D]; tq >= 0 (0 is a no-op); softmax_scale finite and >= 0 (else
 * KVC_EINVAL).  D in {64, 128} (else KVC_EUNSUPPORTED); the sink must be
 * present (else KVC_ESTATE).  A kernel wait that runs out leaves KVC_ETIMEOUT
 * for kvc_last_device_error.  Any tq runs on every SM: queries of a head are cut
 * into 256-row items and items into pieces of K/V tiles when there are fewer
 * items than SMs (pieces merged through attn_ws; without it whole items).
 * Arithmetic: bf16 operands, fp32 accumulation and softmax, bf16 output.  FP4
 * caches are dequantised to f16, K as e2m1 * s (exact), and Q is converted to
 * f16 exactly with a power-of-two scale per row; the regions' K tensor scales
 * enter the logit scale.  Every V tensor scale is first divided by one power
 * of two G covering the largest (G returns in the normalisation, so any
 * finite magnitude of V is representable).  Two ways:
 *  - stage of at least 2 * S * H * D * 2 bytes (S = (1 + W) * Tc;
 *    kvc_cache_bytes(c, 8) is always enough): one launch decodes the visible
 *    regions' K and V into stage, V as f16(e2m1 * s * g_V / G), then the
 *    attention kernel loads those f16 tiles (two launches; stage overwritten);
 *  - otherwise K/V are decoded inside the attention kernel's tile load, V as
 *    e2m1 * s (exact), g_V / G applied to P before it is stored as f16.
 * Defined by: LongLive summary page, 方法 §3 高效长推理 (queries attend to the
 * frame-sink tokens joined with the short window); FP4 read: LongLive 2.0
 * inference blog, "NVFP4 量化与 KV Cache 压缩的工程实现" (fused dequantisation). */
int32_t sinkwin_attn(const kvc_cache* c, const void* q, void* out, int32_t tq,
                     float softmax_scale, kvc_stream_t stream);

/* KV recache at a prompt switch: for the n chunks listed in chunk_ids (host
 * int64, logical order: sink first, then window chunks oldest -> newest; must be
 * exactly the chunks in the cache, else KVC_ESTATE):
 *   [K | V] = hidden @ w_kv;  K <- RoPE3D(RMSNorm(K) * gamma_k);  written to the
 *   chunks' regions.
 * hidden: device bf16 [n*Tc][H*D]; w_kv: device bf16 [H*D][2*H*D], the K columns
 * first; gamma_k: device fp32 [H*D], 16-byte aligned, or NULL (= ones); hidden and
 * w_kv 16-byte aligned (else KVC_EINVAL).  RMSNorm spans the whole
 * H*D-wide K row: x / sqrt(mean(x^2) + eps).  3D RoPE at each chunk's positions
 * (frame0_of_region of its region; see "RoPE positions" above); the D/2 rotation
 * pairs (adjacent elements) are split into [frame | row | column] bands of
 * (P - 2*(P/3), P/3, P/3) pairs, P = D/2; in a band of b dims pair j turns by
 * position * rope_theta^(-2j/b).  grid_h * grid_w == tokens_per_frame.
 * H*D in {64, 128, 256, 512, 768, 1024, 1536, 2048, 3072} (else KVC_EUNSUPPORTED).
 * bf16 cache: H*D a multiple of 512 up to 2048 with D in {64, 128}: one fused
 * launch on `stream` (K and V projections, the norm and rotation applied to K
 * before it is written), plus, when the SMs do not divide into its thread-block
 * clusters, a second launch on a library-owned side stream that waits for the
 * work already in `stream` and that `stream` waits for (event fork and join;
 * this holds under stream capture).  Other shapes: three launches on `stream`
 * (K projection, norm + RoPE, V projection), between which the regions being
 * rebuilt hold intermediate values.  Either way nothing may read those regions
 * until the stream passes the call.
 * FP4 cache: the same launches write bf16 K and V of all n chunks into `stage`
 * (n * Tc * H*D * 4 bytes needed, else KVC_EINVAL), then every region's K and V
 * are FP4-encoded from them with kvc_quant_fp4's rule, each its own tensor
 * with its own tensor scale (one encode over all of them).
 * Defined by: LongLive summary page, 方法 §1 KV 重缓存 (at the switch the cache is
 * recomputed from the generated frames with the new prompt); FP4 store: LongLive
 * 2.0 inference blog, "NVFP4 量化与 KV Cache 压缩的工程实现". */
int32_t kvc_recache(kvc_cache* c, const void* hidden, const void* w_kv, const float* gamma_k,
                    float eps, const int64_t* chunk_ids, int32_t n, int32_t grid_h,
                    int32_t grid_w, float rope_theta, kvc_stream_t stream);

/* Project one new chunk and append its keys and values: 
 *   [Q | K | V] = hidden @ w_qkv;  Q <- RoPE3D(RMSNorm(Q) * gamma_q);
 *   K <- RoPE3D(RMSNorm(K) * gamma_k);  q_out <- Q;  K, V appended as chunk_idx
 * (as kvc_append, or kvc_append_shot when new_shot is nonzero).  hidden: device
 * bf16 [Tc][H*D]; w_qkv: device bf16 [H*D][3*H*D] (Q columns, then K, then V);
 * gamma_q, gamma_k: device fp32 [H*D] or NULL (= ones); q_out: device bf16
 * [Tc][H][D].  Norm, RoPE, eps, rope_theta, grid and the supported H*D as in
 * kvc_recache; positions frame0(chunk_idx).  Uses `stage`: Tc * H*D * 8 bytes
 * (bf16 cache) or 12 (FP4 cache), else KVC_EINVAL.  Two launches (the GEMM over
 * all 3*H*D columns, then norm + RoPE of Q and K), plus the FP4 encode's two.
 * Defined by: LongLive summary page, 方法 (causal frame-level autoregression: each
 * chunk is projected and its keys/values join the cache every later chunk
 * reads) and §3 帧汇聚点. */
int32_t kvc_project_append(kvc_cache* c, const void* hidden, const void* w_qkv,
                           const float* gamma_q, const float* gamma_k, float eps,
                           int64_t chunk_idx, int32_t new_shot, int32_t grid_h, int32_t grid_w,
                           float rope_theta, void* q_out, kvc_stream_t stream);

/* FP4-encode n finite bf16 values (device x, n % 16 == 0, n >= 16; the codes of
 * a tensor holding NaN or infinity are unspecified) as one tensor:
 *   amax = max|x|;  g = fl32(amax / 2688);   (g == 0: all codes and scales 0)
 *   per 16-block b: s = E4M3_rne_satfinite(fl32(fl32(amax_b / 6) / g));
 *   inv = fl32(1 / fl32(s*g));  s == 0, fl32(s*g) == 0 or inv infinite: scale
 *   and codes 0 (only for amax below ~2^-115);  else t = fl32(|x| * inv),
 *   code = signbit(x) << 3 | E2M1_rne_satfinite(t).
 * codes: device uint8 [n/2] (element 2i in the low nibble); scales: device uint8
 * [n/16]; gscale: device float [1]; ws: device scratch of KVC_QUANT_WS_WORDS
 * int32 words that the call overwrites (per-CTA partial maxima; calls that share
 * a ws must be stream-ordered).  n up to 2^31 * 16.
 * Defined by: LongLive 2.0 inference blog, "NVFP4 量化与 KV Cache 压缩的工程实现"
 * (inference.kv_quant: FP4 KV store); the format's rounding details are this
 * library's reading (the page names only FP4/NVFP4). */
int32_t kvc_quant_fp4(const void* x, int64_t n, uint8_t* codes, uint8_t* scales, float* gscale,
                      int32_t* ws, kvc_stream_t stream);

/* kvc_quant_fp4 without caller scratch.  The pages have no counterpart to
 * this call: it exists for callers that cannot allocate device memory when they
 * encode -- e.g. a host program whose device memory is all owned by another
 * allocator, or a latency-critical loop where a cudaMalloc (which may
 * synchronise the device) is not allowed.  Same arguments, encode rule and
 * outputs as kvc_quant_fp4 minus `ws`; the library allocates nothing.
 * Scratch: a static device array of KVC_NOALLOC_SCRATCH_WORDS int32 (1 KiB)
 * inside the library, held by every GPU that loads it until the process exits.
 * Its device address is looked up on every call, with the caller's device
 * current; the first call on a device may load the library's device code
 * there, so make that first call before any stream capture.  All calls share
 * the array: calls that overlap on the GPU (other streams, other threads) race
 * and must be ordered by the caller.  Nothing in it has to start at zero: each
 * call's first pass writes every word its second pass reads.
 * Uses the current device.  n must be a multiple of 16 in [16,
 * KVC_NOALLOC_MAX_ELEMS], else KVC_EINVAL. */
#define KVC_NOALLOC_SCRATCH_WORDS 256
#define KVC_NOALLOC_MAX_ELEMS (((int64_t)1) << 35)
int32_t kvc_quant_fp4_noalloc(const void* x, int64_t n, uint8_t* codes, uint8_t* scales,
                              float* gscale, kvc_stream_t stream);

/* W4A4 projection: out = deq(A) deq(B)^T, both operands FP4 tensors in the
 * encoding kvc_quant_fp4 writes, their 16-element blocks along K.
 *   A (activations):  a_codes  device uint8 [M][K/2] (element 2i in the low nibble),
 *                     a_scales device uint8 [M][K/16] (E4M3), a_gscale device float [1]
 *   B (weight, one row per output feature):
 *                     b_codes [N][K/2], b_scales [N][K/16], b_gscale [1], likewise
 *   out:              device bf16 [M][N], row-major; written, never read
 *   deq(x)[r][k] = e2m1(code) * e4m3(scale of block k/16) * gscale.
 * Each decoded element and each product of two is exact (at most 6 significant
 * bits); the sums are fp32 (tensor-core accumulation order), then scaled by
 * a_gscale * b_gscale and rounded to bf16.
 * ws: NULL, or device scratch of at least KVC_GEMM_FP4_WS_BYTES(M, N, K) bytes
 * (ws_bytes) that the call overwrites.  NULL: one kernel decodes the FP4
 * operands tile by tile inside the GEMM.  Given: A and B are decoded once into
 * ws as f16 and a second kernel multiplies those (faster on this GPU; same
 * result bits, the accumulation order aside).
 * dev_err: optional device int32 word (NULL: none) that records KVC_ETIMEOUT's
 * cause if a kernel wait runs out, as the cache's device error word does.
 * M >= 0 (0: KVC_OK at once, no pointer read), N and K > 0 and < 2^31; N % 32 != 0 or
 * K % 256 != 0: KVC_EUNSUPPORTED.  Codes, scales, out and ws 16-byte aligned, the
 * gscales and dev_err 4-byte aligned, a short ws: KVC_EINVAL.  The call's
 * kernels hold all of an SM's tensor memory while they run.
 * Defined by: LongLive 2.0 inference blog (blog.hotdry.top), "NVFP4 量化与 KV
 * Cache 压缩的工程实现" (NVFP4 W4A4: weights and activations both FP4); NVIDIA
 * infrastructure blog (bittide page), §6 (W4A4 execution in LongLive 2.0). */
#define KVC_GEMM_FP4_WS_BYTES(M, N, K) ((((int64_t)(M)) + ((int64_t)(N))) * ((int64_t)(K)) * 2)
int32_t kvc_gemm_fp4(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_gscale,
                     const uint8_t* b_codes, const uint8_t* b_scales, const float* b_gscale,
                     int64_t M, int64_t N, int64_t K, void* out, void* ws, size_t ws_bytes,
                     int32_t* dev_err, kvc_stream_t stream);

/* Synchronise `stream`, read and clear the cache's device error word.
 * KVC_OK, KVC_ETIMEOUT (a kernel wait ran out), or KVC_ECUDA (a sticky CUDA error). */
int32_t kvc_last_device_error(const kvc_cache* c, kvc_stream_t stream);

/* Diagnostic: one CTA waits on an mbarrier phase that nothing completes, with the
 * same bounded wait the kernels use but a limit of `limit_us` microseconds
 * (1..2000000), then records the timeout in dev_ws[0] and exits.  Exercises the
 * watchdog path without hanging the GPU. */
int32_t kvc_watchdog_selftest(int32_t* dev_ws, int32_t limit_us, kvc_stream_t stream);

/* Human-readable name of a kvc_status value. */
const char* kvc_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
