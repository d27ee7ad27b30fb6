/*
 * cacheblend.h -- C ABI of a GB300 (sm_103a) library for non-prefix KV-cache
 * fusion in RAG prefill: independently precomputed per-chunk K/V caches are
 * re-positioned by composing RoPE rotations, the tokens whose fresh keys
 * deviate most from the reused keys are recomputed, and only those rows run
 * through the layer, attending over the blended cache.
 *
 * Sources of the operations (cited per entry point below):
 *   [QCF]  QCFuse: Query-Aware Cache Fusion via Compressed View for Efficient
 *          RAG Serving (arxiv 2606.05875), §2.1 Eqs. 1-7, §4.1.5.
 *   [CB]   CacheBlend: Reusing KV Caches When Your Text Isn't a Prefix
 *          (blog): "Why You Can't Just Concatenate", "Quantifying the
 *          Damage", "Selective Recompute Without Skipping" (blend_layer),
 *          "The Chicken-and-Egg Problem" (select_hkvd).
 *   [ROM]  Request Order Matters: Cache-History Sensitivity in Selective
 *          KV-Cache Reuse for Rolling Agents: §2.2 Eqs. 1-2, §2.3 Eq. 3.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory    Every buffer argument is caller-owned.  Pointers documented as
 *           "device" must be device memory of the current CUDA device;
 *           "host" pointers are read during the call only.  The library
 *           never allocates device memory on the hot path: scratch space is
 *           the caller's workspace, sized by the matching *_workspace call.
 *           cb_model_create allocates only its small host-side descriptor.
 * Streams   Calls enqueue work on `stream` and return without waiting; a
 *           NULL stream is the legacy default stream.  Arguments read from
 *           host memory are consumed before the call returns.
 * Layout    Row-major.  A "row" of the KV cache is one token's keys (or
 *           values) for all kv heads: n_kv_heads * head_dim contiguous
 *           elements, head h at offset h * head_dim.  Leading dimensions
 *           (ld_*) and strides count elements, not bytes.
 * Dtypes    CB_F32 tensors are float; CB_BF16 tensors are bfloat16.  All
 *           accumulation is fp32.  RMSNorm gains, the residual stream,
 *           deviations and the RoPE table are always float.
 * Alignment Device base pointers and leading dimensions of bf16/f32 tensors
 *           must give 16-byte aligned rows; violations return
 *           CB_ERR_INVALID_ARG.
 * Errors    Host-side validation runs before anything is enqueued and
 *           returns a cb_status; the message is available from
 *           cb_last_error_message() (thread-local).  Failures detected on
 *           the device (an index out of range, a bounded wait that expired)
 *           are recorded in a per-device status word read by
 *           cb_get_device_status(); kernels never trap.
 */
#ifndef CACHEBLEND_H_
#define CACHEBLEND_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *cb_stream; /* same type as cudaStream_t */

typedef enum {
  CB_OK = 0,
  CB_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or layout */
  CB_ERR_UNSUPPORTED = 2,   /* dtype / shape / device not supported */
  CB_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  CB_ERR_TIMEOUT = 4,       /* a bounded device-side wait expired */
  CB_ERR_DEVICE_INDEX = 5,  /* a device-side index check failed */
  CB_ERR_WORKSPACE = 6      /* workspace pointer NULL or too small */
} cb_status;

typedef enum { CB_F32 = 0, CB_BF16 = 1 } cb_dtype;

typedef enum {
  CB_POLICY_TOKEN_TOPK = 0,   /* [ROM] §2.2: the k largest deviations       */
  CB_POLICY_DOC_ALIGNED = 1,  /* [ROM] §2.3: whole spans by mean deviation,
                                 then the best window of the remainder      */
  CB_POLICY_SINGLE_WINDOW = 2,/* [ROM] §2.3: the k-token window of largest
                                 total deviation over all reusable tokens   */
  CB_POLICY_FIXED_CHUNK = 3,  /* [ROM] §2.3, §4.4: equal spans of span_len
                                 tokens shifted by span_offset (they cross
                                 document boundaries), ranked and filled as
                                 DOC_ALIGNED                                 */
  CB_POLICY_RANDOM_DOC = 4,   /* [ROM] §2.3: document spans visited in the
                                 caller's span_order (its random draw),
                                 filled as DOC_ALIGNED                       */
  CB_POLICY_FIRST_TOKENS = 5, /* [QCF] §2 (EPIC's chunk-boundary rule): the
                                 first tokens of every span, k shared out
                                 evenly (the first k mod m spans one more; a
                                 short span passes its surplus on in order)  */
  CB_POLICY_QUERY_PROBE = 6,  /* [QCF] §3.3-3.4: per-chunk anchors (Eq. 14),
                                 the query rows probed over the anchor cache
                                 (Eqs. 15-17), P = top-k of their attention
                                 mass on the context summed over the
                                 critical layers (Eqs. 20, 11)               */
  CB_POLICY_QUERY_FULL = 7    /* [QCF] §3.2.1: the full-view reference
                                 (Eqs. 9-11): every context position is an
                                 anchor and every layer is critical          */
} cb_policy;

/* Anchor rule of [QCF] Eq. 14: the score G_i(r) of chunk-local position r. */
typedef enum {
  CB_ANCHOR_SINK = 0,   /* -r: the chunk's first positions                  */
  CB_ANCHOR_KNORM = 1   /* minus the squared L2 norm of the position's PIC
                           keys summed over all layers and kv heads: the
                           lowest-norm keys first                            */
} cb_anchor_rule;

/* Largest batch of requests one call accepts. */
#define CB_MAX_BATCH 64
/* Largest number of spans (documents) one selection call accepts. */
#define CB_MAX_SPANS 1024

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                              */
/* ------------------------------------------------------------------------ */

/* Message of the last failing call on this thread ("" if none). */
const char *cb_last_error_message(void);

/* Library ABI version (major * 100 + minor). */
int cb_version(void);

/* Reads and clears the device status word of the current device.  Blocks
 * until all work on the device has finished.  *out receives CB_OK or the
 * first device-side failure (CB_ERR_TIMEOUT, CB_ERR_DEVICE_INDEX) recorded
 * since the last read. */
cb_status cb_get_device_status(cb_status *out);

/* Runs one kernel whose single thread waits on a shared-memory mbarrier that
 * nothing ever completes, with a bounded wait of about `limit_us`
 * microseconds; the wait expires, the kernel records CB_ERR_TIMEOUT in the
 * device status word and returns.  Exercises the bounded-wait path used by
 * every pipelined kernel of the library without hanging the device. */
cb_status cb_debug_expire_wait(int limit_us, cb_stream stream);

/* Number of kernels this library has enqueued in this process (all devices,
 * all threads).  Benchmarks difference it around a region to count the
 * library's launches. */
unsigned long long cb_debug_launch_count(void);

/* Which bf16 tensor-core GEMM the library uses for every projection issued
 * after the call (process-wide):
 *   CB_GEMM_AUTO (0)     per epilogue, reduction length and row count, the
 *                        form measured fastest;
 *   CB_GEMM_TOKEN_M (1)  token rows on the MMA's M side (128-row tiles);
 *   CB_GEMM_SWAP_AB (2)  weight rows on M, tokens on N;
 *   CB_GEMM_SWAP_AB_PAIR (3)  the same with each MMA spanning a pair of SMs
 *                        (2-CTA cluster, 256 weight rows per tile).
 * All compute the same function; tests use the switch to check each one
 * on every epilogue.  Returns CB_ERR_INVALID_ARG for any other value. */
#define CB_GEMM_AUTO 0
#define CB_GEMM_TOKEN_M 1
#define CB_GEMM_SWAP_AB 2
#define CB_GEMM_SWAP_AB_PAIR 3
cb_status cb_debug_gemm_path(int path);

/* Whether a bf16 decoder layer runs its MLP (gate/up projection with SiLU
 * gating, then the down projection + residual) as one launch (on = 1, the
 * default) or as two (on = 0), for every call issued after this one
 * (process-wide).  In the one-launch form each down-projection k-block waits
 * only for the gate/up tile that wrote its 64 features (a flag in the
 * workspace), so the down projection starts while the last gate/up tiles
 * finish.  Both forms compute the same function; they differ in the order of
 * fp32 additions (partial sums of split tiles, residual accumulation).  The
 * one-launch form applies where both projections take the same swapped
 * GEMM form (cb_debug_gemm_path) and the flags fit (ceil(rows / 256) * d_ffn /
 * 64 <= 16384); otherwise the two launches run.  Returns CB_ERR_INVALID_ARG
 * for on not 0 or 1. */
cb_status cb_debug_mlp_fusion(int on);

/* 1 if a bf16 decoder layer over n_rows rows with these widths runs its MLP
 * as one launch under the current switches (cb_debug_mlp_fusion,
 * cb_debug_gemm_path), else 0 (two launches, or nonpositive arguments).
 * Host arithmetic only; benchmarks use it to attribute each layer's work to
 * the launch that does it. */
int cb_debug_mlp_one_launch(int n_rows, int d_model, int d_ffn);

/* Debug index checks (process-wide, off by default).  While on, every call
 * also validates the device-side index arrays it consumes before using them:
 * a blended prefill's selected positions (forced or ranked) and each gradual
 * step's kept positions must be strictly ascending per request and inside
 * [0, N_b); an attention call's query positions must ascend per request and
 * lie in [0, kv_len); a selection call's outputs must be strictly ascending
 * inside [0, n_ctx).  A violation records CB_ERR_DEVICE_INDEX in the device
 * status word (read with cb_get_device_status); nothing traps.  The checks
 * are extra launches, so they stay off on the fast path; they never change a
 * result.  Returns CB_ERR_INVALID_ARG for on not 0 or 1. */
cb_status cb_debug_index_checks(int on);

/* Launch probe: times the launches of one kernel class of the decoder layer
 * inside real calls.  After cb_debug_probe_start(kind, max_launches) every
 * launch of that class (up to max_launches, on any call's stream, outside
 * stream capture) is bracketed by two CUDA events on its own stream;
 * cb_debug_probe_stop waits for the recorded launches and returns their
 * count and summed device time in milliseconds, then releases the events.
 * The attention class includes its split-KV combine kernel; classes 6-9
 * bracket the once-per-call steps of cb_blend_prefill.  Debug use only
 * (one probe per process; start discards an unfinished probe). */
#define CB_PROBE_QKV 1       /* fused Q/K/V projection (+ RoPE, cache scatter) */
#define CB_PROBE_O 2         /* attention output projection + residual */
#define CB_PROBE_SWIGLU 3    /* gate/up projection with SiLU gating */
#define CB_PROBE_DOWN 4      /* down projection + residual */
#define CB_PROBE_ATTENTION 5 /* selected-query attention */
#define CB_PROBE_STITCH 6    /* re-position + stitch of the cached segments;
                                in cb_blend_prefill_host_kv, each layer's load
                                on copy_stream (copies, or the zero-copy
                                re-position) */
#define CB_PROBE_SELECT 7    /* deviation + ranking at the selection layer */
#define CB_PROBE_GATHER 8    /* computed-row list + hidden-state gather */
#define CB_PROBE_LM_HEAD 9   /* final norm + tied LM head + arg-max */
#define CB_PROBE_MLP 10      /* gate/up with SiLU gating, then down projection +
                                residual, as one launch (the bf16 default; see
                                cb_debug_mlp_fusion): classes 3 and 4 then
                                record nothing */
cb_status cb_debug_probe_start(int kind, int max_launches);
cb_status cb_debug_probe_stop(int *n_launches, float *total_ms);

/* ------------------------------------------------------------------------ */
/* RoPE table                                                               */
/* ------------------------------------------------------------------------ */

/* Number of floats of a RoPE table for positions [0, max_positions) and
 * head_dim: max_positions * (head_dim / 2) * 2 (cos, sin interleaved). */
size_t cb_rope_table_elems(int max_positions, int head_dim);

/* Fills table[p][e] = (cos(p * theta_e), sin(p * theta_e)) with
 * theta_e = rope_base^(-2e / head_dim), evaluated in double precision and
 * rounded to float.  table: device, cb_rope_table_elems() floats.
 * Errors: CB_ERR_INVALID_ARG for NULL table, head_dim odd or <= 0,
 * max_positions <= 0. */
cb_status cb_rope_table_init(float *table, int max_positions, int head_dim,
                             float rope_base, cb_stream stream);

/* ------------------------------------------------------------------------ */
/* Primitives of the hot path                                               */
/* ------------------------------------------------------------------------ */

/* One cached chunk to place into a request's cache ([QCF] Eq. 4). */
typedef struct {
  const void *k_src;         /* device: layer l, chunk row t at
                                k_src + l * src_layer_stride + t * row_elems */
  const void *v_src;         /* device, same layout as k_src                 */
  int64_t src_layer_stride;  /* elements between consecutive layers          */
  int len;                   /* rows in the chunk                            */
  int dst_row;               /* first destination row in the cache           */
  int delta;                 /* rotation to apply: request offset of the
                                chunk minus the position its keys were
                                computed at (0 for a standalone prefill)     */
} cb_stitch_desc;

/* Pi_i of [QCF] Eq. 4 for every chunk and every layer in
 * [layer_begin, layer_end): keys stored at chunk-local positions t are
 * rotated by delta (rotate-half pairs (e, e + head_dim/2), angle
 * delta * theta_e, [CB] "Why You Can't Just Concatenate": RoPE rotations
 * compose), values are copied unchanged:
 *   k_cache[l][dst_row + t] = R(delta) k_src[l][t]
 *   v_cache[l][dst_row + t] = v_src[l][t]
 * descs: host array of n_desc descriptors (any n_desc >= 0).
 * k_cache / v_cache: device, layer l at k_cache + l * cache_layer_stride.
 * rope_table: device table from cb_rope_table_init with
 *   max_positions > every |delta|.
 * Errors: CB_ERR_INVALID_ARG for NULL pointers, |delta| >= max_positions,
 *   head_dim not dividing row_elems, head_dim % 16 != 0, misalignment. */
cb_status cb_rope_reposition(const cb_stitch_desc *descs, int n_desc,
                             int layer_begin, int layer_end, void *k_cache,
                             void *v_cache, int64_t cache_layer_stride,
                             int row_elems, int head_dim,
                             const float *rope_table, int max_positions,
                             cb_dtype dtype, cb_stream stream);

/* One request of a selection call. */
typedef struct {
  int n_ctx;                 /* reusable context tokens N of the request     */
  int k;                     /* tokens to select, 0 <= k <= n_ctx            */
  int64_t fresh_row0;        /* row of context token 0 in k_fresh            */
  int64_t reused_row0;       /* row of context token 0 in k_reused           */
  int dev_offset;            /* first entry of this request in dev_out       */
  int idx_offset;            /* first entry of this request in idx_out       */
  int n_spans;               /* DOC_ALIGNED, RANDOM_DOC, FIRST_TOKENS: number
                                of spans (documents / chunks)                */
  const int32_t *span_offsets; /* host [n_spans + 1], ascending, from 0 to
                                  n_ctx: span j = [off[j], off[j+1])         */
  const int32_t *span_order; /* RANDOM_DOC: host [n_spans], a permutation of
                                the spans, first visited first               */
  int span_len;              /* FIXED_CHUNK: span length (> 0)              */
  int span_offset;           /* FIXED_CHUNK: the first span is [0, offset),
                                0 <= span_offset <= span_len                */
} cb_select_req;

/* Deviation and selection ([ROM] §2.2 Eqs. 1-2, §2.3 Eq. 3; [CB]
 * "Quantifying the Damage").  For every request b and context token i:
 *   d_i = sum_c (k_fresh[fresh_row0 + i][c] - k_reused[reused_row0 + i][c])^2
 * over the row_elems columns (all kv heads), computed in fp32, written to
 * dev_out[dev_offset + i].  Then the request's k tokens are selected:
 *   CB_POLICY_TOKEN_TOPK  -- the k largest d_i; equal values rank the lower
 *                            index first;
 *   CB_POLICY_DOC_ALIGNED -- spans ranked by mean d (ties: lower span),
 *                            whole spans while they fit, then the window of
 *                            the remaining length with the largest total d
 *                            (ties: leftmost) in the first span that does
 *                            not fit; span sums are accumulated in double;
 *   CB_POLICY_SINGLE_WINDOW, _FIXED_CHUNK, _RANDOM_DOC, _FIRST_TOKENS -- the
 *                            controls of the enum above (spans from
 *                            span_len / span_offset for FIXED_CHUNK, one
 *                            span [0, n_ctx) for SINGLE_WINDOW).
 * The selected context indices are written ascending to
 * idx_out[idx_offset .. idx_offset + k).
 * k_fresh, k_reused: device [rows][ld] of dtype.  dev_out: device float.
 * idx_out: device int32.  ws, ws_bytes: reserved; the selection needs no
 * scratch beyond dev_out, so ws may be NULL with ws_bytes 0 (a non-NULL ws
 * is not touched), and cb_select_workspace_size returns 0.
 * Errors: CB_ERR_INVALID_ARG (n_req > CB_MAX_BATCH, k > n_ctx, spans not
 *   covering [0, n_ctx] ascending, total spans > CB_MAX_SPANS). */
size_t cb_select_workspace_size(int n_req);
cb_status cb_kv_deviation_topk(const void *k_fresh, int64_t ld_fresh,
                               const void *k_reused, int64_t ld_reused,
                               int row_elems, cb_dtype dtype,
                               const cb_select_req *reqs, int n_req,
                               cb_policy policy, float *dev_out,
                               int32_t *idx_out, void *ws, size_t ws_bytes,
                               cb_stream stream);

/* The same deviation and selection as cb_kv_deviation_topk, for callers that
 * cannot allocate device memory (code enqueuing work while another component
 * owns every device allocation, or where an allocation's implicit device
 * synchronisation is not acceptable).  The pages have no counterpart: this
 * is an integration variant.  The per-token deviations live in a fixed 4 MiB
 * device array inside the library instead of caller memory, so a call takes
 * no dev_out and no workspace; req.dev_offset is ignored, whatever its
 * value (the library packs the deviations request after request), and the
 * selected indices go to idx_out exactly as in cb_kv_deviation_topk.
 * Limit: at most 1048576 context tokens (sum of n_ctx) per call; larger calls
 * return CB_ERR_INVALID_ARG and enqueue nothing.
 * The first call on each device resolves the array's device address, so make
 * it before capturing a stream into a CUDA graph.  Every call shares the
 * array (it keeps the last call's contents; nothing in it needs to start at
 * zero), so calls whose execution overlaps on the GPU race and must be
 * serialised by the caller.  The array is held by every device that loads
 * the library until the process exits.  Allocates nothing. */
cb_status cb_kv_deviation_topk_noalloc(const void *k_fresh, int64_t ld_fresh,
                                       const void *k_reused, int64_t ld_reused,
                                       int row_elems, cb_dtype dtype,
                                       const cb_select_req *reqs, int n_req,
                                       cb_policy policy, int32_t *idx_out,
                                       cb_stream stream);

/* Row gather ([CB] blend_layer step 1, h[hkvd_idx]):
 *   dst[i * ld_dst + c] = src[idx[i] * ld_src + c], i < n, c < row_elems.
 * idx: device int32 [n]; every idx[i] must lie in [0, src_rows); an index
 * outside records CB_ERR_DEVICE_INDEX and its row is skipped.
 * dtype applies to src and dst (CB_F32 or CB_BF16). */
cb_status cb_gather_rows(const void *src, int64_t ld_src, int64_t src_rows,
                         const int32_t *idx, int n, int row_elems, void *dst,
                         int64_t ld_dst, cb_dtype dtype, cb_stream stream);

/* Scatter of fresh K/V rows over the reused cache ([CB] blend_layer step 3;
 * [QCF] Eq. 7):
 *   k_cache[rows[i]] = k_new[i],  v_cache[rows[i]] = v_new[i],  i < n.
 * rows: device int32 [n], distinct, each in [0, cache_rows); an index outside
 * records CB_ERR_DEVICE_INDEX and is skipped. */
cb_status cb_scatter_kv(const void *k_new, const void *v_new, int64_t ld_new,
                        const int32_t *rows, int n, void *k_cache,
                        void *v_cache, int64_t ld_cache, int64_t cache_rows,
                        int row_elems, cb_dtype dtype, cb_stream stream);

/* One request of an attention call. */
typedef struct {
  int q_begin, q_end;   /* query rows [q_begin, q_end) of q / q_pos / out   */
  int64_t kv_row0;      /* cache row of position 0 of this request          */
  int kv_len;           /* positions of this request present in the cache   */
} cb_attn_req;

/* Selected-query attention over the blended cache ([CB] blend_layer step 4,
 * n_sel x L work; [QCF] §2.1.3: causal over the partially fused prefix).
 * For query row r of request b at position p = q_pos[r] (0 <= p < kv_len)
 * and q head h (kv head g = h / (n_q_heads / n_kv_heads)):
 *   out[r][h] = sum_{j<=p} softmax_j(scale * q[r][h] . K[j][g]) V[j][g]
 * with K[j] = k_cache[kv_row0 + j].  Queries of a request must have
 * ascending positions.  q, out: device [rows][ld] (n_q_heads * head_dim
 * columns); k_cache, v_cache: device [rows][ld_kv].  dtype applies to q,
 * the cache and out.  ws: device scratch of at least
 * cb_attention_workspace_size(...) bytes for the same requests (partial
 * results when the key range of a query tile is split across SMs; may be
 * 0 bytes).  Errors: CB_ERR_WORKSPACE if ws is too small; CB_ERR_INVALID_ARG (n_req > CB_MAX_BATCH,
 * head counts not dividing, head_dim not 64 or 128); a position outside
 * [0, kv_len) records CB_ERR_DEVICE_INDEX and the row is left unwritten. */
size_t cb_attention_workspace_size(const cb_attn_req *reqs, int n_req,
                                   int n_q_heads, int n_kv_heads, int head_dim,
                                   cb_dtype dtype);
cb_status cb_sparse_query_attention(const void *q, int64_t ld_q,
                                    const int32_t *q_pos,
                                    const cb_attn_req *reqs, int n_req,
                                    const void *k_cache, const void *v_cache,
                                    int64_t ld_kv, int n_q_heads,
                                    int n_kv_heads, int head_dim, float scale,
                                    void *out, int64_t ld_out, cb_dtype dtype,
                                    void *ws, size_t ws_bytes,
                                    cb_stream stream);

/* ------------------------------------------------------------------------ */
/* Model                                                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
  int n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ffn, vocab;
  float rope_base;      /* theta base of the rotary embedding               */
  float norm_eps;       /* RMSNorm epsilon                                   */
  cb_dtype dtype;       /* weights, activations fed to GEMMs, KV cache      */
  int max_positions;    /* rows of rope_table; > every position used        */
} cb_model_config;

/* Device pointers of one decoder layer (pre-norm, no biases):
 *   w_qkv  [(n_q_heads + 2 n_kv_heads) head_dim][d_model]  rows: W_q;W_k;W_v
 *   w_o    [d_model][n_q_heads head_dim]
 *   w_gate [d_ffn][d_model],  w_up [d_ffn][d_model]
 *   w_down [d_model][d_ffn]
 *   norm1, norm2: float [d_model] RMSNorm gains. */
typedef struct {
  const void *w_qkv, *w_o, *w_gate, *w_up, *w_down;
  const float *norm1, *norm2;
} cb_layer_weights;

typedef struct {
  const void *embed;              /* [vocab][d_model]; also the LM head     */
  const float *final_norm;        /* [d_model]                               */
  const cb_layer_weights *layers; /* host array [n_layers], copied           */
  const float *rope_table;        /* device, from cb_rope_table_init         */
} cb_weights;

typedef struct cb_model cb_model;

/* Records the configuration and weight pointers (no device memory is
 * allocated or copied; the weights must outlive the model).  Errors:
 * CB_ERR_INVALID_ARG for inconsistent shapes or NULL weights,
 * CB_ERR_UNSUPPORTED for head_dim not 64/128, d_model % 64 or > 8192, d_ffn % 16,
 * or a device older than sm_103 for CB_BF16. */
cb_status cb_model_create(const cb_model_config *cfg, const cb_weights *w,
                          cb_model **out);
void cb_model_destroy(cb_model *m);

/* ------------------------------------------------------------------------ */
/* Layer and stack                                                          */
/* ------------------------------------------------------------------------ */

/* Dense projection with a fused epilogue, out = f(A W^T):
 *   A [M][K] (ld_a), W [N][K] (ld_w) device, dtype of the model.
 *   CB_EPI_STORE   out[m][n] = acc             (out: dtype, ld_out)
 *   CB_EPI_RESID   out[m][n] += acc            (out: float residual stream)
 *   CB_EPI_SWIGLU  out[m][n] = silu(acc_g) * acc_u, with acc_g from W rows
 *                  and acc_u from W2 rows (W2 [N][K], same ld)
 * Errors: CB_ERR_INVALID_ARG for shapes not multiples of 16 in K, NULLs. */
typedef enum { CB_EPI_STORE = 0, CB_EPI_RESID = 1, CB_EPI_SWIGLU = 2 } cb_epilogue;
cb_status cb_linear(const cb_model *m, const void *A, int64_t ld_a,
                    const void *W, const void *W2, int64_t ld_w, int M, int N,
                    int K, cb_epilogue epi, void *out, int64_t ld_out,
                    cb_stream stream);

/* cb_linear with a device workspace of cb_linear_workspace_size() bytes
 * (16-byte aligned, owned by the caller, contents need no initialisation).
 * With it the bf16 swapped-operand forms split the tiles of a partial last
 * wave along K over the otherwise idle SMs: the later k-segments leave fp32
 * partials there and the unit of segment 0 adds them in segment order, so
 * results stay deterministic.  CB_EPI_RESID does not use it (its stream-K
 * adds into the residual).  Calls that share a workspace must be ordered on
 * one stream.  ws == NULL is cb_linear.  Errors: as cb_linear, and
 * CB_ERR_WORKSPACE when ws is too small or misaligned. */
size_t cb_linear_workspace_size(void);
cb_status cb_linear_ws(const cb_model *m, const void *A, int64_t ld_a,
                       const void *W, const void *W2, int64_t ld_w, int M, int N,
                       int K, cb_epilogue epi, void *out, int64_t ld_out,
                       void *ws, size_t ws_bytes, cb_stream stream);

/* A run of request tokens: cached (k_pic != NULL) or recomputed at every
 * layer (k_pic == NULL: the user query U, or a document that has no cache
 * yet).  All cached segments of a request come before its uncached ones;
 * the N cached tokens are the reusable context C of [QCF] Eq. 1. */
typedef struct {
  int len;
  const void *k_pic;        /* device [n_layers] x [len rows], layer l at
                               k_pic + l * pic_layer_stride; keys computed
                               standalone at positions pic_pos0 ..          */
  const void *v_pic;
  int64_t pic_layer_stride; /* elements between layers of the PIC cache   */
  int pic_pos0;             /* position the chunk's keys were computed at
                               (0 for a standalone chunk prefill)           */
} cb_segment;

typedef struct {
  const int32_t *tokens;        /* device int32 [T], T = sum of lens        */
  const cb_segment *segments;   /* host [n_segments]                         */
  int n_segments;
} cb_request;

/* One gradual-filtering step ([CB] select_hkvd): before layer `layer`, the
 * context rows still selected are ranked again by the deviation of their
 * fresh keys of that layer from the reused keys in its fused cache, and
 * each request keeps its min(keep, current count) largest (ties to the
 * lower position); the uncached rows are always kept. */
typedef struct {
  int layer;  /* > sel_layer (and > the previous step's layer), < n_layers */
  int keep;   /* >= 0: selected rows kept per request from this layer on    */
} cb_schedule_step;

typedef struct {
  int ratio_bp;        /* recompute ratio r in basis points (1500 = 15%)    */
  cb_policy policy;
  int sel_layer;       /* selection layer s; layers < s run on every row    */
  int n_schedule;      /* gradual filtering steps ([CB] select_hkvd), 0 = a
                          single selection reused by every later layer     */
  const cb_schedule_step *schedule;   /* host [n_schedule], layers ascending */
  int span_len;        /* FIXED_CHUNK: span length; 0 = the median length
                          of the request's cached segments, shifted by half
                          a span (the spans then straddle documents)        */
  int span_offset;     /* FIXED_CHUNK with span_len > 0: first span [0, off) */
  const int32_t *span_order;  /* RANDOM_DOC: host, per request in order, a
                          permutation of its cached segments                */
  const int32_t *forced_selected;     /* device [K_total] or NULL: use these
                          request-local context positions (ascending per
                          request, k_b of them) instead of ranking d; d is
                          still computed.  Lets an external selector (or a
                          reference run) fix P.  A position outside
                          [0, N_b) records CB_ERR_DEVICE_INDEX.            */
  /* CB_POLICY_QUERY_PROBE: anchors and critical layers.  Both query
     policies select before layer 0 (sel_layer and the schedule must be 0):
     every layer recomputes P and the uncached rows, and `deviation` of the
     outputs receives the score I(t) in place of d. */
  cb_anchor_rule anchor_rule;
  int anchor_bp;       /* r_a in basis points: ceil(r_a |c_i|) anchors per
                          chunk                                             */
  int n_crit;          /* the critical-layer set L*: n_crit >= 1 distinct  */
  const int32_t *crit_layers; /* host [n_crit] layers in [0, n_layers)     */
  const int32_t *forced_kept; /* device or NULL, used with a schedule: the
                          context positions each gradual step keeps, step
                          after step, each step's requests in order (k'_b
                          ascending request-local positions per request, a
                          subset of the rows selected before the step),
                          taken instead of ranking the step's deviations --
                          the per-step counterpart of forced_selected.  A
                          position that is not in the current selection, or
                          out of order, records CB_ERR_DEVICE_INDEX.       */
  int host_load_ctas;  /* cb_blend_prefill_host_kv only.  0: the copy
                          engines copy each layer's chunk caches into a
                          staging area, then they are re-positioned.  > 0:
                          the re-position kernel itself reads the pinned
                          chunk caches (zero-copy) on copy_stream with at
                          most this many CTAs per layer, which bounds the
                          load bandwidth (a slower storage tier is emulated
                          by a small count) and needs no staging area.
                          0 .. 4096.                                       */
  const int32_t *anchors; /* CB_POLICY_QUERY_PROBE only.  NULL: the library
                          ranks every chunk's anchors by anchor_rule
                          ([QCF] Eq. 14).  Else device int32: the anchors of
                          every cached segment -- request by request,
                          segments in order, each chunk's ceil(anchor_bp
                          |c| / 10^4) chunk-local positions ascending, the
                          layout cb_anchor_select writes.  A store can keep
                          them with its chunks: the Knorm scores depend only
                          on a chunk's own keys.  A position outside its
                          chunk records CB_ERR_DEVICE_INDEX.               */
} cb_blend_params;

/* Per-chunk anchors of [QCF] Eq. 14, as the offline cache preparation of
 * [QCF] §3.1 would store them: for each of n_chunks cached segments (given
 * as for cb_request, k_pic read on the device), the scores G_i(r) of its
 * positions by `rule` (cb_anchor_rule), then A_i = the ceil(ratio_bp |c_i| /
 * 10000) highest (equal scores: the lower position first), ascending
 * chunk-local positions.
 *   scores_out:  device float [sum len] or NULL, chunk after chunk;
 *   anchors_out: device int32 [sum ceil(...)], chunk after chunk.
 * ws: device workspace of cb_anchor_workspace_size(n_chunks) bytes.
 * Errors: CB_ERR_INVALID_ARG (NULL pointers, ratio_bp outside [0, 10000],
 * a bad rule or PIC layout), CB_ERR_WORKSPACE. */
size_t cb_anchor_workspace_size(const cb_model *m, const cb_segment *chunks, int n_chunks);
cb_status cb_anchor_select(const cb_model *m, const cb_segment *chunks, int n_chunks,
                           cb_anchor_rule rule, int ratio_bp, float *scores_out,
                           int32_t *anchors_out, void *ws, size_t ws_bytes, cb_stream stream);

/* Outputs of a prefill call.  The fused cache of request b occupies rows
 * [t_off_b, t_off_b + T_b) of every layer, t_off_b = sum_{c<b} T_c. */
typedef struct {
  void *k_cache, *v_cache;   /* device; layer l at + l * cache_layer_stride */
  int64_t cache_layer_stride;/* elements; 0 means T_total * row_elems       */
  float *deviation;          /* device [N_total] or NULL (d at layer s)     */
  int32_t *selected;         /* device [K_total] or NULL: request-local
                                context positions selected at the last
                                layer, ascending per request; the first
                                K_final entries are used (request b's k'_b
                                after the requests before it)               */
  float *hidden;             /* device [R_total][d_model] or NULL: final
                                hidden states (before the final norm) of the
                                rows computed at the last layer (R_final
                                rows, packed per request)                   */
  int32_t *rows;             /* device [R_total] or NULL: request-local
                                positions of those rows, ascending per
                                request                                      */
  int32_t *first_token;      /* device [B] or NULL: argmax of the last row's
                                logits (LM head tied to the embedding)      */
} cb_blend_out;

typedef struct {
  int64_t T_total;           /* rows of the fused cache (all requests)      */
  int64_t N_total;           /* reusable context tokens                     */
  int64_t K_total;           /* context tokens selected at sel_layer        */
  int64_t R_total;           /* rows computed at sel_layer (K_total plus the
                                uncached rows)                              */
  size_t workspace_bytes;    /* workspace for cb_blend_prefill / full      */
  int64_t K_final;           /* selected tokens after the last gradual step
                                (K_total without a schedule)                */
  int64_t R_final;           /* rows computed at the last layer             */
} cb_plan;

/* Sizes of a blended prefill.  k_b = floor(N_b * ratio_bp / 10000), at
 * least 1 when ratio_bp > 0 and N_b > 0 ([ROM] Eq. 2). */
cb_status cb_blend_plan(const cb_model *m, const cb_request *reqs, int B,
                        const cb_blend_params *p, cb_plan *out);

/* Blended prefill of B independent requests ([QCF] §2.1.3 Eqs. 4-7; [CB]
 * blend_layer; [ROM] §2.2 flow):
 *   1. stitch: every cached segment is re-positioned into the fused cache
 *      at layers >= sel_layer (cb_rope_reposition);
 *   2. layers < sel_layer run on every row (their cache is fresh);
 *   3. at sel_layer every row's keys are projected fresh, d is ranked
 *      (cb_kv_deviation_topk) and the selected context rows plus all
 *      uncached rows form the computed set;
 *   4. layers >= sel_layer compute only that set: fresh K/V replace the
 *      reused rows (Eq. 7) and the set attends over the fused cache;
 *   5. final norm + LM head + argmax of each request's last row.
 * Every step runs in this library's kernels on `stream`; nothing is
 * synchronised.  ws: device workspace of >= cb_plan.workspace_bytes.
 * Recorded calls: on a stream other than the legacy default stream (and one
 * the caller is not capturing), the second call with the same host
 * arguments (every field above, host arrays by content, device buffers by
 * address) records its launches into a CUDA graph held by the model, and
 * later such calls replay it; the device data behind the pointers is read
 * when the replay runs.  The model keeps the 4 most recently used
 * recordings; cb_model_destroy releases them.
 * Errors: CB_ERR_INVALID_ARG (B > CB_MAX_BATCH, a request whose cached
 *   segments do not all precede its uncached ones, a request that ends in
 *   a cached segment, positions >= max_positions), CB_ERR_WORKSPACE. */
cb_status cb_blend_prefill(cb_model *m, const cb_request *reqs, int B,
                           const cb_blend_params *p, const cb_blend_out *out,
                           void *ws, size_t ws_bytes, cb_stream stream);

/* The same blended prefill with the chunk caches in pinned host memory
 * ([CB] "Hiding Recompute Behind I/O"; [QCF] §4.4, layer-wise pipeline):
 * every cached segment's k_pic / v_pic must be pinned (page-locked) host
 * memory with the usual layer stride.  Layer l's slice of every segment is
 * copied by the copy engines, on copy_stream, into a two-layer staging area
 * of the workspace and re-positioned into the fused cache just before
 * layer l runs on `stream`, so loading layer l + 2 overlaps computing layer
 * l.  The copy stream is forked from and joined back into `stream` with the
 * model's events, so a call can be captured into a CUDA graph; calls that
 * share a model must be issued one at a time.  Results are those of
 * cb_blend_prefill.  Workspace: cb_blend_plan_host_kv (cb_blend_plan plus
 * the staging area, 4 * N_total * row_elems * dtype bytes).
 * The query-aware policies load the layers their probe reads first: the
 * anchor probe layers 0 .. max(L*) before its cache gather, the full view
 * each layer just before its probe layer; the later layers' loads overlap
 * the probe and the blend.  With CB_ANCHOR_KNORM the anchor scores read
 * every layer's chunk keys from the host memory in a kernel.
 * Errors: as cb_blend_prefill; CB_ERR_INVALID_ARG when a chunk cache is not
 * pinned host memory, when a kernel reads it (host_load_ctas > 0, or the
 * key-norm anchor rule) and the host pointer is not also its device
 * address, or when copy_stream is NULL or equal to stream. */
cb_status cb_blend_plan_host_kv(const cb_model *m, const cb_request *reqs, int B,
                                const cb_blend_params *p, cb_plan *out);
cb_status cb_blend_prefill_host_kv(cb_model *m, const cb_request *reqs, int B,
                                   const cb_blend_params *p, const cb_blend_out *out,
                                   void *ws, size_t ws_bytes, cb_stream stream,
                                   cb_stream copy_stream);

/* Loading controller of [CB] "Hiding Recompute Behind I/O": with the chunk
 * caches loaded layer by layer, recomputing a fraction r of the tokens is
 * free while its per-layer compute time stays within the per-layer K/V load
 * time, so r = max(r_load, r_min), r_load the largest of the n measured
 * ratios ratio_bp[i] whose recompute_ms_per_layer[i] <= load_ms_per_layer
 * (r_min = min_ratio_bp, the page's 15% quality floor, 1500).
 * ratio_bp, recompute_ms_per_layer: host [n].  *ratio_out: the chosen ratio
 * in basis points.  Host only (no device work).  Errors:
 * CB_ERR_INVALID_ARG for n < 0, NULL arrays with n > 0, ratios outside
 * [0, 10000], a negative or NaN time. */
cb_status cb_loading_ratio(double load_ms_per_layer, const int32_t *ratio_bp,
                           const double *recompute_ms_per_layer, int n,
                           int32_t min_ratio_bp, int32_t *ratio_out);

/* Diagnostics of selections ([ROM] §4.4, Table 2): for request b of a
 * selection (reqs[b].n_ctx, .k, .dev_offset, .idx_offset as for
 * cb_kv_deviation_topk; the other fields are ignored), the number of
 * separate contiguous regions its selected positions occupy (maximal runs
 * of consecutive positions) and the share of the request's total deviation
 * the selected tokens carry (sum of d over the selection / sum over all
 * n_ctx, 0 when the total is 0; sums in double).
 * dev: device float deviations; idx: device int32 selections, ascending per
 * request.  segments_out: device int32 [n_req]; captured_out: device double
 * [n_req].  An index outside [0, n_ctx) records CB_ERR_DEVICE_INDEX and is
 * skipped.  Errors: CB_ERR_INVALID_ARG (NULL pointers, n_req outside
 * [0, CB_MAX_BATCH], k > n_ctx, negative offsets). */
cb_status cb_selection_stats(const float *dev, const int32_t *idx,
                             const cb_select_req *reqs, int n_req,
                             int32_t *segments_out, double *captured_out,
                             cb_stream stream);

/* Number of anchors cb_anchor_select writes for these chunks: the sum over
 * chunks of ceil(ratio_bp |c_i| / 10000) ([QCF] Eq. 14).  Errors:
 * CB_ERR_INVALID_ARG (NULL pointers, n_chunks < 0, a negative length,
 * ratio_bp outside [0, 10000]). */
cb_status cb_anchor_count(const cb_segment *chunks, int n_chunks, int ratio_bp,
                          int64_t *n_anchors);

/* Full prefill ([QCF] Eq. 2): every row of every layer is computed under
 * the whole request (segments' caches are ignored).  Fills k_cache,
 * v_cache, hidden (all T rows), rows (0..T_b-1) and first_token of `out`.
 * A standalone chunk prefill ([QCF] Eq. 3) is a full prefill of a request
 * holding just the chunk's tokens.  Workspace: cb_full_plan. */
cb_status cb_full_plan(const cb_model *m, const cb_request *reqs, int B,
                       cb_plan *out);
cb_status cb_full_prefill(cb_model *m, const cb_request *reqs, int B,
                          const cb_blend_out *out, void *ws, size_t ws_bytes,
                          cb_stream stream);

/* One blended decoder layer on a compact set of rows ([CB] blend_layer
 * with hidden states kept compact):
 *   x = RMSNorm(h; norm1); q, k, v = x W_qkv^T with RoPE on q and k at
 *   pos[i]; k, v written to cache row cache_row[i] (Eq. 7); the rows attend
 *   over the layer's cache; h += attn W_o^T; h += SwiGLU(RMSNorm(h)) W_down^T.
 * h: device float [n_rows][d_model], updated in place.  pos, cache_row:
 * device int32 [n_rows], ascending per request.  reqs: host, one per
 * request (q_begin/q_end index h rows).  k_cache, v_cache: device, this
 * layer's cache [rows][n_kv_heads * head_dim].  ws: device workspace of at
 * least cb_layer_workspace_size(m, n_rows) bytes. */
size_t cb_layer_workspace_size(const cb_model *m, int n_rows);
cb_status cb_blend_layer(cb_model *m, int layer, float *h, int n_rows,
                         const int32_t *pos, const int32_t *cache_row,
                         const cb_attn_req *reqs, int n_req, void *k_cache,
                         void *v_cache, void *ws, size_t ws_bytes,
                         cb_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* CACHEBLEND_H_ */
