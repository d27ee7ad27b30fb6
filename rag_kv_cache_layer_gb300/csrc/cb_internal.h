// Host-side interface between the C ABI (cb_api.cu) and the kernel files.
// Every launcher takes plain device pointers and a stream, enqueues its
// kernel(s) and returns the launch error.  Nothing here allocates.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

#include "cacheblend.h"

namespace cb {

// Per-request row bookkeeping of one call, passed to kernels by value.
//   t_off: first fused-cache row of each request (prefix sums of T_b)
//   n_ctx: reusable context tokens N_b (they are positions 0..N_b-1)
//   k_off: prefix sums of the selected counts k_b
//   r_off: prefix sums of the computed rows R_b = k_b + (T_b - N_b)
struct BatchMeta {
  int B;
  int t_off[CB_MAX_BATCH + 1];
  int n_ctx[CB_MAX_BATCH];
  int k_off[CB_MAX_BATCH + 1];
  int r_off[CB_MAX_BATCH + 1];
};

// Device address of this library's status word on the current device.
int *device_status_ptr();

// Number of devices the per-device caches below cover.
constexpr int kMaxDevices = 64;

// One-time host set-up per device (a kernel's function attributes, an
// occupancy query): such state belongs to each device's context, so it is
// done once for every device the library runs on.  run(f) calls f() with the
// current device's index until it first returns cudaSuccess; concurrent
// first calls from several threads are serialised.
class PerDeviceOnce {
 public:
  template <typename F>
  cudaError_t run(F &&f) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu_);
    if (done_[dev]) return cudaSuccess;
    e = f(dev);
    if (e == cudaSuccess) done_[dev] = true;
    return e;
  }

 private:
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

// Streaming multiprocessors of the current device (queried once per device).
int device_sm_count();

// Sets the thread's cb_last_error_message and returns s.
cb_status record_error(cb_status s, const char *msg);

// Counts kernels enqueued by the library (read through
// cb_debug_launch_count); launchers call launched(n) after n launches.
void note_launches(int n);
inline cudaError_t launched(int n) {
  note_launches(n);
  return cudaGetLastError();
}

// Launches a kernel that follows the grid_dep_wait / grid_dep_launch
// protocol with programmatic stream serialization, so its setup overlaps
// the end of the previous kernel on the stream.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------- RoPE --
cudaError_t launch_rope_table(float *table, int max_pos, int head_dim,
                              float base, cudaStream_t s);
// max_blocks > 0 caps the grid's x extent (a bandwidth-bounded zero-copy
// load when the sources are pinned host memory).
cudaError_t launch_reposition(const cb_stitch_desc *descs, int n_desc,
                              int layer_begin, int layer_end, void *k_cache,
                              void *v_cache, int64_t cache_layer_stride,
                              int row_elems, int head_dim, const float *table,
                              cb_dtype dt, int *status, cudaStream_t s,
                              int max_blocks = 0);

// ------------------------------------------------------------ selection --
struct SelReq {
  int n_ctx, k;
  int64_t fresh_row0, reused_row0;
  int dev_offset, idx_offset;
  int span_begin, n_spans;  // into the packed span-offset array
};
size_t select_ws_bytes(int n_req);
cudaError_t launch_deviation(const void *k_fresh, int64_t ld_fresh,
                             const void *k_reused, int64_t ld_reused,
                             int row_elems, cb_dtype dt, const SelReq *reqs,
                             int n_req, float *dev_out, cudaStream_t s,
                             const int32_t *reused_rows = nullptr);
// With reused_rows, the reused key of fresh row f is row
// reused_row0 + reused_rows[f] instead of reused_row0 + i.
cudaError_t launch_topk(const float *dev, const SelReq *reqs, int n_req,
                        int32_t *idx_out, cudaStream_t s);
// Deviations from per-head partials (EPI_KDEV): d[dev_offset + i] =
// sum over h < n_parts of parts[h * part_stride + dev_offset + i], summed in
// head order (deterministic).  launch_topk_parts also ranks them (token
// top-k, as launch_topk) in the same kernel.
cudaError_t launch_reduce_parts(const float *parts, int n_parts, int64_t part_stride,
                                const SelReq *reqs, int n_req, float *dev_out, cudaStream_t s);
cudaError_t launch_topk_parts(const float *parts, int n_parts, int64_t part_stride,
                              const SelReq *reqs, int n_req, float *dev_out, int32_t *idx_out,
                              cudaStream_t s);
// A selection call after validation: the requests, their packed spans and,
// per span, the visiting order (random document) or the token counts
// (first tokens).  make_sel_plan builds the spans every policy uses.
struct SelPlan {
  cb_policy policy = CB_POLICY_TOKEN_TOPK;
  std::vector<SelReq> reqs;
  std::vector<int32_t> spans, aux;
};
cb_status make_sel_plan(const cb_select_req *reqs, int n_req, cb_policy policy, SelPlan &out,
                        const char **err);
// The ranking of a plan over deviations already in dev (top-k or spans).
cudaError_t launch_selection(const float *dev, const SelPlan &plan, int32_t *idx_out,
                             int *status, cudaStream_t s);
cudaError_t launch_build_rows(const BatchMeta &bm, const int32_t *sel,
                              int32_t *pos, int32_t *glob, int n_rows,
                              int *status, cudaStream_t s);
// launch_build_rows followed by the gather of the rows' hidden states
// (h_dst[r] = h_src[glob[r]], d floats, d % 4 == 0), in one kernel.
cudaError_t launch_rows_gather(const BatchMeta &bm, const int32_t *sel, int32_t *pos,
                               int32_t *glob, int n_rows, const float *h_src, int d,
                               float *h_dst, int *status, cudaStream_t s);
// One gradual-filtering step: from the current rows (cur) to the rows kept
// (nxt, same requests, k'_b <= k_b); keep holds k'_b ascending local
// indices per request at nxt.k_off[b].
cudaError_t launch_filter_rows(const BatchMeta &cur, const BatchMeta &nxt,
                               const int32_t *keep, const int32_t *sel_cur,
                               int32_t *sel_nxt, int32_t *pos, int32_t *glob,
                               int32_t *src, int n_rows, int *status, cudaStream_t s);
// The keep indices of a gradual step whose kept positions are given:
// forced holds each request's k'_b positions at nxt.k_off[b], a subset of
// its current selection sel_cur (cur.k_off[b] ..).
cudaError_t launch_keep_from_positions(const BatchMeta &cur, const BatchMeta &nxt,
                                       const int32_t *forced, const int32_t *sel_cur,
                                       int32_t *keep, int n_keep, int *status, cudaStream_t s);
// dev_idx (may be NULL): for row r of request b at position p, the index
// n_off[b] + p of its deviation when p < n_ctx[b] (reusable context), else
// -1; n_off: prefix sums of n_ctx.
// Debug index check: for each of n_seg segments s, the entries
// idx[off[s] .. off[s + 1]) must lie in [0, hi[s]) and ascend (strictly
// when `strict`); a violation records CB_ERR_DEVICE_INDEX.
struct IndexCheck {
  int n_seg, strict;
  int off[CB_MAX_BATCH + 1];
  int hi[CB_MAX_BATCH];
};
cudaError_t launch_index_check(const int32_t *idx, const IndexCheck &c, int *status,
                               cudaStream_t s);
// Whether the debug index checks are on (cb_debug_index_checks).
bool index_checks_on();
cudaError_t launch_iota_rows(const BatchMeta &bm, int32_t *pos, int32_t *glob,
                             int n_rows, cudaStream_t s, int32_t *dev_idx = nullptr);
// Per request: contiguous regions of its selection and the share of its
// deviation the selection carries (Table 2 diagnostics).
cudaError_t launch_selection_stats(const float *dev, const int32_t *idx, const SelReq *reqs,
                                   int n_req, int32_t *segments, double *captured, int *status,
                                   cudaStream_t s);

// ----------------------------------------------------------------- rows --
cudaError_t launch_embed(const int32_t *const *tokens, const BatchMeta &bm,
                         const void *embed, int vocab, int d, cb_dtype dt,
                         float *h, int *status, cudaStream_t s);
cudaError_t launch_rmsnorm(const float *h, int64_t ld_h, const int32_t *src_rows,
                           int n, int d, const float *gain, float eps,
                           void *out, int64_t ld_out, cb_dtype out_dt,
                           cudaStream_t s);
cudaError_t launch_gather(const void *src, int64_t ld_src, int64_t src_rows,
                          const int32_t *idx, int n, int row_elems, void *dst,
                          int64_t ld_dst, size_t elem_bytes, int *status,
                          cudaStream_t s);
// launch_gather for layers [0, n_layers) in one launch: layer l from
// src + l * src_lstride to dst + l * dst_lstride (elements).
cudaError_t launch_gather_layers(const void *src, int64_t src_lstride, int64_t ld_src,
                                 int64_t src_rows, const int32_t *idx, int n, int row_elems,
                                 void *dst, int64_t dst_lstride, int64_t ld_dst, size_t eb,
                                 int n_layers, int *status, cudaStream_t s);
cudaError_t launch_scatter_kv(const void *k_new, const void *v_new,
                              int64_t ld_new, const int32_t *rows, int n,
                              void *k_cache, void *v_cache, int64_t ld_cache,
                              int64_t cache_rows, int row_elems,
                              size_t elem_bytes, int *status, cudaStream_t s);
// qkv [n][(Hq + 2 Hkv) hd] float -> q (rotated), k (rotated) and v rows.
// k and v go to k_dst[dst_rows[i]] / v_dst[dst_rows[i]] (ld_kv); when
// v_dst is NULL only keys are produced (q_out may be NULL).
cudaError_t launch_qkv_finish(const float *qkv, int64_t ld_qkv, int n,
                              const int32_t *pos, const int32_t *dst_rows,
                              int Hq, int Hkv, int hd, const float *table,
                              void *q_out, int64_t ld_q, void *k_dst,
                              void *v_dst, int64_t ld_kv, cb_dtype dt,
                              int k_col0, cudaStream_t s);
// logits = RMSNorm(h[row_b]) E^T for each request b, argmax -> token[b];
// last_rows_host: host array of the B rows of h to use.
cudaError_t launch_lm_head_argmax(const float *h, int64_t ld_h,
                                  const int32_t *last_rows_host, int B,
                                  const float *final_norm, float eps,
                                  const void *embed, int vocab, int d,
                                  cb_dtype dt, float *x_scratch,
                                  unsigned long long *best_scratch,
                                  int32_t *token_out, cudaStream_t s);
cudaError_t launch_copy_f32(float *dst, const float *src, size_t n,
                            cudaStream_t s);

// ----------------------------------------------------------------- GEMM --
enum GemmEpi {
  EPI_STORE_F32 = 0,
  EPI_STORE = 1,
  EPI_RESID = 2,
  EPI_SWIGLU = 3,
  EPI_QKV = 4,
  EPI_KDEV = 5,  // keys -> per-head deviation partials (bf16 swapped GEMM only)
  EPI_MLP = 6    // gate/up + SwiGLU, then down + residual, in one launch (launch_gemm_mlp)
};
// out = epi(A[M][K] W[N][K]^T); A and W of dtype dt; STORE_F32 and RESID
// write float, STORE and SWIGLU write dt.
cudaError_t launch_gemm_simt(const void *A, int64_t lda, const void *W,
                             const void *W2, int64_t ldw, int M, int N, int K,
                             GemmEpi epi, void *out, int64_t ldo, cb_dtype dt,
                             cudaStream_t s);

// Arguments of the fused Q/K/V epilogue: q heads (rotated at pos[m]) go to
// out[m], k heads (rotated) and v heads to cache row dst_row[m] of k_cache /
// v_cache (this layer's cache, row stride ld_kv).  head_dim must be 128.
//
// EPI_KDEV ("Request Order Matters" §2.2 Eq. 1 at the selection layer): the
// GEMM's weights are the key rows W_k only, so tile h is kv head h.  Each
// token's fresh key head is rotated at pos[m] and compared with the reused
// key in k_cache at row dst_row[m] (this layer's fused cache, holding the
// stitched chunk caches); the squared difference summed over the head's
// 128 features goes to out[h * ldo + dev_idx[m]] (fp32).  Tokens with
// dev_idx[m] < 0 (not reusable context) are skipped.  The fresh keys are
// never stored.
struct QkvEpi {
  const int32_t *pos;
  const int32_t *dst_row;
  void *k_cache, *v_cache;
  int64_t ld_kv;
  const float *rope;  // cb_rope_table_init layout
  int n_q_heads, n_kv_heads;
  const int32_t *dev_idx = nullptr;   // EPI_KDEV only
};
// bf16 tcgen05 GEMM (sm_103a); qkv is read for EPI_QKV only.
cudaError_t launch_gemm_tc(const void *A, int64_t lda, const void *W,
                           const void *W2, int64_t ldw, int M, int N, int K,
                           GemmEpi epi, void *out, int64_t ldo,
                           const QkvEpi *qkv, int *status, cudaStream_t s);
// The same GEMM with the operands swapped (weights on the MMA's M side,
// tokens on N).  gemm_auto_form picks the form for a shape: 0 = token rows
// on M (launch_gemm_tc), 1 or 2 = swapped with that many CTAs per MMA.
int gemm_auto_form(int M, int K, GemmEpi epi);
// cta_group 2 runs each MMA on a pair of SMs (a 2-CTA cluster): 256 weight
// rows per tile, the token operand split between the two CTAs.
// split_ws (may be NULL, gemm_split_ws_bytes() bytes) lets the non-residual
// epilogues split the tiles of a partial last wave along K; the 32-bit
// counters at gemm_split_flags_offset() must be zero before the first launch
// that uses the workspace, and each launch leaves them zero.  Launches that
// share one workspace must be ordered on one stream.
cudaError_t launch_gemm_sab(const void *A, int64_t lda, const void *W,
                            const void *W2, int64_t ldw, int M, int N, int K,
                            GemmEpi epi, void *out, int64_t ldo,
                            const QkvEpi *qkv, int *status, cudaStream_t s,
                            int cta_group = 1, void *split_ws = nullptr);
size_t gemm_split_ws_bytes();
size_t gemm_split_flags_offset();
// The MLP of a decoder layer as one persistent launch of the swapped GEMM:
// g = silu(x Wg^T) * (x Wu^T) (bf16 [M][F]), then h += g Wd^T (fp32,
// stream-K).  Each down-projection k-block waits only for the gate/up tile
// that wrote its 64 features of g for its token tile: that tile's epilogue
// sets a flag to `epoch` after its stores, so the down projection runs
// while the last gate/up tiles drain instead of after the whole launch.
// The flags live in split_ws at gemm_mlp_flags_offset(); they must hold
// values below `epoch` (zero them with the tail-split counters, then give
// every launch on the workspace a larger epoch).  cudaErrorNotSupported:
// the shapes do not fit one launch; run the two projections instead.
cudaError_t launch_gemm_mlp(const void *x, int64_t ldx, const void *w_gate, const void *w_up,
                            int64_t ldw, const void *w_down, int64_t ldwd, int M, int F, int d,
                            void *g, int64_t ldg, float *h, int64_t ldh, int *status,
                            cudaStream_t s, int cta_group, void *split_ws, int epoch);
size_t gemm_mlp_flags_offset();
// Whether launch_gemm_mlp takes M rows with F-wide gate/up features.
bool gemm_mlp_fits(int M, int F, int cta_group);

// ------------------------------------------------------------ attention --
struct AttnReq {
  int q_begin, q_end;
  int64_t kv_row0;
  int kv_len;
};
cudaError_t launch_attention_simt(const void *q, int64_t ld_q,
                                  const int32_t *q_pos, const AttnReq *reqs,
                                  int n_req, const void *k_cache,
                                  const void *v_cache, int64_t ld_kv, int Hq,
                                  int Hkv, int hd, float scale, void *out,
                                  int64_t ld_out, cb_dtype dt, int *status,
                                  cudaStream_t s);

// bf16 tcgen05 attention (head_dim 128, group size 1/2/4/8); queries of a
// request ascending by position.
// Scratch: attention_tc_ws_bytes for a given call (0 when its key ranges
// are not split); attention_tc_ws_bound covers any call on this device.
bool attention_tc_supported(int Hq, int Hkv, int hd);
size_t attention_tc_ws_bytes(const AttnReq *reqs, int n_req, int Hq, int Hkv);
size_t attention_tc_ws_bound();
// plan: a unit table from launch_attention_plan for these requests and query
// positions, or nullptr for a uniform split of every tile's key range.  With
// a table the scratch is at most attention_tc_ws_bound.
cudaError_t launch_attention_tc(const void *q, int64_t ld_q, const int32_t *q_pos,
                                const AttnReq *reqs, int n_req, const void *k_cache,
                                const void *v_cache, int64_t ld_kv, int Hq, int Hkv,
                                float scale, void *out, int64_t ld_out, void *ws,
                                size_t ws_bytes, int *status, cudaStream_t s,
                                const int *plan = nullptr);
// Unit table for launch_attention_tc, built on the device from the query
// positions: every tile's key range is cut so that all units run in one wave
// of CTAs.  Valid for as long as the requests and q_pos stay the same (the
// compact layers of one blended call share it).
size_t attention_plan_bytes(const AttnReq *reqs, int n_req, int Hq, int Hkv);
cudaError_t launch_attention_plan(const int32_t *q_pos, const AttnReq *reqs, int n_req, int Hq,
                                  int Hkv, int *plan, size_t plan_bytes, cudaStream_t s);

// ------------------------------------------------- query-aware selection --
// QCFuse §3.3-3.4 (k_qprobe.cu).  Anchor scores G_i(r) of one chunk's
// positions (CB_ANCHOR_SINK: -r; CB_ANCHOR_KNORM: minus the squared norm of
// its PIC keys over all layers and kv heads) at scores[score_off + r].
struct AnchorChunk {
  const void *k;          // PIC keys, layer l at k + l * layer_stride elements
  int64_t layer_stride;
  int len, score_off;
};
cudaError_t launch_anchor_scores(const AnchorChunk *chunks, int n, int rule, int n_layers,
                                 int kvw, cb_dtype dt, float *scores, cudaStream_t s);
// Layout of the probe cache: request b's rows [probe_off, + n_anchor + n_u)
// hold its anchors (chunk by chunk, ascending) then its query rows.
struct ProbeLayout {
  struct Req {
    int t_off, n_ctx, n_u, seg_begin, seg_end, probe_off, n_anchor, u_off;
  };
  struct Seg {
    int anchor_off, count, ctx_off, len;
  };
  int B = 0, all = 0;            // all: every context position is an anchor
  Req reqs[CB_MAX_BATCH];
  std::vector<Seg> segs;
  int n_probe = 0, n_u = 0;
};
cudaError_t launch_probe_rows(const ProbeLayout &L, const int32_t *anchors, int32_t *probe_rows,
                              int32_t *u_pos, int32_t *u_src, int32_t *u_cache, int32_t *u_mask,
                              int *status, cudaStream_t s);
// mass[t] += sum over the request's query rows u and q heads h of the
// softmax over its n_ctx context keys of q.k / sqrt(hd) (head_dim 128, bf16).
size_t mass_ws_bytes(int n_u, int Hq, int Hkv, int n_ctx);
cudaError_t launch_attention_mass(const void *q, int64_t ld_q, int u_off, int n_u,
                                  const void *k_cache, int64_t ld_k, int t_off, int n_ctx,
                                  int Hq, int Hkv, int hd, void *ws, size_t ws_bytes,
                                  float *mass, int *status, cudaStream_t s);

// ---------------------------------------------------------------- debug --
cudaError_t launch_expire_wait(int limit_us, int *status, cudaStream_t s);

}  // namespace cb
