// C ABI of the blended-prefill library: argument validation, the device
// status word, workspace planning and the layer / stack orchestration.  All
// arithmetic of the path runs in the kernels of the k_*.cu files; this file
// only enqueues them.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "cb_common.cuh"
#include "cb_internal.h"

using namespace cb;

// NVTX range over a host scope: a profiler's timeline shows each call, and
// each decoder layer inside it, as a named range of the enqueueing thread
// (NVTX is inert unless a tool is attached).
namespace {
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  NvtxRange(const char *fmt, int i) {
    char buf[48];
    snprintf(buf, sizeof buf, fmt, i);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};
}  // namespace

// ------------------------------------------------------------------ errors --
static thread_local std::string g_msg;

static cb_status fail(cb_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_msg = buf;
  return s;
}

#define CB_CUDA(expr)                                                        \
  do {                                                                       \
    cudaError_t e_ = (expr);                                                 \
    if (e_ != cudaSuccess)                                                   \
      return fail(CB_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

#define CB_TRY(expr)                  \
  do {                                \
    cb_status s_ = (expr);            \
    if (s_ != CB_OK) return s_;       \
  } while (0)

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
static size_t dtype_bytes(cb_dtype d) { return d == CB_BF16 ? 2 : 4; }

extern "C" const char *cb_last_error_message(void) { return g_msg.c_str(); }

cb_status cb::record_error(cb_status s, const char *msg) {
  g_msg = msg ? msg : "";
  return s;
}
extern "C" int cb_version(void) { return 100; }

// --------------------------------------------------------- launch counter --
#include <atomic>
static std::atomic<unsigned long long> g_launches{0};
void cb::note_launches(int n) { g_launches.fetch_add((unsigned long long)n); }
extern "C" unsigned long long cb_debug_launch_count(void) { return g_launches.load(); }

static std::atomic<int> g_gemm_path{CB_GEMM_AUTO};
static std::atomic<int> g_mlp_fusion{1};
extern "C" cb_status cb_debug_mlp_fusion(int on) {
  if (on != 0 && on != 1) return fail(CB_ERR_INVALID_ARG, "on must be 0 or 1");
  g_mlp_fusion.store(on);
  return CB_OK;
}
static std::atomic<int> g_index_checks{0};
bool cb::index_checks_on() { return g_index_checks.load(std::memory_order_relaxed) != 0; }
extern "C" cb_status cb_debug_index_checks(int on) {
  if (on != 0 && on != 1) return fail(CB_ERR_INVALID_ARG, "on must be 0 or 1");
  g_index_checks.store(on);
  return CB_OK;
}

// The selections of a call: per request, k entries ascending in [0, n).
static cudaError_t check_selection(const int32_t *idx, const int *k_off, const int *n, int B,
                                   int *st, cudaStream_t s) {
  if (!index_checks_on()) return cudaSuccess;
  IndexCheck c;
  c.n_seg = B;
  c.strict = 1;
  for (int b = 0; b <= B; ++b) c.off[b] = k_off[b];
  for (int b = 0; b < B; ++b) c.hi[b] = n[b];
  return launch_index_check(idx, c, st, s);
}
extern "C" cb_status cb_debug_gemm_path(int path) {
  if (path < CB_GEMM_AUTO || path > CB_GEMM_SWAP_AB_PAIR)
    return fail(CB_ERR_INVALID_ARG, "path must be CB_GEMM_AUTO, _TOKEN_M, _SWAP_AB or _SWAP_AB_PAIR");
  g_gemm_path.store(path);
  return CB_OK;
}

// ------------------------------------------------------------ launch probe --
// Brackets the launches of one class of the layer's kernels with CUDA events
// on their own stream, so a caller can time that kernel inside a real step.
static std::mutex g_probe_mu;
static std::atomic<int> g_probe_kind{0};
static std::vector<cudaEvent_t> g_probe_ev;  // start, stop per launch
static int g_probe_n = 0;
static bool g_probe_open = false;

static void probe_mark(int kind, bool begin, cudaStream_t s) {
  if (g_probe_kind.load(std::memory_order_relaxed) != kind) return;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return;  // a captured record would only fire at replay
  std::lock_guard<std::mutex> lk(g_probe_mu);
  if (g_probe_kind.load() != kind) return;
  if (begin) {
    if (2 * (size_t)g_probe_n + 1 >= g_probe_ev.size()) return;
    if (cudaEventRecord(g_probe_ev[2 * g_probe_n], s) == cudaSuccess) g_probe_open = true;
  } else if (g_probe_open) {
    g_probe_open = false;
    if (cudaEventRecord(g_probe_ev[2 * g_probe_n + 1], s) == cudaSuccess) ++g_probe_n;
  }
}

static void probe_release() {
  for (cudaEvent_t e : g_probe_ev) cudaEventDestroy(e);
  g_probe_ev.clear();
  g_probe_n = 0;
  g_probe_open = false;
}

extern "C" cb_status cb_debug_probe_start(int kind, int max_launches) {
  if (kind < CB_PROBE_QKV || kind > CB_PROBE_MLP || max_launches <= 0 ||
      max_launches > 65536)
    return fail(CB_ERR_INVALID_ARG, "bad probe kind or max_launches");
  std::lock_guard<std::mutex> lk(g_probe_mu);
  g_probe_kind.store(0);
  probe_release();
  g_probe_ev.resize(2 * (size_t)max_launches);
  for (auto &e : g_probe_ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      probe_release();
      return fail(CB_ERR_CUDA, "cudaEventCreate failed");
    }
  }
  g_probe_kind.store(kind);
  return CB_OK;
}

extern "C" cb_status cb_debug_probe_stop(int *n_launches, float *total_ms) {
  if (!n_launches || !total_ms) return fail(CB_ERR_INVALID_ARG, "NULL output");
  std::lock_guard<std::mutex> lk(g_probe_mu);
  g_probe_kind.store(0);
  *n_launches = 0;
  *total_ms = 0.f;
  cb_status rc = CB_OK;
  float sum = 0.f;
  for (int i = 0; i < g_probe_n && rc == CB_OK; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_probe_ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_probe_ev[2 * i], g_probe_ev[2 * i + 1]) != cudaSuccess)
      rc = fail(CB_ERR_CUDA, "probe event timing failed");
    sum += ms;
  }
  if (rc == CB_OK) {
    *n_launches = g_probe_n;
    *total_ms = sum;
  }
  probe_release();
  return rc;
}

// ----------------------------------------------------------- status word --
static __device__ int g_status_word;

namespace cb {
int *device_status_ptr() {
  static std::mutex mu;
  static int *ptrs[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = (int *)p;
  }
  return ptrs[dev];
}

int device_sm_count() {
  static std::mutex mu;
  static int n[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if (!n[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return 148;
    n[dev] = v;
  }
  return n[dev];
}
}  // namespace cb

static cb_status status_ptr(int **out) {
  *out = device_status_ptr();
  if (!*out) return fail(CB_ERR_CUDA, "cannot resolve the device status word");
  return CB_OK;
}

extern "C" cb_status cb_get_device_status(cb_status *out) {
  if (!out) return fail(CB_ERR_INVALID_ARG, "out is NULL");
  CB_CUDA(cudaDeviceSynchronize());
  int v = 0;
  CB_CUDA(cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)));
  const int zero = 0;
  CB_CUDA(cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)));
  *out = (cb_status)v;
  return CB_OK;
}

extern "C" cb_status cb_debug_expire_wait(int limit_us, cb_stream stream) {
  if (limit_us < 0 || limit_us > 1000000)
    return fail(CB_ERR_INVALID_ARG, "limit_us must be in [0, 1e6]");
  int *st;
  CB_TRY(status_ptr(&st));
  CB_CUDA(launch_expire_wait(limit_us, st, stream));
  return CB_OK;
}

// ------------------------------------------------------------- RoPE table --
extern "C" size_t cb_rope_table_elems(int max_positions, int head_dim) {
  if (max_positions <= 0 || head_dim <= 0) return 0;
  return (size_t)max_positions * (head_dim / 2) * 2;
}

extern "C" cb_status cb_rope_table_init(float *table, int max_positions,
                                        int head_dim, float rope_base,
                                        cb_stream stream) {
  if (!table) return fail(CB_ERR_INVALID_ARG, "table is NULL");
  if (head_dim <= 0 || head_dim % 2) return fail(CB_ERR_INVALID_ARG, "head_dim must be even and > 0");
  if (max_positions <= 0) return fail(CB_ERR_INVALID_ARG, "max_positions must be > 0");
  if (!(rope_base > 1.f)) return fail(CB_ERR_INVALID_ARG, "rope_base must be > 1");
  CB_CUDA(launch_rope_table(table, max_positions, head_dim, rope_base, stream));
  return CB_OK;
}

// ---------------------------------------------------------- reposition --
static cb_status check_kv_geometry(int row_elems, int head_dim, cb_dtype dt) {
  if (dt != CB_F32 && dt != CB_BF16) return fail(CB_ERR_INVALID_ARG, "bad dtype");
  if (head_dim <= 0 || head_dim % 16) return fail(CB_ERR_INVALID_ARG, "head_dim must be a positive multiple of 16");
  if (row_elems <= 0 || row_elems % head_dim) return fail(CB_ERR_INVALID_ARG, "row_elems must be a multiple of head_dim");
  return CB_OK;
}

extern "C" cb_status cb_rope_reposition(const cb_stitch_desc *descs, int n_desc,
                                        int layer_begin, int layer_end,
                                        void *k_cache, void *v_cache,
                                        int64_t cache_layer_stride,
                                        int row_elems, int head_dim,
                                        const float *rope_table,
                                        int max_positions, cb_dtype dtype,
                                        cb_stream stream) {
  if (n_desc < 0 || (n_desc > 0 && !descs)) return fail(CB_ERR_INVALID_ARG, "descs");
  if (layer_begin < 0 || layer_end < layer_begin) return fail(CB_ERR_INVALID_ARG, "layer range");
  if (!k_cache || !v_cache || !rope_table) return fail(CB_ERR_INVALID_ARG, "NULL cache or table");
  CB_TRY(check_kv_geometry(row_elems, head_dim, dtype));
  const size_t eb = dtype_bytes(dtype);
  if (!aligned16(k_cache) || !aligned16(v_cache) || (cache_layer_stride * eb) % 16)
    return fail(CB_ERR_INVALID_ARG, "cache pointers / layer stride must be 16-byte aligned");
  for (int i = 0; i < n_desc; ++i) {
    const cb_stitch_desc &d = descs[i];
    if (d.len < 0 || d.dst_row < 0) return fail(CB_ERR_INVALID_ARG, "desc %d: negative len/dst_row", i);
    if (d.len == 0) continue;
    if (!d.k_src || !d.v_src || !aligned16(d.k_src) || !aligned16(d.v_src) ||
        (d.src_layer_stride * eb) % 16)
      return fail(CB_ERR_INVALID_ARG, "desc %d: NULL or misaligned source", i);
    if (d.delta >= max_positions || -d.delta >= max_positions)
      return fail(CB_ERR_INVALID_ARG, "desc %d: |delta| %d >= max_positions %d", i, d.delta, max_positions);
  }
  int *st;
  CB_TRY(status_ptr(&st));
  CB_CUDA(launch_reposition(descs, n_desc, layer_begin, layer_end, k_cache, v_cache,
                            cache_layer_stride, row_elems, head_dim, rope_table,
                            dtype, st, stream));
  return CB_OK;
}

// -------------------------------------------------------------- selection --
extern "C" size_t cb_select_workspace_size(int n_req) { return select_ws_bytes(n_req); }

static cb_status run_selection(const void *k_fresh, int64_t ld_fresh,
                               const void *k_reused, int64_t ld_reused,
                               int row_elems, cb_dtype dt, const SelPlan &plan,
                               float *dev, int32_t *idx, int *st, cudaStream_t s) {
  CB_CUDA(launch_deviation(k_fresh, ld_fresh, k_reused, ld_reused, row_elems, dt,
                           plan.reqs.data(), (int)plan.reqs.size(), dev, s));
  CB_CUDA(launch_selection(dev, plan, idx, st, s));
  return CB_OK;
}

extern "C" cb_status cb_kv_deviation_topk(const void *k_fresh, int64_t ld_fresh,
                                          const void *k_reused, int64_t ld_reused,
                                          int row_elems, cb_dtype dtype,
                                          const cb_select_req *reqs, int n_req,
                                          cb_policy policy, float *dev_out,
                                          int32_t *idx_out, void *ws,
                                          size_t ws_bytes, cb_stream stream) {
  if (!k_fresh || !k_reused || !dev_out || !idx_out) return fail(CB_ERR_INVALID_ARG, "NULL pointer");
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(CB_ERR_INVALID_ARG, "bad dtype");
  const size_t eb = dtype_bytes(dtype);
  if (row_elems <= 0 || (row_elems * eb) % 16 || ld_fresh < row_elems || ld_reused < row_elems ||
      (ld_fresh * eb) % 16 || (ld_reused * eb) % 16 || !aligned16(k_fresh) || !aligned16(k_reused))
    return fail(CB_ERR_INVALID_ARG, "rows must be 16-byte aligned and ld >= row_elems");
  (void)ws;        // reserved: the selection needs no scratch beyond dev_out
  (void)ws_bytes;
  SelPlan plan;
  const char *err = "";
  if (make_sel_plan(reqs, n_req, policy, plan, &err) != CB_OK) return fail(CB_ERR_INVALID_ARG, "%s", err);
  int *st;
  CB_TRY(status_ptr(&st));
  CB_TRY(run_selection(k_fresh, ld_fresh, k_reused, ld_reused, row_elems, dtype, plan, dev_out,
                       idx_out, st, stream));
  if (index_checks_on()) {
    // outputs are packed per request at idx_offset; check each run alone
    for (const SelReq &r : plan.reqs) {
      const int off[2] = {0, r.k}, n[1] = {r.n_ctx};
      CB_CUDA(check_selection(idx_out + r.idx_offset, off, n, 1, st, stream));
    }
  }
  return CB_OK;
}

extern "C" cb_status cb_selection_stats(const float *dev, const int32_t *idx,
                                        const cb_select_req *reqs, int n_req,
                                        int32_t *segments_out, double *captured_out,
                                        cb_stream stream) {
  if (n_req < 0 || n_req > CB_MAX_BATCH) return fail(CB_ERR_INVALID_ARG, "n_req must be in [0, %d]", CB_MAX_BATCH);
  if (n_req == 0) return CB_OK;
  if (!dev || !idx || !reqs || !segments_out || !captured_out) return fail(CB_ERR_INVALID_ARG, "NULL pointer");
  std::vector<SelReq> sr(n_req);
  for (int i = 0; i < n_req; ++i) {
    const cb_select_req &r = reqs[i];
    if (r.n_ctx < 0 || r.k < 0 || r.k > r.n_ctx) return fail(CB_ERR_INVALID_ARG, "request %d: need 0 <= k <= n_ctx", i);
    if (r.dev_offset < 0 || r.idx_offset < 0) return fail(CB_ERR_INVALID_ARG, "request %d: negative offset", i);
    sr[i] = SelReq{r.n_ctx, r.k, 0, 0, r.dev_offset, r.idx_offset, 0, 0};
  }
  int *st;
  CB_TRY(status_ptr(&st));
  CB_CUDA(launch_selection_stats(dev, idx, sr.data(), n_req, segments_out, captured_out, st, stream));
  return CB_OK;
}

extern "C" cb_status cb_loading_ratio(double load_ms_per_layer, const int32_t *ratio_bp,
                                      const double *recompute_ms_per_layer, int n,
                                      int32_t min_ratio_bp, int32_t *ratio_out) {
  if (!ratio_out) return fail(CB_ERR_INVALID_ARG, "ratio_out is NULL");
  if (n < 0 || (n > 0 && (!ratio_bp || !recompute_ms_per_layer)))
    return fail(CB_ERR_INVALID_ARG, "need n >= 0 and both arrays");
  if (min_ratio_bp < 0 || min_ratio_bp > 10000) return fail(CB_ERR_INVALID_ARG, "min_ratio_bp must be in [0, 10000]");
  if (!(load_ms_per_layer >= 0.0)) return fail(CB_ERR_INVALID_ARG, "load time must be >= 0");
  int32_t r = min_ratio_bp;
  for (int i = 0; i < n; ++i) {
    if (ratio_bp[i] < 0 || ratio_bp[i] > 10000) return fail(CB_ERR_INVALID_ARG, "ratio %d outside [0, 10000]", i);
    if (!(recompute_ms_per_layer[i] >= 0.0)) return fail(CB_ERR_INVALID_ARG, "time %d must be >= 0", i);
    // recompute at this ratio hides behind the load of the next layer
    if (recompute_ms_per_layer[i] <= load_ms_per_layer && ratio_bp[i] > r) r = ratio_bp[i];
  }
  *ratio_out = r;
  return CB_OK;
}

// -------------------------------------------------------- gather/scatter --
extern "C" cb_status cb_gather_rows(const void *src, int64_t ld_src, int64_t src_rows,
                                    const int32_t *idx, int n, int row_elems,
                                    void *dst, int64_t ld_dst, cb_dtype dtype,
                                    cb_stream stream) {
  if (n < 0) return fail(CB_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return CB_OK;
  if (!src || !idx || !dst) return fail(CB_ERR_INVALID_ARG, "NULL pointer");
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(CB_ERR_INVALID_ARG, "bad dtype");
  const size_t eb = dtype_bytes(dtype);
  if (row_elems <= 0 || (row_elems * eb) % 16 || (ld_src * eb) % 16 || (ld_dst * eb) % 16 ||
      ld_src < row_elems || ld_dst < row_elems || !aligned16(src) || !aligned16(dst))
    return fail(CB_ERR_INVALID_ARG, "rows must be 16-byte aligned and ld >= row_elems");
  int *st;
  CB_TRY(status_ptr(&st));
  CB_CUDA(launch_gather(src, ld_src, src_rows, idx, n, row_elems, dst, ld_dst, eb, st, stream));
  return CB_OK;
}

extern "C" cb_status cb_scatter_kv(const void *k_new, const void *v_new, int64_t ld_new,
                                   const int32_t *rows, int n, void *k_cache,
                                   void *v_cache, int64_t ld_cache, int64_t cache_rows,
                                   int row_elems, cb_dtype dtype, cb_stream stream) {
  if (n < 0) return fail(CB_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return CB_OK;
  if (!k_new || !v_new || !rows || !k_cache || !v_cache) return fail(CB_ERR_INVALID_ARG, "NULL pointer");
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(CB_ERR_INVALID_ARG, "bad dtype");
  const size_t eb = dtype_bytes(dtype);
  if (row_elems <= 0 || (row_elems * eb) % 16 || (ld_new * eb) % 16 || (ld_cache * eb) % 16 ||
      ld_new < row_elems || ld_cache < row_elems || !aligned16(k_new) || !aligned16(v_new) ||
      !aligned16(k_cache) || !aligned16(v_cache))
    return fail(CB_ERR_INVALID_ARG, "rows must be 16-byte aligned and ld >= row_elems");
  int *st;
  CB_TRY(status_ptr(&st));
  CB_CUDA(launch_scatter_kv(k_new, v_new, ld_new, rows, n, k_cache, v_cache, ld_cache,
                            cache_rows, row_elems, eb, st, stream));
  return CB_OK;
}

// -------------------------------------------------------------- attention --
static cb_status check_attn(int Hq, int Hkv, int hd) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return fail(CB_ERR_INVALID_ARG, "n_q_heads must be a multiple of n_kv_heads");
  if (hd != 64 && hd != 128) return fail(CB_ERR_INVALID_ARG, "head_dim must be 64 or 128");
  return CB_OK;
}

static cb_status run_attention(const void *q, int64_t ld_q, const int32_t *q_pos,
                               const std::vector<AttnReq> &reqs, const void *kc,
                               const void *vc, int64_t ld_kv, int Hq, int Hkv, int hd,
                               float scale, void *out, int64_t ld_out, cb_dtype dt,
                               void *ws, size_t ws_bytes, int *st, cudaStream_t s,
                               const int *plan = nullptr) {
  if (index_checks_on()) {
    // query positions ascend per request and lie inside its cache
    IndexCheck c;
    c.n_seg = (int)reqs.size();
    c.strict = 0;
    for (int b = 0; b < c.n_seg; ++b) {
      c.off[b] = reqs[b].q_begin;
      c.hi[b] = reqs[b].kv_len;
    }
    c.off[c.n_seg] = c.n_seg ? reqs[c.n_seg - 1].q_end : 0;
    bool contiguous = true;
    for (int b = 0; b + 1 < c.n_seg; ++b) contiguous &= reqs[b].q_end == reqs[b + 1].q_begin;
    if (contiguous && (c.n_seg == 0 || reqs[0].q_begin >= 0)) CB_CUDA(launch_index_check(q_pos, c, st, s));
  }
  if (dt == CB_BF16 && attention_tc_supported(Hq, Hkv, hd)) {
    const size_t need = plan ? 0 : attention_tc_ws_bytes(reqs.data(), (int)reqs.size(), Hq, Hkv);
    if (need > 0 && (!ws || ws_bytes < need))
      return fail(CB_ERR_WORKSPACE, "attention workspace too small (%zu < %zu)", ws_bytes, need);
    CB_CUDA(launch_attention_tc(q, ld_q, q_pos, reqs.data(), (int)reqs.size(), kc, vc, ld_kv,
                                Hq, Hkv, scale, out, ld_out, ws, ws_bytes, st, s, plan));
  } else {
    CB_CUDA(launch_attention_simt(q, ld_q, q_pos, reqs.data(), (int)reqs.size(), kc, vc,
                                  ld_kv, Hq, Hkv, hd, scale, out, ld_out, dt, st, s));
  }
  return CB_OK;
}

extern "C" size_t cb_attention_workspace_size(const cb_attn_req *reqs, int n_req,
                                              int n_q_heads, int n_kv_heads, int head_dim,
                                              cb_dtype dtype) {
  if (!reqs || n_req <= 0 || n_req > CB_MAX_BATCH || dtype != CB_BF16 || n_kv_heads <= 0 ||
      !attention_tc_supported(n_q_heads, n_kv_heads, head_dim))
    return 256;
  std::vector<AttnReq> ar(n_req);
  for (int i = 0; i < n_req; ++i)
    ar[i] = AttnReq{reqs[i].q_begin, reqs[i].q_end, reqs[i].kv_row0, reqs[i].kv_len};
  const size_t n = attention_tc_ws_bytes(ar.data(), n_req, n_q_heads, n_kv_heads);
  return n > 256 ? n : 256;
}

extern "C" cb_status cb_sparse_query_attention(const void *q, int64_t ld_q,
                                               const int32_t *q_pos,
                                               const cb_attn_req *reqs, int n_req,
                                               const void *k_cache, const void *v_cache,
                                               int64_t ld_kv, int n_q_heads,
                                               int n_kv_heads, int head_dim, float scale,
                                               void *out, int64_t ld_out, cb_dtype dtype,
                                               void *ws, size_t ws_bytes,
                                               cb_stream stream) {
  if (n_req < 0 || n_req > CB_MAX_BATCH) return fail(CB_ERR_INVALID_ARG, "n_req must be in [0, %d]", CB_MAX_BATCH);
  if (n_req == 0) return CB_OK;
  if (!q || !q_pos || !reqs || !k_cache || !v_cache || !out) return fail(CB_ERR_INVALID_ARG, "NULL pointer");
  if (dtype != CB_F32 && dtype != CB_BF16) return fail(CB_ERR_INVALID_ARG, "bad dtype");
  CB_TRY(check_attn(n_q_heads, n_kv_heads, head_dim));
  const size_t eb = dtype_bytes(dtype);
  if (ld_q < (int64_t)n_q_heads * head_dim || ld_out < (int64_t)n_q_heads * head_dim ||
      ld_kv < (int64_t)n_kv_heads * head_dim || (ld_q * eb) % 16 || (ld_out * eb) % 16 ||
      (ld_kv * eb) % 16 || !aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(CB_ERR_INVALID_ARG, "bad leading dimension or alignment");
  std::vector<AttnReq> ar(n_req);
  for (int i = 0; i < n_req; ++i) {
    const cb_attn_req &r = reqs[i];
    if (r.q_begin < 0 || r.q_end < r.q_begin || r.kv_row0 < 0 || r.kv_len < 0)
      return fail(CB_ERR_INVALID_ARG, "req %d: bad ranges", i);
    ar[i] = AttnReq{r.q_begin, r.q_end, r.kv_row0, r.kv_len};
  }
  int *st;
  CB_TRY(status_ptr(&st));
  return run_attention(q, ld_q, q_pos, ar, k_cache, v_cache, ld_kv, n_q_heads, n_kv_heads,
                       head_dim, scale, out, ld_out, dtype, ws, ws_bytes, st, stream);
}

// ------------------------------------------------------------------ model --
// A recorded blended call: the key is its host arguments, serialised.
struct CallGraph {
  std::vector<uint8_t> key;
  cudaGraphExec_t exec = nullptr;
  unsigned long long launches = 0;   // kernels the call launches
  unsigned long long used = 0;       // last use, for eviction
};

struct cb_model {
  cb_model_config cfg;
  cb_weights w;
  std::vector<cb_layer_weights> layers;
  int qw, kvw, qkv_rows;
  size_t eb;
  // ordering events of the host-resident chunk path (copy stream <-> compute
  // stream): fork, per staging buffer "copied" and "consumed"
  cudaEvent_t ev_fork = nullptr, ev_copied[2] = {nullptr, nullptr},
              ev_free[2] = {nullptr, nullptr};
  // recorded blended calls (the most recently used few)
  std::mutex graph_mu;
  std::vector<CallGraph> graphs;
  std::vector<std::vector<uint8_t>> graph_seen;   // keys called once, not yet recorded
  unsigned long long graph_clock = 0;
  ~cb_model() {
    for (cudaEvent_t e : {ev_fork, ev_copied[0], ev_copied[1], ev_free[0], ev_free[1]})
      if (e) cudaEventDestroy(e);
    for (CallGraph &g : graphs)
      if (g.exec) cudaGraphExecDestroy(g.exec);
  }
};

extern "C" cb_status cb_model_create(const cb_model_config *cfg, const cb_weights *w,
                                     cb_model **out) {
  if (!cfg || !w || !out) return fail(CB_ERR_INVALID_ARG, "NULL argument");
  const cb_model_config &c = *cfg;
  if (c.n_layers <= 0 || c.d_model <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 ||
      c.head_dim <= 0 || c.d_ffn <= 0 || c.vocab <= 0 || c.max_positions <= 0)
    return fail(CB_ERR_INVALID_ARG, "non-positive model dimension");
  if (c.n_q_heads % c.n_kv_heads) return fail(CB_ERR_INVALID_ARG, "n_q_heads %% n_kv_heads != 0");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c.d_model % 64 || c.d_ffn % 16) return fail(CB_ERR_UNSUPPORTED, "d_model %% 64 and d_ffn %% 16 must be 0");
  if (c.d_model > 8192) return fail(CB_ERR_UNSUPPORTED, "d_model > 8192");
  if (c.dtype != CB_F32 && c.dtype != CB_BF16) return fail(CB_ERR_INVALID_ARG, "bad dtype");
  if (!(c.norm_eps >= 0.f)) return fail(CB_ERR_INVALID_ARG, "norm_eps < 0");
  if (!w->embed || !w->final_norm || !w->layers || !w->rope_table)
    return fail(CB_ERR_INVALID_ARG, "NULL weight pointer");
  for (int l = 0; l < c.n_layers; ++l) {
    const cb_layer_weights &L = w->layers[l];
    if (!L.w_qkv || !L.w_o || !L.w_gate || !L.w_up || !L.w_down || !L.norm1 || !L.norm2)
      return fail(CB_ERR_INVALID_ARG, "layer %d: NULL weight pointer", l);
    if (!aligned16(L.w_qkv) || !aligned16(L.w_o) || !aligned16(L.w_gate) ||
        !aligned16(L.w_up) || !aligned16(L.w_down) || !aligned16(L.norm1) || !aligned16(L.norm2))
      return fail(CB_ERR_INVALID_ARG, "layer %d: weights must be 16-byte aligned", l);
  }
  int dev = 0;
  cudaDeviceProp prop;
  CB_CUDA(cudaGetDevice(&dev));
  CB_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(CB_ERR_UNSUPPORTED, "device sm_%d%d: this library is built for sm_103a", prop.major, prop.minor);
  cb_model *m = new cb_model;
  for (cudaEvent_t *e : {&m->ev_fork, &m->ev_copied[0], &m->ev_copied[1], &m->ev_free[0],
                         &m->ev_free[1]}) {
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) {
      delete m;
      return fail(CB_ERR_CUDA, "cudaEventCreate failed");
    }
  }
  m->cfg = c;
  m->w = *w;
  m->layers.assign(w->layers, w->layers + c.n_layers);
  m->w.layers = m->layers.data();
  m->qw = c.n_q_heads * c.head_dim;
  m->kvw = c.n_kv_heads * c.head_dim;
  m->qkv_rows = m->qw + 2 * m->kvw;
  m->eb = dtype_bytes(c.dtype);
  *out = m;
  return CB_OK;
}

extern "C" void cb_model_destroy(cb_model *m) { delete m; }

// ----------------------------------------------------------------- linear --
// bf16 projections run on the tcgen05 kernel; the fp32 parity path keeps
// CUDA-core FMAs (tensor cores would round its operands).
// split_ws: the swapped GEMM's tail-split workspace (NULL: no split).
static cb_status run_linear(const cb_model *m, const void *A, int64_t lda, const void *W,
                            const void *W2, int64_t ldw, int M, int N, int K, GemmEpi epi,
                            void *out, int64_t ldo, cudaStream_t s,
                            const QkvEpi *qkv = nullptr, void *split_ws = nullptr) {
  if (m->cfg.dtype == CB_BF16) {
    int *st;
    CB_TRY(status_ptr(&st));
    const int path = g_gemm_path.load(std::memory_order_relaxed);
    int form = path == CB_GEMM_AUTO        ? gemm_auto_form(M, K, epi)
               : path == CB_GEMM_SWAP_AB      ? 1
               : path == CB_GEMM_SWAP_AB_PAIR ? 2
                                              : 0;
    if (epi == EPI_KDEV && form == 0) form = 1;   // the key-deviation epilogue is swapped-only
    if (form)
      CB_CUDA(launch_gemm_sab(A, lda, W, W2, ldw, M, N, K, epi, out, ldo, qkv, st, s, form,
                              split_ws));
    else
      CB_CUDA(launch_gemm_tc(A, lda, W, W2, ldw, M, N, K, epi, out, ldo, qkv, st, s));
  } else {
    if (epi == EPI_QKV) return fail(CB_ERR_UNSUPPORTED, "fused QKV epilogue is bf16-only");
    CB_CUDA(launch_gemm_simt(A, lda, W, W2, ldw, M, N, K, epi, out, ldo, m->cfg.dtype, s));
  }
  return CB_OK;
}

extern "C" size_t cb_linear_workspace_size(void) { return gemm_split_ws_bytes(); }

extern "C" cb_status cb_linear(const cb_model *m, const void *A, int64_t ld_a,
                               const void *W, const void *W2, int64_t ld_w, int M,
                               int N, int K, cb_epilogue epi, void *out, int64_t ld_out,
                               cb_stream stream) {
  return cb_linear_ws(m, A, ld_a, W, W2, ld_w, M, N, K, epi, out, ld_out, nullptr, 0, stream);
}

extern "C" cb_status cb_linear_ws(const cb_model *m, const void *A, int64_t ld_a,
                                  const void *W, const void *W2, int64_t ld_w, int M,
                                  int N, int K, cb_epilogue epi, void *out, int64_t ld_out,
                                  void *ws, size_t ws_bytes, cb_stream stream) {
  if (!m || !A || !W || !out) return fail(CB_ERR_INVALID_ARG, "NULL pointer");
  if (ws && (ws_bytes < gemm_split_ws_bytes() || !aligned16(ws)))
    return fail(CB_ERR_WORKSPACE, "linear workspace too small or misaligned (%zu < %zu)", ws_bytes,
                gemm_split_ws_bytes());
  if (M < 0 || N <= 0 || K <= 0 || K % 16) return fail(CB_ERR_INVALID_ARG, "need M >= 0, N > 0, K %% 16 == 0");
  if (ld_a < K || ld_w < K || ld_out < N) return fail(CB_ERR_INVALID_ARG, "leading dimension too small");
  if (m->cfg.dtype == CB_BF16) {
    // TMA: 16-byte aligned bases and row strides; 16-byte output vectors
    if (!aligned16(A) || !aligned16(W) || (W2 && !aligned16(W2)) || !aligned16(out) ||
        (ld_a * 2) % 16 || (ld_w * 2) % 16 || N % 8 || (ld_out * (epi == CB_EPI_RESID ? 4 : 2)) % 16)
      return fail(CB_ERR_INVALID_ARG, "bf16 GEMM needs 16-byte aligned rows and N %% 8 == 0");
  }
  GemmEpi e;
  switch (epi) {
    case CB_EPI_STORE: e = EPI_STORE; break;
    case CB_EPI_RESID: e = EPI_RESID; break;
    case CB_EPI_SWIGLU:
      if (!W2) return fail(CB_ERR_INVALID_ARG, "SWIGLU needs W2");
      e = EPI_SWIGLU;
      break;
    default: return fail(CB_ERR_INVALID_ARG, "unknown epilogue");
  }
  if (M == 0) return CB_OK;
  if (ws && m->cfg.dtype == CB_BF16)
    CB_CUDA(cudaMemsetAsync((char *)ws + gemm_split_flags_offset(), 0,
                            gemm_split_ws_bytes() - gemm_split_flags_offset(), stream));
  return run_linear(m, A, ld_a, W, W2, ld_w, M, N, K, e, out, ld_out, stream, nullptr,
                    m->cfg.dtype == CB_BF16 ? ws : nullptr);
}

// ------------------------------------------------------------------- plan --
namespace {

struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  }
};

// Scratch of one decoder layer over n rows.
struct LayerScratch {
  void *x, *q, *o, *g;
  float *qkv32;
  void *attn;          // attention partials (split key ranges)
  size_t attn_bytes;
  void *split;         // the swapped GEMM's tail-split partials and counters (bf16)
  int *mlp_epoch;      // the call's last fused-MLP epoch (host counter; NULL: no fusion)
};

struct LayerOffsets {
  size_t x, q, o, g, qkv32, attn, attn_bytes, split, split_bytes;
};

LayerOffsets carve_layer(Carver &c, const cb_model *m, int64_t n) {
  LayerOffsets L;
  const cb_model_config &cf = m->cfg;
  L.x = c.take(n * cf.d_model * m->eb);
  L.q = c.take(n * m->qw * m->eb);
  L.o = c.take(n * m->qw * m->eb);
  L.g = c.take(n * cf.d_ffn * m->eb);
  L.qkv32 = c.take(n * m->qkv_rows * sizeof(float));
  L.attn_bytes = (cf.dtype == CB_BF16 &&
                  attention_tc_supported(cf.n_q_heads, cf.n_kv_heads, cf.head_dim))
                     ? attention_tc_ws_bound()
                     : 0;
  L.attn = c.take(L.attn_bytes);
  L.split_bytes = cf.dtype == CB_BF16 ? gemm_split_ws_bytes() : 0;
  L.split = c.take(L.split_bytes);
  return L;
}

LayerScratch bind_layer(char *ws, const LayerOffsets &L) {
  return LayerScratch{ws + L.x, ws + L.q, ws + L.o, ws + L.g, (float *)(ws + L.qkv32),
                      ws + L.attn, L.attn_bytes, L.split_bytes ? ws + L.split : nullptr,
                      nullptr};
}

// The tail-split counters start at zero in every call (each GEMM leaves them
// zero), and so do the fused MLP's flags (each launch of the call takes the
// next epoch, counted from 1 in *S.mlp_epoch).
cudaError_t reset_split(const LayerScratch &S, cudaStream_t s) {
  if (!S.split) return cudaSuccess;
  return cudaMemsetAsync((char *)S.split + gemm_split_flags_offset(), 0,
                         gemm_split_ws_bytes() - gemm_split_flags_offset(), s);
}

struct Plan {
  int B = 0;
  BatchMeta bm;
  std::vector<int> T, N, k, R;
  std::vector<std::vector<int>> seg_start;  // position of each segment
  int64_t T_total = 0, N_total = 0, K_total = 0, R_total = 0;
  int n_off[CB_MAX_BATCH + 1];
  // gradual filtering: the rows of every request from `layer` on
  struct Step {
    int layer;
    BatchMeta bm;
    int64_t K_total, R_total;
  };
  std::vector<Step> sched;
  int64_t K_final = 0, R_final = 0;
  // workspace
  LayerOffsets lay;
  size_t h_all, kf, dev, sel, pos_all, glob_all, pos_c, glob_c, h_c, lm_x, lm_best, total;
  size_t kdev = 0, dev_idx = 0;   // fused key deviation: per-head partials, row -> d index
  size_t attn_plan = 0, attn_plan_bytes = 0;   // unit table of the compact layers' attention
  // query-aware selection ([QCF] §3.3-3.4)
  ProbeLayout probe;
  int n_anchor_total = 0;
  size_t qp_scores = 0, qp_anchors = 0, qp_rows = 0, qp_u = 0, qp_k = 0, qp_v = 0, qp_h = 0,
         qp_mass = 0, qp_mass_bytes = 0;
  size_t g_dev = 0, g_keep = 0, g_sel = 0, g_pos = 0, g_glob = 0, g_src = 0, g_h = 0;
  // host-resident chunk path: two layers of the context K/V in flight
  size_t stage = 0, stage_bytes = 0;     // stage_bytes: K of one layer (V follows)
};

}  // namespace

static cb_status validate_requests(const cb_model *m, const cb_request *reqs, int B,
                                   bool blend) {
  if (!m) return fail(CB_ERR_INVALID_ARG, "model is NULL");
  if (B <= 0 || B > CB_MAX_BATCH) return fail(CB_ERR_INVALID_ARG, "B must be in [1, %d]", CB_MAX_BATCH);
  if (!reqs) return fail(CB_ERR_INVALID_ARG, "reqs is NULL");
  for (int b = 0; b < B; ++b) {
    const cb_request &r = reqs[b];
    if (!r.tokens || r.n_segments <= 0 || !r.segments)
      return fail(CB_ERR_INVALID_ARG, "request %d: tokens/segments missing", b);
    bool seen_uncached = false;
    int64_t T = 0;
    for (int i = 0; i < r.n_segments; ++i) {
      const cb_segment &s = r.segments[i];
      if (s.len < 0) return fail(CB_ERR_INVALID_ARG, "request %d segment %d: len < 0", b, i);
      const bool cached = s.k_pic != nullptr;
      if (blend) {
        if (cached != (s.v_pic != nullptr))
          return fail(CB_ERR_INVALID_ARG, "request %d segment %d: k_pic and v_pic must both be set or both NULL", b, i);
        if (cached && seen_uncached)
          return fail(CB_ERR_INVALID_ARG, "request %d: cached segments must precede uncached ones", b);
        if (cached && s.len > 0) {
          if (!aligned16(s.k_pic) || !aligned16(s.v_pic) || (s.pic_layer_stride * (int64_t)m->eb) % 16 ||
              s.pic_layer_stride < (int64_t)s.len * m->kvw)
            return fail(CB_ERR_INVALID_ARG, "request %d segment %d: bad PIC layout", b, i);
          if (s.pic_pos0 < 0) return fail(CB_ERR_INVALID_ARG, "request %d segment %d: pic_pos0 < 0", b, i);
        }
      }
      if (!cached) seen_uncached = true;
      T += s.len;
    }
    if (T <= 0) return fail(CB_ERR_INVALID_ARG, "request %d is empty", b);
    if (T > m->cfg.max_positions)
      return fail(CB_ERR_INVALID_ARG, "request %d: %lld positions exceed max_positions %d", b, (long long)T, m->cfg.max_positions);
    if (blend) {
      const cb_segment &last = r.segments[r.n_segments - 1];
      if (last.k_pic != nullptr || last.len == 0)
        return fail(CB_ERR_INVALID_ARG, "request %d must end in a non-empty uncached segment (the query)", b);
    }
  }
  return CB_OK;
}

static int select_count(int n_ctx, int ratio_bp) {
  if (ratio_bp <= 0 || n_ctx <= 0) return 0;
  const int64_t k = ((int64_t)n_ctx * ratio_bp) / 10000;
  return (int)(k < 1 ? 1 : k);
}

static bool is_query_policy(cb_policy p) {
  return p == CB_POLICY_QUERY_PROBE || p == CB_POLICY_QUERY_FULL;
}

static cb_status make_plan(const cb_model *m, const cb_request *reqs, int B,
                           const cb_blend_params *p, bool blend, Plan &P,
                           bool host_kv = false) {
  CB_TRY(validate_requests(m, reqs, B, blend));
  if (blend) {
    if (!p) return fail(CB_ERR_INVALID_ARG, "params is NULL");
    if (p->ratio_bp < 0 || p->ratio_bp > 10000) return fail(CB_ERR_INVALID_ARG, "ratio_bp must be in [0, 10000]");
    if (p->sel_layer < 0 || p->sel_layer >= m->cfg.n_layers)
      return fail(CB_ERR_INVALID_ARG, "sel_layer must be in [0, n_layers)");
    if (p->policy < CB_POLICY_TOKEN_TOPK || p->policy > CB_POLICY_QUERY_FULL)
      return fail(CB_ERR_INVALID_ARG, "unknown policy");
    if (is_query_policy(p->policy)) {
      // [QCF] §3.5: P exists before layer 0, every layer recomputes it
      if (p->sel_layer != 0 || p->n_schedule != 0)
        return fail(CB_ERR_INVALID_ARG, "query-aware policies select before layer 0: sel_layer and n_schedule must be 0");
      if (m->cfg.dtype != CB_BF16 || m->cfg.head_dim != 128)
        return fail(CB_ERR_UNSUPPORTED, "query-aware policies run on bf16 models with head_dim 128");
      if (p->policy == CB_POLICY_QUERY_PROBE) {
        if (p->anchor_rule != CB_ANCHOR_SINK && p->anchor_rule != CB_ANCHOR_KNORM)
          return fail(CB_ERR_INVALID_ARG, "unknown anchor rule");
        if (p->anchor_bp < 0 || p->anchor_bp > 10000)
          return fail(CB_ERR_INVALID_ARG, "anchor_bp must be in [0, 10000]");
        if (p->n_crit < 1 || p->n_crit > m->cfg.n_layers || !p->crit_layers)
          return fail(CB_ERR_INVALID_ARG, "the critical-layer set needs 1..n_layers layers");
        for (int i = 0; i < p->n_crit; ++i) {
          if (p->crit_layers[i] < 0 || p->crit_layers[i] >= m->cfg.n_layers)
            return fail(CB_ERR_INVALID_ARG, "critical layer out of range");
          for (int j = 0; j < i; ++j)
            if (p->crit_layers[j] == p->crit_layers[i])
              return fail(CB_ERR_INVALID_ARG, "critical layers must be distinct");
        }
      }
    }
    if (p->host_load_ctas < 0 || p->host_load_ctas > 4096)
      return fail(CB_ERR_INVALID_ARG, "host_load_ctas must be in [0, 4096]");
    if (p->policy == CB_POLICY_RANDOM_DOC && !p->span_order)
      return fail(CB_ERR_INVALID_ARG, "random-document needs span_order");
    if (p->policy == CB_POLICY_FIXED_CHUNK &&
        (p->span_len < 0 || (p->span_len > 0 && (p->span_offset < 0 || p->span_offset > p->span_len))))
      return fail(CB_ERR_INVALID_ARG, "fixed-chunk needs 0 <= span_offset <= span_len");
    if (p->n_schedule < 0 || p->n_schedule > m->cfg.n_layers)
      return fail(CB_ERR_INVALID_ARG, "n_schedule must be in [0, n_layers]");
    if (p->n_schedule > 0 && !p->schedule) return fail(CB_ERR_INVALID_ARG, "schedule is NULL");
    for (int i = 0; i < p->n_schedule; ++i) {
      const cb_schedule_step &st = p->schedule[i];
      const int prev = i ? p->schedule[i - 1].layer : p->sel_layer;
      if (st.layer <= prev || st.layer >= m->cfg.n_layers)
        return fail(CB_ERR_INVALID_ARG, "schedule layers must ascend strictly, above sel_layer and below n_layers");
      if (st.keep < 0) return fail(CB_ERR_INVALID_ARG, "schedule keep must be >= 0");
    }
  }
  P.B = B;
  P.bm.B = B;
  P.T.resize(B); P.N.resize(B); P.k.resize(B); P.R.resize(B); P.seg_start.resize(B);
  P.bm.t_off[0] = P.bm.k_off[0] = P.bm.r_off[0] = 0;
  P.n_off[0] = 0;
  for (int b = 0; b < B; ++b) {
    int T = 0, N = 0;
    for (int i = 0; i < reqs[b].n_segments; ++i) {
      const cb_segment &s = reqs[b].segments[i];
      P.seg_start[b].push_back(T);
      T += s.len;
      if (blend && s.k_pic) N += s.len;
    }
    const int k = blend ? select_count(N, p->ratio_bp) : 0;
    P.T[b] = T; P.N[b] = N; P.k[b] = k;
    P.R[b] = blend ? k + (T - N) : T;
    P.bm.n_ctx[b] = N;
    P.bm.t_off[b + 1] = P.bm.t_off[b] + T;
    P.bm.k_off[b + 1] = P.bm.k_off[b] + k;
    P.bm.r_off[b + 1] = P.bm.r_off[b] + P.R[b];
    P.n_off[b + 1] = P.n_off[b] + N;
  }
  P.T_total = P.bm.t_off[B];
  P.N_total = P.n_off[B];
  P.K_total = P.bm.k_off[B];
  P.R_total = P.bm.r_off[B];
  P.K_final = P.K_total;
  P.R_final = P.R_total;
  if (blend) {
    // every request keeps min(keep, its current count) at each step
    BatchMeta cur = P.bm;
    for (int i = 0; i < p->n_schedule; ++i) {
      Plan::Step st{p->schedule[i].layer, cur, 0, 0};
      for (int b = 0; b < B; ++b) {
        const int kc = cur.k_off[b + 1] - cur.k_off[b];
        const int kn = p->schedule[i].keep < kc ? p->schedule[i].keep : kc;
        st.bm.k_off[b + 1] = st.bm.k_off[b] + kn;
        st.bm.r_off[b + 1] = st.bm.r_off[b] + kn + (P.T[b] - P.N[b]);
      }
      st.K_total = st.bm.k_off[B];
      st.R_total = st.bm.r_off[B];
      P.sched.push_back(st);
      cur = st.bm;
      P.K_final = st.K_total;
      P.R_final = st.R_total;
    }
  }
  if (P.T_total >= (1ll << 31) / 2) return fail(CB_ERR_INVALID_ARG, "too many rows in one call");
  const cb_model_config &c = m->cfg;
  Carver cv;
  P.lay = carve_layer(cv, m, P.T_total);
  P.h_all = cv.take(P.T_total * c.d_model * sizeof(float));
  P.kf = cv.take(P.T_total * m->kvw * m->eb);
  P.dev = cv.take((P.N_total + 1) * sizeof(float));
  P.sel = cv.take((P.K_total + 1) * sizeof(int32_t));
  P.pos_all = cv.take(P.T_total * sizeof(int32_t));
  P.glob_all = cv.take(P.T_total * sizeof(int32_t));
  P.pos_c = cv.take((P.R_total + 1) * sizeof(int32_t));
  P.glob_c = cv.take((P.R_total + 1) * sizeof(int32_t));
  P.h_c = cv.take((P.R_total + 1) * c.d_model * sizeof(float));
  P.lm_x = cv.take((size_t)B * c.d_model * sizeof(float));
  P.lm_best = cv.take((size_t)B * sizeof(unsigned long long));
  if (blend) {
    P.kdev = cv.take((size_t)c.n_kv_heads * (P.N_total + 1) * sizeof(float));
    P.dev_idx = cv.take((P.T_total + 1) * sizeof(int32_t));
  }
  if (c.dtype == CB_BF16 && attention_tc_supported(c.n_q_heads, c.n_kv_heads, c.head_dim)) {
    // the compact rows of each request (the largest set; filtering only shrinks it)
    std::vector<AttnReq> ar(B);
    for (int b = 0; b < B; ++b)
      ar[b] = AttnReq{P.bm.r_off[b], P.bm.r_off[b + 1], (int64_t)P.bm.t_off[b], P.T[b]};
    P.attn_plan_bytes = attention_plan_bytes(ar.data(), B, c.n_q_heads, c.n_kv_heads);
    P.attn_plan = cv.take(P.attn_plan_bytes);
  }
  if (!P.sched.empty()) {
    // second set of compact buffers; the filtered rows ping-pong between them
    P.g_dev = cv.take((P.K_total + 1) * sizeof(float));
    P.g_keep = cv.take((P.K_total + 1) * sizeof(int32_t));
    P.g_sel = cv.take((P.K_total + 1) * sizeof(int32_t));
    P.g_pos = cv.take((P.R_total + 1) * sizeof(int32_t));
    P.g_glob = cv.take((P.R_total + 1) * sizeof(int32_t));
    P.g_src = cv.take((P.R_total + 1) * sizeof(int32_t));
    P.g_h = cv.take((P.R_total + 1) * c.d_model * sizeof(float));
  }
  if (blend && is_query_policy(p->policy)) {
    // [QCF] Eqs. 14-17: anchors, the probe cache [anchors; query rows] of
    // each request, the query rows' hidden states and the mass scratch
    const bool all = p->policy == CB_POLICY_QUERY_FULL;
    ProbeLayout &Q = P.probe;
    Q.B = B;
    Q.all = all;
    int probe_off = 0, u_off = 0, anchor_off = 0;
    size_t mass = 0;
    for (int b = 0; b < B; ++b) {
      ProbeLayout::Req r{};
      r.t_off = P.bm.t_off[b];
      r.n_ctx = P.N[b];
      r.n_u = P.T[b] - P.N[b];
      r.seg_begin = (int)Q.segs.size();
      for (int i = 0; i < reqs[b].n_segments; ++i) {
        const cb_segment &sg = reqs[b].segments[i];
        if (!sg.k_pic || sg.len == 0) continue;
        const int cnt = all ? sg.len : (int)(((int64_t)sg.len * p->anchor_bp + 9999) / 10000);
        Q.segs.push_back(ProbeLayout::Seg{anchor_off, cnt, P.seg_start[b][i], sg.len});
        anchor_off += cnt;
        r.n_anchor += cnt;
      }
      r.seg_end = (int)Q.segs.size();
      r.probe_off = probe_off;
      r.u_off = u_off;
      Q.reqs[b] = r;
      probe_off += r.n_anchor + r.n_u;
      u_off += r.n_u;
      const size_t mb = mass_ws_bytes(r.n_u, c.n_q_heads, c.n_kv_heads, r.n_ctx);
      if (mb > mass) mass = mb;
    }
    if ((int)Q.segs.size() > CB_MAX_SPANS)
      return fail(CB_ERR_INVALID_ARG, "more than %d cached segments in one query-aware call", CB_MAX_SPANS);
    Q.n_probe = probe_off;
    Q.n_u = u_off;
    P.n_anchor_total = anchor_off;
    P.qp_scores = cv.take((P.N_total + 1) * sizeof(float));
    P.qp_anchors = cv.take((size_t)(anchor_off + 1) * sizeof(int32_t));
    P.qp_rows = cv.take((size_t)(probe_off + 1) * sizeof(int32_t));
    P.qp_u = cv.take((size_t)4 * (u_off + 1) * sizeof(int32_t));
    // the anchor probe's cache for layers 0 .. max(L*) (the full view works
    // in the fused cache)
    int probe_layers = 0;
    if (!all)
      for (int i = 0; i < p->n_crit; ++i)
        probe_layers = std::max(probe_layers, p->crit_layers[i] + 1);
    const size_t pcache = (size_t)probe_layers * probe_off * m->kvw * m->eb + 256;
    P.qp_k = cv.take(pcache);
    P.qp_v = cv.take(pcache);
    P.qp_h = cv.take((size_t)(u_off + 1) * c.d_model * sizeof(float));
    P.qp_mass_bytes = mass;
    P.qp_mass = cv.take(mass);
  }
  if (host_kv && p->host_load_ctas == 0) {
    P.stage_bytes = (size_t)(P.N_total + 1) * m->kvw * m->eb;
    P.stage_bytes = (P.stage_bytes + 255) / 256 * 256;
    P.stage = cv.take(4 * P.stage_bytes);         // [buffer][K, V]
  }
  P.total = cv.off;
  return CB_OK;
}

static void fill_plan(const Plan &P, cb_plan *out) {
  out->T_total = P.T_total;
  out->N_total = P.N_total;
  out->K_total = P.K_total;
  out->R_total = P.R_total;
  out->workspace_bytes = P.total;
  out->K_final = P.K_final;
  out->R_final = P.R_final;
}

extern "C" cb_status cb_blend_plan(const cb_model *m, const cb_request *reqs, int B,
                                   const cb_blend_params *p, cb_plan *out) {
  if (!out) return fail(CB_ERR_INVALID_ARG, "out is NULL");
  Plan P;
  CB_TRY(make_plan(m, reqs, B, p, true, P));
  fill_plan(P, out);
  return CB_OK;
}

extern "C" cb_status cb_full_plan(const cb_model *m, const cb_request *reqs, int B,
                                  cb_plan *out) {
  if (!out) return fail(CB_ERR_INVALID_ARG, "out is NULL");
  Plan P;
  CB_TRY(make_plan(m, reqs, B, nullptr, false, P));
  fill_plan(P, out);
  return CB_OK;
}

// ------------------------------------------------------------------ layer --
// The swapped GEMM form (1 or 2 CTAs per MMA) in which a bf16 layer over n
// rows runs its MLP as one launch, or 0 when it runs the two projections:
// the one-launch form is switched on, both projections take the same swapped
// form, and the flags fit.
static int mlp_one_launch_form(int n, int d, int F) {
  if (!g_mlp_fusion.load(std::memory_order_relaxed) || n <= 0 || d <= 0 || F <= 0) return 0;
  const int path = g_gemm_path.load(std::memory_order_relaxed);
  const int form = path == CB_GEMM_AUTO        ? gemm_auto_form(n, d, EPI_SWIGLU)
                   : path == CB_GEMM_SWAP_AB      ? 1
                   : path == CB_GEMM_SWAP_AB_PAIR ? 2
                                                  : 0;
  const int form_down = path == CB_GEMM_AUTO ? gemm_auto_form(n, F, EPI_RESID) : form;
  return form && form == form_down && gemm_mlp_fits(n, F, form) ? form : 0;
}

extern "C" int cb_debug_mlp_one_launch(int n_rows, int d_model, int d_ffn) {
  return mlp_one_launch_form(n_rows, d_model, d_ffn) != 0;
}

static inline char *layer_ptr(void *base, int l, int64_t stride, size_t eb) {
  return (char *)base + (int64_t)l * stride * (int64_t)eb;
}

// One decoder layer over n rows of h (see cb_blend_layer).  q_only: stop
// once the rows' rotated queries are in S.q (bf16: only the W_q rows of the
// projection run; h, kc and vc are left as they are).
static cb_status layer_forward(cb_model *m, int l, float *h, int n, const int32_t *pos,
                               const int32_t *cache_row, const std::vector<AttnReq> &ar,
                               void *kc, void *vc, const LayerScratch &S, int *st,
                               cudaStream_t s, const int *attn_plan = nullptr,
                               const int32_t *attn_pos = nullptr, bool q_only = false) {
  const NvtxRange range("layer %d", l);
  const cb_model_config &c = m->cfg;
  const cb_layer_weights &L = m->layers[l];
  const int d = c.d_model, F = c.d_ffn, hd = c.head_dim;
  const cb_dtype dt = c.dtype;
  CB_CUDA(launch_rmsnorm(h, d, nullptr, n, d, L.norm1, c.norm_eps, S.x, d, dt, s));
  probe_mark(CB_PROBE_QKV, true, s);
  if (dt == CB_BF16 && hd == 128) {
    // projection, RoPE and the Eq. 7 scatter in one kernel
    const QkvEpi q{pos, cache_row, kc, vc, m->kvw, m->w.rope_table, c.n_q_heads, c.n_kv_heads};
    CB_TRY(run_linear(m, S.x, d, L.w_qkv, nullptr, d, n, q_only ? m->qw : m->qkv_rows, d,
                      EPI_QKV, S.q, m->qw, s, &q, S.split));
  } else {
    CB_TRY(run_linear(m, S.x, d, L.w_qkv, nullptr, d, n, m->qkv_rows, d, EPI_STORE_F32,
                      S.qkv32, m->qkv_rows, s));
    CB_CUDA(launch_qkv_finish(S.qkv32, m->qkv_rows, n, pos, cache_row, c.n_q_heads,
                              c.n_kv_heads, hd, m->w.rope_table, S.q, m->qw, kc, vc, m->kvw,
                              dt, 0, s));
  }
  probe_mark(CB_PROBE_QKV, false, s);
  if (q_only) return CB_OK;
  probe_mark(CB_PROBE_ATTENTION, true, s);
  // attn_pos: the rows' causal-mask positions in kc / vc when these are not
  // their request positions (the query probe's compact cache)
  CB_TRY(run_attention(S.q, m->qw, attn_pos ? attn_pos : pos, ar, kc, vc, m->kvw, c.n_q_heads,
                       c.n_kv_heads, hd,
                       1.f / sqrtf((float)hd), S.o, m->qw, dt, S.attn, S.attn_bytes, st, s,
                       attn_plan));
  probe_mark(CB_PROBE_ATTENTION, false, s);
  probe_mark(CB_PROBE_O, true, s);
  CB_TRY(run_linear(m, S.o, m->qw, L.w_o, nullptr, m->qw, n, d, m->qw, EPI_RESID, h, d, s));
  probe_mark(CB_PROBE_O, false, s);
  CB_CUDA(launch_rmsnorm(h, d, nullptr, n, d, L.norm2, c.norm_eps, S.x, d, dt, s));
  if (dt == CB_BF16 && S.split && S.mlp_epoch) {
    // gate/up and down in one launch (the swapped form both take)
    const int form = mlp_one_launch_form(n, d, F);
    if (form) {
      probe_mark(CB_PROBE_MLP, true, s);
      const cudaError_t e = launch_gemm_mlp(S.x, d, L.w_gate, L.w_up, d, L.w_down, F, n, F, d,
                                            S.g, F, h, d, st, s, form, S.split,
                                            ++*S.mlp_epoch);
      probe_mark(CB_PROBE_MLP, false, s);
      CB_CUDA(e);
      return CB_OK;
    }
  }
  probe_mark(CB_PROBE_SWIGLU, true, s);
  CB_TRY(run_linear(m, S.x, d, L.w_gate, L.w_up, d, n, F, d, EPI_SWIGLU, S.g, F, s, nullptr,
                    S.split));
  probe_mark(CB_PROBE_SWIGLU, false, s);
  probe_mark(CB_PROBE_DOWN, true, s);
  CB_TRY(run_linear(m, S.g, F, L.w_down, nullptr, F, n, d, F, EPI_RESID, h, d, s));
  probe_mark(CB_PROBE_DOWN, false, s);
  return CB_OK;
}

extern "C" size_t cb_layer_workspace_size(const cb_model *m, int n_rows) {
  if (!m || n_rows < 0) return 0;
  Carver c;
  carve_layer(c, m, n_rows);
  return c.off;
}

extern "C" cb_status cb_blend_layer(cb_model *m, int layer, float *h, int n_rows,
                                    const int32_t *pos, const int32_t *cache_row,
                                    const cb_attn_req *reqs, int n_req, void *k_cache,
                                    void *v_cache, void *ws, size_t ws_bytes,
                                    cb_stream stream) {
  if (!m) return fail(CB_ERR_INVALID_ARG, "model is NULL");
  if (layer < 0 || layer >= m->cfg.n_layers) return fail(CB_ERR_INVALID_ARG, "layer out of range");
  if (n_rows < 0) return fail(CB_ERR_INVALID_ARG, "n_rows < 0");
  if (n_rows == 0) return CB_OK;
  if (!h || !pos || !cache_row || !reqs || !k_cache || !v_cache) return fail(CB_ERR_INVALID_ARG, "NULL pointer");
  if (n_req <= 0 || n_req > CB_MAX_BATCH) return fail(CB_ERR_INVALID_ARG, "n_req must be in [1, %d]", CB_MAX_BATCH);
  if (!aligned16(h) || !aligned16(k_cache) || !aligned16(v_cache)) return fail(CB_ERR_INVALID_ARG, "misaligned");
  Carver c;
  LayerOffsets L = carve_layer(c, m, n_rows);
  if (!ws || ws_bytes < c.off) return fail(CB_ERR_WORKSPACE, "workspace too small (%zu < %zu)", ws_bytes, c.off);
  std::vector<AttnReq> ar(n_req);
  for (int i = 0; i < n_req; ++i) {
    const cb_attn_req &r = reqs[i];
    if (r.q_begin < 0 || r.q_end < r.q_begin || r.q_end > n_rows || r.kv_row0 < 0 || r.kv_len < 0)
      return fail(CB_ERR_INVALID_ARG, "req %d: bad ranges", i);
    ar[i] = AttnReq{r.q_begin, r.q_end, r.kv_row0, r.kv_len};
  }
  int *st;
  CB_TRY(status_ptr(&st));
  LayerScratch S = bind_layer((char *)ws, L);
  int mlp_epoch = 0;
  S.mlp_epoch = &mlp_epoch;
  CB_CUDA(reset_split(S, stream));
  return layer_forward(m, layer, h, n_rows, pos, cache_row, ar, k_cache, v_cache, S, st, stream);
}

// ------------------------------------------------------------------ stack --
static cb_status check_out(const cb_model *m, const cb_blend_out *out) {
  if (!out) return fail(CB_ERR_INVALID_ARG, "out is NULL");
  if (!out->k_cache || !out->v_cache) return fail(CB_ERR_INVALID_ARG, "out cache is NULL");
  if (!aligned16(out->k_cache) || !aligned16(out->v_cache) ||
      (out->cache_layer_stride * (int64_t)m->eb) % 16)
    return fail(CB_ERR_INVALID_ARG, "out cache must be 16-byte aligned");
  if (out->hidden && !aligned16(out->hidden)) return fail(CB_ERR_INVALID_ARG, "out hidden misaligned");
  return CB_OK;
}

static void full_attn_reqs(const Plan &P, std::vector<AttnReq> &ar) {
  ar.resize(P.B);
  for (int b = 0; b < P.B; ++b)
    ar[b] = AttnReq{P.bm.t_off[b], P.bm.t_off[b + 1], (int64_t)P.bm.t_off[b], P.T[b]};
}

// Final norm + tied LM head + arg-max of each request's last row of h:
// row r_off[b+1]-1 of the compact rows, or t_off[b+1]-1 of all rows.
// row_end: per request, one past its last row of h (B + 1 prefix sums)
static cb_status run_lm_head(cb_model *m, const Plan &P, const float *h, const int *row_end,
                             char *ws, int32_t *first_token, cudaStream_t s) {
  const cb_model_config &c = m->cfg;
  int32_t last[CB_MAX_BATCH];
  for (int b = 0; b < P.B; ++b) last[b] = row_end[b + 1] - 1;
  CB_CUDA(launch_lm_head_argmax(h, c.d_model, last, P.B, m->w.final_norm, c.norm_eps,
                                m->w.embed, c.vocab, c.d_model, c.dtype,
                                (float *)(ws + P.lm_x), (unsigned long long *)(ws + P.lm_best),
                                first_token, s));
  return CB_OK;
}

// One gradual-filtering step before layer l (CacheBlend blog, select_hkvd):
// the current rows' fresh keys of layer l are compared with the reused keys
// still in the layer's fused cache at the selected rows, each request keeps
// its k'_b largest deviations among its selected rows, and the hidden
// states of the kept rows (and of the uncached rows) are gathered.
static cb_status filter_rows(cb_model *m, int l, const BatchMeta &cur, const BatchMeta &nxt,
                             int R_nxt, const float *h, const int32_t *pos,
                             const int32_t *glob, const int32_t *sel, float *h_n,
                             int32_t *pos_n, int32_t *glob_n, int32_t *sel_n, int R_cur,
                             char *ws, const Plan &P, const LayerScratch &S,
                             const cb_blend_out *out, int64_t lstride, int *st,
                             cudaStream_t s, const int32_t *forced = nullptr) {
  const cb_model_config &c = m->cfg;
  const cb_layer_weights &Lw = m->layers[l];
  const int d = c.d_model, B = cur.B;
  void *kf = ws + P.kf;
  float *dp = (float *)(ws + P.g_dev);
  int32_t *keep = (int32_t *)(ws + P.g_keep);
  int32_t *src = (int32_t *)(ws + P.g_src);
  if (forced) {
    // the caller gives the kept positions: no ranking at this step
    CB_CUDA(check_selection(forced, nxt.k_off, nxt.n_ctx, B, st, s));
    CB_CUDA(launch_keep_from_positions(cur, nxt, forced, sel, keep, nxt.k_off[B], st, s));
    CB_CUDA(launch_filter_rows(cur, nxt, keep, sel, sel_n, pos_n, glob_n, src, R_nxt, st, s));
    CB_CUDA(launch_gather(h, d, R_cur, src, R_nxt, d, h_n, d, sizeof(float), st, s));
    return CB_OK;
  }
  CB_CUDA(launch_rmsnorm(h, d, nullptr, R_cur, d, Lw.norm1, c.norm_eps, S.x, d, c.dtype, s));
  const char *wk = (const char *)Lw.w_qkv + (int64_t)m->qw * d * m->eb;
  CB_TRY(run_linear(m, S.x, d, wk, nullptr, d, R_cur, m->kvw, d, EPI_STORE_F32, S.qkv32,
                    m->kvw, s));
  CB_CUDA(launch_qkv_finish(S.qkv32, m->kvw, R_cur, pos, nullptr, c.n_q_heads, c.n_kv_heads,
                            c.head_dim, m->w.rope_table, nullptr, 0, kf, nullptr, m->kvw,
                            c.dtype, 0, s));
  std::vector<SelReq> sr(B);
  for (int b = 0; b < B; ++b) {
    const int kc = cur.k_off[b + 1] - cur.k_off[b];
    sr[b] = SelReq{kc, nxt.k_off[b + 1] - nxt.k_off[b], (int64_t)cur.r_off[b], 0,
                   cur.k_off[b], nxt.k_off[b], 0, 0};
  }
  CB_CUDA(launch_deviation(kf, m->kvw, layer_ptr(out->k_cache, l, lstride, m->eb), m->kvw,
                           m->kvw, c.dtype, sr.data(), B, dp, s, glob));
  CB_CUDA(launch_topk(dp, sr.data(), B, keep, s));
  CB_CUDA(launch_filter_rows(cur, nxt, keep, sel, sel_n, pos_n, glob_n, src, R_nxt, st, s));
  CB_CUDA(launch_gather(h, d, R_cur, src, R_nxt, d, h_n, d, sizeof(float), st, s));
  return CB_OK;
}

// host_kv: the cached segments' K/V are in pinned host memory; each layer's
// slice is copied (copy engines, on copy_stream) into a two-layer staging
// area and stitched right before the layer runs, so the load of layer l + 1
// overlaps the compute of layer l ([CB] "Hiding Recompute Behind I/O").
// Per-chunk anchors ([QCF] Eq. 14): scores of every position, then each
// chunk's count highest (ties to the lower position), ascending.
static cb_status rank_anchors(const cb_model *m, const std::vector<AnchorChunk> &ch,
                              const std::vector<ProbeLayout::Seg> &segs, int rule,
                              float *scores, int32_t *anchors, cudaStream_t s) {
  CB_CUDA(launch_anchor_scores(ch.data(), (int)ch.size(), rule, m->cfg.n_layers, m->kvw,
                               m->cfg.dtype, scores, s));
  for (size_t base = 0; base < ch.size(); base += CB_MAX_BATCH) {
    SelReq r[CB_MAX_BATCH];
    int n = 0;
    for (size_t i = base; i < ch.size() && n < CB_MAX_BATCH; ++i, ++n)
      r[n] = SelReq{ch[i].len, segs[i].count, 0, 0, ch[i].score_off, segs[i].anchor_off, 0, 0};
    CB_CUDA(launch_topk(scores, r, n, anchors, s));
  }
  return CB_OK;
}

// [QCF] §3.3-3.4: every request's query rows (its uncached rows) run layers
// 0 .. max(L*) over the probe cache [anchors; query rows] (Eqs. 15-17: the
// anchors' stitched PIC entries at their request positions, read only);
// after each critical layer their attention mass on the request's context
// keys is added into I (Eq. 20).  QUERY_FULL: every position is an anchor
// and every layer critical (Eqs. 9-10).
// ready(l): layers 0 .. l of the fused cache hold the stitched chunk caches.
// layerwise (host-resident chunks, which arrive layer by layer): the anchor
// probe gathers each layer's probe cache just before its probe layer, so
// the probe overlaps the loads of its later layers.
static cb_status query_probe(cb_model *m, const cb_request *reqs, int B,
                             const cb_blend_params *p, const Plan &P, char *ws,
                             const cb_blend_out *out, int64_t lstride, const LayerScratch &S,
                             const float *h_all, float *I, int *st, cudaStream_t s,
                             const std::function<cb_status(int)> &ready, bool layerwise) {
  const cb_model_config &c = m->cfg;
  const ProbeLayout &Q = P.probe;
  const int d = c.d_model;
  const int32_t *anchors = p->anchors ? p->anchors : (const int32_t *)(ws + P.qp_anchors);
  if (!Q.all && !p->anchors) {
    std::vector<AnchorChunk> ch;
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < reqs[b].n_segments; ++i) {
        const cb_segment &sg = reqs[b].segments[i];
        if (!sg.k_pic || sg.len == 0) continue;
        ch.push_back(AnchorChunk{sg.k_pic, sg.pic_layer_stride, sg.len,
                                 P.n_off[b] + P.seg_start[b][i]});
      }
    CB_TRY(rank_anchors(m, ch, Q.segs, p->anchor_rule, (float *)(ws + P.qp_scores),
                        (int32_t *)(ws + P.qp_anchors), s));
  }
  const int nu = Q.n_u;
  int32_t *u = (int32_t *)(ws + P.qp_u);
  int32_t *u_pos = u, *u_src = u + (nu + 1), *u_cache = u + 2 * (nu + 1), *u_mask = u + 3 * (nu + 1);
  int32_t *rows = (int32_t *)(ws + P.qp_rows);
  CB_CUDA(launch_probe_rows(Q, anchors, rows, u_pos, u_src, u_cache, u_mask, st, s));
  float *h_u = (float *)(ws + P.qp_h);
  CB_CUDA(launch_gather(h_all, d, P.T_total, u_src, nu, d, h_u, d, sizeof(float), st, s));
  CB_CUDA(cudaMemsetAsync(I, 0, (size_t)P.N_total * sizeof(float), s));
  std::vector<char> crit(c.n_layers, p->policy == CB_POLICY_QUERY_FULL ? 1 : 0);
  int last = c.n_layers - 1;
  if (p->policy == CB_POLICY_QUERY_PROBE) {
    last = 0;
    for (int i = 0; i < p->n_crit; ++i) {
      crit[p->crit_layers[i]] = 1;
      if (p->crit_layers[i] > last) last = p->crit_layers[i];
    }
  }
  std::vector<AttnReq> ar(B);
  for (int b = 0; b < B; ++b) {
    const ProbeLayout::Req &r = Q.reqs[b];
    ar[b] = AttnReq{r.u_off, r.u_off + r.n_u, (int64_t)r.probe_off, r.n_anchor + r.n_u};
  }
  // The probe cache of every probe layer.  Full view: every context
  // position is an anchor, so the probe cache is the fused cache itself, row
  // for row (the query rows' K/V written there are recomputed by the blend
  // before it reads them).  Anchor probe: the anchors' stitched rows of all
  // probe layers, gathered at once.
  const int64_t pstride = (int64_t)Q.n_probe * m->kvw;    // elements per probe layer
  if (!Q.all && !layerwise) {
    CB_TRY(ready(last));
    CB_CUDA(launch_gather_layers(out->k_cache, lstride, m->kvw, P.T_total, rows, Q.n_probe,
                                 m->kvw, ws + P.qp_k, pstride, m->kvw, m->eb, last + 1, st, s));
    CB_CUDA(launch_gather_layers(out->v_cache, lstride, m->kvw, P.T_total, rows, Q.n_probe,
                                 m->kvw, ws + P.qp_v, pstride, m->kvw, m->eb, last + 1, st, s));
  }
  for (int l = 0; l <= last; ++l) {
    if (Q.all) CB_TRY(ready(l));
    if (!Q.all && layerwise) {
      CB_TRY(ready(l));
      CB_CUDA(launch_gather_layers(layer_ptr(out->k_cache, l, lstride, m->eb), lstride, m->kvw,
                                   P.T_total, rows, Q.n_probe, m->kvw,
                                   layer_ptr(ws + P.qp_k, l, pstride, m->eb), pstride, m->kvw,
                                   m->eb, 1, st, s));
      CB_CUDA(launch_gather_layers(layer_ptr(out->v_cache, l, lstride, m->eb), lstride, m->kvw,
                                   P.T_total, rows, Q.n_probe, m->kvw,
                                   layer_ptr(ws + P.qp_v, l, pstride, m->eb), pstride, m->kvw,
                                   m->eb, 1, st, s));
    }
    const char *kl = layer_ptr(out->k_cache, l, lstride, m->eb);
    void *pk = Q.all ? layer_ptr(out->k_cache, l, lstride, m->eb) : layer_ptr(ws + P.qp_k, l, pstride, m->eb);
    void *pv = Q.all ? layer_ptr(out->v_cache, l, lstride, m->eb) : layer_ptr(ws + P.qp_v, l, pstride, m->eb);
    // the last probe layer only feeds its queries to the mass: nothing after
    // its Q projection is read
    CB_TRY(layer_forward(m, l, h_u, nu, u_pos, u_cache, ar, pk, pv, S, st, s, nullptr, u_mask,
                         l == last));
    if (!crit[l]) continue;
    for (int b = 0; b < B; ++b) {
      const ProbeLayout::Req &r = Q.reqs[b];
      CB_CUDA(launch_attention_mass(S.q, m->qw, r.u_off, r.n_u, kl, m->kvw, r.t_off, r.n_ctx,
                                    c.n_q_heads, c.n_kv_heads, c.head_dim, ws + P.qp_mass,
                                    P.qp_mass_bytes, I + P.n_off[b], st, s));
    }
  }
  return CB_OK;
}

extern "C" cb_status cb_anchor_count(const cb_segment *chunks, int n_chunks, int ratio_bp,
                                     int64_t *n_anchors) {
  if (!n_anchors || (n_chunks > 0 && !chunks) || n_chunks < 0)
    return fail(CB_ERR_INVALID_ARG, "NULL pointer or n_chunks < 0");
  if (ratio_bp < 0 || ratio_bp > 10000) return fail(CB_ERR_INVALID_ARG, "ratio_bp must be in [0, 10000]");
  int64_t total = 0;
  for (int i = 0; i < n_chunks; ++i) {
    if (chunks[i].len < 0) return fail(CB_ERR_INVALID_ARG, "chunk %d: len < 0", i);
    total += ((int64_t)chunks[i].len * ratio_bp + 9999) / 10000;
  }
  *n_anchors = total;
  return CB_OK;
}

extern "C" size_t cb_anchor_workspace_size(const cb_model *m, const cb_segment *chunks,
                                           int n_chunks) {
  if (!m || !chunks || n_chunks <= 0) return 256;
  int64_t total = 0;
  for (int i = 0; i < n_chunks; ++i) total += chunks[i].len > 0 ? chunks[i].len : 0;
  return (size_t)(total + 1) * sizeof(float) + 256;
}

extern "C" cb_status cb_anchor_select(const cb_model *m, const cb_segment *chunks, int n_chunks,
                                      cb_anchor_rule rule, int ratio_bp, float *scores_out,
                                      int32_t *anchors_out, void *ws, size_t ws_bytes,
                                      cb_stream stream) {
  if (!m || !chunks || !anchors_out) return fail(CB_ERR_INVALID_ARG, "NULL pointer");
  if (n_chunks <= 0) return fail(CB_ERR_INVALID_ARG, "n_chunks must be >= 1");
  if (rule != CB_ANCHOR_SINK && rule != CB_ANCHOR_KNORM) return fail(CB_ERR_INVALID_ARG, "unknown anchor rule");
  if (ratio_bp < 0 || ratio_bp > 10000) return fail(CB_ERR_INVALID_ARG, "ratio_bp must be in [0, 10000]");
  std::vector<AnchorChunk> ch;
  std::vector<ProbeLayout::Seg> segs;
  int score_off = 0, anchor_off = 0;
  for (int i = 0; i < n_chunks; ++i) {
    const cb_segment &sg = chunks[i];
    if (sg.len < 0) return fail(CB_ERR_INVALID_ARG, "chunk %d: len < 0", i);
    if (rule == CB_ANCHOR_KNORM && sg.len > 0 &&
        (!sg.k_pic || !aligned16(sg.k_pic) || (sg.pic_layer_stride * (int64_t)m->eb) % 16 ||
         sg.pic_layer_stride < (int64_t)sg.len * m->kvw))
      return fail(CB_ERR_INVALID_ARG, "chunk %d: bad PIC layout", i);
    const int cnt = (int)(((int64_t)sg.len * ratio_bp + 9999) / 10000);
    ch.push_back(AnchorChunk{sg.k_pic, sg.pic_layer_stride, sg.len, score_off});
    segs.push_back(ProbeLayout::Seg{anchor_off, cnt, 0, sg.len});
    score_off += sg.len;
    anchor_off += cnt;
  }
  float *scores = scores_out;
  if (!scores) {
    if (!ws || ws_bytes < (size_t)(score_off + 1) * sizeof(float))
      return fail(CB_ERR_WORKSPACE, "anchor workspace too small");
    scores = (float *)ws;
  }
  return rank_anchors(m, ch, segs, rule, scores, anchors_out, stream);
}

static cb_status blend_impl(cb_model *m, const cb_request *reqs, int B,
                            const cb_blend_params *p, const cb_blend_out *out, void *ws_v,
                            size_t ws_bytes, cudaStream_t stream, bool host_kv,
                            cudaStream_t copy_stream) {
  const NvtxRange range(host_kv ? "cb_blend_prefill_host_kv" : "cb_blend_prefill");
  Plan P;
  CB_TRY(make_plan(m, reqs, B, p, true, P, host_kv));
  CB_TRY(check_out(m, out));
  if (!ws_v || ws_bytes < P.total) return fail(CB_ERR_WORKSPACE, "workspace too small (%zu < %zu)", ws_bytes, P.total);
  char *ws = (char *)ws_v;
  const cb_model_config &c = m->cfg;
  const int L = c.n_layers, s_layer = p->sel_layer, d = c.d_model;
  const int64_t lstride = out->cache_layer_stride ? out->cache_layer_stride : P.T_total * m->kvw;
  int *st;
  CB_TRY(status_ptr(&st));
  cudaStream_t s = stream;
  float *h_all = (float *)(ws + P.h_all);
  float *dev = out->deviation ? out->deviation : (float *)(ws + P.dev);
  int32_t *sel = out->selected ? out->selected : (int32_t *)(ws + P.sel);
  int32_t *pos_all = (int32_t *)(ws + P.pos_all), *glob_all = (int32_t *)(ws + P.glob_all);
  int32_t *pos_c = out->rows ? out->rows : (int32_t *)(ws + P.pos_c);
  int32_t *glob_c = (int32_t *)(ws + P.glob_c);
  float *h_c = out->hidden ? out->hidden : (float *)(ws + P.h_c);
  LayerScratch S = bind_layer(ws, P.lay);
  int mlp_epoch = 0;
  S.mlp_epoch = &mlp_epoch;
  CB_CUDA(reset_split(S, stream));

  // 1. re-position + stitch of every cached segment, layers [s, L)
  std::vector<cb_stitch_desc> descs;
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < reqs[b].n_segments; ++i) {
      const cb_segment &sg = reqs[b].segments[i];
      if (!sg.k_pic || sg.len == 0) continue;
      const int pos0 = P.seg_start[b][i];
      descs.push_back(cb_stitch_desc{sg.k_pic, sg.v_pic, sg.pic_layer_stride, sg.len,
                                     P.bm.t_off[b] + pos0, pos0 - sg.pic_pos0});
    }
  // host-resident chunks: per-layer copies into the staging area, stitched
  // one layer at a time; stage[l & 1] holds layer l as [N_total][kvw]
  const size_t sb = P.stage_bytes;
  auto stage_k = [&](int l) { return ws + P.stage + (size_t)(l & 1) * 2 * sb; };
  auto stage_v = [&](int l) { return ws + P.stage + (size_t)(l & 1) * 2 * sb + sb; };
  const int zc_ctas = host_kv ? p->host_load_ctas : 0;
  auto issue_copies = [&](int l) -> cb_status {
    if (zc_ctas > 0) {
      // zero-copy: the re-position kernel reads layer l of the pinned chunk
      // caches itself, with a capped grid, straight into the fused cache
      probe_mark(CB_PROBE_STITCH, true, copy_stream);
      CB_CUDA(launch_reposition(descs.data(), (int)descs.size(), l, l + 1, out->k_cache,
                                out->v_cache, lstride, m->kvw, c.head_dim, m->w.rope_table,
                                c.dtype, st, copy_stream, zc_ctas));
      probe_mark(CB_PROBE_STITCH, false, copy_stream);
      CB_CUDA(cudaEventRecord(m->ev_copied[l & 1], copy_stream));
      return CB_OK;
    }
    CB_CUDA(cudaStreamWaitEvent(copy_stream, m->ev_free[l & 1], 0));
    probe_mark(CB_PROBE_STITCH, true, copy_stream);
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < reqs[b].n_segments; ++i) {
        const cb_segment &sg = reqs[b].segments[i];
        if (!sg.k_pic || sg.len == 0) continue;
        const size_t off = ((size_t)P.n_off[b] + P.seg_start[b][i]) * m->kvw * m->eb;
        const size_t bytes = (size_t)sg.len * m->kvw * m->eb;
        const size_t src = (size_t)l * sg.pic_layer_stride * m->eb;
        CB_CUDA(cudaMemcpyAsync(stage_k(l) + off, (const char *)sg.k_pic + src, bytes,
                                cudaMemcpyHostToDevice, copy_stream));
        CB_CUDA(cudaMemcpyAsync(stage_v(l) + off, (const char *)sg.v_pic + src, bytes,
                                cudaMemcpyHostToDevice, copy_stream));
      }
    probe_mark(CB_PROBE_STITCH, false, copy_stream);
    CB_CUDA(cudaEventRecord(m->ev_copied[l & 1], copy_stream));
    return CB_OK;
  };
  auto stitch_layer = [&](int l) -> cb_status {
    if (zc_ctas > 0) {
      CB_CUDA(cudaStreamWaitEvent(s, m->ev_copied[l & 1], 0));
      return CB_OK;
    }
    std::vector<cb_stitch_desc> ld;
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < reqs[b].n_segments; ++i) {
        const cb_segment &sg = reqs[b].segments[i];
        if (!sg.k_pic || sg.len == 0) continue;
        const int pos0 = P.seg_start[b][i];
        const size_t off = ((size_t)P.n_off[b] + pos0) * m->kvw * m->eb;
        ld.push_back(cb_stitch_desc{stage_k(l) + off, stage_v(l) + off, 0, sg.len,
                                    P.bm.t_off[b] + pos0, pos0 - sg.pic_pos0});
      }
    CB_CUDA(cudaStreamWaitEvent(s, m->ev_copied[l & 1], 0));
    CB_CUDA(launch_reposition(ld.data(), (int)ld.size(), l, l + 1, out->k_cache, out->v_cache,
                              lstride, m->kvw, c.head_dim, m->w.rope_table, c.dtype, st, s));
    CB_CUDA(cudaEventRecord(m->ev_free[l & 1], s));
    return CB_OK;
  };
  // Host-resident chunks: layer l is loaded (issue_copies) at most two
  // layers ahead of the last one stitched, since its staging buffer (or its
  // copy-done event) is that of layer l - 2; stitch_through(l) stitches every
  // layer up to l, keeping the loads two layers ahead.
  int next_issue = s_layer, next_stitch = s_layer;
  auto prefetch = [&]() -> cb_status {
    while (next_issue < L && next_issue < next_stitch + 2) CB_TRY(issue_copies(next_issue++));
    return CB_OK;
  };
  auto stitch_through = [&](int upto) -> cb_status {
    if (!host_kv) return CB_OK;
    while (next_stitch <= upto && next_stitch < L) {
      CB_TRY(prefetch());
      CB_TRY(stitch_layer(next_stitch++));
    }
    return prefetch();
  };
  if (host_kv) {
    // fork the copy stream from the compute stream (a graph capture then
    // covers both); both staging buffers start free
    CB_CUDA(cudaEventRecord(m->ev_fork, s));
    CB_CUDA(cudaStreamWaitEvent(copy_stream, m->ev_fork, 0));
    CB_CUDA(cudaEventRecord(m->ev_free[0], s));
    CB_CUDA(cudaEventRecord(m->ev_free[1], s));
    CB_TRY(prefetch());
  } else {
    probe_mark(CB_PROBE_STITCH, true, s);
    CB_CUDA(launch_reposition(descs.data(), (int)descs.size(), s_layer, L, out->k_cache,
                              out->v_cache, lstride, m->kvw, c.head_dim, m->w.rope_table,
                              c.dtype, st, s));
    probe_mark(CB_PROBE_STITCH, false, s);
  }
  // 2. embeddings of every row, full layers below the selection layer
  const int32_t *toks[CB_MAX_BATCH];
  for (int b = 0; b < B; ++b) toks[b] = reqs[b].tokens;
  CB_CUDA(launch_embed(toks, P.bm, m->w.embed, c.vocab, d, c.dtype, h_all, st, s));
  int32_t *dev_idx = (int32_t *)(ws + P.dev_idx);
  CB_CUDA(launch_iota_rows(P.bm, pos_all, glob_all, (int)P.T_total, s, dev_idx));
  std::vector<AttnReq> ar_full;
  full_attn_reqs(P, ar_full);
  for (int l = 0; l < s_layer; ++l)
    CB_TRY(layer_forward(m, l, h_all, (int)P.T_total, pos_all, glob_all, ar_full,
                         layer_ptr(out->k_cache, l, lstride, m->eb),
                         layer_ptr(out->v_cache, l, lstride, m->eb), S, st, s));
  // 3. selection layer: fresh keys of every row, deviation, ranking; the
  // query-aware policies score the context with the query probe instead
  const bool query = is_query_policy(p->policy);
  // the key projection compares with the stitched layer s; the query probe
  // asks for its layers itself
  if (!query) CB_TRY(stitch_through(s_layer));
  // bf16 with 128-wide heads: the key projection's epilogue compares the
  // fresh keys with the stitched ones and leaves per-head squared
  // differences; the fresh keys are never stored
  const bool fused_dev = !query && c.dtype == CB_BF16 && c.head_dim == 128;
  float *kparts = (float *)(ws + P.kdev);
  const int64_t kstride = P.N_total + 1;
  {
    const cb_layer_weights &Ls = m->layers[s_layer];
    void *kf = ws + P.kf;
    if (!query) {
      CB_CUDA(launch_rmsnorm(h_all, d, nullptr, (int)P.T_total, d, Ls.norm1, c.norm_eps, S.x, d,
                             c.dtype, s));
      const char *wk = (const char *)Ls.w_qkv + (int64_t)m->qw * d * m->eb;
      if (fused_dev) {
        QkvEpi q{pos_all, glob_all, layer_ptr(out->k_cache, s_layer, lstride, m->eb), nullptr,
                 m->kvw, m->w.rope_table, c.n_q_heads, c.n_kv_heads, dev_idx};
        CB_TRY(run_linear(m, S.x, d, wk, nullptr, d, (int)P.T_total, m->kvw, d, EPI_KDEV, kparts,
                          kstride, s, &q));
      } else {
        CB_TRY(run_linear(m, S.x, d, wk, nullptr, d, (int)P.T_total, m->kvw, d, EPI_STORE_F32,
                          S.qkv32, m->kvw, s));
        CB_CUDA(launch_qkv_finish(S.qkv32, m->kvw, (int)P.T_total, pos_all, nullptr, c.n_q_heads,
                                  c.n_kv_heads, c.head_dim, m->w.rope_table, nullptr, 0, kf,
                                  nullptr, m->kvw, c.dtype, 0, s));
      }
    }
    // selection requests: every request's cached segments are its spans
    std::vector<cb_select_req> cr(B);
    std::vector<std::vector<int32_t>> seg_offs(B);
    int order_at = 0;
    for (int b = 0; b < B; ++b) {
      std::vector<int32_t> &o = seg_offs[b];
      std::vector<int> lens;
      for (int i = 0; i < reqs[b].n_segments; ++i) {
        if (!reqs[b].segments[i].k_pic) break;
        o.push_back(P.seg_start[b][i]);
        lens.push_back(reqs[b].segments[i].len);
      }
      o.push_back(P.N[b]);
      int L_ = p->span_len, off_ = p->span_offset;
      if (L_ == 0) {
        // the median cached-segment length, shifted by half a span
        std::vector<int> sl = lens;
        std::sort(sl.begin(), sl.end());
        L_ = sl.empty() ? 1 : (sl.size() % 2 ? sl[sl.size() / 2]
                                             : (sl[sl.size() / 2 - 1] + sl[sl.size() / 2]) / 2);
        if (L_ < 1) L_ = 1;
        off_ = L_ / 2;
      }
      cr[b] = cb_select_req{P.N[b], P.k[b], (int64_t)P.bm.t_off[b], (int64_t)P.bm.t_off[b],
                            P.n_off[b], P.bm.k_off[b], (int)o.size() - 1, o.data(),
                            p->span_order ? p->span_order + order_at : nullptr, L_, off_};
      order_at += (int)o.size() - 1;
    }
    SelPlan plan;
    const char *err = "";
    if (make_sel_plan(cr.data(), B, query ? CB_POLICY_TOKEN_TOPK : p->policy, plan, &err) !=
        CB_OK)
      return fail(CB_ERR_INVALID_ARG, "%s", err);
    const std::vector<SelReq> &sr = plan.reqs;
    probe_mark(CB_PROBE_SELECT, true, s);
    if (query) {
      // I(t) in the deviation buffer, then P = TopK(I, k) ([QCF] Eq. 11)
      CB_TRY(query_probe(m, reqs, B, p, P, ws, out, lstride, S, h_all, dev, st, s,
                         stitch_through, host_kv));
      if (p->forced_selected) {
        if (sel != p->forced_selected && P.K_total > 0)
          CB_CUDA(cudaMemcpyAsync(sel, p->forced_selected, P.K_total * sizeof(int32_t),
                                  cudaMemcpyDeviceToDevice, s));
      } else {
        CB_CUDA(launch_selection(dev, plan, sel, st, s));
      }
    } else if (p->forced_selected) {
      // the caller fixes P; d is still produced for inspection
      if (fused_dev)
        CB_CUDA(launch_reduce_parts(kparts, c.n_kv_heads, kstride, sr.data(), B, dev, s));
      else
        CB_CUDA(launch_deviation(kf, m->kvw, layer_ptr(out->k_cache, s_layer, lstride, m->eb),
                                 m->kvw, m->kvw, c.dtype, sr.data(), B, dev, s));
      if (sel != p->forced_selected && P.K_total > 0)
        CB_CUDA(cudaMemcpyAsync(sel, p->forced_selected, P.K_total * sizeof(int32_t),
                                cudaMemcpyDeviceToDevice, s));
    } else if (fused_dev && p->policy == CB_POLICY_TOKEN_TOPK) {
      CB_CUDA(launch_topk_parts(kparts, c.n_kv_heads, kstride, sr.data(), B, dev, sel, s));
    } else if (fused_dev) {
      CB_CUDA(launch_reduce_parts(kparts, c.n_kv_heads, kstride, sr.data(), B, dev, s));
      CB_CUDA(launch_selection(dev, plan, sel, st, s));
    } else {
      CB_TRY(run_selection(kf, m->kvw, layer_ptr(out->k_cache, s_layer, lstride, m->eb),
                           m->kvw, m->kvw, c.dtype, plan, dev, sel, st, s));
    }
    probe_mark(CB_PROBE_SELECT, false, s);
  }
  CB_CUDA(check_selection(sel, P.bm.k_off, P.bm.n_ctx, B, st, s));
  // 4. computed rows: selected context rows + uncached rows, gathered once
  probe_mark(CB_PROBE_GATHER, true, s);
  CB_CUDA(launch_rows_gather(P.bm, sel, pos_c, glob_c, (int)P.R_total, h_all, d, h_c, st, s));
  probe_mark(CB_PROBE_GATHER, false, s);
  // 5. layers >= s on the computed rows; gradual filtering steps shrink the
  // set between layers (the rows alternate between two buffer sets)
  int32_t *sel_b[2] = {sel, (int32_t *)(ws + P.g_sel)};
  int32_t *pos_b[2] = {pos_c, (int32_t *)(ws + P.g_pos)};
  int32_t *glob_b[2] = {glob_c, (int32_t *)(ws + P.g_glob)};
  float *h_b[2] = {h_c, (float *)(ws + P.g_h)};
  int cur = 0;
  BatchMeta bm = P.bm;
  int R_cur = (int)P.R_total;
  size_t next_step = 0;
  int64_t forced_at = 0;    // this step's part of p->forced_kept
  std::vector<AttnReq> ar_c(B);
  // the compact layers' attention units, planned from the rows' positions
  // whenever the set changes (its first layer, each filtering step)
  int *attn_plan = P.attn_plan_bytes ? (int *)(ws + P.attn_plan) : nullptr;
  bool plan_stale = true;
  for (int l = s_layer; l < L; ++l) {
    CB_TRY(stitch_through(l));
    if (next_step < P.sched.size() && P.sched[next_step].layer == l) {
      const Plan::Step &stp = P.sched[next_step++];
      CB_TRY(filter_rows(m, l, bm, stp.bm, (int)stp.R_total, h_b[cur], pos_b[cur], glob_b[cur],
                         sel_b[cur], h_b[cur ^ 1], pos_b[cur ^ 1], glob_b[cur ^ 1],
                         sel_b[cur ^ 1], R_cur, ws, P, S, out, lstride, st, s,
                         p->forced_kept ? p->forced_kept + forced_at : nullptr));
      forced_at += stp.K_total;
      cur ^= 1;
      bm = stp.bm;
      R_cur = (int)stp.R_total;
      plan_stale = true;
    }
    for (int b = 0; b < B; ++b)
      ar_c[b] = AttnReq{bm.r_off[b], bm.r_off[b + 1], (int64_t)P.bm.t_off[b], P.T[b]};
    if (attn_plan && plan_stale) {
      CB_CUDA(launch_attention_plan(pos_b[cur], ar_c.data(), B, c.n_q_heads, c.n_kv_heads,
                                    attn_plan, P.attn_plan_bytes, s));
      plan_stale = false;
    }
    CB_TRY(layer_forward(m, l, h_b[cur], R_cur, pos_b[cur], glob_b[cur], ar_c,
                         layer_ptr(out->k_cache, l, lstride, m->eb),
                         layer_ptr(out->v_cache, l, lstride, m->eb), S, st, s, attn_plan));
  }
  if (cur == 1) {
    // the final set is in the second buffers: move it to the outputs
    CB_CUDA(cudaMemcpyAsync(sel_b[0], sel_b[1], P.K_final * sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, s));
    CB_CUDA(cudaMemcpyAsync(pos_b[0], pos_b[1], P.R_final * sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, s));
    CB_CUDA(cudaMemcpyAsync(h_b[0], h_b[1], P.R_final * d * sizeof(float),
                            cudaMemcpyDeviceToDevice, s));
  }
  // 6. first token from each request's last computed row (its last position)
  probe_mark(CB_PROBE_LM_HEAD, true, s);
  if (out->first_token) CB_TRY(run_lm_head(m, P, h_b[0], bm.r_off, ws, out->first_token, s));
  probe_mark(CB_PROBE_LM_HEAD, false, s);
  return CB_OK;
}

// ----------------------------------------------------------- call graphs --
// The kernels of a blended call and every argument they receive follow from
// its host arguments alone: device data is read through pointers, and the
// call neither synchronises nor reads anything back.  The first call with a
// given argument set therefore records its launches into a CUDA graph, and
// later calls with the same set replay it, which removes the host's launch
// cost and most of the gaps between the launches.  A set is recorded on its
// second call (the first runs directly and also does the one-time host
// set-up of the kernels).  The call runs its launches directly on the legacy
// default stream (which cannot be captured), on a stream that the caller is
// capturing, and while the launch probe is on.
namespace {
constexpr size_t kCallGraphs = 4;

struct KeyWriter {
  std::vector<uint8_t> v;
  template <class T>
  void put(const T &x) {
    const uint8_t *b = reinterpret_cast<const uint8_t *>(&x);
    v.insert(v.end(), b, b + sizeof(T));
  }
};

// Every host argument of cb_blend_prefill, field by field (no padding bytes).
std::vector<uint8_t> call_key(const cb_model *m, const cb_request *reqs, int B,
                              const cb_blend_params *p, const cb_blend_out *out, void *ws,
                              size_t ws_bytes, cudaStream_t stream) {
  KeyWriter k;
  int dev = -1;
  cudaGetDevice(&dev);
  k.put(dev);
  k.put(m);
  k.put(g_gemm_path.load(std::memory_order_relaxed));
  k.put(B);
  int n_cached = 0;
  for (int b = 0; b < B; ++b) {
    k.put(reqs[b].tokens);
    k.put(reqs[b].n_segments);
    for (int i = 0; i < reqs[b].n_segments; ++i) {
      const cb_segment &g = reqs[b].segments[i];
      k.put(g.len);
      k.put(g.k_pic);
      k.put(g.v_pic);
      k.put(g.pic_layer_stride);
      k.put(g.pic_pos0);
      n_cached += g.k_pic != nullptr;
    }
  }
  k.put(p->ratio_bp);
  k.put(p->policy);
  k.put(p->sel_layer);
  k.put(p->n_schedule);
  for (int i = 0; i < p->n_schedule; ++i) {
    k.put(p->schedule[i].layer);
    k.put(p->schedule[i].keep);
  }
  k.put(p->span_len);
  k.put(p->span_offset);
  k.put(p->span_order != nullptr);
  if (p->span_order)
    for (int i = 0; i < n_cached; ++i) k.put(p->span_order[i]);
  k.put(p->forced_selected);
  k.put(p->forced_kept);
  k.put(p->host_load_ctas);
  k.put(p->anchors);
  k.put(p->anchor_rule);
  k.put(p->anchor_bp);
  k.put(p->n_crit);
  for (int i = 0; i < p->n_crit && p->crit_layers; ++i) k.put(p->crit_layers[i]);
  k.put(out->k_cache);
  k.put(out->v_cache);
  k.put(out->cache_layer_stride);
  k.put(out->deviation);
  k.put(out->selected);
  k.put(out->hidden);
  k.put(out->rows);
  k.put(out->first_token);
  k.put(ws);
  k.put(ws_bytes);
  k.put(stream);
  return std::move(k.v);
}
}  // namespace

extern "C" cb_status cb_blend_prefill(cb_model *m, const cb_request *reqs, int B,
                                      const cb_blend_params *p, const cb_blend_out *out,
                                      void *ws, size_t ws_bytes, cb_stream stream) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool direct = !m || !reqs || B <= 0 || B > CB_MAX_BATCH || !p || !out ||
                      stream == nullptr || stream == cudaStreamLegacy ||
                      stream == cudaStreamPerThread ||
                      g_probe_kind.load(std::memory_order_relaxed) != 0 ||
                      cudaStreamIsCapturing(stream, &cap) != cudaSuccess ||
                      cap != cudaStreamCaptureStatusNone;
  if (direct) return blend_impl(m, reqs, B, p, out, ws, ws_bytes, stream, false, nullptr);
  for (int b = 0; b < B; ++b)
    if (!reqs[b].segments || reqs[b].n_segments <= 0)
      return blend_impl(m, reqs, B, p, out, ws, ws_bytes, stream, false, nullptr);
  std::vector<uint8_t> key = call_key(m, reqs, B, p, out, ws, ws_bytes, stream);
  std::lock_guard<std::mutex> lk(m->graph_mu);
  for (CallGraph &g : m->graphs)
    if (g.key == key) {
      const NvtxRange range("cb_blend_prefill (recorded call)");
      g.used = ++m->graph_clock;
      CB_CUDA(cudaGraphLaunch(g.exec, stream));
      g_launches.fetch_add(g.launches);
      return CB_OK;
    }
  auto seen = std::find(m->graph_seen.begin(), m->graph_seen.end(), key);
  if (seen == m->graph_seen.end()) {
    const cb_status rc = blend_impl(m, reqs, B, p, out, ws, ws_bytes, stream, false, nullptr);
    if (rc == CB_OK) {
      if (m->graph_seen.size() >= 2 * kCallGraphs) m->graph_seen.erase(m->graph_seen.begin());
      m->graph_seen.push_back(std::move(key));
    }
    return rc;
  }
  m->graph_seen.erase(seen);
  // record the call (nothing runs while the stream captures), then run it
  const unsigned long long n0 = g_launches.load();
  CB_CUDA(cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal));
  const cb_status rc = blend_impl(m, reqs, B, p, out, ws, ws_bytes, stream, false, nullptr);
  cudaGraph_t graph = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(stream, &graph);
  if (rc != CB_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (ce != cudaSuccess) return fail(CB_ERR_CUDA, "recording the call: %s", cudaGetErrorString(ce));
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ie != cudaSuccess) return fail(CB_ERR_CUDA, "instantiating the call: %s", cudaGetErrorString(ie));
  CallGraph g;
  g.key = std::move(key);
  g.exec = exec;
  g.launches = g_launches.load() - n0;
  g.used = ++m->graph_clock;
  if (m->graphs.size() >= kCallGraphs) {
    auto lru = std::min_element(m->graphs.begin(), m->graphs.end(),
                                [](const CallGraph &a, const CallGraph &b) { return a.used < b.used; });
    cudaGraphExecDestroy(lru->exec);
    *lru = std::move(g);
  } else {
    m->graphs.push_back(std::move(g));
  }
  CB_CUDA(cudaGraphLaunch(exec, stream));
  return CB_OK;
}

extern "C" cb_status cb_blend_plan_host_kv(const cb_model *m, const cb_request *reqs, int B,
                                           const cb_blend_params *p, cb_plan *out) {
  if (!out) return fail(CB_ERR_INVALID_ARG, "out is NULL");
  Plan P;
  CB_TRY(make_plan(m, reqs, B, p, true, P, true));
  fill_plan(P, out);
  return CB_OK;
}

extern "C" cb_status cb_blend_prefill_host_kv(cb_model *m, const cb_request *reqs, int B,
                                              const cb_blend_params *p,
                                              const cb_blend_out *out, void *ws,
                                              size_t ws_bytes, cb_stream stream,
                                              cb_stream copy_stream) {
  if (!copy_stream || copy_stream == stream)
    return fail(CB_ERR_INVALID_ARG, "copy_stream must be a stream other than stream");
  if (!m || !reqs || B <= 0 || B > CB_MAX_BATCH) return fail(CB_ERR_INVALID_ARG, "bad model or requests");
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < reqs[b].n_segments; ++i) {
      const cb_segment &sg = reqs[b].segments[i];
      if (!sg.k_pic || sg.len == 0) continue;
      for (const void *ptr : {sg.k_pic, sg.v_pic}) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess || a.type != cudaMemoryTypeHost)
          return fail(CB_ERR_INVALID_ARG, "request %d segment %d: chunk caches must be pinned host memory", b, i);
        // the zero-copy load, and the key-norm anchor scores of the query
        // probe, dereference the host pointer in a kernel: it must be the
        // allocation's device address as well (unified addressing)
        const bool kernel_reads =
            p && (p->host_load_ctas > 0 ||
                  (p->policy == CB_POLICY_QUERY_PROBE && p->anchor_rule == CB_ANCHOR_KNORM &&
                   !p->anchors));
        if (kernel_reads && a.devicePointer != ptr)
          return fail(CB_ERR_INVALID_ARG, "request %d segment %d: chunk cache is not mapped at the same device address (read by a kernel)", b, i);
      }
    }
  return blend_impl(m, reqs, B, p, out, ws, ws_bytes, stream, true, copy_stream);
}

extern "C" cb_status cb_full_prefill(cb_model *m, const cb_request *reqs, int B,
                                     const cb_blend_out *out, void *ws_v, size_t ws_bytes,
                                     cb_stream stream) {
  const NvtxRange range("cb_full_prefill");
  Plan P;
  CB_TRY(make_plan(m, reqs, B, nullptr, false, P));
  CB_TRY(check_out(m, out));
  if (!ws_v || ws_bytes < P.total) return fail(CB_ERR_WORKSPACE, "workspace too small (%zu < %zu)", ws_bytes, P.total);
  char *ws = (char *)ws_v;
  const cb_model_config &c = m->cfg;
  const int64_t lstride = out->cache_layer_stride ? out->cache_layer_stride : P.T_total * m->kvw;
  int *st;
  CB_TRY(status_ptr(&st));
  float *h = out->hidden ? out->hidden : (float *)(ws + P.h_all);
  int32_t *pos_all = out->rows ? out->rows : (int32_t *)(ws + P.pos_all);
  int32_t *glob_all = (int32_t *)(ws + P.glob_all);
  LayerScratch S = bind_layer(ws, P.lay);
  int mlp_epoch = 0;
  S.mlp_epoch = &mlp_epoch;
  CB_CUDA(reset_split(S, stream));
  const int32_t *toks[CB_MAX_BATCH];
  for (int b = 0; b < B; ++b) toks[b] = reqs[b].tokens;
  CB_CUDA(launch_embed(toks, P.bm, m->w.embed, c.vocab, c.d_model, c.dtype, h, st, stream));
  CB_CUDA(launch_iota_rows(P.bm, pos_all, glob_all, (int)P.T_total, stream));
  std::vector<AttnReq> ar;
  full_attn_reqs(P, ar);
  for (int l = 0; l < c.n_layers; ++l)
    CB_TRY(layer_forward(m, l, h, (int)P.T_total, pos_all, glob_all, ar,
                         layer_ptr(out->k_cache, l, lstride, m->eb),
                         layer_ptr(out->v_cache, l, lstride, m->eb), S, st, stream));
  if (out->first_token) CB_TRY(run_lm_head(m, P, h, P.bm.t_off, ws, out->first_token, stream));
  return CB_OK;
}
