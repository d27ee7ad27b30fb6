// Deviation ranking and selection.
//
//  * deviation_kernel -- d_i = ||K_i^fresh - K_i^reused||_2^2 over all kv
//    heads, fp32 ("Request Order Matters" §2.2 Eq. 1).  One warp per token
//    row, 16-byte loads; HBM-bound.
//  * topk_kernel -- exact k largest d_i per request, ties to the lower
//    index, indices written ascending (token top-k, same page §2.2 Eq. 2).
//    One CTA per request: a 4-pass 8-bit radix select over the order-
//    preserving integer image of the floats finds the k-th largest key,
//    then a block-wide ordered compaction emits the winners by index.
//  * doc_aligned_kernel -- document-aligned spans (same page §2.3 Eq. 3).
//  * build_rows / iota_rows -- positions and fused-cache rows of the rows a
//    layer computes.
#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

constexpr int kSelThreads = 1024;

struct SelParams {
  int n_req;
  SelReq r[CB_MAX_BATCH];
  int row_prefix[CB_MAX_BATCH + 1];  // context rows before request i
};

// -------------------------------------------------------------- deviation --
template <typename T>
__global__ void __launch_bounds__(256)
deviation_kernel(const __grid_constant__ SelParams p, const T *__restrict__ kf,
                 int64_t ld_f, const T *__restrict__ kr, int64_t ld_r,
                 const int32_t *__restrict__ reused_rows, int row_elems,
                 float *__restrict__ dev_out) {
  constexpr int VEC = 16 / sizeof(T);
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int total = p.row_prefix[p.n_req];
  if (warp >= total) return;
  int b = 0;
  while (p.row_prefix[b + 1] <= warp) ++b;
  const SelReq &q = p.r[b];
  const int i = warp - p.row_prefix[b];
  const T *a = kf + (q.fresh_row0 + i) * ld_f;

  const int64_t fr = q.fresh_row0 + i;
  const int64_t rr = reused_rows ? q.reused_row0 + reused_rows[fr] : q.reused_row0 + i;
  const T *c = kr + rr * ld_r;
  float acc = 0.f;
  for (int col = lane * VEC; col < row_elems; col += 32 * VEC) {
    float x[VEC], y[VEC];
    load16<T>(a + col, x);
    load16<T>(c + col, y);
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      const float t = x[j] - y[j];
      acc = fmaf(t, t, acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) dev_out[q.dev_offset + i] = acc;
}

static void fill_params(SelParams &p, const SelReq *reqs, int n_req) {
  p.n_req = n_req;
  p.row_prefix[0] = 0;
  for (int i = 0; i < n_req; ++i) {
    p.r[i] = reqs[i];
    p.row_prefix[i + 1] = p.row_prefix[i] + reqs[i].n_ctx;
  }
}

// The selection keeps its working state in shared memory and dev_out.
size_t select_ws_bytes(int) { return 0; }

cudaError_t launch_deviation(const void *k_fresh, int64_t ld_fresh,
                             const void *k_reused, int64_t ld_reused,
                             int row_elems, cb_dtype dt, const SelReq *reqs,
                             int n_req, float *dev_out, cudaStream_t s,
                             const int32_t *reused_rows) {
  SelParams p;
  fill_params(p, reqs, n_req);
  const int rows = p.row_prefix[n_req];
  if (rows == 0) return cudaSuccess;
  const int blocks = (rows + 7) / 8;
  if (dt == CB_BF16)
    deviation_kernel<bf16><<<blocks, 256, 0, s>>>(
        p, reinterpret_cast<const bf16 *>(k_fresh), ld_fresh,
        reinterpret_cast<const bf16 *>(k_reused), ld_reused, reused_rows, row_elems, dev_out);
  else
    deviation_kernel<float><<<blocks, 256, 0, s>>>(
        p, reinterpret_cast<const float *>(k_fresh), ld_fresh,
        reinterpret_cast<const float *>(k_reused), ld_reused, reused_rows, row_elems,
        dev_out);
  return launched(1);
}

// ------------------------------------------------------------------ top-k --
// Order-preserving map of float bits to unsigned integers: larger float ->
// larger key (negative values below positive ones, -0 just below +0).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan of one int per thread (kSelThreads threads); returns
// the exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_buf,
                                                    int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < (kSelThreads / 32) ? warp_buf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_buf[lane] = t;  // inclusive prefix of warp sums
  }
  __syncthreads();
  const int before = (w > 0 ? warp_buf[w - 1] : 0) + x - v;
  *total = warp_buf[kSelThreads / 32 - 1];
  __syncthreads();
  return before;
}

// The k largest of d[0 .. n) (ties to the lower index), their indices
// written ascending to out: the body of the top-k kernels, one CTA.  d is a
// generic pointer (global or shared memory) that the whole CTA reads.
__device__ void topk_block(const float *d, int n, int k, int32_t *__restrict__ out) {
  __shared__ uint32_t hist[256];
  __shared__ int warp_buf[32];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_remaining;
  const int tid = threadIdx.x;

  if (tid == 0) { s_prefix = 0; s_mask = 0; s_remaining = k; }
  // ---- radix select of the k-th largest key, 8 bits per pass, MSB first
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int j = tid; j < 256; j += kSelThreads) hist[j] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int base = 0; base < n; base += kSelThreads) {
      const int i = base + tid;
      bool active = false;
      uint32_t digit = 0;
      if (i < n) {
        const uint32_t key = float_key(d[i]);
        if ((key & mask) == prefix) { active = true; digit = (key >> shift) & 255u; }
      }
      // warp-aggregated histogram update: one atomic per distinct digit
      // (deviations share their leading bits, so plain atomics would pile
      // onto a few bins)
      const unsigned act = __ballot_sync(0xffffffffu, active);
      if (active) {
        const unsigned peers = __match_any_sync(act, digit);
        if ((tid & 31) == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
    }
    __syncthreads();
    if (tid < 32) {
      // find the digit holding the remaining-th largest: walk digits from
      // 255 down; each lane owns 8 consecutive digits.
      const int lane = tid;
      const int hi = 255 - lane * 8;
      uint32_t cnt[8];
      uint32_t mysum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { cnt[j] = hist[hi - j]; mysum += cnt[j]; }
      // inclusive scan over lanes (lane 0 holds the highest digits)
      uint32_t incl = mysum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - mysum;
      const uint32_t rem = (uint32_t)s_remaining;
      if (excl < rem && incl >= rem) {
        uint32_t acc = excl;
        int j = 0;
        for (; j < 8; ++j) {
          if (acc + cnt[j] >= rem) break;
          acc += cnt[j];
        }
        const uint32_t dig = (uint32_t)(hi - j);
        s_prefix = prefix | (dig << shift);
        s_mask = mask | (255u << shift);
        s_remaining = (int)(rem - acc);
      }
    }
    __syncthreads();
  }
  const uint32_t thr = s_prefix;     // key of the k-th largest value
  const int need_eq = s_remaining;   // how many keys equal to thr to take
  // ---- ordered compaction: keep key > thr, and the first need_eq keys
  // equal to thr in index order.  Thread t owns the contiguous range
  // [t * per, (t + 1) * per); one block scan of its packed (greater, equal)
  // counts gives every output position (a key's position is the number of
  // greater keys before it plus the taken equal keys before it).
  if (n < 32768) {     // both packed counts stay below 2^15
    const int per = (n + kSelThreads - 1) / kSelThreads;
    const int i0 = tid * per, i1 = min(n, i0 + per);
    int gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = float_key(d[i]);
      gt += key > thr;
      eq += key == thr;
    }
    int total;
    const int before = block_exclusive_scan((gt << 16) | eq, warp_buf, &total);
    int g = before >> 16, e = before & 0xFFFF;
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = float_key(d[i]);
      if (key > thr) {
        out[g + min(e, need_eq)] = i;
        ++g;
      } else if (key == thr) {
        if (e < need_eq) out[g + e] = i;
        ++e;
      }
    }
    return;
  }
  int taken_eq = 0, written = 0;
  for (int base = 0; base < n; base += kSelThreads) {
    const int i = base + tid;
    uint32_t key = 0;
    if (i < n) key = float_key(d[i]);
    const int gt = (i < n && key > thr) ? 1 : 0;
    const int eq = (i < n && key == thr) ? 1 : 0;
    int eq_total;
    const int eq_before = block_exclusive_scan(eq, warp_buf, &eq_total);
    const int sel = gt || (eq && (taken_eq + eq_before) < need_eq);
    int sel_total;
    const int pos = block_exclusive_scan(sel, warp_buf, &sel_total);
    if (sel) out[written + pos] = i;
    written += sel_total;
    taken_eq += eq_total;
    if (written >= k) break;
  }
}

__global__ void __launch_bounds__(kSelThreads)
topk_kernel(const __grid_constant__ SelParams p, const float *__restrict__ dev,
            int32_t *__restrict__ idx_out) {
  const SelReq &q = p.r[blockIdx.x];
  if (q.k <= 0) return;
  topk_block(dev + q.dev_offset, q.n_ctx, q.k, idx_out + q.idx_offset);
}

// Deviations of the selection layer from the per-head partials that the key
// projection's epilogue leaves (EPI_KDEV), summed in head order, then (with
// rank) the request's token top-k over them.  One CTA per request; with
// rank the deviations stay in shared memory (kSmemCtx floats at most; a
// longer request reads them back from dev_out) for the select's passes.
constexpr int kSmemCtx = 40960;
constexpr int kPartsUnroll = 8;            // head partials loaded at once (more: one by one)
constexpr int kPartsTok = 3;               // tokens per thread per pass
template <bool RANK>
__global__ void __launch_bounds__(kSelThreads)
parts_kernel(const __grid_constant__ SelParams p, const float *__restrict__ parts, int n_parts,
             int64_t part_stride, float *__restrict__ dev_out, int32_t *__restrict__ idx_out) {
  extern __shared__ float s_d[];
  grid_dep_wait();      // the partials come from the previous kernel
  grid_dep_launch();
  const SelReq &q = p.r[blockIdx.x];
  const int n = q.n_ctx;
  const bool in_smem = RANK && n <= kSmemCtx;
  if (n_parts <= kPartsUnroll) {
    // every load of a thread's kPartsTok tokens is issued before the first
    // add (one memory round trip); the adds keep the head order
    for (int i0 = threadIdx.x; i0 < n; i0 += kSelThreads * kPartsTok) {
      float x[kPartsTok][kPartsUnroll];
#pragma unroll
      for (int u = 0; u < kPartsTok; ++u) {
        const int i = i0 + u * kSelThreads;
        const float *src = parts + q.dev_offset + i;
#pragma unroll
        for (int h = 0; h < kPartsUnroll; ++h)
          x[u][h] = (i < n && h < n_parts) ? __ldg(src + h * part_stride) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kPartsTok; ++u) {
        const int i = i0 + u * kSelThreads;
        if (i >= n) break;
        float v = 0.f;
#pragma unroll
        for (int h = 0; h < kPartsUnroll; ++h)
          if (h < n_parts) v += x[u][h];
        dev_out[q.dev_offset + i] = v;
        if (in_smem) s_d[i] = v;
      }
    }
  } else {
    for (int i = threadIdx.x; i < n; i += kSelThreads) {
      const float *src = parts + q.dev_offset + i;
      float v = 0.f;
      for (int h = 0; h < n_parts; ++h) v += __ldg(src + h * part_stride);
      dev_out[q.dev_offset + i] = v;
      if (in_smem) s_d[i] = v;
    }
  }
  if (!RANK || q.k <= 0) return;
  __syncthreads();
  topk_block(in_smem ? s_d : dev_out + q.dev_offset, n, q.k, idx_out + q.idx_offset);
}

cudaError_t launch_reduce_parts(const float *parts, int n_parts, int64_t part_stride,
                                const SelReq *reqs, int n_req, float *dev_out, cudaStream_t s) {
  if (n_req == 0) return cudaSuccess;
  SelParams p;
  fill_params(p, reqs, n_req);
  cudaError_t e = launch_pdl(parts_kernel<false>, dim3(n_req), dim3(kSelThreads), 0, s, p, parts,
                             n_parts, part_stride, dev_out, (int32_t *)nullptr);
  return e != cudaSuccess ? e : launched(1);
}

cudaError_t launch_topk_parts(const float *parts, int n_parts, int64_t part_stride,
                              const SelReq *reqs, int n_req, float *dev_out, int32_t *idx_out,
                              cudaStream_t s) {
  if (n_req == 0) return cudaSuccess;
  SelParams p;
  fill_params(p, reqs, n_req);
  int n_max = 0;
  for (int i = 0; i < n_req; ++i) n_max = reqs[i].n_ctx > n_max ? reqs[i].n_ctx : n_max;
  const size_t smem = (size_t)(n_max < kSmemCtx ? n_max : kSmemCtx) * sizeof(float);
  static PerDeviceOnce attr;
  cudaError_t e = attr.run([](int) {
    return cudaFuncSetAttribute(parts_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemCtx * (int)sizeof(float));
  });
  if (e != cudaSuccess) return e;
  e = launch_pdl(parts_kernel<true>, dim3(n_req), dim3(kSelThreads), smem, s, p, parts, n_parts,
                 part_stride, dev_out, idx_out);
  return e != cudaSuccess ? e : launched(1);
}

cudaError_t launch_topk(const float *dev, const SelReq *reqs, int n_req,
                        int32_t *idx_out, cudaStream_t s) {
  if (n_req == 0) return cudaSuccess;
  SelParams p;
  fill_params(p, reqs, n_req);
  topk_kernel<<<n_req, kSelThreads, 0, s>>>(p, dev, idx_out);
  return launched(1);
}

// ----------------------------------------------------------- span policies --
// One CTA per request.  Spans: offsets spans[span_begin .. +n_spans] (local
// context positions).  Modes:
//   kSpanMean  -- rank spans by mean deviation (ties: lower span), take whole
//                 spans while they fit, then the max-total window (ties:
//                 leftmost) of the remainder inside the first span that does
//                 not fit (document-aligned, fixed-chunk and single-window,
//                 "Request Order Matters" §2.3 Eq. 3);
//   kSpanOrder -- the same fill with the visiting order given in aux (the
//                 random-document control of §2.3);
//   kSpanFirst -- the first aux[j] tokens of every span j (EPIC's
//                 chunk-boundary rule).
// Span sums are accumulated in double in a fixed order; the chosen positions
// are written ascending by a block-wide ordered compaction.
enum { kSpanMean = 0, kSpanOrder = 1, kSpanFirst = 2 };

struct DocParams {
  SelParams sel;
  int n_spans_total, mode;
  int32_t spans[CB_MAX_SPANS + CB_MAX_BATCH];
  int32_t aux[CB_MAX_SPANS + CB_MAX_BATCH];    // order or counts, per span
};

__global__ void __launch_bounds__(kSelThreads)
doc_aligned_kernel(const __grid_constant__ DocParams P,
                   const float *__restrict__ dev, int32_t *__restrict__ idx_out,
                   int *status) {
  __shared__ double s_sum[CB_MAX_SPANS];
  __shared__ int s_rank_of[CB_MAX_SPANS];    // span id at rank r
  __shared__ unsigned char s_take[CB_MAX_SPANS];
  __shared__ int warp_buf[32];
  __shared__ double s_best[32];
  __shared__ int s_best_i[32];
  __shared__ int s_part_span, s_rem;
  const SelReq &q = P.sel.r[blockIdx.x];
  const int k = q.k;
  if (k <= 0) return;
  const int m = q.n_spans;
  const int32_t *off = P.spans + q.span_begin;
  const int32_t *aux = P.aux + q.span_begin;
  const float *d = dev + q.dev_offset;
  int32_t *out = idx_out + q.idx_offset;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int mode = P.mode;

  int rem = 0, win_start = -1;
  if (mode != kSpanFirst) {
    for (int j = w; j < m; j += kSelThreads / 32) {
      double acc = 0.0;
      for (int i = off[j] + lane; i < off[j + 1]; i += 32) acc += (double)__ldg(d + i);
      acc = warp_sum_d(acc);
      if (lane == 0) s_sum[j] = acc;
    }
    for (int j = tid; j < m; j += kSelThreads) s_take[j] = 0;
    __syncthreads();
    if (mode == kSpanOrder) {
      for (int r = tid; r < m; r += kSelThreads) s_rank_of[r] = aux[r];
    } else {
      // rank of span j by (mean desc, index asc); empty spans after all
      // non-empty ones, by index
      for (int j = tid; j < m; j += kSelThreads) {
        const int lj = off[j + 1] - off[j];
        int rank = 0;
        if (lj > 0) {
          const double rj = s_sum[j] / lj;
          for (int i = 0; i < m; ++i) {
            const int li = off[i + 1] - off[i];
            if (li <= 0 || i == j) continue;
            const double ri = s_sum[i] / li;
            if (ri > rj || (ri == rj && i < j)) ++rank;
          }
        } else {
          for (int i = 0; i < m; ++i) rank += (off[i + 1] > off[i]) || (i < j);
        }
        s_rank_of[rank] = j;
      }
    }
    __syncthreads();
    if (tid == 0) {
      int left = k, part = -1;
      for (int r = 0; r < m && left > 0; ++r) {
        const int j = s_rank_of[r];
        const int lj = off[j + 1] - off[j];
        if (lj <= 0) continue;
        if (lj <= left) { s_take[j] = 1; left -= lj; }
        else { part = j; break; }
      }
      s_part_span = part;
      s_rem = part >= 0 ? left : 0;
      if (left > 0 && part < 0) report(status, CB_ERR_INVALID_ARG);  // k > N
    }
    __syncthreads();
    rem = s_rem;
    if (rem > 0) {
      const int a = off[s_part_span], b = off[s_part_span + 1];
      const int n_win = b - a - rem + 1;
      double best = -1.0;
      int best_i = 0x7fffffff;
      for (int t = tid; t < n_win; t += kSelThreads) {
        double acc = 0.0;
        for (int i = a + t; i < a + t + rem; ++i) acc += (double)__ldg(d + i);
        if (acc > best || (acc == best && a + t < best_i)) { best = acc; best_i = a + t; }
      }
      // block arg-max, ties to the lower start
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const double ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
        if (ob > best || (ob == best && oi < best_i)) { best = ob; best_i = oi; }
      }
      if (lane == 0) { s_best[w] = best; s_best_i[w] = best_i; }
      __syncthreads();
      if (tid == 0) {
        double bb = s_best[0];
        int bi = s_best_i[0];
        for (int j = 1; j < kSelThreads / 32; ++j)
          if (s_best[j] > bb || (s_best[j] == bb && s_best_i[j] < bi)) { bb = s_best[j]; bi = s_best_i[j]; }
        s_best_i[0] = bi;
      }
      __syncthreads();
      win_start = s_best_i[0];
    }
  }
  // ordered compaction over the context positions
  const int n = q.n_ctx;
  int written = 0;
  for (int base = 0; base < n; base += kSelThreads) {
    const int i = base + tid;
    int sel = 0;
    if (i < n) {
      // span of position i (binary search, spans cover [0, n))
      int lo = 0, hi = m - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= i) lo = mid; else hi = mid - 1;
      }
      if (mode == kSpanFirst)
        sel = i - off[lo] < aux[lo];
      else
        sel = s_take[lo] || (rem > 0 && i >= win_start && i < win_start + rem);
    }
    int total;
    const int pos = block_exclusive_scan(sel, warp_buf, &total);
    if (sel) out[written + pos] = i;
    written += total;
  }
}

cudaError_t launch_selection(const float *dev, const SelPlan &plan, int32_t *idx_out,
                             int *status, cudaStream_t s) {
  const int n_req = (int)plan.reqs.size();
  if (n_req == 0) return cudaSuccess;
  if (plan.policy == CB_POLICY_TOKEN_TOPK) return launch_topk(dev, plan.reqs.data(), n_req, idx_out, s);
  DocParams *P = new DocParams;
  fill_params(P->sel, plan.reqs.data(), n_req);
  P->n_spans_total = (int)plan.spans.size();
  P->mode = plan.policy == CB_POLICY_RANDOM_DOC    ? kSpanOrder
            : plan.policy == CB_POLICY_FIRST_TOKENS ? kSpanFirst
                                                    : kSpanMean;
  for (size_t i = 0; i < plan.spans.size(); ++i) P->spans[i] = plan.spans[i];
  for (size_t i = 0; i < plan.aux.size(); ++i) P->aux[i] = plan.aux[i];
  doc_aligned_kernel<<<n_req, kSelThreads, 0, s>>>(*P, dev, idx_out, status);
  delete P;
  return launched(1);
}

// Tokens each span contributes under the chunk-boundary rule: k shared out
// evenly over the non-empty spans (the first k mod m one more), a short span
// passing what it cannot hold to the following spans in order.
static void first_token_counts(const int32_t *off, int n_spans, int k, int32_t *cnt) {
  int m = 0;
  for (int j = 0; j < n_spans; ++j) m += off[j + 1] > off[j];
  int left = k, r = 0;
  for (int j = 0; j < n_spans; ++j) {
    cnt[j] = 0;
    const int lj = off[j + 1] - off[j];
    if (lj <= 0) continue;
    const int quota = k / m + (r < k % m ? 1 : 0);
    ++r;
    cnt[j] = quota < lj ? quota : lj;
    left -= cnt[j];
  }
  for (int j = 0; j < n_spans && left > 0; ++j) {
    const int room = (off[j + 1] - off[j]) - cnt[j];
    const int e = room < left ? room : left;
    cnt[j] += e;
    left -= e;
  }
}

cb_status make_sel_plan(const cb_select_req *reqs, int n_req, cb_policy policy, SelPlan &out,
                        const char **err) {
  auto bad = [&](const char *msg) { *err = msg; return CB_ERR_INVALID_ARG; };
  if (n_req < 0 || n_req > CB_MAX_BATCH) return bad("n_req must be in [0, CB_MAX_BATCH]");
  if (n_req > 0 && !reqs) return bad("reqs is NULL");
  if (policy < CB_POLICY_TOKEN_TOPK || policy > CB_POLICY_FIRST_TOKENS) return bad("unknown policy");
  out.policy = policy;
  out.reqs.assign(n_req, SelReq{});
  out.spans.clear();
  out.aux.clear();
  std::vector<int32_t> offs;
  for (int i = 0; i < n_req; ++i) {
    const cb_select_req &r = reqs[i];
    if (r.n_ctx < 0 || r.k < 0 || r.k > r.n_ctx) return bad("need 0 <= k <= n_ctx");
    if (r.fresh_row0 < 0 || r.reused_row0 < 0 || r.dev_offset < 0 || r.idx_offset < 0)
      return bad("negative offset");
    SelReq s{r.n_ctx, r.k, r.fresh_row0, r.reused_row0, r.dev_offset, r.idx_offset, 0, 0};
    if (policy != CB_POLICY_TOKEN_TOPK && r.k > 0) {
      offs.clear();
      if (policy == CB_POLICY_SINGLE_WINDOW) {
        offs = {0, r.n_ctx};
      } else if (policy == CB_POLICY_FIXED_CHUNK) {
        if (r.span_len <= 0 || r.span_offset < 0 || r.span_offset > r.span_len)
          return bad("fixed-chunk needs span_len > 0 and 0 <= span_offset <= span_len");
        offs.push_back(0);
        if (r.span_offset > 0 && r.span_offset < r.n_ctx) offs.push_back(r.span_offset);
        while (offs.back() < r.n_ctx) {
          const int64_t nx = (int64_t)offs.back() + r.span_len;
          offs.push_back((int32_t)(nx < r.n_ctx ? nx : r.n_ctx));
          if ((int)offs.size() > CB_MAX_SPANS + 1) return bad("too many fixed-chunk spans");
        }
      } else {
        if (r.n_spans < 1 || !r.span_offsets) return bad("this policy needs spans");
        if (r.n_spans > CB_MAX_SPANS) return bad("too many spans");
        if (r.span_offsets[0] != 0 || r.span_offsets[r.n_spans] != r.n_ctx)
          return bad("spans must cover [0, n_ctx]");
        for (int j = 0; j < r.n_spans; ++j)
          if (r.span_offsets[j + 1] < r.span_offsets[j]) return bad("spans not ascending");
        offs.assign(r.span_offsets, r.span_offsets + r.n_spans + 1);
      }
      const int ns = (int)offs.size() - 1;
      if (ns > CB_MAX_SPANS || (int)out.spans.size() + ns + 1 > CB_MAX_SPANS + CB_MAX_BATCH)
        return bad("too many spans in one call");
      s.span_begin = (int)out.spans.size();
      s.n_spans = ns;
      out.spans.insert(out.spans.end(), offs.begin(), offs.end());
      // aux shares the span indexing (one entry per offset; the last unused)
      std::vector<int32_t> a(ns + 1, 0);
      if (policy == CB_POLICY_RANDOM_DOC) {
        if (!r.span_order) return bad("random-document needs span_order");
        std::vector<unsigned char> seen(ns, 0);
        for (int j = 0; j < ns; ++j) {
          const int o = r.span_order[j];
          if (o < 0 || o >= ns || seen[o]) return bad("span_order must be a permutation of the spans");
          seen[o] = 1;
          a[j] = o;
        }
      } else if (policy == CB_POLICY_FIRST_TOKENS) {
        first_token_counts(offs.data(), ns, r.k, a.data());
      }
      out.aux.insert(out.aux.end(), a.begin(), a.end());
    }
    out.reqs[i] = s;
  }
  return CB_OK;
}

// ------------------------------------------------------------- row maps --
// Computed row r of request b: the first k_b rows are the selected context
// positions, the remaining ones the uncached positions N_b .. T_b-1; both
// parts are ascending, so the rows are ascending by position.
__global__ void build_rows_kernel(const __grid_constant__ BatchMeta bm,
                                  const int32_t *__restrict__ sel,
                                  int32_t *__restrict__ pos,
                                  int32_t *__restrict__ glob, int n_rows,
                                  int *status) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows) return;
  int b = 0;
  while (bm.r_off[b + 1] <= r) ++b;
  const int j = r - bm.r_off[b];
  const int kb = bm.k_off[b + 1] - bm.k_off[b];
  int p = j < kb ? sel[bm.k_off[b] + j] : bm.n_ctx[b] + (j - kb);
  if (p < 0 || p >= (j < kb ? bm.n_ctx[b] : bm.t_off[b + 1] - bm.t_off[b])) {
    report(status, CB_ERR_DEVICE_INDEX);
    p = 0;
  }
  pos[r] = p;
  glob[r] = bm.t_off[b] + p;
}

// build_rows_kernel and the gather of the rows' hidden states in one
// launch: block r computes row r's position and cache row, then copies its
// d floats of h (16-byte vectors).
__global__ void __launch_bounds__(256)
rows_gather_kernel(const __grid_constant__ BatchMeta bm, const int32_t *__restrict__ sel,
                   int32_t *__restrict__ pos, int32_t *__restrict__ glob,
                   const float *__restrict__ h_src, int d, float *__restrict__ h_dst,
                   int *status) {
  grid_dep_wait();      // the selection comes from the previous kernel
  grid_dep_launch();
  __shared__ int64_t s_src;
  const int r = blockIdx.x;
  if (threadIdx.x == 0) {
    int b = 0;
    while (bm.r_off[b + 1] <= r) ++b;
    const int j = r - bm.r_off[b];
    const int kb = bm.k_off[b + 1] - bm.k_off[b];
    int p = j < kb ? sel[bm.k_off[b] + j] : bm.n_ctx[b] + (j - kb);
    if (p < 0 || p >= (j < kb ? bm.n_ctx[b] : bm.t_off[b + 1] - bm.t_off[b])) {
      report(status, CB_ERR_DEVICE_INDEX);
      p = 0;
    }
    pos[r] = p;
    glob[r] = bm.t_off[b] + p;
    s_src = (int64_t)(bm.t_off[b] + p) * d;
  }
  __syncthreads();
  const float4 *src = reinterpret_cast<const float4 *>(h_src + s_src);
  float4 *dst = reinterpret_cast<float4 *>(h_dst + (int64_t)r * d);
  for (int i = threadIdx.x; i < d / 4; i += 256) dst[i] = __ldg(src + i);
}

cudaError_t launch_rows_gather(const BatchMeta &bm, const int32_t *sel, int32_t *pos,
                               int32_t *glob, int n_rows, const float *h_src, int d,
                               float *h_dst, int *status, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(rows_gather_kernel, dim3(n_rows), dim3(256), 0, s, bm, sel, pos, glob,
                             h_src, d, h_dst, status);
  return e != cudaSuccess ? e : launched(1);
}

cudaError_t launch_build_rows(const BatchMeta &bm, const int32_t *sel,
                              int32_t *pos, int32_t *glob, int n_rows,
                              int *status, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  build_rows_kernel<<<(n_rows + 255) / 256, 256, 0, s>>>(bm, sel, pos, glob, n_rows,
                                                         status);
  return launched(1);
}

// Rows of the next layer after a gradual-filtering step (CacheBlend blog,
// select_hkvd): request b keeps keep[j], j < k'_b (ascending local indices
// into its current selection) and all its uncached rows.  Writes the new
// selection, the rows' positions and fused-cache rows, and the current row
// each new row comes from (src) for the hidden-state gather.
__global__ void filter_rows_kernel(const __grid_constant__ BatchMeta cur,
                                   const __grid_constant__ BatchMeta nxt,
                                   const int32_t *__restrict__ keep,
                                   const int32_t *__restrict__ sel_cur,
                                   int32_t *__restrict__ sel_nxt,
                                   int32_t *__restrict__ pos, int32_t *__restrict__ glob,
                                   int32_t *__restrict__ src, int n_rows, int *status) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows) return;
  int b = 0;
  while (nxt.r_off[b + 1] <= r) ++b;
  const int j = r - nxt.r_off[b];
  const int kn = nxt.k_off[b + 1] - nxt.k_off[b];
  const int kc = cur.k_off[b + 1] - cur.k_off[b];
  int p, from;
  if (j < kn) {
    int kk = keep[nxt.k_off[b] + j];
    if (kk < 0 || kk >= kc) {
      report(status, CB_ERR_DEVICE_INDEX);
      kk = 0;
    }
    p = sel_cur[cur.k_off[b] + kk];
    sel_nxt[nxt.k_off[b] + j] = p;
    from = cur.r_off[b] + kk;
  } else {
    p = nxt.n_ctx[b] + (j - kn);
    from = cur.r_off[b] + kc + (j - kn);
  }
  pos[r] = p;
  glob[r] = nxt.t_off[b] + p;
  src[r] = from;
}

cudaError_t launch_filter_rows(const BatchMeta &cur, const BatchMeta &nxt,
                               const int32_t *keep, const int32_t *sel_cur,
                               int32_t *sel_nxt, int32_t *pos, int32_t *glob,
                               int32_t *src, int n_rows, int *status, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  filter_rows_kernel<<<(n_rows + 255) / 256, 256, 0, s>>>(cur, nxt, keep, sel_cur, sel_nxt, pos,
                                                          glob, src, n_rows, status);
  return launched(1);
}

// A gradual step whose kept rows are given (cb_blend_params.forced_kept):
// request b's k'_b positions forced[nxt.k_off[b] ..] become indices into its
// current selection sel_cur (ascending, so a binary search finds them),
// which is the form filter_rows_kernel takes.  A position that is not
// selected, or not above the previous one, records CB_ERR_DEVICE_INDEX.
__global__ void keep_from_positions_kernel(const __grid_constant__ BatchMeta cur,
                                           const __grid_constant__ BatchMeta nxt,
                                           const int32_t *__restrict__ forced,
                                           const int32_t *__restrict__ sel_cur,
                                           int32_t *__restrict__ keep, int n_keep,
                                           int *status) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_keep) return;
  int b = 0;
  while (nxt.k_off[b + 1] <= r) ++b;
  const int p = forced[r];
  const int32_t *sel = sel_cur + cur.k_off[b];
  int lo = 0, hi = cur.k_off[b + 1] - cur.k_off[b];
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sel[mid] < p) lo = mid + 1; else hi = mid;
  }
  const bool found = lo < cur.k_off[b + 1] - cur.k_off[b] && sel[lo] == p;
  const bool ordered = r == nxt.k_off[b] || forced[r - 1] < p;
  if (!found || !ordered) {
    report(status, CB_ERR_DEVICE_INDEX);
    lo = 0;
  }
  keep[r] = lo;
}

cudaError_t launch_keep_from_positions(const BatchMeta &cur, const BatchMeta &nxt,
                                       const int32_t *forced, const int32_t *sel_cur,
                                       int32_t *keep, int n_keep, int *status, cudaStream_t s) {
  if (n_keep == 0) return cudaSuccess;
  keep_from_positions_kernel<<<(n_keep + 255) / 256, 256, 0, s>>>(cur, nxt, forced, sel_cur, keep,
                                                                  n_keep, status);
  return launched(1);
}

// Table 2 diagnostics of "Request Order Matters" §4.4, one CTA per request:
// segments = maximal runs of consecutive selected positions (the number of
// j with j == 0 or idx[j] != idx[j-1] + 1), captured = sum of d over the
// selection / sum of d over the request, both sums in double in a fixed
// order (per-thread strides, then a fixed tree), so results are
// deterministic.
__global__ void __launch_bounds__(256)
selection_stats_kernel(const __grid_constant__ SelParams p, const float *__restrict__ dev,
                       const int32_t *__restrict__ idx, int32_t *__restrict__ segments,
                       double *__restrict__ captured, int *status) {
  __shared__ double s_tot[8], s_sel[8];
  __shared__ int s_seg[8];
  const SelReq &q = p.r[blockIdx.x];
  const float *d = dev + q.dev_offset;
  const int32_t *sel = idx + q.idx_offset;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  double tot = 0.0, got = 0.0;
  int seg = 0;
  for (int i = tid; i < q.n_ctx; i += blockDim.x) tot += (double)__ldg(d + i);
  for (int j = tid; j < q.k; j += blockDim.x) {
    const int t = sel[j];
    if (t < 0 || t >= q.n_ctx) {
      report(status, CB_ERR_DEVICE_INDEX);
      continue;
    }
    got += (double)__ldg(d + t);
    seg += (j == 0 || sel[j - 1] + 1 != t) ? 1 : 0;
  }
  tot = warp_sum_d(tot);
  got = warp_sum_d(got);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) seg += __shfl_xor_sync(0xffffffffu, seg, o);
  if (lane == 0) { s_tot[w] = tot; s_sel[w] = got; s_seg[w] = seg; }
  __syncthreads();
  if (tid == 0) {
    double a = 0.0, b = 0.0;
    int c = 0;
    for (int i = 0; i < 8; ++i) { a += s_tot[i]; b += s_sel[i]; c += s_seg[i]; }
    segments[blockIdx.x] = c;
    captured[blockIdx.x] = a > 0.0 ? b / a : 0.0;
  }
}

cudaError_t launch_selection_stats(const float *dev, const int32_t *idx, const SelReq *reqs,
                                   int n_req, int32_t *segments, double *captured, int *status,
                                   cudaStream_t s) {
  if (n_req == 0) return cudaSuccess;
  SelParams p;
  fill_params(p, reqs, n_req);
  selection_stats_kernel<<<n_req, 256, 0, s>>>(p, dev, idx, segments, captured, status);
  return launched(1);
}

__global__ void index_check_kernel(const int32_t *__restrict__ idx,
                                   const __grid_constant__ IndexCheck c, int *status) {
  const int total = c.off[c.n_seg];
  for (int i = c.off[0] + blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += gridDim.x * blockDim.x) {
    int sg = 0;
    while (c.off[sg + 1] <= i) ++sg;
    const int v = idx[i];
    bool bad = v < 0 || v >= c.hi[sg];
    if (i > c.off[sg]) {
      const int prev = idx[i - 1];
      bad |= c.strict ? !(prev < v) : !(prev <= v);
    }
    if (bad) report(status, CB_ERR_DEVICE_INDEX);
  }
}

cudaError_t launch_index_check(const int32_t *idx, const IndexCheck &c, int *status,
                               cudaStream_t s) {
  const int total = c.off[c.n_seg] - c.off[0];
  if (total <= 0) return cudaSuccess;
  const int blocks = (total + 255) / 256 < 1024 ? (total + 255) / 256 : 1024;
  index_check_kernel<<<blocks, 256, 0, s>>>(idx, c, status);
  return launched(1);
}

__global__ void iota_rows_kernel(const __grid_constant__ BatchMeta bm,
                                 int32_t *__restrict__ pos,
                                 int32_t *__restrict__ glob, int n_rows,
                                 int32_t *__restrict__ dev_idx) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows) return;
  int b = 0, n_off = 0;
  while (bm.t_off[b + 1] <= r) n_off += bm.n_ctx[b++];
  const int p = r - bm.t_off[b];
  pos[r] = p;
  glob[r] = r;
  if (dev_idx) dev_idx[r] = p < bm.n_ctx[b] ? n_off + p : -1;
}

cudaError_t launch_iota_rows(const BatchMeta &bm, int32_t *pos, int32_t *glob,
                             int n_rows, cudaStream_t s, int32_t *dev_idx) {
  if (n_rows == 0) return cudaSuccess;
  iota_rows_kernel<<<(n_rows + 255) / 256, 256, 0, s>>>(bm, pos, glob, n_rows, dev_idx);
  return launched(1);
}

}  // namespace cb
