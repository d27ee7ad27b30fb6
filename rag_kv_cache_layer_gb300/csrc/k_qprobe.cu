// Query-aware selection of QCFuse on the device (§3.3-3.4):
//   * per-chunk anchor scores G_i(r) for Eq. 14 (Sink: -r; Knorm: minus the
//     squared L2 norm of the position's PIC keys over all layers and kv
//     heads);
//   * the rows of the anchor-conditioned query probe (Eqs. 15-17): each
//     request's probe cache is [its anchors in order; its query rows], the
//     anchors keeping their request positions;
//   * the user-query-to-context attention mass of one layer (the summand of
//     Eq. 20): for every query row u and q head h, the softmax of q.k/sqrt(hd)
//     over the request's N context keys, summed over u and h for each key.
// All sums run in a fixed order, so a call's results do not depend on
// scheduling.
#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {
namespace qp {

// ------------------------------------------------------------ anchor scores
constexpr int kMaxSeg = 128;            // chunks per launch (metadata in the parameters)
struct AnchorParams {
  int n, rule, n_layers, kvw;
  int row_prefix[kMaxSeg + 1];          // positions before chunk i
  const void *k[kMaxSeg];               // chunk i's PIC keys, layer l at + l * stride
  int64_t stride[kMaxSeg];
  int out_off[kMaxSeg];                 // chunk i's first score
};

// One warp per chunk position.
template <typename T>
__global__ void anchor_score_kernel(const __grid_constant__ AnchorParams p,
                                    float *__restrict__ scores) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int VEC = 16 / sizeof(T);
  const int lane = threadIdx.x & 31;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (w >= p.row_prefix[p.n]) return;
  int i = 0;
  while (p.row_prefix[i + 1] <= w) ++i;
  const int r = (int)(w - p.row_prefix[i]);
  float score;
  if (p.rule == CB_ANCHOR_KNORM) {
    const T *k = reinterpret_cast<const T *>(p.k[i]);
    float acc = 0.f;
    for (int l = 0; l < p.n_layers; ++l) {
      const T *row = k + (int64_t)l * p.stride[i] + (int64_t)r * p.kvw;
      for (int e = lane * VEC; e < p.kvw; e += 32 * VEC) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(row + e);
        const T *v = reinterpret_cast<const T *>(&raw);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          const float x = to_f(v[j]);
          acc = fmaf(x, x, acc);
        }
      }
    }
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    score = -acc;
  } else {
    score = -(float)r;
  }
  if (lane == 0) scores[p.out_off[i] + r] = score;
}

// --------------------------------------------------------------- probe rows
struct ProbeReq {
  int t_off;       // first fused-cache row of the request
  int n_ctx;       // N: context positions
  int n_u;         // query rows (every uncached row, after the context)
  int seg_begin, seg_end;
  int probe_off;   // first probe-cache row of the request
  int n_anchor;    // anchors of the request
  int u_off;       // first query row in the packed query arrays
};
struct ProbeSeg {
  int anchor_off;  // first anchor (chunk-local position) of the chunk
  int count;       // anchors of the chunk
  int ctx_off;     // the chunk's first context position in its request
  int len;
};
struct ProbeParams {
  int B, n_probe, all;                  // all: every context position is an anchor
  int probe_prefix[CB_MAX_BATCH + 1];
  ProbeReq r[CB_MAX_BATCH];
  ProbeSeg s[CB_MAX_SPANS];
};

// One thread per probe-cache row: the fused-cache row it reads, and for the
// query rows their request position (RoPE), source row (embedding), probe
// cache row (K/V write) and position within the request's probe cache
// (causal mask).
__global__ void probe_rows_kernel(const __grid_constant__ ProbeParams p,
                                  const int32_t *__restrict__ anchors,
                                  int32_t *__restrict__ probe_rows, int32_t *__restrict__ u_pos,
                                  int32_t *__restrict__ u_src, int32_t *__restrict__ u_cache,
                                  int32_t *__restrict__ u_mask, int *status) {
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= p.n_probe) return;
  int b = 0;
  while (p.probe_prefix[b + 1] <= i) ++b;
  const ProbeReq &R = p.r[b];
  const int j = i - R.probe_off;
  if (j < R.n_anchor) {
    int ctx;
    if (p.all) {
      ctx = j;
    } else {
      int k = R.seg_begin, cum = 0;
      while (k + 1 < R.seg_end && cum + p.s[k].count <= j) cum += p.s[k++].count;
      const ProbeSeg &S = p.s[k];
      int local = anchors[S.anchor_off + (j - cum)];
      if (local < 0 || local >= S.len) {
        report(status, CB_ERR_DEVICE_INDEX);
        local = 0;
      }
      ctx = S.ctx_off + local;
    }
    probe_rows[i] = R.t_off + ctx;
  } else {
    const int u = j - R.n_anchor;
    const int ui = R.u_off + u;
    probe_rows[i] = R.t_off + R.n_ctx + u;
    u_pos[ui] = R.n_ctx + u;
    u_src[ui] = R.t_off + R.n_ctx + u;
    u_cache[ui] = i;
    u_mask[ui] = j;
  }
}

// ---------------------------------------------------------- attention mass
// One request: query rows q[u_off + u] (n_u of them, q head h at column
// h * 128), context keys in the fused cache rows t_off + t, t < N.  Score
// rows are ordered r = h * n_u + u, so a kv head's rows are contiguous.
constexpr int HD = 128;
constexpr int KC = 32;                  // keys per CTA of the score pass
constexpr int kRowThreads = 256;

// Scores s[t][r] = log2(e) q_r.k_t / sqrt(hd) of the chunk's keys for the
// rows of kv head g, and each row's (max, sum of 2^(s - max)) over the chunk.
__global__ void __launch_bounds__(kRowThreads)
mass_score_kernel(const bf16 *__restrict__ q, int64_t ld_q, int u_off, int n_u,
                  const bf16 *__restrict__ kc, int64_t ld_k, int t_off, int n_ctx, int Hq,
                  int Hkv, float scale_log2, float *__restrict__ s,
                  float2 *__restrict__ part) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float ks[KC][HD + 4];
  const int chunk = blockIdx.x, g = blockIdx.y;
  const int G = Hq / Hkv;
  const int t0 = chunk * KC;
  const int nk = min(KC, n_ctx - t0);
  const int n_rows = Hq * n_u;
  for (int e = threadIdx.x; e < KC * HD; e += kRowThreads) {
    const int t = e / HD, c = e % HD;
    ks[t][c] = t < nk ? __bfloat162float(kc[(int64_t)(t_off + t0 + t) * ld_k + g * HD + c]) : 0.f;
  }
  __syncthreads();
  for (int rr = threadIdx.x; rr < G * n_u; rr += kRowThreads) {
    const int r = g * G * n_u + rr;           // row of q head g*G + rr / n_u
    const int h = r / n_u, u = r % n_u;
    float qv[HD];
    const bf16 *qr = q + (int64_t)(u_off + u) * ld_q + h * HD;
#pragma unroll
    for (int c = 0; c < HD; c += 8) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(qr + c);
      const bf16 *v = reinterpret_cast<const bf16 *>(&raw);
#pragma unroll
      for (int j = 0; j < 8; ++j) qv[c + j] = __bfloat162float(v[j]) * scale_log2;
    }
    float mx = -INFINITY, sum = 0.f;
    for (int t = 0; t < nk; ++t) {
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int c = 0; c < HD; c += 4) {
        const float4 k4 = *reinterpret_cast<const float4 *>(&ks[t][c]);
        a0 = fmaf(qv[c], k4.x, a0);
        a1 = fmaf(qv[c + 1], k4.y, a1);
        a2 = fmaf(qv[c + 2], k4.z, a2);
        a3 = fmaf(qv[c + 3], k4.w, a3);
      }
      const float sc = (a0 + a1) + (a2 + a3);
      s[(int64_t)(t0 + t) * n_rows + r] = sc;
      if (sc > mx) {
        sum = sum * exp2f(mx - sc) + 1.f;
        mx = sc;
      } else {
        sum += exp2f(sc - mx);
      }
    }
    part[(int64_t)chunk * n_rows + r] = make_float2(mx, sum);
  }
}

// Each row's softmax statistics over all of the request's keys.
__global__ void mass_stats_kernel(const float2 *__restrict__ part, int n_chunks, int n_rows,
                                  float2 *__restrict__ ml) {
  grid_dep_wait();
  grid_dep_launch();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows) return;
  float M = -INFINITY;
  for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, part[(int64_t)c * n_rows + r].x);
  float L = 0.f;
  for (int c = 0; c < n_chunks; ++c) {
    const float2 v = part[(int64_t)c * n_rows + r];
    L += v.y * exp2f(v.x - M);
  }
  ml[r] = make_float2(M, L);
}

// One warp per key: I[t] += sum over every row of 2^(s - m_r) / l_r, lanes
// striding the rows, then a fixed-order butterfly.
__global__ void mass_sum_kernel(const float *__restrict__ s, const float2 *__restrict__ ml,
                                int n_rows, int n_ctx, float *__restrict__ mass) {
  grid_dep_wait();
  grid_dep_launch();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= n_ctx) return;
  const float *row = s + (int64_t)t * n_rows;
  float acc = 0.f;
  for (int r = lane; r < n_rows; r += 32) {
    const float2 v = ml[r];
    acc += exp2f(row[r] - v.x) / v.y;
  }
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) mass[t] += acc;
}

}  // namespace qp

// --------------------------------------------------------------------- host
cudaError_t launch_anchor_scores(const AnchorChunk *chunks, int n, int rule, int n_layers,
                                 int kvw, cb_dtype dt, float *scores, cudaStream_t s) {
  using namespace qp;
  for (int base = 0; base < n; base += kMaxSeg) {
    AnchorParams p{};
    p.n = n - base < kMaxSeg ? n - base : kMaxSeg;
    p.rule = rule;
    p.n_layers = n_layers;
    p.kvw = kvw;
    p.row_prefix[0] = 0;
    for (int i = 0; i < p.n; ++i) {
      const AnchorChunk &c = chunks[base + i];
      p.k[i] = c.k;
      p.stride[i] = c.layer_stride;
      p.out_off[i] = c.score_off;
      p.row_prefix[i + 1] = p.row_prefix[i] + c.len;
    }
    const int64_t warps = p.row_prefix[p.n];
    if (warps == 0) continue;
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    cudaError_t e = dt == CB_BF16
                        ? launch_pdl(anchor_score_kernel<bf16>, dim3(blocks), dim3(256), 0, s, p,
                                     scores)
                        : launch_pdl(anchor_score_kernel<float>, dim3(blocks), dim3(256), 0, s, p,
                                     scores);
    if (e != cudaSuccess) return e;
    e = launched(1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_probe_rows(const ProbeLayout &L, const int32_t *anchors, int32_t *probe_rows,
                              int32_t *u_pos, int32_t *u_src, int32_t *u_cache, int32_t *u_mask,
                              int *status, cudaStream_t s) {
  using namespace qp;
  if (L.B > CB_MAX_BATCH || (int)L.segs.size() > CB_MAX_SPANS) return cudaErrorInvalidValue;
  ProbeParams p{};
  p.B = L.B;
  p.all = L.all;
  p.n_probe = 0;
  for (int b = 0; b < L.B; ++b) {
    const ProbeLayout::Req &q = L.reqs[b];
    p.r[b] = ProbeReq{q.t_off, q.n_ctx, q.n_u, q.seg_begin, q.seg_end, q.probe_off, q.n_anchor,
                      q.u_off};
    p.probe_prefix[b] = q.probe_off;
    p.n_probe = q.probe_off + q.n_anchor + q.n_u;
  }
  p.probe_prefix[L.B] = p.n_probe;
  for (size_t k = 0; k < L.segs.size(); ++k)
    p.s[k] = ProbeSeg{L.segs[k].anchor_off, L.segs[k].count, L.segs[k].ctx_off, L.segs[k].len};
  if (p.n_probe == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(probe_rows_kernel, dim3((p.n_probe + 255) / 256), dim3(256), 0, s, p,
                             anchors, probe_rows, u_pos, u_src, u_cache, u_mask, status);
  if (e != cudaSuccess) return e;
  return launched(1);
}

size_t mass_ws_bytes(int n_u, int Hq, int n_ctx) {
  const int64_t rows = (int64_t)Hq * n_u;
  const int64_t chunks = (n_ctx + qp::KC - 1) / qp::KC;
  return (size_t)(rows * n_ctx * 4 + chunks * rows * 8 + rows * 8) + 3 * 256;
}

cudaError_t launch_attention_mass(const void *q, int64_t ld_q, int u_off, int n_u,
                                  const void *k_cache, int64_t ld_k, int t_off, int n_ctx,
                                  int Hq, int Hkv, int hd, void *ws, size_t ws_bytes,
                                  float *mass, cudaStream_t s) {
  using namespace qp;
  if (n_u <= 0 || n_ctx <= 0) return cudaSuccess;
  if (hd != HD || Hq % Hkv) return cudaErrorInvalidValue;
  if (!ws || ws_bytes < mass_ws_bytes(n_u, Hq, n_ctx)) return cudaErrorInvalidValue;
  const int n_rows = Hq * n_u;
  const int n_chunks = (n_ctx + KC - 1) / KC;
  char *w = reinterpret_cast<char *>(ws);
  float *sc = reinterpret_cast<float *>(w);
  w += ((size_t)n_rows * n_ctx * 4 + 255) / 256 * 256;
  float2 *part = reinterpret_cast<float2 *>(w);
  w += ((size_t)n_chunks * n_rows * 8 + 255) / 256 * 256;
  float2 *ml = reinterpret_cast<float2 *>(w);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  cudaError_t e = launch_pdl(mass_score_kernel, dim3(n_chunks, Hkv), dim3(kRowThreads), 0, s,
                             reinterpret_cast<const bf16 *>(q), ld_q, u_off, n_u,
                             reinterpret_cast<const bf16 *>(k_cache), ld_k, t_off, n_ctx, Hq, Hkv,
                             scale_log2, sc, part);
  if (e != cudaSuccess) return e;
  e = launch_pdl(mass_stats_kernel, dim3((n_rows + 255) / 256), dim3(256), 0, s,
                 (const float2 *)part, n_chunks, n_rows, ml);
  if (e != cudaSuccess) return e;
  e = launch_pdl(mass_sum_kernel, dim3((n_ctx * 32 + 255) / 256), dim3(256), 0, s,
                 (const float *)sc, (const float2 *)ml, n_rows, n_ctx, mass);
  if (e != cudaSuccess) return e;
  return launched(3);
}

}  // namespace cb
