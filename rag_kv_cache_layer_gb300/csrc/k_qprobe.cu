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
constexpr int KC = 64;                  // keys per score tile
constexpr int RC = 128;                 // rows per score tile
constexpr int kTileThreads = 256;       // 16 x 16 threads, 8 rows x 4 keys each
constexpr int kScoreSmem = HD * (RC + KC) * 4;

// Scores s[t][r] = log2(e) q_r.k_t / sqrt(hd) of a 64-row x 64-key tile
// (all rows of one kv head's group), and each row's (max, sum of
// 2^(s - max)) over the tile's keys.  Q and K are staged transposed in shared
// memory ([dim][row], [dim][key]), so each step of the dot products reads
// one float4 of rows and one of keys for 16 FMAs.
__global__ void __launch_bounds__(kTileThreads)
mass_score_kernel(const bf16 *__restrict__ q, int64_t ld_q, int u_off, int n_u,
                  const bf16 *__restrict__ kc, int64_t ld_k, int t_off, int n_ctx, int Hq,
                  int Hkv, float scale_log2, float *__restrict__ s,
                  float2 *__restrict__ part) {
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ __align__(16) float sm[];
  float *qs = sm;                        // [HD][RC]
  float *ks = sm + HD * RC;              // [HD][KC]
  const int G = Hq / Hkv;
  const int group_rows = G * n_u;
  const int tiles_per_group = (group_rows + RC - 1) / RC;
  const int g = blockIdx.y / tiles_per_group;
  const int rt = blockIdx.y % tiles_per_group;
  const int r0 = g * group_rows + rt * RC;           // first row of the tile
  const int nr = min(RC, group_rows - rt * RC);
  const int t0 = blockIdx.x * KC;
  const int nk = min(KC, n_ctx - t0);
  const int n_rows = Hq * n_u;
  // stage: entry i is row i % RC (key i % KC), dims 8 * (i / RC) .. + 7
  for (int i = threadIdx.x; i < RC * (HD / 8); i += kTileThreads) {
    const int row = i % RC, e = 8 * (i / RC);
    float qv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (row < nr) {
      const int r = r0 + row, h = r / n_u, u = r % n_u;
      const uint4 raw =
          *reinterpret_cast<const uint4 *>(q + (int64_t)(u_off + u) * ld_q + h * HD + e);
      const bf16 *v = reinterpret_cast<const bf16 *>(&raw);
#pragma unroll
      for (int j = 0; j < 8; ++j) qv[j] = __bfloat162float(v[j]) * scale_log2;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) qs[(e + j) * RC + row] = qv[j];
  }
  for (int i = threadIdx.x; i < KC * (HD / 8); i += kTileThreads) {
    const int row = i % KC, e = 8 * (i / KC);
    float kv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (row < nk) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(
          kc + (int64_t)(t_off + t0 + row) * ld_k + g * HD + e);
      const bf16 *v = reinterpret_cast<const bf16 *>(&raw);
#pragma unroll
      for (int j = 0; j < 8; ++j) kv[j] = __bfloat162float(v[j]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) ks[(e + j) * KC + row] = kv[j];
  }
  __syncthreads();
  // thread (ty, tx): rows 8 ty .. 8 ty + 7, keys 4 tx .. 4 tx + 3
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
  for (int e = 0; e < HD; ++e) {
    const float4 a0 = *reinterpret_cast<const float4 *>(qs + e * RC + 8 * ty);
    const float4 a1 = *reinterpret_cast<const float4 *>(qs + e * RC + 8 * ty + 4);
    const float4 b = *reinterpret_cast<const float4 *>(ks + e * KC + 4 * tx);
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
  // scores out (8 consecutive rows per key), then each row's statistics over
  // the tile's keys: the 16 threads of a row group are 16 consecutive lanes
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int t = 4 * tx + j;
    if (t < nk && 8 * ty < nr) {
      float *dst = s + (int64_t)(t0 + t) * n_rows + r0 + 8 * ty;
      if (8 * ty + 8 <= nr && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
        reinterpret_cast<float4 *>(dst)[0] = make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
        reinterpret_cast<float4 *>(dst)[1] = make_float4(acc[4][j], acc[5][j], acc[6][j], acc[7][j]);
      } else {
        for (int i = 0; i < 8 && 8 * ty + i < nr; ++i) dst[i] = acc[i][j];
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (4 * tx + j < nk) mx = fmaxf(mx, acc[i][j]);
    for (int o = 8; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (4 * tx + j < nk) sum += exp2f(acc[i][j] - mx);
    for (int o = 8; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (tx == 0 && 8 * ty + i < nr)
      part[(int64_t)blockIdx.x * n_rows + r0 + 8 * ty + i] = make_float2(mx, sum);
  }
}

// Each row's softmax statistics over all of the request's keys: the maximum
// and the reciprocal of the sum (the sum pass multiplies).
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
  ml[r] = make_float2(M, 1.f / L);
}

// One warp per key: I[t] += sum over every row of 2^(s - m_r) / l_r (ml holds
// m_r and 1 / l_r), lanes striding the rows, then a fixed-order butterfly.
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
    acc += exp2f(row[r] - v.x) * v.y;
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
  static PerDeviceOnce attr;
  cudaError_t ea = attr.run([](int) {
    return cudaFuncSetAttribute(mass_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kScoreSmem);
  });
  if (ea != cudaSuccess) return ea;
  const int tiles_per_group = ((Hq / Hkv) * n_u + RC - 1) / RC;
  cudaError_t e = launch_pdl(mass_score_kernel, dim3(n_chunks, Hkv * tiles_per_group),
                             dim3(kTileThreads), kScoreSmem, s,
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
