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
#include "cb_tc.cuh"

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
// rows are ordered r = h * n_u + u, so kv head g's rows are the contiguous
// range [g * R_g, (g + 1) * R_g), R_g = G * n_u.
//
// Both contractions run on the tensor cores (tcgen05, fp32 accumulators in
// TMEM), with the scores never stored:
//   1. gather: each group's query rows, contiguous and zero-padded to a
//      multiple of 256 rows (qg[g][i], i = h_local * n_u + u);
//   2. statistics: tiles S = Q_g K^T of 128 rows x 256 keys; epilogue thread
//      i holds row i's 256 scores, so the tile's (max, sum of 2^(s - max))
//      per row needs no exchange;
//   3. combine: every row's max M_r and 1 / L_r over all key tiles;
//   4. mass: the swapped tiles S^T = K Q_g^T of 128 keys x 256 rows; thread
//      t holds key t's 256 scores, so sum_r 2^(s - M_r) / L_r is again a
//      per-thread sum, left per (row tile, key);
//   5. the row tiles' sums are added to I in a fixed order.
// One CTA per tile, four warps: warp 0 issues the copies and the eight
// MMAs (K = 16 each over the head dimension), all four drain TMEM.  Every
// wait is bounded.
constexpr int HD = 128;
constexpr int kMassThreads = 128;
constexpr int kRowsA = 128;                 // MMA M
constexpr int kRowsB = 256;                 // MMA N
constexpr int kAtomA = kRowsA * 128;        // one 64-wide swizzle atom of A (bytes)
constexpr int kAtomB = kRowsB * 128;
constexpr int kMassSmem = 2 * kAtomA + 2 * kAtomB + 1024 + 64;
constexpr int kMassCols = 256;              // TMEM columns: the 128 x 256 accumulator

__host__ __device__ inline int group_pad(int group_rows) { return (group_rows + 255) / 256 * 256; }

// qg[g * pad + i] = q row (u_off + u), columns (g * G + h) * 128 .. + 127,
// for i = h * n_u + u < G * n_u; zero above.  One thread per 16 bytes.
__global__ void mass_gather_kernel(const bf16 *__restrict__ q, int64_t ld_q, int u_off, int n_u,
                                   int G, int Hkv, bf16 *__restrict__ qg) {
  grid_dep_wait();
  grid_dep_launch();
  const int rows = G * n_u, pad = group_pad(rows);
  const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // 16-byte unit
  if (v >= (int64_t)Hkv * pad * 16) return;
  const int e = (int)(v % 16) * 8;
  const int64_t gi = v / 16;
  const int g = (int)(gi / pad), i = (int)(gi % pad);
  uint4 val = make_uint4(0u, 0u, 0u, 0u);
  if (i < rows) {
    const int h = g * G + i / n_u, u = i % n_u;
    val = *reinterpret_cast<const uint4 *>(q + (int64_t)(u_off + u) * ld_q + h * HD + e);
  }
  *reinterpret_cast<uint4 *>(qg + gi * HD + e) = val;
}

struct MassParams {
  int n_ctx, n_u, G, Hkv, pad;
  int rt_per_g;          // row tiles per group (128 rows in STATS, 256 in MASS)
  int n_kt;              // key tiles (256 keys in STATS, 128 in MASS)
  float scale_log2;      // log2(e) / sqrt(hd)
  int key_row0;          // fused-cache row of context key 0
};

// MASS == false: statistics tiles (A = 128 query rows, B = 256 keys); part0
// gets (max, sum) per (key tile, row).  MASS == true: mass tiles (A = 128
// keys, B = 256 query rows); partI gets sum_r 2^(s - M_r) / L_r per (row
// tile, key), with ml = (M_r, 1 / L_r).
template <bool MASS>
__global__ void __launch_bounds__(kMassThreads)
mass_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ MassParams p, float2 *__restrict__ part0,
               const float2 *__restrict__ ml, float *__restrict__ partI, int *status) {
  using namespace tcx;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sa = smem, *sb = smem + 2 * kAtomA;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 2 * kAtomA + 2 * kAtomB);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 2);
  __shared__ float2 s_ml[kRowsB];
  __shared__ int s_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // tile: blockIdx.x = key tile, blockIdx.y = g * rt_per_g + row tile
  const int kt = blockIdx.x, g = blockIdx.y / p.rt_per_g, rt = blockIdx.y % p.rt_per_g;
  const int group_rows = p.G * p.n_u;
  const int q_row0 = g * p.pad + rt * (MASS ? kRowsB : kRowsA);   // first qg row of the tile
  const int key0 = kt * (MASS ? kRowsA : kRowsB);                 // first key of the tile
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 1);
    s_ok = 1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kMassCols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();      // q (gathered) and the statistics come from earlier kernels
  grid_dep_launch();
  if (MASS) {
    // the tile's 256 rows: (M_r, 1 / L_r); rows past the group weigh 0
    for (int c = threadIdx.x; c < kRowsB; c += kMassThreads) {
      const int i = rt * kRowsB + c;
      s_ml[c] = i < group_rows ? ml[g * group_rows + i] : make_float2(0.f, 0.f);
    }
  }
  if (warp == 0) {
    if (elect_one()) {
      const uint32_t b = smem_u32(&bar[0]);
      expect_tx(b, 2 * kAtomA + 2 * kAtomB);
      for (int half = 0; half < 2; ++half) {
        // MASS: A = keys, B = query rows; statistics: the other way round
        if (MASS) {
          tma_load_2d(smem_u32(sa + half * kAtomA), &mapK, b, g * HD + half * 64, p.key_row0 + key0);
          tma_load_2d(smem_u32(sb + half * kAtomB), &mapQ, b, half * 64, q_row0);
        } else {
          tma_load_2d(smem_u32(sa + half * kAtomA), &mapQ, b, half * 64, q_row0);
          tma_load_2d(smem_u32(sb + half * kAtomB), &mapK, b, g * HD + half * 64, p.key_row0 + key0);
        }
      }
    }
    __syncwarp();
    const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar[0]), 0, kWaitLimitNs, status));
    if (got) {
      fence_after();
      if (elect_one()) {
        const uint32_t a = smem_u32(sa), bb = smem_u32(sb);
        constexpr uint32_t id = idesc_bf16(kRowsA, kRowsB);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t o = (k & 3) * 32;
          mma(tmem, desc_kmajor(a + (k >> 2) * kAtomA + o), desc_kmajor(bb + (k >> 2) * kAtomB + o),
              id, k > 0);
        }
        commit(smem_u32(&bar[1]));
      }
      __syncwarp();
    } else if (lane == 0) {
      s_ok = 0;
      // let the copies land before this CTA's shared memory goes away
      mbar_wait_bounded(smem_u32(&bar[0]), 0, 10000000ull, nullptr);
    }
  }
  __syncthreads();
  bool ok = s_ok != 0;
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bar[1]), 0, kWaitLimitNs, status));
  if (ok) {
    fence_after();
    const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
    const int me = warp * 32 + lane;               // this thread's A row
    const float sl2 = p.scale_log2;
    if (!MASS) {
      // row me of the tile over its 256 keys: running (max, sum)
      const int i = rt * kRowsA + me;
      float m = -INFINITY, l = 0.f;
#pragma unroll 1
      for (int c = 0; c < kRowsB; c += 32) {
        float x[32];
        tmem_ld32(tbase + c, x);
        const int n_vis = min(32, p.n_ctx - (key0 + c));
        float mc = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) if (j < n_vis) mc = fmaxf(mc, x[j] * sl2);
        if (mc == -INFINITY) continue;
        const float mn = fmaxf(m, mc);
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) if (j < n_vis) sum += exp2f(x[j] * sl2 - mn);
        l = l * exp2f(m - mn) + sum;
        m = mn;
      }
      if (i < group_rows) part0[(int64_t)kt * (p.Hkv * group_rows) + g * group_rows + i] = make_float2(m, l);
    } else {
      // key me of the tile over its 256 query rows
      const int t = key0 + me;
      float acc = 0.f;
#pragma unroll 1
      for (int c = 0; c < kRowsB; c += 32) {
        float x[32];
        tmem_ld32(tbase + c, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 w = s_ml[c + j];
          acc += exp2f(x[j] * sl2 - w.x) * w.y;
        }
      }
      if (t < p.n_ctx) partI[(int64_t)blockIdx.y * p.n_ctx + t] = acc;
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kMassCols);
  }
}

// Each row's softmax statistics over all of the request's keys: the maximum
// and the reciprocal of the sum.
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
    if (v.x != -INFINITY) L += v.y * exp2f(v.x - M);
  }
  ml[r] = make_float2(M, L > 0.f ? 1.f / L : 0.f);
}

// I[t] += the row tiles' sums for key t, in row-tile order.
__global__ void mass_final_kernel(const float *__restrict__ partI, int n_parts, int n_ctx,
                                  float *__restrict__ mass) {
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n_ctx) return;
  float acc = 0.f;
  for (int j = 0; j < n_parts; ++j) acc += partI[(int64_t)j * n_ctx + t];
  mass[t] += acc;
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

// Scratch of one request's mass: the gathered query rows, the statistics
// tiles' (max, sum), the rows' (max, 1 / sum), the mass tiles' key sums.
struct MassLayout {
  size_t qg, part0, ml, partI, total;
  int pad, n_kt0, n_kt1, rt0, rt1;
};
static MassLayout mass_layout(int n_u, int Hq, int Hkv, int n_ctx) {
  MassLayout L;
  const int G = Hq / Hkv, rows = G * n_u;
  L.pad = qp::group_pad(rows);
  L.rt0 = (rows + qp::kRowsA - 1) / qp::kRowsA;
  L.rt1 = L.pad / qp::kRowsB;
  L.n_kt0 = (n_ctx + qp::kRowsB - 1) / qp::kRowsB;
  L.n_kt1 = (n_ctx + qp::kRowsA - 1) / qp::kRowsA;
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  size_t off = 0;
  L.qg = off;
  off += up((size_t)Hkv * L.pad * qp::HD * sizeof(bf16));
  L.part0 = off;
  off += up((size_t)L.n_kt0 * Hq * n_u * sizeof(float2));
  L.ml = off;
  off += up((size_t)Hq * n_u * sizeof(float2));
  L.partI = off;
  off += up((size_t)Hkv * L.rt1 * n_ctx * sizeof(float));
  L.total = off;
  return L;
}

size_t mass_ws_bytes(int n_u, int Hq, int Hkv, int n_ctx) {
  if (n_u <= 0 || n_ctx <= 0 || Hkv <= 0) return 256;
  return mass_layout(n_u, Hq, Hkv, n_ctx).total;
}

cudaError_t launch_attention_mass(const void *q, int64_t ld_q, int u_off, int n_u,
                                  const void *k_cache, int64_t ld_k, int t_off, int n_ctx,
                                  int Hq, int Hkv, int hd, void *ws, size_t ws_bytes,
                                  float *mass, int *status, cudaStream_t s) {
  using namespace qp;
  if (n_u <= 0 || n_ctx <= 0) return cudaSuccess;
  if (hd != HD || Hq % Hkv) return cudaErrorInvalidValue;
  const MassLayout Lo = mass_layout(n_u, Hq, Hkv, n_ctx);
  if (!ws || ws_bytes < Lo.total) return cudaErrorInvalidValue;
  char *w = reinterpret_cast<char *>(ws);
  bf16 *qg = reinterpret_cast<bf16 *>(w + Lo.qg);
  float2 *part0 = reinterpret_cast<float2 *>(w + Lo.part0);
  float2 *ml = reinterpret_cast<float2 *>(w + Lo.ml);
  float *partI = reinterpret_cast<float *>(w + Lo.partI);
  const int G = Hq / Hkv, n_rows = Hq * n_u;
  MassParams p{n_ctx, n_u, G, Hkv, Lo.pad, Lo.rt0, Lo.n_kt0,
               1.4426950408889634f / sqrtf((float)hd), t_off};
  // keys: the context rows only (rows past them read as zeros and are masked)
  CUtensorMap mq0, mq1, mk0, mk1;
  if (!tcx::make_map(&mq0, qg, (int64_t)Hkv * Lo.pad, HD, HD, kRowsA) ||
      !tcx::make_map(&mq1, qg, (int64_t)Hkv * Lo.pad, HD, HD, kRowsB) ||
      !tcx::make_map(&mk0, k_cache, (int64_t)t_off + n_ctx, (int64_t)Hkv * HD, ld_k, kRowsB) ||
      !tcx::make_map(&mk1, k_cache, (int64_t)t_off + n_ctx, (int64_t)Hkv * HD, ld_k, kRowsA))
    return cudaErrorInvalidValue;
  static PerDeviceOnce attr;
  cudaError_t e = attr.run([](int) {
    cudaError_t r = cudaFuncSetAttribute(mass_tc_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMassSmem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(mass_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMassSmem);
    return r;
  });
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)Hkv * Lo.pad * 16;
  e = launch_pdl(mass_gather_kernel, dim3((unsigned)((units + 255) / 256)), dim3(256), 0, s,
                 reinterpret_cast<const bf16 *>(q), ld_q, u_off, n_u, G, Hkv, qg);
  if (e != cudaSuccess) return e;
  e = launch_pdl(mass_tc_kernel<false>, dim3(Lo.n_kt0, Hkv * Lo.rt0), dim3(kMassThreads),
                 kMassSmem, s, mq0, mk0, p, part0, (const float2 *)nullptr, (float *)nullptr,
                 status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(mass_stats_kernel, dim3((n_rows + 255) / 256), dim3(256), 0, s,
                 (const float2 *)part0, Lo.n_kt0, n_rows, ml);
  if (e != cudaSuccess) return e;
  MassParams p1 = p;
  p1.rt_per_g = Lo.rt1;
  p1.n_kt = Lo.n_kt1;
  e = launch_pdl(mass_tc_kernel<true>, dim3(Lo.n_kt1, Hkv * Lo.rt1), dim3(kMassThreads),
                 kMassSmem, s, mq1, mk1, p1, (float2 *)nullptr, (const float2 *)ml, partI,
                 status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(mass_final_kernel, dim3((n_ctx + 255) / 256), dim3(256), 0, s,
                 (const float *)partI, Hkv * Lo.rt1, n_ctx, mass);
  if (e != cudaSuccess) return e;
  return launched(5);
}

}  // namespace cb
