// CUDA-core selected-query attention (fp32 parity path).
//
// For each computed row r at request position p and q head h (kv head
// g = h / (Hq / Hkv)): out = softmax_{j<=p}(scale q.K_j) V_j over the fused
// cache of the row's request -- n_sel x L work, not L x L (CacheBlend blog,
// blend_layer step 4).  One warp per (row, head): lane j scores key j of a
// 32-key tile, the tile is folded into a running (max, sum, acc) online
// softmax, and each lane accumulates head_dim / 32 output columns.
#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

struct AttnParams {
  int n_req;
  AttnReq r[CB_MAX_BATCH];
};

template <typename T, int HD>
__global__ void __launch_bounds__(128)
attn_simt_kernel(const __grid_constant__ AttnParams P, const T *__restrict__ q,
                 int64_t ld_q, const int32_t *__restrict__ q_pos,
                 const T *__restrict__ kc, const T *__restrict__ vc,
                 int64_t ld_kv, int Hq, int Hkv, float scale, T *__restrict__ out,
                 int64_t ld_out, int n_rows_total, int *status) {
  constexpr int PER = HD / 32;
  __shared__ float qs[4][HD];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int64_t gw = (int64_t)blockIdx.x * 4 + wl;
  if (gw >= (int64_t)n_rows_total * Hq) return;
  const int row_i = (int)(gw / Hq), h = (int)(gw % Hq);
  // request of this row (row_i counts rows over all requests in order)
  int b = 0, acc_rows = 0;
  for (; b < P.n_req; ++b) {
    const int nr = P.r[b].q_end - P.r[b].q_begin;
    if (row_i < acc_rows + nr) break;
    acc_rows += nr;
  }
  const AttnReq &R = P.r[b];
  const int row = R.q_begin + (row_i - acc_rows);
  const int p = q_pos[row];
  if (p < 0 || p >= R.kv_len) {
    if (lane == 0) report(status, CB_ERR_DEVICE_INDEX);
    return;
  }
  const int g = h / (Hq / Hkv);
  for (int c = lane; c < HD; c += 32) qs[wl][c] = to_f(q[(int64_t)row * ld_q + h * HD + c]) * scale;
  __syncwarp();
  const T *kbase = kc + R.kv_row0 * ld_kv + g * HD;
  const T *vbase = vc + R.kv_row0 * ld_kv + g * HD;
  float m = -INFINITY, l = 0.f, acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 <= p; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j <= p) {
      const T *kr = kbase + (int64_t)j * ld_kv;
      float dot = 0.f;
      for (int c = 0; c < HD; ++c) dot = fmaf(qs[wl][c], to_f(kr[c]), dot);
      s = dot;
    }
    const float mt = warp_max(s);
    const float m_new = fmaxf(m, mt);
    const float pj = (j <= p) ? expf(s - m_new) : 0.f;
    const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
    l = l * corr + warp_sum(pj);
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] *= corr;
    const int nk = (p - j0 + 1) < 32 ? (p - j0 + 1) : 32;
    for (int t = 0; t < nk; ++t) {
      const float pt = __shfl_sync(0xffffffffu, pj, t);
      const T *vr = vbase + (int64_t)(j0 + t) * ld_kv;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(pt, to_f(vr[lane + 32 * i]), acc[i]);
    }
    m = m_new;
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    out[(int64_t)row * ld_out + h * HD + lane + 32 * i] = from_f<T>(acc[i] * inv);
}

template <typename T>
static cudaError_t attn_dispatch(const AttnParams &P, const void *q, int64_t ld_q,
                                 const int32_t *q_pos, const void *k,
                                 const void *v, int64_t ld_kv, int Hq, int Hkv,
                                 int hd, float scale, void *out, int64_t ld_out,
                                 int n_rows, int *status, cudaStream_t s) {
  const int64_t warps = (int64_t)n_rows * Hq;
  const int blocks = (int)((warps + 3) / 4);
  if (hd == 64)
    attn_simt_kernel<T, 64><<<blocks, 128, 0, s>>>(P, (const T *)q, ld_q, q_pos, (const T *)k,
                                                   (const T *)v, ld_kv, Hq, Hkv, scale,
                                                   (T *)out, ld_out, n_rows, status);
  else
    attn_simt_kernel<T, 128><<<blocks, 128, 0, s>>>(P, (const T *)q, ld_q, q_pos, (const T *)k,
                                                    (const T *)v, ld_kv, Hq, Hkv, scale,
                                                    (T *)out, ld_out, n_rows, status);
  return launched(1);
}

cudaError_t launch_attention_simt(const void *q, int64_t ld_q,
                                  const int32_t *q_pos, const AttnReq *reqs,
                                  int n_req, const void *k_cache,
                                  const void *v_cache, int64_t ld_kv, int Hq,
                                  int Hkv, int hd, float scale, void *out,
                                  int64_t ld_out, cb_dtype dt, int *status,
                                  cudaStream_t s) {
  AttnParams P;
  P.n_req = n_req;
  int n_rows = 0;
  for (int i = 0; i < n_req; ++i) {
    P.r[i] = reqs[i];
    n_rows += reqs[i].q_end - reqs[i].q_begin;
  }
  if (n_rows == 0) return cudaSuccess;
  if (dt == CB_BF16)
    return attn_dispatch<bf16>(P, q, ld_q, q_pos, k_cache, v_cache, ld_kv, Hq, Hkv, hd,
                               scale, out, ld_out, n_rows, status, s);
  return attn_dispatch<float>(P, q, ld_q, q_pos, k_cache, v_cache, ld_kv, Hq, Hkv, hd,
                              scale, out, ld_out, n_rows, status, s);
}

// ------------------------------------------------------------------ debug --
// A single thread waits on an mbarrier that is never completed; the bounded
// wait expires after limit_us and records CB_ERR_TIMEOUT.
__global__ void expire_wait_kernel(uint64_t limit_ns, int *status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = smem_u32(&bar);
  mbar_init(a, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  (void)mbar_wait_bounded(a, 0, limit_ns, status);
}

cudaError_t launch_expire_wait(int limit_us, int *status, cudaStream_t s) {
  expire_wait_kernel<<<1, 1, 0, s>>>((uint64_t)limit_us * 1000ull, status);
  return launched(1);
}

}  // namespace cb
