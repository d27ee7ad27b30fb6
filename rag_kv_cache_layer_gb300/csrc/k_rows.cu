// Row-wise kernels of the decoder stack: embedding gather, RMSNorm (with an
// optional row gather), generic row gather, K/V scatter into the fused
// cache (QCFuse Eq. 7; CacheBlend blog blend_layer step 3), the RoPE +
// scatter step that follows a Q/K/V projection, and the first-token LM head
// (GEMV over the tied embedding + arg-max).  All are HBM-bound streams with
// 16-byte vector accesses.
#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

// -------------------------------------------------------------- embedding --
struct TokPtrs {
  const int32_t *p[CB_MAX_BATCH];
};

template <typename T>
__global__ void __launch_bounds__(256)
embed_kernel(const __grid_constant__ TokPtrs tp, const __grid_constant__ BatchMeta bm,
             const T *__restrict__ E, int vocab, int d, float *__restrict__ h,
             int *status) {
  constexpr int VEC = 16 / sizeof(T);
  const int row = blockIdx.x;
  int b = 0;
  while (bm.t_off[b + 1] <= row) ++b;
  int tok = tp.p[b][row - bm.t_off[b]];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) report(status, CB_ERR_DEVICE_INDEX);
    tok = 0;
  }
  const T *src = E + (int64_t)tok * d;
  float *dst = h + (int64_t)row * d;
  for (int c = threadIdx.x * VEC; c < d; c += blockDim.x * VEC) {
    float x[VEC];
    load16<T>(src + c, x);
#pragma unroll
    for (int i = 0; i < VEC; i += 4)
      *reinterpret_cast<float4 *>(dst + c + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
  }
}

cudaError_t launch_embed(const int32_t *const *tokens, const BatchMeta &bm,
                         const void *embed, int vocab, int d, cb_dtype dt,
                         float *h, int *status, cudaStream_t s) {
  TokPtrs tp;
  for (int b = 0; b < bm.B; ++b) tp.p[b] = tokens[b];
  const int rows = bm.t_off[bm.B];
  if (rows == 0) return cudaSuccess;
  if (dt == CB_BF16)
    embed_kernel<bf16><<<rows, 256, 0, s>>>(tp, bm, reinterpret_cast<const bf16 *>(embed),
                                            vocab, d, h, status);
  else
    embed_kernel<float><<<rows, 256, 0, s>>>(tp, bm, reinterpret_cast<const float *>(embed),
                                             vocab, d, h, status);
  return launched(1);
}

// ---------------------------------------------------------------- RMSNorm --
// out[i] = h[src(i)] / sqrt(mean(h[src(i)]^2) + eps) * gain, written as
// 16-byte bf16 vectors (or float4 pairs).
template <typename T>
__device__ __forceinline__ void store8(T *p, const float (&v)[8]);
template <>
__device__ __forceinline__ void store8<bf16>(bf16 *p, const float (&v)[8]) {
  uint4 pk;
  __nv_bfloat162 *e = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
  for (int i = 0; i < 4; ++i) e[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(p) = pk;
}
template <>
__device__ __forceinline__ void store8<float>(float *p, const float (&v)[8]) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// Rows of up to kNormMaxD floats; 128 threads per row, two rows per CTA.
// Every load of a thread is issued before the first is used (the row stays
// in registers), so a row costs one memory round trip.
constexpr int kNormMaxD = 8192;
constexpr int kNormSteps = kNormMaxD / (128 * 8);

template <typename T>
__global__ void __launch_bounds__(256)
rmsnorm_kernel(const float *__restrict__ h, int64_t ld_h,
               const int32_t *__restrict__ src_rows, int n, int d,
               const float *__restrict__ gain, float eps, T *__restrict__ out,
               int64_t ld_out) {
  __shared__ float red[2][4];
  grid_dep_wait();
  grid_dep_launch();
  const int sub = threadIdx.x >> 7, t = threadIdx.x & 127;
  const int i = blockIdx.x * 2 + sub;
  const bool ok = i < n;
  const int64_t src = ok ? (src_rows ? src_rows[i] : i) : 0;
  const float *x = h + src * ld_h;
  float v[kNormSteps][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kNormSteps; ++k) {
    const int c = (k * 128 + t) * 8;
    if (ok && c < d) {
      const float4 a = *reinterpret_cast<const float4 *>(x + c);
      const float4 b = *reinterpret_cast<const float4 *>(x + c + 4);
      v[k][0] = a.x; v[k][1] = a.y; v[k][2] = a.z; v[k][3] = a.w;
      v[k][4] = b.x; v[k][5] = b.y; v[k][6] = b.z; v[k][7] = b.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[k][e] = 0.f;
    }
  }
#pragma unroll
  for (int k = 0; k < kNormSteps; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(v[k][e], v[k][e], ss);
  ss = warp_sum(ss);
  if ((t & 31) == 0) red[sub][t >> 5] = ss;
  __syncthreads();
  if (!ok) return;
  const float tot = red[sub][0] + red[sub][1] + red[sub][2] + red[sub][3];
  const float inv = rsqrtf(tot / (float)d + eps);
  T *o = out + (int64_t)i * ld_out;
#pragma unroll
  for (int k = 0; k < kNormSteps; ++k) {
    const int c = (k * 128 + t) * 8;
    if (c < d) {
      const float4 ga = *reinterpret_cast<const float4 *>(gain + c);
      const float4 gb = *reinterpret_cast<const float4 *>(gain + c + 4);
      const float y[8] = {v[k][0] * inv * ga.x, v[k][1] * inv * ga.y, v[k][2] * inv * ga.z,
                          v[k][3] * inv * ga.w, v[k][4] * inv * gb.x, v[k][5] * inv * gb.y,
                          v[k][6] * inv * gb.z, v[k][7] * inv * gb.w};
      store8<T>(o + c, y);
    }
  }
}

cudaError_t launch_rmsnorm(const float *h, int64_t ld_h, const int32_t *src_rows,
                           int n, int d, const float *gain, float eps,
                           void *out, int64_t ld_out, cb_dtype out_dt,
                           cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (d > kNormMaxD) return cudaErrorInvalidValue;
  const int blocks = (n + 1) / 2;
  cudaError_t e;
  if (out_dt == CB_BF16)
    e = launch_pdl(rmsnorm_kernel<bf16>, dim3(blocks), dim3(256), 0, s, h, ld_h, src_rows, n, d,
                   gain, eps, reinterpret_cast<bf16 *>(out), ld_out);
  else
    e = launch_pdl(rmsnorm_kernel<float>, dim3(blocks), dim3(256), 0, s, h, ld_h, src_rows, n, d,
                   gain, eps, reinterpret_cast<float *>(out), ld_out);
  if (e != cudaSuccess) return e;
  return launched(1);
}

// ---------------------------------------------------------- gather / scatter --
// Byte-level row moves in 16-byte units (row bytes are multiples of 16).
__global__ void __launch_bounds__(256)
gather_kernel(const char *__restrict__ src, int64_t ld_src_b, int64_t src_rows,
              const int32_t *__restrict__ idx, int n, int row_units,
              char *__restrict__ dst, int64_t ld_dst_b, int *status) {
  const int64_t total = (int64_t)n * row_units;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(t / row_units), u = (int)(t % row_units);
    const int r = idx[i];
    if (r < 0 || r >= src_rows) { report(status, CB_ERR_DEVICE_INDEX); continue; }
    stg16(dst + i * ld_dst_b + (int64_t)u * 16, ldg16(src + r * ld_src_b + (int64_t)u * 16));
  }
}

static int grid_for(int64_t work, int threads) {
  int64_t b = (work + threads - 1) / threads;
  if (b > 152 * 16) b = 152 * 16;
  return b < 1 ? 1 : (int)b;
}

cudaError_t launch_gather(const void *src, int64_t ld_src, int64_t src_rows,
                          const int32_t *idx, int n, int row_elems, void *dst,
                          int64_t ld_dst, size_t eb, int *status,
                          cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int units = (int)(row_elems * eb / 16);
  gather_kernel<<<grid_for((int64_t)n * units, 256), 256, 0, s>>>(
      (const char *)src, ld_src * (int64_t)eb, src_rows, idx, n, units,
      (char *)dst, ld_dst * (int64_t)eb, status);
  return launched(1);
}

// The same row gather for layers [0, n_layers) at once: layer l reads
// src + l * src_lstride and writes dst + l * dst_lstride (elements).
__global__ void __launch_bounds__(256)
gather_layers_kernel(const char *__restrict__ src, int64_t src_lstride_b, int64_t ld_src_b,
                     int64_t src_rows, const int32_t *__restrict__ idx, int n, int row_units,
                     char *__restrict__ dst, int64_t dst_lstride_b, int64_t ld_dst_b,
                     int *status) {
  const char *sl = src + (int64_t)blockIdx.y * src_lstride_b;
  char *dl = dst + (int64_t)blockIdx.y * dst_lstride_b;
  const int64_t total = (int64_t)n * row_units;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(t / row_units), u = (int)(t % row_units);
    const int r = idx[i];
    if (r < 0 || r >= src_rows) { report(status, CB_ERR_DEVICE_INDEX); continue; }
    stg16(dl + i * ld_dst_b + (int64_t)u * 16, ldg16(sl + r * ld_src_b + (int64_t)u * 16));
  }
}

cudaError_t launch_gather_layers(const void *src, int64_t src_lstride, int64_t ld_src,
                                 int64_t src_rows, const int32_t *idx, int n, int row_elems,
                                 void *dst, int64_t dst_lstride, int64_t ld_dst, size_t eb,
                                 int n_layers, int *status, cudaStream_t s) {
  if (n == 0 || n_layers <= 0) return cudaSuccess;
  const int units = (int)(row_elems * eb / 16);
  const int bx = grid_for((int64_t)n * units, 256);   // a full grid's worth per layer
  gather_layers_kernel<<<dim3(bx, n_layers), 256, 0, s>>>(
      (const char *)src, src_lstride * (int64_t)eb, ld_src * (int64_t)eb, src_rows, idx, n, units,
      (char *)dst, dst_lstride * (int64_t)eb, ld_dst * (int64_t)eb, status);
  return launched(1);
}

__global__ void __launch_bounds__(256)
scatter_kv_kernel(const char *__restrict__ kn, const char *__restrict__ vn,
                  int64_t ld_new_b, const int32_t *__restrict__ rows, int n,
                  char *__restrict__ kc, char *__restrict__ vc,
                  int64_t ld_cache_b, int64_t cache_rows, int row_units,
                  int *status) {
  const int64_t total = (int64_t)n * row_units * 2;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int which = (int)(t / ((int64_t)n * row_units));
    const int64_t tt = t - (int64_t)which * n * row_units;
    const int i = (int)(tt / row_units), u = (int)(tt % row_units);
    const int r = rows[i];
    if (r < 0 || r >= cache_rows) { report(status, CB_ERR_DEVICE_INDEX); continue; }
    const char *src = (which ? vn : kn) + i * ld_new_b + (int64_t)u * 16;
    char *dst = (which ? vc : kc) + r * ld_cache_b + (int64_t)u * 16;
    stg16(dst, ldg16(src));
  }
}

cudaError_t launch_scatter_kv(const void *k_new, const void *v_new,
                              int64_t ld_new, const int32_t *rows, int n,
                              void *k_cache, void *v_cache, int64_t ld_cache,
                              int64_t cache_rows, int row_elems, size_t eb,
                              int *status, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int units = (int)(row_elems * eb / 16);
  scatter_kv_kernel<<<grid_for((int64_t)n * units * 2, 256), 256, 0, s>>>(
      (const char *)k_new, (const char *)v_new, ld_new * (int64_t)eb, rows, n,
      (char *)k_cache, (char *)v_cache, ld_cache * (int64_t)eb, cache_rows,
      units, status);
  return launched(1);
}

// ------------------------------------------------------------- QKV finish --
// One CTA per row.  Column blocks of the projection: [0, Hq hd) -> q,
// [Hq hd, (Hq+Hkv) hd) -> k, the rest -> v.  q and k are rotated at pos[i]
// (rotate-half pairs); k and v land in cache row dst_rows[i].  When v_dst is
// NULL the input holds keys only (k_col0 = column of key 0).
template <typename T>
__global__ void __launch_bounds__(128)
qkv_finish_kernel(const float *__restrict__ qkv, int64_t ld_qkv,
                  const int32_t *__restrict__ pos, const int32_t *__restrict__ dst_rows,
                  int Hq, int Hkv, int hd, const float2 *__restrict__ table,
                  T *__restrict__ q_out, int64_t ld_q, T *__restrict__ k_dst,
                  T *__restrict__ v_dst, int64_t ld_kv, int k_col0) {
  const int i = blockIdx.x;
  const int p = pos[i];
  const int64_t dr = dst_rows ? dst_rows[i] : i;
  const float *src = qkv + (int64_t)i * ld_qkv;
  const int half = hd / 2;
  const float2 *cs = table + (int64_t)p * half;
  const bool keys_only = v_dst == nullptr;
  const int n_rot_heads = keys_only ? Hkv : Hq + Hkv;
  // rotated heads: q heads then k heads
  for (int t = threadIdx.x; t < n_rot_heads * half; t += blockDim.x) {
    const int hh = t / half, e = t % half;
    const int col = keys_only ? k_col0 + hh * hd : hh * hd;
    const float x1 = src[col + e], x2 = src[col + e + half];
    const float2 w = __ldg(cs + e);
    const float o1 = x1 * w.x - x2 * w.y;
    const float o2 = x2 * w.x + x1 * w.y;
    if (!keys_only && hh < Hq) {
      q_out[(int64_t)i * ld_q + hh * hd + e] = from_f<T>(o1);
      q_out[(int64_t)i * ld_q + hh * hd + e + half] = from_f<T>(o2);
    } else {
      const int kh = keys_only ? hh : hh - Hq;
      k_dst[dr * ld_kv + kh * hd + e] = from_f<T>(o1);
      k_dst[dr * ld_kv + kh * hd + e + half] = from_f<T>(o2);
    }
  }
  if (!keys_only) {
    const int v0 = (Hq + Hkv) * hd;
    for (int c = threadIdx.x; c < Hkv * hd; c += blockDim.x)
      v_dst[dr * ld_kv + c] = from_f<T>(src[v0 + c]);
  }
}

cudaError_t launch_qkv_finish(const float *qkv, int64_t ld_qkv, int n,
                              const int32_t *pos, const int32_t *dst_rows,
                              int Hq, int Hkv, int hd, const float *table,
                              void *q_out, int64_t ld_q, void *k_dst,
                              void *v_dst, int64_t ld_kv, cb_dtype dt,
                              int k_col0, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const float2 *tab = reinterpret_cast<const float2 *>(table);
  if (dt == CB_BF16)
    qkv_finish_kernel<bf16><<<n, 128, 0, s>>>(qkv, ld_qkv, pos, dst_rows, Hq, Hkv, hd, tab,
                                              (bf16 *)q_out, ld_q, (bf16 *)k_dst,
                                              (bf16 *)v_dst, ld_kv, k_col0);
  else
    qkv_finish_kernel<float><<<n, 128, 0, s>>>(qkv, ld_qkv, pos, dst_rows, Hq, Hkv, hd, tab,
                                               (float *)q_out, ld_q, (float *)k_dst,
                                               (float *)v_dst, ld_kv, k_col0);
  return launched(1);
}

// -------------------------------------------------------------- LM head --
// Stage 1: x_b = RMSNorm(h[last_b]) (float, one CTA per request) and reset
// of the packed arg-max words.  Stage 2: every CTA takes a slice of the
// vocabulary; a warp computes whole dot products x_b . E[v] (16-byte loads
// of E, which is read exactly once), the best (value, lowest id) per CTA is
// merged with a 64-bit atomicMax on (order-preserving value bits, ~id).
__device__ __forceinline__ unsigned long long pack_best(float v, int id) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)key << 32) | (unsigned long long)(~(uint32_t)id);
}

struct LastRows {
  int r[CB_MAX_BATCH];
};

__global__ void lm_norm_kernel(const float *__restrict__ h, int64_t ld_h,
                               const __grid_constant__ LastRows last_rows, int d,
                               const float *__restrict__ g, float eps,
                               float *__restrict__ x,
                               unsigned long long *__restrict__ best) {
  __shared__ float red[8];
  const int b = blockIdx.x;
  const float *src = h + (int64_t)last_rows.r[b] * ld_h;
  float ss = 0.f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) ss = fmaf(src[c], src[c], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = rsqrtf(tot / (float)d + eps);
  for (int c = threadIdx.x; c < d; c += blockDim.x) x[(int64_t)b * d + c] = src[c] * inv * g[c];
  if (threadIdx.x == 0) best[b] = 0ull;
}

template <typename T>
__global__ void __launch_bounds__(256)
lm_head_kernel(const float *__restrict__ x, int B, const T *__restrict__ E,
               int vocab, int d, unsigned long long *__restrict__ best) {
  constexpr int VEC = 16 / sizeof(T);
  extern __shared__ float xs[];  // [B][d]
  for (int i = threadIdx.x; i < B * d; i += blockDim.x) xs[i] = x[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int gw = blockIdx.x * warps + (threadIdx.x >> 5);
  const int nw = gridDim.x * warps;
  unsigned long long mine[CB_MAX_BATCH > 8 ? 8 : CB_MAX_BATCH];
  const int bl = B < 8 ? B : 8;
  for (int b = 0; b < bl; ++b) mine[b] = 0ull;
  for (int v = gw; v < vocab; v += nw) {
    const T *row = E + (int64_t)v * d;
    float acc[8];
    for (int b = 0; b < bl; ++b) acc[b] = 0.f;
    for (int c = lane * VEC; c < d; c += 32 * VEC) {
      float e[VEC];
      load16<T>(row + c, e);
      for (int b = 0; b < bl; ++b) {
        const float *xb = xs + b * d + c;
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[b] = fmaf(e[j], xb[j], acc[b]);
      }
    }
    for (int b = 0; b < bl; ++b) {
      const float s = warp_sum(acc[b]);
      const unsigned long long pk = pack_best(s, v);
      if (pk > mine[b]) mine[b] = pk;
    }
  }
  for (int b = 0; b < bl; ++b)
    if (lane == 0) atomicMax(best + b, mine[b]);
}

// SMs of the current device (one persistent CTA each for the GEMV).
static int num_sms_rows() { return device_sm_count(); }

// One request, d = 4096, bf16 embedding: each lane holds its 128 entries of
// the normed hidden state in registers (dims 8 * lane + 256 k) and issues the
// 16 loads of a vocabulary row before using any of them, so a warp keeps the
// whole 8 KB row in flight.  Same ranking as lm_head_kernel.
constexpr int kLmD = 4096;
__global__ void __launch_bounds__(256, 1)
lm_head_one_kernel(const float *__restrict__ x, const bf16 *__restrict__ E, int vocab,
                   unsigned long long *__restrict__ best) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int nw = gridDim.x * 8;
  float xr[kLmD / 32];
#pragma unroll
  for (int k = 0; k < kLmD / 256; ++k) {
    const float4 a = *reinterpret_cast<const float4 *>(x + 256 * k + 8 * lane);
    const float4 b = *reinterpret_cast<const float4 *>(x + 256 * k + 8 * lane + 4);
    xr[8 * k] = a.x; xr[8 * k + 1] = a.y; xr[8 * k + 2] = a.z; xr[8 * k + 3] = a.w;
    xr[8 * k + 4] = b.x; xr[8 * k + 5] = b.y; xr[8 * k + 6] = b.z; xr[8 * k + 7] = b.w;
  }
  unsigned long long mine = 0ull;
  for (int v = gw; v < vocab; v += nw) {
    const uint4 *row = reinterpret_cast<const uint4 *>(E + (int64_t)v * kLmD) + lane;
    uint4 raw[kLmD / 256];
#pragma unroll
    for (int k = 0; k < kLmD / 256; ++k) raw[k] = __ldg(row + 32 * k);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kLmD / 256; ++k) {
      const __nv_bfloat162 *e = reinterpret_cast<const __nv_bfloat162 *>(&raw[k]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(e[j]);
        acc[j] = fmaf(f.x, xr[8 * k + 2 * j], acc[j]);
        acc[j] = fmaf(f.y, xr[8 * k + 2 * j + 1], acc[j]);
      }
    }
    const float sum = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
    const unsigned long long pk = pack_best(sum, v);
    if (pk > mine) mine = pk;
  }
  if (lane == 0) atomicMax(best, mine);
}

__global__ void lm_unpack_kernel(const unsigned long long *__restrict__ best,
                                 int B, int32_t *__restrict__ token) {
  const int b = threadIdx.x;
  if (b < B) token[b] = (int32_t)(~(uint32_t)(best[b] & 0xffffffffull));
}

cudaError_t launch_lm_head_argmax(const float *h, int64_t ld_h,
                                  const int32_t *last_rows_host, int B,
                                  const float *final_norm, float eps,
                                  const void *embed, int vocab, int d,
                                  cb_dtype dt, float *x_scratch,
                                  unsigned long long *best, int32_t *token_out,
                                  cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  LastRows lr;
  for (int b = 0; b < B; ++b) lr.r[b] = last_rows_host[b];
  lm_norm_kernel<<<B, 256, 0, s>>>(h, ld_h, lr, d, final_norm, eps, x_scratch, best);
  if (B == 1 && d == kLmD && dt == CB_BF16) {
    lm_head_one_kernel<<<num_sms_rows(), 256, 0, s>>>(x_scratch, (const bf16 *)embed, vocab,
                                                      best);
    lm_unpack_kernel<<<1, 32, 0, s>>>(best, B, token_out);
    return launched(3);
  }
  // up to 8 requests per pass over the vocabulary
  for (int b0 = 0; b0 < B; b0 += 8) {
    const int nb = B - b0 < 8 ? B - b0 : 8;
    const size_t smem = (size_t)nb * d * sizeof(float);
    const int blocks = 152 * 4;
    if (dt == CB_BF16) {
      cudaFuncSetAttribute(lm_head_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      lm_head_kernel<bf16><<<blocks, 256, smem, s>>>(x_scratch + (int64_t)b0 * d, nb,
                                                     (const bf16 *)embed, vocab, d, best + b0);
    } else {
      cudaFuncSetAttribute(lm_head_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      lm_head_kernel<float><<<blocks, 256, smem, s>>>(x_scratch + (int64_t)b0 * d, nb,
                                                      (const float *)embed, vocab, d, best + b0);
    }
  }
  lm_unpack_kernel<<<1, CB_MAX_BATCH, 0, s>>>(best, B, token_out);
  return launched(2 + (B + 7) / 8);
}

// ------------------------------------------------------------------- copy --
__global__ void copy_f32_kernel(float *__restrict__ dst, const float *__restrict__ src, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

cudaError_t launch_copy_f32(float *dst, const float *src, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  copy_f32_kernel<<<grid_for((int64_t)n, 256), 256, 0, s>>>(dst, src, n);
  return launched(1);
}

}  // namespace cb
