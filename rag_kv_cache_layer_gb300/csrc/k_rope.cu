// RoPE table and the re-position + stitch kernel (Pi_i of QCFuse Eq. 4).
//
// Keys of a chunk prefilled standalone carry rotations for chunk-local
// positions t.  RoPE rotations compose (CacheBlend blog, "Why You Can't Just
// Concatenate"), so placing the chunk at request offset o applies one more
// rotation by delta = o to every rotate-half pair (e, e + hd/2); values are
// copied unchanged in token order.
//
// The kernel is a pure HBM stream: every byte of the stored K and V is read
// once and written once.  Work is flattened over (row, 16-byte unit) so that
// consecutive threads touch consecutive 16-byte vectors of a row, and one
// launch covers every chunk and every layer (grid.y = layer).
#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

// ------------------------------------------------------------ RoPE table --
__global__ void rope_table_kernel(float2 *table, int max_pos, int half,
                                  double base) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)max_pos * half) return;
  const int p = (int)(i / half);
  const int e = (int)(i % half);
  // theta_e = base^(-2e/hd) with hd = 2 * half; angle evaluated in double.
  const double theta = pow(base, -(double)e / (double)half);
  double s, c;
  sincos((double)p * theta, &s, &c);
  table[i] = make_float2((float)c, (float)s);
}

cudaError_t launch_rope_table(float *table, int max_pos, int head_dim,
                              float base, cudaStream_t s) {
  const int half = head_dim / 2;
  const int64_t n = (int64_t)max_pos * half;
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads);
  rope_table_kernel<<<blocks, threads, 0, s>>>(reinterpret_cast<float2 *>(table),
                                               max_pos, half, (double)base);
  return launched(1);
}

// ------------------------------------------------------------ reposition --
constexpr int kMaxStitch = 96;

struct StitchParams {
  int n;
  int row_prefix[kMaxStitch + 1];  // rows before descriptor i
  cb_stitch_desc d[kMaxStitch];
};

template <typename T>
__global__ void __launch_bounds__(256)
reposition_kernel(const __grid_constant__ StitchParams p, int layer_begin,
                  T *__restrict__ k_cache, T *__restrict__ v_cache,
                  int64_t cache_layer_stride, int row_elems, int head_dim,
                  const float2 *__restrict__ table, int *status) {
  constexpr int VEC = 16 / sizeof(T);
  const int layer = layer_begin + blockIdx.y;
  const int total_rows = p.row_prefix[p.n];
  const int k_units = row_elems / (2 * VEC);      // pair units per row
  const int v_units = row_elems / VEC;
  const int per_row = k_units + v_units;
  const int64_t total = (int64_t)total_rows * per_row;
  const int half = head_dim / 2;
  const int units_per_head = half / VEC;

  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    // Units are ordered [K pair units of all rows][V units of all rows] so
    // that a warp's 32 threads always read contiguous memory.
    int row, unit;
    bool is_k;
    if (t < (int64_t)total_rows * k_units) {
      row = (int)(t / k_units);
      unit = (int)(t % k_units);
      is_k = true;
    } else {
      const int64_t tv = t - (int64_t)total_rows * k_units;
      row = (int)(tv / v_units);
      unit = (int)(tv % v_units);
      is_k = false;
    }
    // descriptor holding this row (binary search over the prefix)
    int lo = 0, hi = p.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.row_prefix[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const cb_stitch_desc &d = p.d[lo];
    const int r = row - p.row_prefix[lo];
    const T *ksrc = reinterpret_cast<const T *>(d.k_src) +
                    (int64_t)layer * d.src_layer_stride + (int64_t)r * row_elems;
    const T *vsrc = reinterpret_cast<const T *>(d.v_src) +
                    (int64_t)layer * d.src_layer_stride + (int64_t)r * row_elems;
    const int64_t dst = (int64_t)layer * cache_layer_stride +
                        (int64_t)(d.dst_row + r) * row_elems;
    if (!is_k) {
      stg16(v_cache + dst + (int64_t)unit * VEC, ldg16(vsrc + (int64_t)unit * VEC));
      continue;
    }
    const int h = unit / units_per_head;
    const int e0 = (unit % units_per_head) * VEC;
    const int c1 = h * head_dim + e0;
    const int c2 = c1 + half;
    float x1[VEC], x2[VEC], o1[VEC], o2[VEC];
    load16<T>(ksrc + c1, x1);
    load16<T>(ksrc + c2, x2);
    const int ad = d.delta < 0 ? -d.delta : d.delta;
    const float sgn = d.delta < 0 ? -1.f : 1.f;
    const float2 *cs = table + (int64_t)ad * half + e0;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const float2 w = __ldg(cs + i);
      const float c = w.x, s = sgn * w.y;
      o1[i] = x1[i] * c - x2[i] * s;
      o2[i] = x2[i] * c + x1[i] * s;
    }
    store16<T>(k_cache + dst + c1, o1);
    store16<T>(k_cache + dst + c2, o2);
  }
  (void)status;
}

cudaError_t launch_reposition(const cb_stitch_desc *descs, int n_desc,
                              int layer_begin, int layer_end, void *k_cache,
                              void *v_cache, int64_t cache_layer_stride,
                              int row_elems, int head_dim, const float *table,
                              cb_dtype dt, int *status, cudaStream_t s, int max_blocks) {
  if (layer_end <= layer_begin) return cudaSuccess;
  for (int base = 0; base < n_desc; base += kMaxStitch) {
    StitchParams p;
    p.n = n_desc - base < kMaxStitch ? n_desc - base : kMaxStitch;
    p.row_prefix[0] = 0;
    for (int i = 0; i < p.n; ++i) {
      p.d[i] = descs[base + i];
      p.row_prefix[i + 1] = p.row_prefix[i] + descs[base + i].len;
    }
    const int rows = p.row_prefix[p.n];
    if (rows == 0) continue;
    const int vec = dt == CB_BF16 ? 8 : 4;
    const int64_t units = (int64_t)rows * (row_elems / (2 * vec) + row_elems / vec);
    int64_t blocks = (units + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    if (max_blocks > 0 && blocks > max_blocks) blocks = max_blocks;
    dim3 grid((unsigned)blocks, (unsigned)(layer_end - layer_begin));
    const float2 *tab = reinterpret_cast<const float2 *>(table);
    if (dt == CB_BF16)
      reposition_kernel<bf16><<<grid, 256, 0, s>>>(
          p, layer_begin, reinterpret_cast<bf16 *>(k_cache),
          reinterpret_cast<bf16 *>(v_cache), cache_layer_stride, row_elems,
          head_dim, tab, status);
    else
      reposition_kernel<float><<<grid, 256, 0, s>>>(
          p, layer_begin, reinterpret_cast<float *>(k_cache),
          reinterpret_cast<float *>(v_cache), cache_layer_stride, row_elems,
          head_dim, tab, status);
    cudaError_t e = launched(1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace cb
