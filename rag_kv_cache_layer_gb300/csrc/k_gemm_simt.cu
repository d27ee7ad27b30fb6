// CUDA-core GEMM, out = epi(A W^T) with A [M][K] and W [N][K] both K-major.
// This is the fp32 parity path (tensor cores would round operands to
// tf32/bf16), with fused epilogues:
//   EPI_STORE_F32  out (float)  = acc
//   EPI_STORE      out (T)      = acc
//   EPI_RESID      out (float) += acc            (residual stream)
//   EPI_SWIGLU     out (T)      = silu(acc_W) * acc_W2
// 64x64 output tile per 256-thread CTA, 4x4 outputs per thread, K in steps
// of 16 staged through shared memory.
#include "cb_common.cuh"
#include "cb_internal.h"

namespace cb {

constexpr int BM = 64, BN = 64, BK = 16;

template <typename T, int EPI>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const T *__restrict__ A, int64_t lda, const T *__restrict__ W,
                 const T *__restrict__ W2, int64_t ldw, int M, int N, int K,
                 void *__restrict__ out, int64_t ldo) {
  constexpr bool DUAL = EPI == EPI_SWIGLU;
  __shared__ float As[BK][BM + 4];
  __shared__ float Ws[BK][BN + 4];
  __shared__ float W2s[DUAL ? BK : 1][BN + 4];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tr = tid / 16, tc = tid % 16;   // 16x16 thread grid, 4x4 each
  float acc[4][4] = {}, acc2[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    // each thread loads 4 elements of each tile: row = tid/4 (0..63),
    // k = (tid%4)*4 .. +3
    const int lr = tid / 4, lk = (tid % 4) * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gm = m0 + lr, gn = n0 + lr, gk = k0 + lk + j;
      As[lk + j][lr] = (gm < M) ? to_f(A[(int64_t)gm * lda + gk]) : 0.f;
      Ws[lk + j][lr] = (gn < N) ? to_f(W[(int64_t)gn * ldw + gk]) : 0.f;
      if (DUAL) W2s[lk + j][lr] = (gn < N) ? to_f(W2[(int64_t)gn * ldw + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], w[4], w2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][tr * 4 + i];
        w[i] = Ws[kk][tc * 4 + i];
        if (DUAL) w2[i] = W2s[kk][tc * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
          if (DUAL) acc2[i][j] = fmaf(a[i], w2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + tr * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tc * 4 + j;
      if (gn >= N) continue;
      const int64_t o = (int64_t)gm * ldo + gn;
      if (EPI == EPI_STORE_F32) {
        reinterpret_cast<float *>(out)[o] = acc[i][j];
      } else if (EPI == EPI_STORE) {
        reinterpret_cast<T *>(out)[o] = from_f<T>(acc[i][j]);
      } else if (EPI == EPI_RESID) {
        reinterpret_cast<float *>(out)[o] += acc[i][j];
      } else {
        const float g = acc[i][j];
        const float sg = g / (1.f + expf(-g));
        reinterpret_cast<T *>(out)[o] = from_f<T>(sg * acc2[i][j]);
      }
    }
  }
}

template <typename T>
static cudaError_t gemm_dispatch(const void *A, int64_t lda, const void *W,
                                 const void *W2, int64_t ldw, int M, int N,
                                 int K, GemmEpi epi, void *out, int64_t ldo,
                                 cudaStream_t s) {
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  const T *a = (const T *)A, *w = (const T *)W, *w2 = (const T *)W2;
  switch (epi) {
    case EPI_STORE_F32: gemm_simt_kernel<T, EPI_STORE_F32><<<grid, 256, 0, s>>>(a, lda, w, w2, ldw, M, N, K, out, ldo); break;
    case EPI_STORE: gemm_simt_kernel<T, EPI_STORE><<<grid, 256, 0, s>>>(a, lda, w, w2, ldw, M, N, K, out, ldo); break;
    case EPI_RESID: gemm_simt_kernel<T, EPI_RESID><<<grid, 256, 0, s>>>(a, lda, w, w2, ldw, M, N, K, out, ldo); break;
    case EPI_SWIGLU: gemm_simt_kernel<T, EPI_SWIGLU><<<grid, 256, 0, s>>>(a, lda, w, w2, ldw, M, N, K, out, ldo); break;
  }
  return launched(1);
}

cudaError_t launch_gemm_simt(const void *A, int64_t lda, const void *W,
                             const void *W2, int64_t ldw, int M, int N, int K,
                             GemmEpi epi, void *out, int64_t ldo, cb_dtype dt,
                             cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (dt == CB_BF16) return gemm_dispatch<bf16>(A, lda, W, W2, ldw, M, N, K, epi, out, ldo, s);
  return gemm_dispatch<float>(A, lda, W, W2, ldw, M, N, K, epi, out, ldo, s);
}

}  // namespace cb
