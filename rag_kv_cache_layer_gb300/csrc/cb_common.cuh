// Device-side helpers shared by the library's kernels: typed loads/stores of
// float and bfloat16 rows, the device status word, warp reductions and the
// bounded mbarrier wait used by every pipelined kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cacheblend.h"

namespace cb {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- status --
// The first failure recorded on the device wins; later ones are dropped.
__device__ __forceinline__ void report(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ conversions --
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) {
  return __float2bfloat16_rn(x);
}

// A 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  T v[N];
};

template <typename T>
__device__ __forceinline__ void load16(const T *p, float (&out)[16 / sizeof(T)]) {
  uint4 raw = *reinterpret_cast<const uint4 *>(p);
  const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
  for (int i = 0; i < (int)(16 / sizeof(T)); ++i) out[i] = to_f(e[i]);
}

template <typename T>
__device__ __forceinline__ void store16(T *p, const float (&in)[16 / sizeof(T)]) {
  uint4 raw;
  T *e = reinterpret_cast<T *>(&raw);
#pragma unroll
  for (int i = 0; i < (int)(16 / sizeof(T)); ++i) e[i] = from_f<T>(in[i]);
  *reinterpret_cast<uint4 *>(p) = raw;
}

__device__ __forceinline__ uint4 ldg16(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void stg16(void *p, uint4 v) {
  *reinterpret_cast<uint4 *>(p) = v;
}

// ------------------------------------------------------------- reductions --
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// -------------------------------------------------------- bounded waits --
// Wall-clock limit of every spin-wait in the library.  A wait that runs
// past it records CB_ERR_TIMEOUT and reports failure to its caller, which
// then leaves its pipeline in an orderly way instead of hanging the device.
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of the mbarrier at shared address `bar`.
// Returns false (after recording CB_ERR_TIMEOUT) once `limit_ns` has passed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns, int *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) {
      report(status, CB_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialization may start while the previous kernel of the stream is
// still running.  It does only shared-memory / TMEM setup before
// grid_dep_wait(), which returns once the previous grid has completed and
// its writes are visible; it then calls grid_dep_launch() so that the next
// kernel may start its own setup.  The next grid is scheduled only after
// every CTA of this grid has called grid_dep_launch() or exited.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Default limit for pipeline waits: two seconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

}  // namespace cb
