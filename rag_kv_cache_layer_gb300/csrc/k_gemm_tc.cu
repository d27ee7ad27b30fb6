// bf16 tensor-core GEMM for sm_103a: out = epi(A W^T), A [M][K] and W [N][K]
// both K-major, fp32 accumulation in tensor memory.
//
// Structure (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: one thread streams 128x64 A tiles and BNx64 W
//               tiles (128-byte swizzle) into a ring of shared-memory stages;
//   warp 1      owns the TMEM allocation; one thread issues tcgen05.mma
//               (M=128, N=BN, K=16) and commits stage releases / accumulator
//               completion to mbarriers;
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator (each thread one
//               row), fused epilogue, global stores.
// The accumulator is double-buffered in TMEM so that the epilogue of one
// tile overlaps the main loop of the next.  Every mbarrier wait is bounded:
// on expiry the kernel records CB_ERR_TIMEOUT, drains its own copies and
// frees TMEM before returning.
//
// Epilogues: STORE (bf16), STORE_F32, RESID (float += acc; split-K units add
// with vector atomics), SWIGLU (MMA N = 256 over [W_gate tile; W_up tile],
// out = silu(gate) * up, 128 output columns per tile), QKV (RoPE at the
// row's position for q and k heads, k and v rows written to fused-cache
// rows, QCFuse Eq. 7).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "cb_common.cuh"
#include "cb_internal.h"
#include "cb_tc.cuh"

namespace cb {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                 // one 128-byte swizzle row of bf16
constexpr int kThreads = 192;
constexpr int kTileA = BM * BK * 2;    // 16 KB

// --------------------------------------------------------------- PTX ops --
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused, SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                      // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: D f32, A/B bf16, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map,
                                            uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b,
                                     uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 accumulator columns of one row -> bf16; `valid` columns remain in the
// row (16-byte stores when all 32 fit, element stores for a ragged tail).
__device__ __forceinline__ void store_bf16_chunk(bf16 *dst, const float (&x)[32], int valid) {
  if (valid >= 32) {
    uint4 pk[4];
    bf16 *pe = reinterpret_cast<bf16 *>(pk);
#pragma unroll
    for (int i = 0; i < 32; ++i) pe[i] = __float2bfloat16_rn(x[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i) reinterpret_cast<uint4 *>(dst)[i] = pk[i];
  } else {
    for (int i = 0; i < valid; ++i) dst[i] = __float2bfloat16_rn(x[i]);
  }
}

// -------------------------------------------------------------- params --
struct EpiParams {
  void *out;            // STORE / STORE_F32 / RESID / SWIGLU destination, QKV: q
  int64_t ldo;
  // QKV epilogue
  const int32_t *pos;   // row position (RoPE angle)
  const int32_t *dst_row;  // fused-cache row of each A row
  void *k_cache, *v_cache;
  int64_t ld_kv;
  const float2 *rope;   // [max_pos][hd/2] (cos, sin)
  int n_q_heads, n_kv_heads;
};

template <int BN, int EPI>
struct Cfg {
  static constexpr bool kDual = EPI == EPI_SWIGLU;
  static constexpr int kMmaN = kDual ? 256 : BN;        // MMA N
  static constexpr int kOutN = kDual ? 128 : BN;        // output columns per tile
  static constexpr int kTileB = kMmaN * BK * 2;
  static constexpr int kStage = kTileA + kTileB;
  static constexpr int kStages = kStage <= 32768 ? 6 : 4;
  static constexpr int kTmemCols = 2 * kMmaN;           // double buffer
  static constexpr int kSmem = kStages * kStage + 1024 /*align*/ + 256 /*barriers*/;
};

// Work of one persistent CTA.  Tile mode: output tiles blockIdx.x,
// blockIdx.x + gridDim.x, ... over the whole K range.  Stream-K mode (the
// residual epilogue, whose atomic add makes any K split legal): the
// tiles x k-blocks of the GEMM are laid end to end and every CTA takes an
// equal contiguous share, which may start or end inside a tile.  Tiles are
// numbered M-fastest so that CTAs running together share weight tiles.
struct Work {
  int n_m, num_kb;
  bool sk;
  int64_t w, w_end;
  __device__ Work(int n_m_, int n_n, int num_kb_, bool sk_) : n_m(n_m_), num_kb(num_kb_), sk(sk_) {
    const int64_t tiles = (int64_t)n_m_ * n_n;
    if (sk) {
      const int64_t total = tiles * num_kb_;
      w = total * blockIdx.x / gridDim.x;
      w_end = total * (blockIdx.x + 1) / gridDim.x;
    } else {
      w = blockIdx.x;
      w_end = tiles;
    }
  }
  __device__ bool next(int &m_blk, int &n_blk, int &kb0, int &kb1) {
    if (w >= w_end) return false;
    int tile;
    if (sk) {
      tile = (int)(w / num_kb);
      kb0 = (int)(w % num_kb);
      const int64_t left = w_end - w;
      kb1 = (int)(kb0 + left < num_kb ? kb0 + left : num_kb);
      w += kb1 - kb0;
    } else {
      tile = (int)w;
      kb0 = 0;
      kb1 = num_kb;
      w += gridDim.x;
    }
    m_blk = tile % n_m;
    n_blk = tile / n_m;
    return true;
  }
};

// ---------------------------------------------------------------- kernel --
template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA,
               const __grid_constant__ CUtensorMap mapB,
               const __grid_constant__ CUtensorMap mapB2, int M, int N, int K,
               int stream_k, const EpiParams ep, int *status) {
  using C = Cfg<BN, EPI>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStage);
  uint64_t *full = bars;                       // [kStages]
  uint64_t *empty = bars + C::kStages;         // [kStages]
  uint64_t *tfull = bars + 2 * C::kStages;     // [2]
  uint64_t *tempty = tfull + 2;                // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  volatile int *fail_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_m = (M + BM - 1) / BM;
  const int n_n = (N + C::kOutN - 1) / C::kOutN;
  const int num_kb = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 128);
    }
    *fail_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&mapA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&mapB) : "memory");
    if (C::kDual) asm volatile("prefetch.tensormap [%0];" ::"l"(&mapB2) : "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_wait();      // inputs of the previous kernel are visible from here
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The warp runs the loop converged; the elected lane issues the copies.
    int stage = 0;
    uint32_t phase = 0;
    int issued[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    bool ok = true;
    Work wk(n_m, n_n, num_kb, stream_k != 0);
    int m_blk, n_blk, kb0, kb1;
    while (ok && wk.next(m_blk, n_blk, kb0, kb1)) {
      for (int kb = kb0; kb < kb1; ++kb) {
        const bool got = mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, kWaitLimitNs,
                                           status) &&
                         !*fail_flag;
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        if (tcx::elect_one()) {
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_expect_tx(fb, C::kStage);
          uint8_t *sa = smem + stage * C::kStage;
          uint8_t *sb = sa + kTileA;
          tma_load_2d(smem_u32(sa), &mapA, fb, kb * BK, m_blk * BM);
          if (C::kDual) {
            tma_load_2d(smem_u32(sb), &mapB, fb, kb * BK, n_blk * 128);
            tma_load_2d(smem_u32(sb + 128 * BK * 2), &mapB2, fb, kb * BK, n_blk * 128);
          } else {
            tma_load_2d(smem_u32(sb), &mapB, fb, kb * BK, n_blk * BN);
          }
        }
        __syncwarp();
        ++issued[stage];
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok && lane == 0) {
      *fail_flag = 1;
      // drain this warp's copies still in flight before the CTA exits
      for (int s = 0; s < C::kStages; ++s)
        if (issued[s] > 0)
          mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((issued[s] - 1) & 1), 10000000ull,
                            nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // Converged warp, elected lane issues; the failure flag is polled once
    // per tile (a stalled producer also ends the bounded waits below).
    constexpr uint32_t idesc = make_idesc(BM, C::kMmaN);
    int stage = 0;
    uint32_t phase = 0;
    int buf = 0;
    uint32_t bphase = 0;
    bool ok = true;
    Work wk(n_m, n_n, num_kb, stream_k != 0);
    int m_blk, n_blk, kb0, kb1;
    while (ok && wk.next(m_blk, n_blk, kb0, kb1)) {
      const bool got =
          mbar_wait_bounded(smem_u32(&tempty[buf]), bphase ^ 1, kWaitLimitNs, status) &&
          !*fail_flag;
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + buf * C::kMmaN;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(smem_u32(&full[stage]), phase, kWaitLimitNs, status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (tcx::elect_one()) {
          const uint32_t sa = smem_u32(smem + stage * C::kStage);
          const uint64_t da = smem_desc(sa), db = smem_desc(sa + kTileA);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma(d, da + 2 * k, db + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&empty[stage]));
        }
        __syncwarp();
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (tcx::elect_one()) umma_commit(smem_u32(&tfull[buf]));
      __syncwarp();
      if (++buf == 2) { buf = 0; bphase ^= 1; }
    }
    if (!ok && lane == 0) *fail_flag = 1;
  } else {
    // ----------------------------------------------------------- epilogue
    const int quad = warp & 3;                 // TMEM lanes 32*quad .. +31
    const int row_in_tile = quad * 32 + lane;
    int buf = 0;
    uint32_t bphase = 0;
    Work wk(n_m, n_n, num_kb, stream_k != 0);
    int m_blk, n_blk, kb0, kb1;
    while (wk.next(m_blk, n_blk, kb0, kb1)) {
      // a tile covered by one CTA alone is updated in place; pieces of a
      // tile shared between CTAs are added atomically
      const bool whole = kb0 == 0 && kb1 == num_kb;
      // leave warp-uniformly on failure: the TMEM loads are .sync.aligned
      const bool bad =
          !mbar_wait_bounded(smem_u32(&tfull[buf]), bphase, kWaitLimitNs, status) || *fail_flag;
      if (__any_sync(0xffffffffu, bad)) {
        *fail_flag = 1;
        break;
      }
      tc_fence_after();
      const int m = m_blk * BM + row_in_tile;
      const bool row_ok = m < M;
      const uint32_t tbase = tmem_base + buf * C::kMmaN + ((uint32_t)(quad * 32) << 16);
      const int n0 = n_blk * C::kOutN;
      if (EPI == EPI_SWIGLU) {
        bf16 *o = reinterpret_cast<bf16 *>(ep.out) + (int64_t)m * ep.ldo + n0;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          float g[32], v[32];
          tmem_ld32(tbase + c, g);
          tmem_ld32(tbase + 128 + c, v);
          if (row_ok && n0 + c < N) {
            float y[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = __fdividef(g[i], 1.f + __expf(-g[i])) * v[i];
            store_bf16_chunk(o + c, y, N - (n0 + c));
          }
        }
      } else if (EPI == EPI_QKV) {
        // head_dim 128: the tile holds BN / 128 consecutive heads of the
        // stacked [q heads | k heads | v heads] projection.
        const int Hq = ep.n_q_heads, Hkv = ep.n_kv_heads;
        const int p = row_ok ? ep.pos[m] : 0;
        const int64_t dr = row_ok ? ep.dst_row[m] : 0;
        const float2 *cs = ep.rope + (int64_t)p * 64;
#pragma unroll 1
        for (int hh = 0; hh < BN / 128; ++hh) {
          const int head = n_blk * (BN / 128) + hh;
          if (head >= Hq + 2 * Hkv) break;               // uniform across the warp
          const uint32_t hbase = tbase + hh * 128;
          if (head < Hq + Hkv) {
            bf16 *dst = head < Hq
                            ? reinterpret_cast<bf16 *>(ep.out) + (int64_t)m * ep.ldo + head * 128
                            : reinterpret_cast<bf16 *>(ep.k_cache) + dr * ep.ld_kv + (head - Hq) * 128;
#pragma unroll 1
            for (int c = 0; c < 64; c += 32) {
              float x1[32], x2[32];
              tmem_ld32(hbase + c, x1);
              tmem_ld32(hbase + 64 + c, x2);
              if (row_ok) {
                uint4 p1[4], p2[4];
                bf16 *e1 = reinterpret_cast<bf16 *>(p1);
                bf16 *e2 = reinterpret_cast<bf16 *>(p2);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const float2 w = __ldg(cs + c + i);
                  e1[i] = __float2bfloat16_rn(x1[i] * w.x - x2[i] * w.y);
                  e2[i] = __float2bfloat16_rn(x2[i] * w.x + x1[i] * w.y);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  reinterpret_cast<uint4 *>(dst + c)[i] = p1[i];
                  reinterpret_cast<uint4 *>(dst + 64 + c)[i] = p2[i];
                }
              }
            }
          } else {
            bf16 *dst = reinterpret_cast<bf16 *>(ep.v_cache) + dr * ep.ld_kv +
                        (head - Hq - Hkv) * 128;
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
              float x[32];
              tmem_ld32(hbase + c, x);
              if (row_ok) store_bf16_chunk(dst + c, x, 32);
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float x[32];
          tmem_ld32(tbase + c, x);
          if (!row_ok || n0 + c >= N) continue;
          const int valid = N - (n0 + c);     // columns left in this row
          if (EPI == EPI_STORE) {
            store_bf16_chunk(reinterpret_cast<bf16 *>(ep.out) + (int64_t)m * ep.ldo + n0 + c, x,
                             valid);
          } else if (valid < 32) {            // ragged tail: element by element
            float *o = reinterpret_cast<float *>(ep.out) + (int64_t)m * ep.ldo + n0 + c;
            for (int i = 0; i < valid; ++i) {
              if (EPI == EPI_STORE_F32) o[i] = x[i];
              else if (whole) o[i] += x[i];
              else atomicAdd(o + i, x[i]);
            }
          } else if (EPI == EPI_STORE_F32) {
            float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(ep.out) +
                                                   (int64_t)m * ep.ldo + n0 + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              o[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
          } else {  // EPI_RESID
            float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(ep.out) +
                                                   (int64_t)m * ep.ldo + n0 + c);
            if (whole) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float4 h = o[i];
                h.x += x[4 * i]; h.y += x[4 * i + 1]; h.z += x[4 * i + 2]; h.w += x[4 * i + 3];
                o[i] = h;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                atomicAdd(o + i, make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[buf]));
      if (++buf == 2) { buf = 0; bphase ^= 1; }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host --
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor [rows][cols] (cols contiguous, row stride ld elements);
// box = 64 columns x box_rows rows, 128-byte swizzle, zero fill outside.
static bool make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                     int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int num_sms() { return device_sm_count(); }

template <int BN, int EPI>
static cudaError_t run(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mb2,
                       int M, int N, int K, bool stream_k, const EpiParams &ep, int *status,
                       cudaStream_t s) {
  using C = Cfg<BN, EPI>;
  static PerDeviceOnce attr;
  cudaError_t ea = attr.run([](int) {
    return cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmem);
  });
  if (ea != cudaSuccess) return ea;
  const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + C::kOutN - 1) / C::kOutN);
  const int64_t work = stream_k ? tiles * ((K + BK - 1) / BK) : tiles;
  const int grid = work < num_sms() ? (int)work : num_sms();
  cudaError_t e = launch_pdl(gemm_tc_kernel<BN, EPI>, dim3(grid), dim3(kThreads), C::kSmem, s,
                             ma, mb, mb2, M, N, K, stream_k ? 1 : 0, ep, status);
  if (e != cudaSuccess) return e;
  return launched(1);
}

}  // namespace tc

cudaError_t launch_gemm_tc(const void *A, int64_t lda, const void *W, const void *W2,
                           int64_t ldw, int M, int N, int K, GemmEpi epi, void *out,
                           int64_t ldo, const QkvEpi *qkv, int *status, cudaStream_t s) {
  using namespace tc;
  if (M == 0 || N == 0) return cudaSuccess;
  CUtensorMap ma, mb, mb2;
  EpiParams ep{};
  ep.out = out;
  ep.ldo = ldo;
  if (!make_map(&ma, A, M, K, lda, BM)) return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_SWIGLU: {
      if (!make_map(&mb, W, N, K, ldw, 128) || !make_map(&mb2, W2, N, K, ldw, 128))
        return cudaErrorInvalidValue;
      return run<128, EPI_SWIGLU>(ma, mb, mb2, M, N, K, false, ep, status, s);
    }
    case EPI_QKV: {
      if (!qkv || !make_map(&mb, W, N, K, ldw, 256)) return cudaErrorInvalidValue;
      ep.pos = qkv->pos;
      ep.dst_row = qkv->dst_row;
      ep.k_cache = qkv->k_cache;
      ep.v_cache = qkv->v_cache;
      ep.ld_kv = qkv->ld_kv;
      ep.rope = reinterpret_cast<const float2 *>(qkv->rope);
      ep.n_q_heads = qkv->n_q_heads;
      ep.n_kv_heads = qkv->n_kv_heads;
      return run<256, EPI_QKV>(ma, mb, mb, M, N, K, false, ep, status, s);
    }
    case EPI_RESID: {
      const bool wide = N % 256 == 0;
      if (!make_map(&mb, W, N, K, ldw, wide ? 256 : 128)) return cudaErrorInvalidValue;
      if (wide) return run<256, EPI_RESID>(ma, mb, mb, M, N, K, true, ep, status, s);
      return run<128, EPI_RESID>(ma, mb, mb, M, N, K, true, ep, status, s);
    }
    case EPI_STORE:
    case EPI_STORE_F32: {
      const bool wide = N % 256 == 0;
      if (!make_map(&mb, W, N, K, ldw, wide ? 256 : 128)) return cudaErrorInvalidValue;
      if (epi == EPI_STORE) {
        if (wide) return run<256, EPI_STORE>(ma, mb, mb, M, N, K, false, ep, status, s);
        return run<128, EPI_STORE>(ma, mb, mb, M, N, K, false, ep, status, s);
      }
      if (wide) return run<256, EPI_STORE_F32>(ma, mb, mb, M, N, K, false, ep, status, s);
      return run<128, EPI_STORE_F32>(ma, mb, mb, M, N, K, false, ep, status, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace cb
