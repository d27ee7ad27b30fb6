// bf16 tensor-core selected-query attention for sm_103a (CacheBlend blog,
// blend_layer step 4: the computed rows attend over the whole fused cache,
// n_sel x L work; QCFuse §2.1.3: causal over the partially fused prefix).
//
// Work unit: one request, one kv head g and a tile of QT = 128 / G query
// rows, where G = n_q_heads / n_kv_heads; the G q heads of the group share
// the kv head, so the tile is 128 MMA rows (row = h * QT + query).  Queries
// of a request are sorted by position, so a tile only visits keys up to its
// last query's position.
//
// Roles (192 threads, two CTAs per SM): warp 0 TMA producer (Q once, then
// double-buffered 64-key K and V blocks, 128-byte swizzle); warp 1 owns 256
// TMEM columns and issues tcgen05.mma: S_j = Q K_j^T into slot j & 1
// (columns 0..63 or 64..127, K-major operands) and O += P_j V_j into columns
// 128..255 with P_j read from TMEM (it overwrites S_j in its slot) and V
// MN-major from shared memory; warps 2..5 do the online softmax (one row
// per thread, log2 domain, causal mask) and store P_j as packed bf16 into
// TMEM.  With two S slots the tensor core computes S_{j+1} while the
// softmax works on S_j, so the softmax warps run block after block; the
// SM's other CTA fills the remaining tensor-core time.  The row's reference
// maximum m only moves when a block raises the maximum by more than
// 2^kRescale: then O (after P_{j-1} V_{j-1} has landed) and l are scaled by
// 2^(m_old - m_new).  Between moves the probabilities stay below
// 2^kRescale, and O / l does not depend on the reference, so the result is
// the same softmax.  Every exponential runs on the SFU (ex2.approx): with
// two CTAs per SM it is under half busy.  All waits are bounded.
//
// When the query tiles alone cannot fill the SMs (the compact layers), the
// key range of every tile is split into chunks processed by separate CTAs;
// each writes its normalised output O_c / l_c (bf16) with (m_c, l_c), and a
// combine kernel merges them: O = sum_c w_c (O_c / l_c) / sum_c w_c with
// w_c = 2^(m_c - M) l_c.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "cb_common.cuh"
#include "cb_internal.h"
#include "cb_tc.cuh"

namespace cb {
namespace attn {

constexpr int kThreads = 192;
constexpr float kRescale = 8.f;            // log2 of the largest p between rescales
constexpr int HD = 128;
constexpr int BN = 64;                     // keys per block
constexpr int kAtom = 128 * 64 * 2;        // one [128 rows x 64 bf16] swizzle tile (Q)
constexpr int kAtomKV = BN * 64 * 2;       // one [64 keys x 64 bf16] swizzle tile
constexpr int kQ = 2 * kAtom;              // Q tile: 128 rows x 128 dims
constexpr int kKV = 2 * kAtomKV;           // K or V block: 64 keys x 128 dims
// smem: Q | K[2] | V[2] | barriers   (96 KB + barriers): two CTAs fit on an SM
constexpr int kOffK = kQ;
constexpr int kOffV = kOffK + 2 * kKV;
constexpr int kOffBar = kOffV + 2 * kKV;
constexpr int kSmem = kOffBar + 256 + 1024;
constexpr int kCtasPerSm = 2;
constexpr int kTmemCols = 256;             // S/P slots 0..63, 64..127; O 128..255
static_assert(kCtasPerSm * (kSmem + 1024) <= 233472, "two attention CTAs must fit an SM");

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                // leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;      // 8-row groups 1024 B apart
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;                // 128-byte swizzle
  return d;
}

// MN-major (N contiguous) operand: 64-element N atoms lbo bytes apart,
// 8-row K groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr, uint32_t lbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

constexpr uint32_t idesc(bool b_mn_major, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map,
                                            uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                    uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
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

// 32 consecutive fp32 columns of this thread's lane, without waiting: the
// registers are valid after wait_ld(), so several loads share one latency.
__device__ __forceinline__ void ld32_nw(uint32_t taddr, float *v) {
  uint32_t *r = reinterpret_cast<uint32_t *>(v);
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
}
__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Writes 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x with the SFU's approximate base-2 exponential (PTX ex2.approx.ftz;
// documented maximum relative error about 2^-22), far below the bf16
// rounding of the probabilities it feeds.
// Packed fp32 pairs (fma / add on .f32x2 of the sm_100 family): two
// softmax elements per instruction.
__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  return ((unsigned long long)__float_as_uint(b) << 32) | __float_as_uint(a);
}
__device__ __forceinline__ float lo2(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(unsigned long long v) {
  return __uint_as_float((uint32_t)(v >> 32));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c) in one instruction (three-input max.f32 of the sm_100 family).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Writes 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

// D (TMEM) += A (TMEM, M lanes x K packed in columns) * B (shared memory).
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}

struct Params {
  int n_req;
  int G, QT, Hkv;
  float scale_log2;            // softmax scale times log2(e)
  int n_chunks, chunk_blocks;  // uniform key-range split of every tile (plan == nullptr)
  const int *plan;             // device unit table (attn_plan_kernel) or nullptr
  int tile_off[CB_MAX_BATCH + 1];
  AttnReq r[CB_MAX_BATCH];
};

// Unit table written by attn_plan_kernel (int32 words): [0] units, [1] key
// blocks per unit at most, [2] tiles, [3] 0; then per tile t the pair
// (first unit, unit count) at [4 + 2t]; then, 16-byte aligned, one int4
// {tile, first key block, end key block, 0} per unit, the units of a tile
// consecutive.
__host__ __device__ inline size_t plan_units_off(int tiles) {
  return ((size_t)(4 + 2 * tiles) * 4 + 15) / 16 * 16;
}

// (request, kv head, query tile) of a tile index; longest tiles first
// within a request.
struct TileId {
  int b, g, t;
};
__device__ __forceinline__ TileId decode_tile(const Params &P, int tile) {
  int b = 0;
  while (P.tile_off[b + 1] <= tile) ++b;
  const int local = tile - P.tile_off[b];
  const int n_rows = P.r[b].q_end - P.r[b].q_begin;
  const int n_t = (n_rows + P.QT - 1) / P.QT;
  return TileId{b, local % P.Hkv, n_t - 1 - local / P.Hkv};
}


// ------------------------------------------------------------ unit plan --
// Splits the tiles' key ranges so that every unit fits in one wave of CTA
// slots: B, the key blocks per unit at most, is the smallest value for which
// sum_t ceil(nb_t / B) <= slots (nb_t: key blocks up to the tile's last query
// position); tile t is cut into ceil(nb_t / B) near-equal consecutive
// ranges.  With at least as many tiles as slots nothing is split.  One CTA.
// Entry u of the table is {tile, first block, end block, partial slot}; the
// slots of a tile's units are consecutive (the combine reads them there).
// Split plans of at most kPlanSort units are stored longest unit first: a
// launch places blocks 0 .. SMs-1 one per SM before the second CTA of each
// SM, and that second wave starts a few microseconds later, so it gets the
// shorter units.
constexpr int kPlanThreads = 1024;
constexpr int kPlanCache = 8192;           // tiles whose block counts stay in smem
constexpr int kPlanSort = 512;
static_assert(kPlanThreads == 1024, "the block reductions assume 32 warps");

__device__ int block_sum(int v, int *red) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = red[threadIdx.x & 31];               // 32 warps: every warp reduces all
  for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;                                  // every warp of the block holds the sum
}
__device__ int block_max(int v, int *red) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = red[threadIdx.x & 31];               // 32 warps: every warp reduces all
  for (int o = 16; o; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

__global__ void __launch_bounds__(kPlanThreads)
attn_plan_kernel(const __grid_constant__ Params P, const int32_t *__restrict__ q_pos, int slots,
                 int *__restrict__ plan) {
  __shared__ int red[kPlanThreads / 32];
  __shared__ int s_nb[kPlanCache];
  __shared__ int4 s_units[kPlanSort];
  __shared__ int s_len[kPlanSort];
  grid_dep_wait();      // q_pos comes from earlier kernels
  grid_dep_launch();
  const int tiles = P.tile_off[P.n_req];
  auto nb_of = [&](int tile) -> int {
    const TileId id = decode_tile(P, tile);
    const AttnReq &R = P.r[id.b];
    const int last = min(R.q_end - R.q_begin, (id.t + 1) * P.QT) - 1;
    const int pmax = q_pos[R.q_begin + last];
    return (pmax < 0 || pmax >= R.kv_len) ? 0 : pmax / BN + 1;   // the kernel reports bad rows
  };
  auto nb_at = [&](int tile) -> int { return tile < kPlanCache ? s_nb[tile] : nb_of(tile); };
  int mx = 0, sum = 0;
  for (int t = threadIdx.x; t < tiles; t += kPlanThreads) {
    const int nb = nb_of(t);
    if (t < kPlanCache) s_nb[t] = nb;
    mx = max(mx, nb);
    sum += nb;
  }
  const int max_nb = block_max(mx, red);
  const int total = block_sum(sum, red);
  int B = max(max_nb, 1);
  if (tiles < slots && max_nb > 1) {
    int lo = max(1, (total + slots - 1) / slots), hi = max_nb;
    while (lo < hi) {                           // uniform across the block
      const int mid = (lo + hi) / 2;
      int cnt = 0;
      for (int t = threadIdx.x; t < tiles; t += kPlanThreads)
        cnt += max(1, (nb_at(t) + mid - 1) / mid);
      if (block_sum(cnt, red) <= slots) hi = mid;
      else lo = mid + 1;
    }
    B = lo;
  }
  int4 *units = reinterpret_cast<int4 *>(reinterpret_cast<char *>(plan) + plan_units_off(tiles));
  int n_cnt = 0;
  for (int t = threadIdx.x; t < tiles; t += kPlanThreads) n_cnt += max(1, (nb_at(t) + B - 1) / B);
  const int n_units = block_sum(n_cnt, red);
  const bool sorted = tiles < slots && n_units <= kPlanSort;
  int base = 0;
  for (int t0 = 0; t0 < tiles; t0 += kPlanThreads) {
    const int t = t0 + threadIdx.x;
    const int nb = t < tiles ? nb_at(t) : 0;
    const int cnt = t < tiles ? max(1, (nb + B - 1) / B) : 0;
    // exclusive scan of cnt over the block
    int incl = cnt;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    __syncthreads();
    if (lane == 31) red[w] = incl;
    __syncthreads();
    if (w == 0) {
      int x = red[lane];
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += v;
      }
      red[lane] = x;                           // inclusive warp totals
    }
    __syncthreads();
    const int first = base + (w ? red[w - 1] : 0) + incl - cnt;
    if (t < tiles) {
      plan[4 + 2 * t] = first;
      plan[5 + 2 * t] = cnt;
      for (int u = 0; u < cnt; ++u) {
        const int4 e = make_int4(t, nb * u / cnt, nb * (u + 1) / cnt, first + u);
        if (sorted) {
          s_units[first + u] = e;
          s_len[first + u] = e.z - e.y;
        } else {
          units[first + u] = e;
        }
      }
    }
    base += red[kPlanThreads / 32 - 1];
    __syncthreads();
  }
  if (sorted) {
    // stable order by length, longest first: the rank of unit u
    for (int u = threadIdx.x; u < n_units; u += kPlanThreads) {
      const int len = s_len[u];
      int pos = 0;
      for (int v = 0; v < n_units; ++v) {
        const int lv = s_len[v];
        pos += (lv > len) || (lv == len && v < u);
      }
      units[pos] = s_units[u];
    }
  }
  if (threadIdx.x == 0) {
    plan[0] = base;
    plan[1] = B;
    plan[2] = tiles;
    plan[3] = 0;
  }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
attn_tc_kernel(const __grid_constant__ CUtensorMap mapQ,
               const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV, const __grid_constant__ Params P,
               const int32_t *__restrict__ q_pos, bf16 *__restrict__ out, int64_t ld_out,
               bf16 *__restrict__ part_o, float2 *__restrict__ part_ml, int *status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *q_full = bar + 0;
  uint64_t *k_full = bar + 1;      // [2] K_j landed
  uint64_t *k_empty = bar + 3;     // [2] S_j = Q K_j^T done with K_j
  uint64_t *v_full = bar + 5;      // [2] V_j landed
  uint64_t *v_empty = bar + 7;     // [2] P_j V_j done with V_j
  uint64_t *s_full = bar + 9;      // [2] S_j in its TMEM slot
  uint64_t *p_full = bar + 11;     // [2] P_j in the slot (and O rescaled)
  uint64_t *pv_done = bar + 13;    // [2] O += P_j V_j has landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 15);
  volatile int *fail = reinterpret_cast<volatile int *>(tmem_slot + 1);
  __shared__ int s_unit[7];        // b, g, tile, first block, end block, split (-1: none), slot

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_wait();      // q, the cache and q_pos come from earlier kernels
  grid_dep_launch();
  if (threadIdx.x == 0) {
    // this CTA's unit: a tile and a range of its key blocks
    int tile, jb, jcap, split;
    int pslot = blockIdx.x;        // partial slot of a split tile's unit
    if (P.plan) {
      if ((int)blockIdx.x >= P.plan[0]) {
        tile = -1;
        jb = jcap = split = 0;
      } else {
        const int4 u = reinterpret_cast<const int4 *>(
            reinterpret_cast<const char *>(P.plan) + plan_units_off(P.plan[2]))[blockIdx.x];
        tile = u.x;
        jb = u.y;
        jcap = u.z;
        pslot = u.w;
        split = P.plan[5 + 2 * tile] > 1;
      }
    } else {
      tile = blockIdx.x / P.n_chunks;
      jb = (blockIdx.x % P.n_chunks) * P.chunk_blocks;
      jcap = jb + P.chunk_blocks;
      split = P.n_chunks > 1;
    }
    s_unit[5] = tile < 0 ? -1 : split;
    s_unit[6] = pslot;
    if (tile >= 0) {
      const TileId id = decode_tile(P, tile);
      const AttnReq &R = P.r[id.b];
      const int n_rows = R.q_end - R.q_begin;
      const int last = min(n_rows, (id.t + 1) * P.QT) - 1;
      int pmax = q_pos[R.q_begin + last];
      if (pmax < 0 || pmax >= R.kv_len) { report(status, CB_ERR_DEVICE_INDEX); pmax = -1; }
      const int nb_tile = pmax < 0 ? 0 : pmax / BN + 1;
      s_unit[0] = id.b; s_unit[1] = id.g; s_unit[2] = id.t;
      s_unit[3] = jb;
      s_unit[4] = max(jb, min(nb_tile, jcap));
    }
    mbar_init(smem_u32(q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&k_full[i]), 1);
      mbar_init(smem_u32(&k_empty[i]), 1);
      mbar_init(smem_u32(&v_full[i]), 1);
      mbar_init(smem_u32(&v_empty[i]), 1);
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&p_full[i]), 128);
      mbar_init(smem_u32(&pv_done[i]), 1);
    }
    *fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (s_unit[5] < 0) return;                      // no unit for this CTA
  const bool split = s_unit[5] != 0;              // partial of a split tile
  const int b = s_unit[0], g = s_unit[1], t = s_unit[2], jb = s_unit[3], je = s_unit[4];
  const int64_t pslot = s_unit[6];
  const int nb = je - jb;                         // key blocks of this unit
  const AttnReq &R = P.r[b];
  const int row0 = R.q_begin + t * P.QT;          // first q row of the tile
  const int n_valid = min(P.QT, R.q_end - row0);  // q rows of the request in the tile
  if (nb == 0) {
    // a key chunk past the tile's last query: an empty partial, nothing else
    if (split && threadIdx.x < 128 && (int)threadIdx.x % P.QT < n_valid)
      part_ml[pslot * 128 + threadIdx.x] = make_float2(-INFINITY, 0.f);
    return;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane < 2) {
    // ----------------------------------------------- producers (K: lane 0, V: lane 1)
    const CUtensorMap *map = lane == 0 ? &mapK : &mapV;
    uint64_t *full = lane == 0 ? k_full : v_full;
    uint64_t *empty = lane == 0 ? k_empty : v_empty;
    const int off = lane == 0 ? kOffK : kOffV;
    if (lane == 0) {
      const uint32_t qb = smem_u32(q_full);
      expect_tx(qb, kQ);
      for (int h = 0; h < P.G; ++h)
        for (int half = 0; half < 2; ++half)
          tma_load_2d(smem_u32(smem + half * kAtom + h * P.QT * 128), &mapQ, qb,
                      (g * P.G + h) * HD + half * 64, row0);
    }
    for (int j = 0; j < nb; ++j) {
      const int sl = j & 1;
      if (!mbar_wait_bounded(smem_u32(&empty[sl]), ((j >> 1) & 1) ^ 1, kWaitLimitNs, status) ||
          *fail) {
        *fail = 1;
        break;
      }
      const uint32_t fb = smem_u32(&full[sl]);
      expect_tx(fb, kKV);
      const int key_row = (int)R.kv_row0 + (jb + j) * BN;
      for (int half = 0; half < 2; ++half)
        tma_load_2d(smem_u32(smem + off + sl * kKV + half * kAtomKV), map, fb,
                    g * HD + half * 64, key_row);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    // The warp waits converged and one elected lane issues: tcgen05.mma from
    // a lone diverged lane costs several times more issue time.
    const uint32_t idS = idesc(false, BN), idPV = idesc(true, HD);
    const uint32_t q_addr = smem_u32(smem);
    auto wait_all = [&](uint64_t *b, uint32_t ph) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(b), ph, kWaitLimitNs, status));
    };
    bool ok = wait_all(q_full, 0);
    // S_j into slot j & 1; the slot held P_{j-2}, so P_{j-2} V_{j-2} must be done
    auto issue_s = [&](int j) -> bool {
      const int sl = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!wait_all(&k_full[sl], ph)) return false;
      if (j >= 2 && !wait_all(&pv_done[sl], ph ^ 1)) return false;
      fence_after();
      if (tcx::elect_one()) {
        const uint32_t k_addr = smem_u32(smem + kOffK + sl * kKV);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t qo = (k >> 2) * kAtom + (k & 3) * 32;
          const uint32_t ko = (k >> 2) * kAtomKV + (k & 3) * 32;
          mma(tmem + sl * BN, desc_kmajor(q_addr + qo), desc_kmajor(k_addr + ko), idS, k > 0);
        }
        commit(smem_u32(&s_full[sl]));
        commit(smem_u32(&k_empty[sl]));
      }
      __syncwarp();
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int j = 0; j < nb && ok; ++j) {
      if (__any_sync(0xffffffffu, *fail != 0)) break;
      const int sl = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (j + 1 < nb && !issue_s(j + 1)) { ok = false; break; }
      if (!wait_all(&p_full[sl], ph) || !wait_all(&v_full[sl], ph)) {
        ok = false;
        break;
      }
      fence_after();
      if (tcx::elect_one()) {
        const uint32_t v_addr = smem_u32(smem + kOffV + sl * kKV);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts(tmem + 2 * BN, tmem + sl * BN + k * 8,
                 desc_mnmajor(v_addr + k * 16 * 128, kAtomKV), idPV,
                 (j > 0 || k > 0) ? 1u : 0u);
        commit(smem_u32(&pv_done[sl]));
        commit(smem_u32(&v_empty[sl]));
      }
      __syncwarp();
    }
    if (!ok && lane == 0) *fail = 1;
  } else if (warp >= 2) {
    // ------------------------------------------------------------- softmax
    const int quad = warp & 3;
    const int row = quad * 32 + lane;             // MMA row = h * QT + qi
    const int h = row / P.QT, qi = row % P.QT;
    const bool valid = qi < n_valid;
    int p = valid ? q_pos[row0 + qi] : 0;
    if (p < 0 || p >= R.kv_len) p = 0;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t obase = tmem + lane_off + 2 * BN;
    float m = -INFINITY, l = 0.f;                 // reference max (log2 domain), sum
    const float sl2 = P.scale_log2;
    bool failed = false;
    auto pv_landed = [&](int j) -> bool {
      const bool bad = !mbar_wait_bounded(smem_u32(&pv_done[j & 1]), (j >> 1) & 1,
                                          kWaitLimitNs, status) || *fail;
      if (__any_sync(0xffffffffu, bad)) return false;
      fence_after();
      return true;
    };
    for (int j = 0; j < nb; ++j) {
      const int sl = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      const bool bad =
          !mbar_wait_bounded(smem_u32(&s_full[sl]), ph, kWaitLimitNs, status) || *fail;
      if (__any_sync(0xffffffffu, bad)) { failed = true; break; }
      fence_after();
      const uint32_t sbase = tmem + lane_off + sl * BN;
      const int key0 = (jb + j) * BN;
      // Keys visible to this row: key0 .. p.  Blocks wholly at or before p
      // take the mask-free path.  Four partial maxima / sums keep the
      // dependency chains short.
      const int n_vis = p - key0 + 1;               // >= BN: no masking
      float x[BN];
      ld32_nw(sbase, x);
      ld32_nw(sbase + 32, x + 32);
      wait_ld();
      float mx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
      if (n_vis >= BN) {
#pragma unroll
        for (int i = 0; i < BN; i += 8) {
          mx[0] = max3(mx[0], x[i], x[i + 1]);
          mx[1] = max3(mx[1], x[i + 2], x[i + 3]);
          mx[2] = max3(mx[2], x[i + 4], x[i + 5]);
          mx[3] = max3(mx[3], x[i + 6], x[i + 7]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < BN; ++i)
          if (i < n_vis) mx[i & 3] = fmaxf(mx[i & 3], x[i]);
      }
      const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
      // move the reference only for a large rise; the first visible key
      // always sets it (m = -inf before)
      const bool move = mloc > m + kRescale;
      const bool rescale = move && m != -INFINITY;  // O and l hold earlier blocks
      if (__any_sync(0xffffffffu, rescale) && j > 0) {
        // O must hold P_{j-1} V_{j-1} first; the TMEM loads / stores are
        // warp-wide, rows that keep m scale by 1
        if (!pv_landed(j - 1)) { failed = true; break; }
        const float corr = rescale ? fast_exp2(m - mloc) : 1.f;
#pragma unroll 1
        for (int c = 0; c < HD; c += 32) {
          float y[32];
          ld32(obase + c, y);
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] *= corr;
          st32(obase + c, y);
        }
        l *= corr;
      }
      if (move) m = mloc;
      // P_j for keys c..c+31 -> slot columns c/2 .. c/2+15 (S_j is in
      // registers); the scale-and-shift and the sums run on packed pairs
      const unsigned long long s2 = pack2(sl2, sl2), nm2 = pack2(-m, -m);
      unsigned long long ls2[2] = {0ull, 0ull};
#pragma unroll
      for (int c = 0; c < BN; c += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const unsigned long long a = fma2(pack2(x[c + i], x[c + i + 1]), s2, nm2);
          float p0 = fast_exp2(lo2(a));
          float p1 = fast_exp2(hi2(a));
          if (n_vis < BN) {
            p0 = c + i < n_vis ? p0 : 0.f;
            p1 = c + i + 1 < n_vis ? p1 : 0.f;
          }
          ls2[(i >> 1) & 1] = add2(ls2[(i >> 1) & 1], pack2(p0, p1));
          __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
          pk[i / 2] = *reinterpret_cast<uint32_t *>(&v2);
        }
        st16(sbase + c / 2, pk);
      }
      wait_st();
      l += (lo2(ls2[0]) + hi2(ls2[0])) + (lo2(ls2[1]) + hi2(ls2[1]));
      fence_before();
      arrive(smem_u32(&p_full[sl]));
    }
    // the whole key range is in O once the last P V has landed
    if (!failed && !pv_landed(nb - 1)) failed = true;
    if (failed) *fail = 1;
    const bool ok = !failed && !*fail;
    if (__any_sync(0xffffffffu, ok)) {
      // O chunks straight from TMEM to the output (warp-wide loads)
      const int q_row = row0 + qi, head = g * P.G + h;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t slot = pslot * 128 + row;
#pragma unroll 1
      for (int c = 0; c < HD; c += 32) {
        float o[32];
        ld32(obase + c, o);
        if (!(valid && ok)) continue;
        // the output row, or this key chunk's normalised partial (bf16, with
        // its (m, l) beside it for the combine)
        bf16 *dst = split ? part_o + slot * HD + c : out + (int64_t)q_row * ld_out + head * HD + c;
#pragma unroll
        for (int c8 = 0; c8 < 32; c8 += 8) {
          uint4 pk;
          __nv_bfloat162 *e = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            e[i] = __floats2bfloat162_rn(o[c8 + 2 * i] * inv, o[c8 + 2 * i + 1] * inv);
          *reinterpret_cast<uint4 *>(dst + c8) = pk;
        }
      }
      if (valid && ok && split) part_ml[slot] = make_float2(m, l);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *fail) {
    // drain the K/V copies this CTA may still have in flight
    for (int i = 0; i < 2; ++i) {
      mbar_wait_bounded(smem_u32(&k_full[i]), 0, 10000000ull, nullptr);
      mbar_wait_bounded(smem_u32(&v_full[i]), 0, 10000000ull, nullptr);
    }
  }
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// Merges the key-chunk partials of every (query row, q head).  A CTA of
// eight warps takes 32 rows of a tile, four per warp, and issues the loads
// of all four rows before using them; each lane owns four of the 128 output
// dimensions, so every partial row (bf16) is read as one coalesced 256-byte
// access.
constexpr int kCombineRows = 4;            // rows per warp
__global__ void __launch_bounds__(256)
attn_combine_kernel(const __grid_constant__ Params P, const bf16 *__restrict__ part_o,
                    const float2 *__restrict__ part_ml, bf16 *__restrict__ out, int64_t ld_out) {
  grid_dep_wait();
  grid_dep_launch();
  const int tile = blockIdx.x / 4;
  const int lane = threadIdx.x & 31;
  const int row_base = (blockIdx.x % 4) * 32 + (threadIdx.x >> 5);   // rows row_base + 8 r
  // the tile's partial units: consecutive slots from `first`
  int first = tile * P.n_chunks, count = P.n_chunks;
  if (P.plan) {
    first = P.plan[4 + 2 * tile];
    count = P.plan[5 + 2 * tile];
    if (count <= 1) return;                       // written directly by its unit
  }
  const TileId id = decode_tile(P, tile);
  const AttnReq &R = P.r[id.b];
  const int row0 = R.q_begin + id.t * P.QT;
  const int n_valid = min(P.QT, R.q_end - row0);
  // lane c holds partial c's (m, l) of each row: the weights come from warp
  // reductions, then the partial rows are read back to back
  float M[kCombineRows], l[kCombineRows];
  float4 o[kCombineRows];
#pragma unroll
  for (int r = 0; r < kCombineRows; ++r) {
    M[r] = -INFINITY;
    l[r] = 0.f;
    o[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int c = lane; c < count; c += 32) {
#pragma unroll
    for (int r = 0; r < kCombineRows; ++r)
      M[r] = fmaxf(M[r], part_ml[((int64_t)first + c) * 128 + row_base + 8 * r].x);
  }
#pragma unroll
  for (int r = 0; r < kCombineRows; ++r)
    for (int s = 16; s; s >>= 1) M[r] = fmaxf(M[r], __shfl_xor_sync(0xffffffffu, M[r], s));
  for (int c0 = 0; c0 < count; c0 += 32) {
    float w[kCombineRows];
#pragma unroll
    for (int r = 0; r < kCombineRows; ++r) {
      const float2 ml = c0 + lane < count
                            ? part_ml[((int64_t)first + c0 + lane) * 128 + row_base + 8 * r]
                            : make_float2(-INFINITY, 0.f);
      // a chunk's weight is its sum l rescaled to the common maximum (its
      // partial is already divided by l); an empty chunk has none
      w[r] = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M[r]) * ml.y;
      l[r] += w[r];
    }
    const int n = min(32, count - c0);
    for (int i = 0; i < n; ++i) {
#pragma unroll
      for (int r = 0; r < kCombineRows; ++r) {
        const float wi = __shfl_sync(0xffffffffu, w[r], i);
        if (wi != 0.f) {
          const uint2 raw = reinterpret_cast<const uint2 *>(
              part_o + (((int64_t)first + c0 + i) * 128 + row_base + 8 * r) * HD)[lane];
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
          const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
          o[r].x += wi * a.x; o[r].y += wi * a.y; o[r].z += wi * b.x; o[r].w += wi * b.y;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kCombineRows; ++r) {
    for (int s = 16; s; s >>= 1) l[r] += __shfl_xor_sync(0xffffffffu, l[r], s);
    const int row = row_base + 8 * r;
    const int h = row / P.QT, qi = row % P.QT;
    if (qi >= n_valid) continue;
    const float inv = 1.f / l[r];
    bf16 *dst = out + (int64_t)(row0 + qi) * ld_out + (id.g * P.G + h) * HD + lane * 4;
    __nv_bfloat162 lo = __floats2bfloat162_rn(o[r].x * inv, o[r].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(o[r].z * inv, o[r].w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(dst) = pk;
  }
}

// ------------------------------------------------------------------ host --
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static bool make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                     int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() { return device_sm_count(); }

// Tiles of a call and the key-range split: tiles that alone fill fewer than
// all SMs get their key blocks split into chunks so that about two waves of
// CTAs run; chunks past a tile's last query position exit at once.  A chunk
// holds at least kMinChunkBlocks blocks: a CTA's fixed cost (set-up, first
// loads, writing O) is worth about six blocks of its loop, and a split also
// needs the combine, so shorter ranges run unsplit.
constexpr int kMinChunkBlocks = 8;
static void plan_split(Params &P, const AttnReq *reqs, int n_req, int Hq, int Hkv) {
  P.n_req = n_req;
  P.plan = nullptr;
  P.G = Hq / Hkv;
  P.QT = 128 / P.G;
  P.Hkv = Hkv;
  P.tile_off[0] = 0;
  int max_nb = 0;
  for (int i = 0; i < n_req; ++i) {
    P.r[i] = reqs[i];
    const int n = reqs[i].q_end - reqs[i].q_begin;
    P.tile_off[i + 1] = P.tile_off[i] + Hkv * ((n + P.QT - 1) / P.QT);
    const int nb = (reqs[i].kv_len + BN - 1) / BN;
    if (n > 0 && nb > max_nb) max_nb = nb;
  }
  const int tiles = P.tile_off[n_req];
  P.n_chunks = 1;
  P.chunk_blocks = max_nb > 0 ? max_nb : 1;
  const int sms = num_sms();
  const int slots = kCtasPerSm * sms;            // CTAs resident at once
  if (tiles > 0 && tiles < slots && max_nb > kMinChunkBlocks) {
    int want = (2 * slots + tiles - 1) / tiles;
    if (want > max_nb) want = max_nb;
    P.chunk_blocks = max((max_nb + want - 1) / want, kMinChunkBlocks);
    P.n_chunks = (max_nb + P.chunk_blocks - 1) / P.chunk_blocks;
  }
}

constexpr size_t kPartBytes = 128 * (HD * sizeof(bf16) + sizeof(float2));

}  // namespace attn

bool attention_tc_supported(int Hq, int Hkv, int hd) {
  if (hd != attn::HD || Hq % Hkv) return false;
  const int G = Hq / Hkv;
  return G == 1 || G == 2 || G == 4 || G == 8;
}

// tiles * chunks < 2 slots + tiles < 3 slots whenever the key range is split
size_t attention_tc_ws_bound() {
  return (size_t)3 * attn::kCtasPerSm * attn::num_sms() * attn::kPartBytes + 256;
}

size_t attention_plan_bytes(const AttnReq *reqs, int n_req, int Hq, int Hkv) {
  attn::Params P;
  attn::plan_split(P, reqs, n_req, Hq, Hkv);
  const int tiles = P.tile_off[n_req];
  const int slots = attn::kCtasPerSm * attn::num_sms();
  return attn::plan_units_off(tiles) + (size_t)16 * (tiles > slots ? tiles : slots) + 256;
}

cudaError_t launch_attention_plan(const int32_t *q_pos, const AttnReq *reqs, int n_req, int Hq,
                                  int Hkv, int *plan, size_t plan_bytes, cudaStream_t s) {
  using namespace attn;
  Params P;
  plan_split(P, reqs, n_req, Hq, Hkv);
  if (!plan || plan_bytes < attention_plan_bytes(reqs, n_req, Hq, Hkv))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(attn_plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, P, q_pos,
                             kCtasPerSm * num_sms(), plan);
  if (e != cudaSuccess) return e;
  return launched(1);
}

size_t attention_tc_ws_bytes(const AttnReq *reqs, int n_req, int Hq, int Hkv) {
  attn::Params P;
  attn::plan_split(P, reqs, n_req, Hq, Hkv);
  if (P.n_chunks == 1) return 0;
  return (size_t)P.tile_off[n_req] * P.n_chunks * attn::kPartBytes + 256;
}

cudaError_t launch_attention_tc(const void *q, int64_t ld_q, const int32_t *q_pos,
                                const AttnReq *reqs, int n_req, const void *k_cache,
                                const void *v_cache, int64_t ld_kv, int Hq, int Hkv,
                                float scale, void *out, int64_t ld_out, void *ws,
                                size_t ws_bytes, int *status, cudaStream_t s, const int *plan) {
  using namespace attn;
  Params P;
  plan_split(P, reqs, n_req, Hq, Hkv);
  P.plan = plan;
  P.scale_log2 = scale * 1.4426950408889634f;
  int64_t q_rows = 0, kv_rows = 0;
  for (int i = 0; i < n_req; ++i) {
    if (reqs[i].q_end > q_rows) q_rows = reqs[i].q_end;
    if (reqs[i].kv_row0 + reqs[i].kv_len > kv_rows) kv_rows = reqs[i].kv_row0 + reqs[i].kv_len;
  }
  const int tiles = P.tile_off[n_req];
  if (tiles == 0) return cudaSuccess;
  // CTAs and partial slots: with a unit table, one wave of slots (or one
  // unit per tile when the tiles alone fill the slots); else tiles x chunks
  const int slots = kCtasPerSm * num_sms();
  const int grid = plan ? (tiles > slots ? tiles : slots) : tiles * P.n_chunks;
  const bool split = plan ? tiles < slots : P.n_chunks > 1;
  bf16 *part_o = nullptr;
  float2 *part_ml = nullptr;
  if (split) {
    const size_t need = (size_t)grid * kPartBytes;
    if (!ws || ws_bytes < need) return cudaErrorInvalidValue;
    part_o = reinterpret_cast<bf16 *>(ws);
    part_ml = reinterpret_cast<float2 *>(reinterpret_cast<char *>(ws) +
                                         (size_t)grid * 128 * HD * sizeof(bf16));
  }
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, q_rows, (int64_t)Hq * HD, ld_q, P.QT) ||
      !make_map(&mk, k_cache, kv_rows, (int64_t)Hkv * HD, ld_kv, BN) ||
      !make_map(&mv, v_cache, kv_rows, (int64_t)Hkv * HD, ld_kv, BN))
    return cudaErrorInvalidValue;
  static PerDeviceOnce attr;
  cudaError_t e = attr.run([](int) {
    return cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_tc_kernel, dim3(grid), dim3(kThreads), kSmem, s,
                             mq, mk, mv, P, q_pos, reinterpret_cast<bf16 *>(out), ld_out, part_o,
                             part_ml, status);
  if (e != cudaSuccess) return e;
  if (!split) return launched(1);
  e = launch_pdl(attn_combine_kernel, dim3(tiles * 4), dim3(256), 0, s, P,
                 (const bf16 *)part_o, (const float2 *)part_ml, reinterpret_cast<bf16 *>(out),
                 ld_out);
  if (e != cudaSuccess) return e;
  return launched(2);
}

}  // namespace cb
