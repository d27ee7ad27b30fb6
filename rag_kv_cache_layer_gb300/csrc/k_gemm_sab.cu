// bf16 tcgen05 GEMM for few rows (the compact layers' ~500 rows), operands
// swapped: out[tok][f] = epi(sum_k A[tok][k] W[f][k]) is computed as
// D[f][tok] = W_tile A_tile^T with the 128 weight rows of a tile as the MMA's
// M side and the tokens as its N side (N = BT, a multiple of 16 up to 256).
// Splitting M_tok rows into ceil(M_tok / 256) token tiles of equal width
// (176 for 524 rows) wastes 1% of the work where 128-row tiles waste 18%.
//
// Roles: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps 2..9
// epilogue in two groups of four (warps 2..5 and 6..9, each covering the
// four TMEM lane quarters) that take alternate 32-token chunks of a tile,
// each with its own transpose buffer; the fp32 accumulator [128 features][BT
// tokens] is double-buffered in TMEM (columns 0 and 256).  Epilogue thread r
// of a group owns feature r of the tile, so for every token the 32 lanes of
// a warp write 32 consecutive features.  Two epilogues pair feature r with r + 64
// through a shared-memory exchange: SwiGLU (tile rows 0..63 are W_gate rows,
// 64..127 the matching W_up rows) and the QKV RoPE (rotate-half pairs
// (e, e + 64) of a 128-wide head).  The key-deviation epilogue rotates the
// same way and, instead of storing the keys, compares each token's head with
// the reused key in the fused cache and leaves the head's squared
// difference.  Residual outputs may use stream-K.
// Other outputs may split the tiles of a partial last wave along K: the
// units that run the later k-segments leave fp32 partials in a workspace
// and the unit that runs segment 0 adds them, in segment order, before its
// epilogue.
#include <type_traits>

#include "cb_internal.h"
#include "cb_tc.cuh"

namespace cb {
namespace sab {

using namespace tcx;

constexpr int FM = 128;                      // weight rows per tile
constexpr int BK = 64;
constexpr int kThreads = 320;
constexpr int kTileW = FM * BK * 2;          // 16 KB
constexpr int kTrStride = 132;               // floats per transposed token row
constexpr int kTr = 32 * kTrStride * 4;      // 32 tokens x 128 features, fp32
constexpr int kTokTab = 256 * 16;            // Q/K/V, K-deviation: positions, cache rows, d index
constexpr int kSmemMax = 232448;
constexpr int kPartFloats = 8 * FM * 32;     // one CTA's partial: 8 chunks x 128 features x 32 tokens
constexpr int kSplitFlagBytes = 4096;       // arrival counters: one per tail tile and CTA (<= SMs)
constexpr int kMlpFlags = 16384;            // fused MLP: one flag per (gate/up CTA tile, token tile)
// Epilogues that take the tail split (the residual one uses stream-K), and
// the kernel compiled with it.  The Q/K/V epilogue is at its register limit
// (168 for 320 threads): it has a second instantiation with the split, used
// only by launches that do split, so that the others keep their registers.
template <int EPI>
constexpr bool can_split() { return EPI != EPI_RESID && EPI != EPI_KDEV; }
template <int EPI>
constexpr bool split_by_default() { return can_split<EPI>() && EPI != EPI_QKV; }

struct Params {
  int M, N, K;           // tokens, output features, reduction
  int BT, n_tt, n_ft;    // token tile width, token tiles, feature tiles
  int stream_k;
  // stream-K with defer: a range that crosses a weight tile's end runs the
  // part after the crossing first (the fused MLP's down projection, whose
  // last k-blocks wait for the last gate/up tiles)
  int defer;
  // tail split: tiles [0, n_whole) run whole; every later tile runs as
  // `split` k-segments on as many units (split = 1: no split).  tail_first:
  // the split tiles are [0, n_tail) instead and the whole ones follow, so
  // the last tiles to finish hold the highest features (the fused MLP)
  int n_whole, split, tail_first;
  float *part;           // [tail tile][segment][CG][kPartFloats] partials
  int *flag;             // [tail tile][CG] arrivals of segments 1.., zero between launches
  int stages, stage_bytes;
  uint32_t idesc;
  // epilogue
  void *out;
  int64_t ldo;
  const int32_t *pos, *dst_row, *dev_idx;
  void *k_cache, *v_cache;
  int64_t ld_kv;
  const float2 *rope;
  int Hq, Hkv;
  // fused MLP: flag[fct * n_tt + tt] = epoch once gate/up CTA tile fct has
  // written its 64 features of token tile tt
  int *mlp_flag;
  int epoch;
};

// Work decomposition.  Whole tiles: tile index with the token tile fastest,
// so the CTAs running together share a weight tile.  Stream-K: the grid is
// n_tt-CTA groups; group g owns a contiguous range of the n_ft x num_kb
// (weight tile, k-block) units and each CTA of the group runs that range
// for its own token tile, so the group reads every weight tile at the same
// time and HBM serves it once (the other n_tt - 1 reads hit L2).
// Whole tiles with a tail split: item j * split + g (< n_seg) is k-segment g
// of tile n_whole + j, and item n_seg + i is whole tile i.  The segments
// come first, at most one per unit, so those of a tile start together on
// different units and the fixup of segment 0 overlaps its unit's next tile
// (the accumulator is double-buffered).  n_whole is a multiple of the unit
// count, so every unit still ends after the same number of whole tiles.
// A "unit" is one CTA, or one CTA pair when the MMA spans two SMs (CG = 2);
// both CTAs of a pair walk the same sequence, ft then counting pair tiles.
// With tail_first the split tiles are the first n_tail tiles.  With defer
// (stream-K) a range that starts inside a weight tile and runs past its end
// takes the part after that end first and the first part last.
template <int CG, bool EXT = false>   // EXT: tail_first and defer are read (the fused MLP)
struct Work {
  int n_tt, num_kb, my_tt;
  bool sk, tail_first;
  int n_whole, split;
  int seg, tj;           // tail split: k-segment of the current item (-1: whole) and tail tile
  int64_t n_seg, n_tail; // items that are k-segments; tiles that are split
  int64_t w, w_end, step;
  int64_t dw0, dw1;      // stream-K: the deferred first part of the range
  __device__ Work(const Params &p, int num_kb_)
      : n_tt(p.n_tt), num_kb(num_kb_), sk(p.stream_k != 0), tail_first(EXT && p.tail_first != 0),
        n_whole(p.n_whole), split(p.split), seg(-1), tj(0), n_seg(0), n_tail(0), dw0(0), dw1(0) {
    const int unit = blockIdx.x / CG, n_units = gridDim.x / CG;
    const int n_ft = (p.n_ft + CG - 1) / CG;
    step = n_units;
    if (sk) {
      const int64_t total = (int64_t)n_ft * num_kb_;
      int64_t groups = n_units / p.n_tt;
      if (groups > total) groups = total;
      const int g = unit / p.n_tt;
      my_tt = unit % p.n_tt;
      w = g < groups ? total * g / groups : 0;
      w_end = g < groups ? total * (g + 1) / groups : 0;
      if (EXT && p.defer && w < w_end && w % num_kb_) {
        const int64_t cross = (w / num_kb_ + 1) * num_kb_;
        if (cross < w_end) {
          dw0 = w;
          dw1 = cross;
          w = cross;
        }
      }
    } else {
      my_tt = 0;
      w = unit;
      n_tail = split > 1 ? (int64_t)p.n_tt * n_ft - n_whole : 0;
      n_seg = n_tail * split;
      w_end = n_seg + n_whole;
    }
  }
  __device__ bool next(int &tt, int &ft, int &kb0, int &kb1) {
    if (w >= w_end) {
      if (!EXT || dw0 >= dw1) return false;
      w = dw0;
      w_end = dw1;
      dw0 = dw1;
    }
    if (sk) {
      ft = (int)(w / num_kb);
      kb0 = (int)(w % num_kb);
      const int64_t left = w_end - w;
      kb1 = (int)(kb0 + left < num_kb ? kb0 + left : num_kb);
      w += kb1 - kb0;
      tt = my_tt;
    } else {
      int64_t tile = w - n_seg + (tail_first ? n_tail : 0);
      kb0 = 0;
      kb1 = num_kb;
      seg = -1;
      if (w < n_seg) {
        tj = (int)(w / split);
        seg = (int)(w % split);
        tile = tail_first ? tj : n_whole + tj;
        kb0 = num_kb * seg / split;
        kb1 = num_kb * (seg + 1) / split;
      }
      tt = (int)(tile % n_tt);
      ft = (int)(tile / n_tt);
      w += step;
    }
    return true;
  }
};

// Barriers of one epilogue group (128 threads) and of all eight epilogue warps.
__device__ __forceinline__ void epi_bar(int grp) {
  if (grp == 0) asm volatile("bar.sync 1, 128;" ::: "memory");
  else asm volatile("bar.sync 2, 128;" ::: "memory");
}
__device__ __forceinline__ void epi_all_bar() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

// Arrival counters of the tail split (global memory, GPU scope).
__device__ __forceinline__ void signal_add(int *flag) {
  asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(flag) : "memory");
}
__device__ __forceinline__ int load_acquire(const int *flag) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  return v;
}
// Waits until *flag == want; false (after recording CB_ERR_TIMEOUT) past the limit.
__device__ __forceinline__ bool flag_wait_bounded(const int *flag, int want, uint64_t limit_ns,
                                                  int *status) {
  if (load_acquire(flag) == want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (load_acquire(flag) == want) return true;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > limit_ns) {
      report(status, CB_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ int load_relaxed(const int *flag) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  return v;
}
// Fused MLP, down projection: waits until the k-block kb of its token tile
// has been written by the gate/up tile (flag[kb * stride] >= epoch), looking
// ahead over at most 256 k-blocks in one round of loads; returns the end of
// the run of written k-blocks from kb (<= kb1), or -1 (after recording
// CB_ERR_TIMEOUT) past the limit.  Called by a whole warp; the acquire and
// proxy fences order the TMA loads that follow after the flags.
__device__ int wait_written(const int *flag, int stride, int kb, int kb1, int epoch,
                            int *status) {
  const int lane = threadIdx.x & 31;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (it > 0) {
      // until kb itself is written, one lane polls it alone (the whole
      // warp's look-ahead loads would load L2 while gate/up tiles stream)
      for (uint32_t w = 0;; ++w) {
        int f = 0;
        if (lane == 0) f = load_relaxed(flag + (int64_t)kb * stride);
        if (__shfl_sync(0xffffffffu, f, 0) >= epoch) break;
        if ((w & 15u) == 15u && globaltimer_ns() - t0 > kWaitLimitNs) {
          if (lane == 0) report(status, CB_ERR_TIMEOUT);
          return -1;
        }
        __nanosleep(256);
      }
    }
    int v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = kb + 32 * j + lane;
      v[j] = i < kb1 ? load_relaxed(flag + (int64_t)i * stride) : epoch;
    }
    int end = kb1 < kb + 256 ? kb1 : kb + 256;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      const unsigned nw = __ballot_sync(0xffffffffu, v[j] < epoch);
      if (nw) end = kb + 32 * j + __ffs(nw) - 1;
    }
    if (end > kb) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return end;
    }
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      if (lane == 0) report(status, CB_ERR_TIMEOUT);
      return -1;
    }
  }
}

__device__ __forceinline__ void store_bf16x8(bf16 *dst, const float *v) {
  uint4 pk;
  __nv_bfloat162 *e = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
  for (int i = 0; i < 4; ++i) e[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(dst) = pk;
}

// The phase's operand (p and the maps of phase 0, or p2 and those of phase
// 1), chosen at compile time: each role's loop is instantiated per phase.
template <int PH, typename T>
__device__ __forceinline__ const T &pick(const T &a, const T &b) {
  if constexpr (PH == 0) return a;
  else return b;
}
template <int PH>
__device__ __forceinline__ const CUtensorMap *pick(const CUtensorMap *a, const CUtensorMap *b) {
  if constexpr (PH == 0) return a;
  else return b;
}

// The kernel body.  EPI_MLP runs two GEMMs one after the other on the same
// units, pipeline stages and accumulators: phase 0 the gate/up projection
// (mapX, mapW, mapW2, p; SwiGLU epilogue), phase 1 the down projection
// (mapX2 over phase 0's output, mapW3, p2; residual epilogue, stream-K).
// The other epilogues run phase 0 only.
template <int EPI, int CG, bool TS>
__device__ __forceinline__ void gemm_body(const CUtensorMap *mapX, const CUtensorMap *mapW,
                                          const CUtensorMap *mapW2, const CUtensorMap *mapX2,
                                          const CUtensorMap *mapW3, const Params &p,
                                          const Params &p2, int *status) {
  constexpr bool MLP = EPI == EPI_MLP;
  constexpr int kPhases = MLP ? 2 : 1;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.stages * p.stage_bytes + 2 * kTr);
  int64_t *s_dst = reinterpret_cast<int64_t *>(smem + p.stages * p.stage_bytes + 2 * kTr + 256);
  int32_t *s_pos = reinterpret_cast<int32_t *>(s_dst + 256);
  int32_t *s_dev = s_pos + 256;                  // EPI_KDEV: deviation index (-1: none)
  uint64_t *full = bars;                 // [stages]
  uint64_t *empty = bars + 8;            // [stages]
  uint64_t *tfull = bars + 16;           // [2]
  uint64_t *tempty = bars + 18;          // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 20);
  volatile int *fail = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // epilogue stop votes [tile parity][epilogue warp] (bytes 192..255 of the barrier area)
  volatile int *vote = reinterpret_cast<volatile int *>(bars + 24);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CG = 2: this CTA's rank in its pair; the leader (rank 0) issues the MMAs
  const uint32_t rank = CG == 2 ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      // CG = 2: lane 0 of each epilogue warp of both CTAs
      mbar_init(smem_u32(&tempty[b]), CG == 2 ? 16 : 256);
    }
    *fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if (CG == 2) tmem_alloc_pair(smem_u32(tmem_slot), 512);
    else tmem_alloc(smem_u32(tmem_slot), 512);
  }
  fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();   // the peer's barriers exist before any remote use
  fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();      // inputs of the previous kernel are visible from here
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The warp runs the loop converged; the elected lane issues the copies.
    int stage = 0;
    uint32_t phase = 0;
    int issued[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    bool ok = true;
    auto produce = [&](auto phase_c) {
      constexpr int ph = decltype(phase_c)::value;
      const Params &pq = pick<ph>(p, p2);
      const CUtensorMap *mx = pick<ph>(mapX, mapX2), *mw = pick<ph>(mapW, mapW3);
      const bool swiglu = MLP ? ph == 0 : EPI == EPI_SWIGLU;
      const bool gated = MLP && ph == 1;    // B rows come from phase 0 of this launch
      const int num_kb = (pq.K + BK - 1) / BK;
      Work<CG, MLP> wk(pq, num_kb);
      int tt, ft, kb0, kb1;
      const int bt = pq.BT / CG;             // token rows of B held by this CTA
      while (ok && wk.next(tt, ft, kb0, kb1)) {
        const int fct = ft * CG + (int)rank;   // this CTA's 128-row weight tile
        const int ty = tt * pq.BT + (int)rank * bt;
        int written = gated ? kb0 : kb1;       // B k-blocks known to be written
        for (int kb = kb0; kb < kb1; ++kb) {
          const bool got =
              mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, kWaitLimitNs, status) && !*fail;
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          // the pair's operands all complete on the leader's barrier
          uint32_t fb = smem_u32(&full[stage]);
          if (CG == 2) fb = map_to_rank(fb, 0);
          uint8_t *sw = smem + stage * p.stage_bytes;
          uint8_t *sx = sw + kTileW;
          // a gated k-block whose token rows are not yet known to be written
          // issues its weights first and waits for the gate/up tile after
          const bool wait_x = gated && kb >= written;
          if (elect_one()) {
            if (leader) expect_tx(smem_u32(&full[stage]), CG * p.stage_bytes);
            if (CG == 2) {
              if (swiglu) {
                tma_load_2d_pair(smem_u32(sw), mw, fb, kb * BK, fct * 64);
                tma_load_2d_pair(smem_u32(sw + 64 * 128), mapW2, fb, kb * BK, fct * 64);
              } else {
                tma_load_2d_pair(smem_u32(sw), mw, fb, kb * BK, fct * FM);
              }
              if (!wait_x) tma_load_2d_pair(smem_u32(sx), mx, fb, kb * BK, ty);
            } else {
              if (swiglu) {
                tma_load_2d(smem_u32(sw), mw, fb, kb * BK, fct * 64);
                tma_load_2d(smem_u32(sw + 64 * 128), mapW2, fb, kb * BK, fct * 64);
              } else {
                tma_load_2d(smem_u32(sw), mw, fb, kb * BK, fct * FM);
              }
              if (!wait_x) tma_load_2d(smem_u32(sx), mx, fb, kb * BK, ty);
            }
          }
          __syncwarp();
          if (wait_x) {
            written = wait_written(pq.mlp_flag + tt, pq.n_tt, kb, kb1, pq.epoch, status);
            if (!__all_sync(0xffffffffu, written > kb && !*fail)) {
              ok = false;
              ++issued[stage];     // the weight copy above completes on this stage's barrier
              break;
            }
            if (elect_one()) {
              if (CG == 2) tma_load_2d_pair(smem_u32(sx), mx, fb, kb * BK, ty);
              else tma_load_2d(smem_u32(sx), mx, fb, kb * BK, ty);
            }
            __syncwarp();
          }
          ++issued[stage];
          if (++stage == p.stages) { stage = 0; phase ^= 1; }
        }
      }
    };
    produce(std::integral_constant<int, 0>());
    if constexpr (kPhases > 1) {
      if (ok) produce(std::integral_constant<int, 1>());
    }
    if (!ok && lane == 0) {
      *fail = 1;
      if (CG == 1 || leader) {
        for (int s = 0; s < p.stages; ++s)
          if (issued[s] > 0)
            mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((issued[s] - 1) & 1), 10000000ull,
                              nullptr);
      } else {
        // this CTA's copies complete on the leader's barriers: give them
        // time to land before the pair can retire
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // Converged warp, elected lane issues; the failure flag is polled once
    // per tile (a stalled producer also ends the bounded waits below).
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t bphase = 0;
      bool ok = true;
      auto issue = [&](auto phase_c) {
        constexpr int ph = decltype(phase_c)::value;
        const Params &pq = pick<ph>(p, p2);
        const int num_kb = (pq.K + BK - 1) / BK;
        Work<CG, MLP> wk(pq, num_kb);
        int tt, ft, kb0, kb1;
        while (ok && wk.next(tt, ft, kb0, kb1)) {
          const bool got =
              mbar_wait_bounded(smem_u32(&tempty[buf]), bphase ^ 1, kWaitLimitNs, status) && !*fail;
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t d = tmem + buf * 256;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[stage]), phase,
                                                            kWaitLimitNs, status))) {
              ok = false;
              break;
            }
            fence_after();
            if (elect_one()) {
              const uint32_t sw = smem_u32(smem + stage * p.stage_bytes);
              const uint64_t dw = desc_kmajor(sw), dx = desc_kmajor(sw + kTileW);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                if (CG == 2)
                  mma_pair(d, dw + 2 * k, dx + 2 * k, pq.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                else
                  mma(d, dw + 2 * k, dx + 2 * k, pq.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
              }
              if (CG == 2) commit_pair(smem_u32(&empty[stage]), 3);
              else commit(smem_u32(&empty[stage]));
            }
            __syncwarp();
            if (++stage == p.stages) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          if (elect_one()) {
            if (CG == 2) commit_pair(smem_u32(&tfull[buf]), 3);
            else commit(smem_u32(&tfull[buf]));
          }
          __syncwarp();
          if (++buf == 2) { buf = 0; bphase ^= 1; }
        }
      };
      issue(std::integral_constant<int, 0>());
      if constexpr (kPhases > 1) {
        if (ok) issue(std::integral_constant<int, 1>());
      }
      if (!ok && lane == 0) *fail = 1;
    }
  } else {
    // ----------------------------------------------------------- epilogue
    // Every decision to stop is taken by all eight warps together (a vote
    // behind a barrier), so no group waits at a barrier for a warp that left.
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                 // feature row of the tile
    const int grp = (threadIdx.x - 64) >> 7;        // epilogue group 0 / 1
    const int t = (threadIdx.x - 64) & 127;         // 0..127 within the group
    float *tr = reinterpret_cast<float *>(smem + p.stages * p.stage_bytes) + grp * (kTr / 4);
    int buf = 0;
    uint32_t bphase = 0;
    int n_tile = 0;
    bool stop = false;
    auto drain = [&](auto phase_c) {
      constexpr int ph = decltype(phase_c)::value;
      const Params &pq = pick<ph>(p, p2);
      constexpr int epi = MLP ? (ph ? EPI_RESID : EPI_SWIGLU) : EPI;
      constexpr bool kSplit = TS && !(MLP && ph == 1);   // the down projection never splits
      const int num_kb = (pq.K + BK - 1) / BK;
      Work<CG, MLP> wk(pq, num_kb);
      int tt, ft, kb0, kb1;
      while (wk.next(tt, ft, kb0, kb1)) {
        const bool whole = kb0 == 0 && kb1 == num_kb;
        if (EPI == EPI_QKV || EPI == EPI_KDEV) {
          // the tile's positions and fused-cache rows, read while the MMAs run,
          // once every warp is done with the previous tile's table
          epi_all_bar();
          for (int i = threadIdx.x - 64; i < pq.BT; i += 256) {
            const int tok = tt * pq.BT + i;
            s_pos[i] = tok < pq.M ? pq.pos[tok] : 0;
            s_dst[i] = tok < pq.M ? (int64_t)pq.dst_row[tok] : 0;
            if (EPI == EPI_KDEV) s_dev[i] = tok < pq.M ? pq.dev_idx[tok] : -1;
          }
        }
        // tail split: segment 0 finishes the tile once the other segments'
        // partials have arrived; the later segments only leave partials
        const bool helper = kSplit && wk.seg > 0;
        const bool finisher = kSplit && wk.seg == 0 && wk.split > 1;
        int *flag = wk.split > 1 ? pq.flag + (int64_t)wk.tj * CG + rank : nullptr;
        bool bad_l = !mbar_wait_bounded(smem_u32(&tfull[buf]), bphase, kWaitLimitNs, status) || *fail;
        if (finisher && warp == 2 && lane == 0 && !bad_l) {
          bad_l = !flag_wait_bounded(flag, wk.split - 1, kWaitLimitNs, status);
          if (!bad_l) *flag = 0;        // every segment has arrived: ready for the next launch
        }
        const bool bad_w = __any_sync(0xffffffffu, bad_l);
        if (lane == 0) vote[(n_tile & 1) * 8 + warp - 2] = bad_w ? 1 : 0;
        epi_all_bar();               // also publishes the table to both groups
        bool bad = false;
#pragma unroll
        for (int w = 0; w < 8; ++w) bad |= vote[(n_tile & 1) * 8 + w] != 0;
        if (bad) {
          if (lane == 0) *fail = 1;
          stop = true;
          break;
        }
        ++n_tile;
        fence_after();
        ft = ft * CG + (int)rank;                      // this CTA's 128 weight rows
        const uint32_t tbase = tmem + buf * 256 + ((uint32_t)(quad * 32) << 16);
        const int tok0 = tt * pq.BT;
        int head = 0;
        bool rotate = false;
        if (EPI == EPI_QKV) {
          head = ft;
          rotate = head < pq.Hq + pq.Hkv;
        } else if (EPI == EPI_KDEV) {
          head = ft;                                   // tile h = kv head h of W_k
          rotate = true;
        }
        // this tile's partial slots: [segment][CG][kPartFloats]
        float *part = wk.split > 1 ? pq.part + ((int64_t)wk.tj * wk.split * CG + rank) * kPartFloats
                                   : nullptr;
#pragma unroll 1
        for (int c = 32 * grp; c < pq.BT; c += 64) {
          float x[32];
          tmem_ld32(tbase + c, x);
          // partial layout: [chunk][token quad v][feature] float4s, so the 32
          // lanes of a warp move 512 contiguous bytes per instruction
          const int64_t po = (int64_t)(c >> 5) * (FM * 32) + r * 4;
          if (helper) {
            float4 *dst = reinterpret_cast<float4 *>(part + (int64_t)wk.seg * CG * kPartFloats + po);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              __stcg(dst + v * FM, make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]));
            continue;
          }
          if (finisher) {
#pragma unroll 1
            for (int g = 1; g < wk.split; ++g) {
              const float4 *src =
                  reinterpret_cast<const float4 *>(part + (int64_t)g * CG * kPartFloats + po);
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const float4 a = __ldcg(src + v * FM);
                x[4 * v] += a.x;
                x[4 * v + 1] += a.y;
                x[4 * v + 2] += a.z;
                x[4 * v + 3] += a.w;
              }
            }
          }
          // Q/K heads: this thread's rotation factors for the chunk, loaded
          // before the transpose so that their latency overlaps it
          constexpr bool kRope = EPI == EPI_QKV || EPI == EPI_KDEV;
          float4 rf[kRope ? 4 : 1][kRope ? 4 : 1];
          if (kRope && rotate) {
            const int e0 = 8 * ((t & 15) & 7);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = (t >> 4) + 8 * q;
              const int ci = (c + i < pq.BT && tok0 + c + i < pq.M) ? c + i : 0;
              const float4 *src = reinterpret_cast<const float4 *>(pq.rope + (int64_t)s_pos[ci] * 64 + e0);
#pragma unroll
              for (int u = 0; u < 4; ++u) rf[q][u] = __ldg(src + u);
            }
          }
          // K-deviation: the reused keys this thread compares, also loaded
          // before the transpose
          uint4 kraw[EPI == EPI_KDEV ? 4 : 1];
          if (EPI == EPI_KDEV) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = (t >> 4) + 8 * q;
              const bool use = c + i < pq.BT && tok0 + c + i < pq.M && s_dev[c + i] >= 0;
              kraw[q] = use ? __ldg(reinterpret_cast<const uint4 *>(
                                  reinterpret_cast<const bf16 *>(pq.k_cache) + s_dst[c + i] * pq.ld_kv +
                                  head * 128 + 8 * (t & 15)))
                            : make_uint4(0u, 0u, 0u, 0u);
            }
          }
          // transpose: feature column r of 32 tokens -> rows of the chunk
#pragma unroll
          for (int i = 0; i < 32; ++i) tr[i * kTrStride + r] = x[i];
          epi_bar(grp);
          if (EPI == EPI_STORE) {
            // 32 tokens x 16 vectors of 8 bf16 features
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int v = t + 128 * q, i = v >> 4, j = v & 15;
              const int tok = tok0 + c + i, f = ft * FM + 8 * j;
              if (c + i < pq.BT && tok < pq.M && f < pq.N)
                store_bf16x8(reinterpret_cast<bf16 *>(pq.out) + (int64_t)tok * pq.ldo + f,
                             tr + i * kTrStride + 8 * j);
            }
          } else if (epi == EPI_STORE_F32 || epi == EPI_RESID) {
            // 32 tokens x 32 vectors of 4 fp32 features; one loop per kind of
            // store (with the read-modify-write and the atomic add in one loop
            // the two-phase kernel's residual epilogue took 13 us a tile
            // instead of 3)
            float *const o0 = reinterpret_cast<float *>(pq.out);
            if (epi == EPI_STORE_F32 || whole) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int v = t + 128 * q, i = v >> 5, j = v & 31;
                const int tok = tok0 + c + i, f = ft * FM + 4 * j;
                if (c + i < pq.BT && tok < pq.M && f < pq.N) {
                  const float4 a = *reinterpret_cast<const float4 *>(tr + i * kTrStride + 4 * j);
                  float4 *o = reinterpret_cast<float4 *>(o0 + (int64_t)tok * pq.ldo + f);
                  if (epi == EPI_STORE_F32) {
                    *o = a;
                  } else {
                    float4 h = *o;
                    h.x += a.x; h.y += a.y; h.z += a.z; h.w += a.w;
                    *o = h;
                  }
                }
              }
            } else {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int v = t + 128 * q, i = v >> 5, j = v & 31;
                const int tok = tok0 + c + i, f = ft * FM + 4 * j;
                if (c + i < pq.BT && tok < pq.M && f < pq.N)
                  atomicAdd(reinterpret_cast<float4 *>(o0 + (int64_t)tok * pq.ldo + f),
                            *reinterpret_cast<const float4 *>(tr + i * kTrStride + 4 * j));
              }
            }
          } else if (epi == EPI_SWIGLU) {
            // tile rows 0..63 gate, 64..127 up: 32 tokens x 8 vectors of 8.  The
            // fast divide (2 ulp; 0 once the denominator passes 2^126, where SiLU
            // is 0 to fp32 precision) is well inside the bf16 output's rounding.
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int v = t + 128 * q, i = v >> 3, j = v & 7;
              const int tok = tok0 + c + i, f = ft * 64 + 8 * j;
              if (c + i < pq.BT && tok < pq.M && f < pq.N) {
                const float *g = tr + i * kTrStride + 8 * j;
                const float *u = g + 64;
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __fdividef(g[e], 1.f + __expf(-g[e])) * u[e];
                store_bf16x8(reinterpret_cast<bf16 *>(pq.out) + (int64_t)tok * pq.ldo + f, y);
              }
            }
          } else if (EPI == EPI_KDEV) {
            // 32 tokens x 16 groups of 8 features; the 16 threads of a token
            // are one half-warp, which sums the head's squared differences
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int v = t + 128 * q, i = v >> 4, j = v & 15;
              const int tok = tok0 + c + i;
              const int di = (c + i < pq.BT && tok < pq.M) ? s_dev[c + i] : -1;
              float acc = 0.f;
              if (di >= 0) {
                const float *row = tr + i * kTrStride;
                const int e0 = 8 * (j & 7);
                const float *w = reinterpret_cast<const float *>(rf[q]);   // (cos, sin) x 8
                const bf16 *kb = reinterpret_cast<const bf16 *>(&kraw[q]);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float x1 = row[e0 + e], x2 = row[64 + e0 + e];
                  const float co = w[2 * e], si = w[2 * e + 1];
                  const float y = j < 8 ? x1 * co - x2 * si : x2 * co + x1 * si;
                  const float dlt = y - __bfloat162float(kb[e]);
                  acc = fmaf(dlt, dlt, acc);
                }
              }
#pragma unroll
              for (int o = 8; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
              if (j == 0 && di >= 0) reinterpret_cast<float *>(pq.out)[head * pq.ldo + di] = acc;
            }
          } else if (EPI == EPI_QKV) {  // one head per tile
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int v = t + 128 * q, i = v >> 4, j = v & 15;
              const int tok = tok0 + c + i;
              if (c + i >= pq.BT || tok >= pq.M) continue;
              const float *row = tr + i * kTrStride;
              float y[8];
              bf16 *dst;
              if (rotate) {
                // rotate-half pairs (e, e + 64) at the token's position
                const int e0 = 8 * (j & 7);
                const float *w = reinterpret_cast<const float *>(rf[q]);   // (cos, sin) x 8
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float x1 = row[e0 + e], x2 = row[64 + e0 + e];
                  const float co = w[2 * e], si = w[2 * e + 1];
                  y[e] = j < 8 ? x1 * co - x2 * si : x2 * co + x1 * si;
                }
                dst = head < pq.Hq
                          ? reinterpret_cast<bf16 *>(pq.out) + (int64_t)tok * pq.ldo + head * 128
                          : reinterpret_cast<bf16 *>(pq.k_cache) + s_dst[c + i] * pq.ld_kv +
                                (head - pq.Hq) * 128;
              } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = row[8 * j + e];
                dst = reinterpret_cast<bf16 *>(pq.v_cache) + s_dst[c + i] * pq.ld_kv +
                      (head - pq.Hq - pq.Hkv) * 128;
              }
              store_bf16x8(dst + 8 * j, y);
            }
          }
          epi_bar(grp);
        }
        if (helper) {
          // every epilogue thread's partial is written before the arrival
          __threadfence();
          epi_all_bar();
          if (threadIdx.x == 64) signal_add(flag);
        } else if (MLP && ph == 0) {
          // this CTA's 64 features of g for the token tile are written: publish
          // them to the down projection's copies (async proxy, other SMs)
          asm volatile("fence.proxy.async.global;" ::: "memory");
          epi_all_bar();
          if (threadIdx.x == 64) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            int *const written = pq.mlp_flag + (int64_t)ft * pq.n_tt + tt;
            asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(written), "r"(pq.epoch)
                         : "memory");
          }
        }
        fence_before();
        if (CG == 2) {
          __syncwarp();
          if (lane == 0) arrive_remote(map_to_rank(smem_u32(&tempty[buf]), 0));
        } else {
          arrive(smem_u32(&tempty[buf]));
        }
        if (++buf == 2) { buf = 0; bphase ^= 1; }
      }
    };
    drain(std::integral_constant<int, 0>());
    if constexpr (kPhases > 1) {
      if (!stop) drain(std::integral_constant<int, 1>());
    }
  }
  fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();   // neither CTA retires while the pair may touch it
  if (warp == 1) {
    fence_after();
    if (CG == 2) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
}

template <int EPI, int CG, bool TS>
__global__ void __launch_bounds__(kThreads, 1)
gemm_sab_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW,
                const __grid_constant__ CUtensorMap mapW2, const __grid_constant__ Params p,
                int *status) {
  gemm_body<EPI, CG, TS>(&mapX, &mapW, &mapW2, &mapX, &mapW, p, p, status);
}

// The fused MLP: gate/up + SwiGLU into g, then h += g W_down^T.
template <int CG>
__global__ void __launch_bounds__(kThreads, 1)
gemm_mlp_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapWg,
                const __grid_constant__ CUtensorMap mapWu, const __grid_constant__ CUtensorMap mapG,
                const __grid_constant__ CUtensorMap mapWd, const __grid_constant__ Params p,
                const __grid_constant__ Params p2, int *status) {
  gemm_body<EPI_MLP, CG, true>(&mapX, &mapWg, &mapWu, &mapG, &mapWd, p, p2, status);
}

// Largest number of CTA pairs of this kernel that fit on the device at once
// (a pair needs two SMs of one GPC).
template <int EPI>
static int max_pairs(int smem) {
  static std::mutex mu;
  static int cached[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return num_sms() / 2;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev]) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_sms(), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_sab_kernel<EPI, 2, split_by_default<EPI>()>, &cfg) !=
          cudaSuccess ||
      n <= 0)
    n = num_sms() / 2;
  cached[dev] = n;
  return n;
}

// Function attributes of one instantiation, set once.
template <int EPI, int CG, bool TS>
static cudaError_t prepare() {
  static PerDeviceOnce once;
  return once.run([](int) {
    cudaError_t e = cudaFuncSetAttribute(gemm_sab_kernel<EPI, CG, TS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e == cudaSuccess && CG == 2)
      e = cudaFuncSetAttribute(gemm_sab_kernel<EPI, CG, TS>,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    return e;
  });
}

template <int EPI, int CG, bool TS>
static cudaError_t launch(int units, int smem, const CUtensorMap &mx, const CUtensorMap &mw,
                          const CUtensorMap &mw2, const Params &p, int *status, cudaStream_t s) {
  cudaError_t e = prepare<EPI, CG, TS>();
  if (e != cudaSuccess) return e;
  if (CG == 1)
    return launch_pdl(gemm_sab_kernel<EPI, 1, TS>, dim3(units), dim3(kThreads), smem, s, mx, mw,
                      mw2, p, status);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * units, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_sab_kernel<EPI, 2, TS>, mx, mw, mw2, p, status);
}

template <int EPI, int CG>
static cudaError_t run(const CUtensorMap &mx, const CUtensorMap &mw, const CUtensorMap &mw2,
                       Params &p, int *status, cudaStream_t s) {
  const int fixed = 2 * kTr + 256 + (EPI == EPI_QKV || EPI == EPI_KDEV ? kTokTab : 0) + 1024;
  p.stage_bytes = kTileW + (p.BT / CG) * BK * 2;
  p.stages = (kSmemMax - fixed) / p.stage_bytes;
  if (p.stages > 8) p.stages = 8;
  if (p.stages < 2) return cudaErrorInvalidValue;
  const int smem = p.stages * p.stage_bytes + fixed;
  cudaError_t e = prepare<EPI, CG, split_by_default<EPI>()>();
  if (e != cudaSuccess) return e;
  // units: CTAs, or CTA pairs
  const int max_units = CG == 2 ? max_pairs<EPI>(kSmemMax) : num_sms();
  const int n_ft = (p.n_ft + CG - 1) / CG;
  const int64_t tiles = (int64_t)p.n_tt * n_ft;
  int units;
  p.n_whole = (int)tiles;
  p.split = 1;
  if (p.stream_k) {
    // whole groups of n_tt units, at most one group per weight unit
    const int64_t wunits = (int64_t)n_ft * ((p.K + BK - 1) / BK);
    int64_t groups = max_units / p.n_tt;
    if (groups < 1) groups = 1;
    if (groups > wunits) groups = wunits;
    units = (int)(groups * p.n_tt);
  } else {
    units = tiles < max_units ? (int)tiles : max_units;
    if (p.part && can_split<EPI>()) {
      // the partial last wave: split its tiles along K over the idle units
      const int64_t rem = tiles % max_units;
      const int num_kb = (p.K + BK - 1) / BK;
      int split = rem ? (int)(max_units / rem) : 1;
      if (split > num_kb / 8) split = num_kb / 8;     // segments of at least 8 k-blocks
      if (split > 8) split = 8;
      if (split >= 2) {
        p.split = split;
        p.n_whole = (int)(tiles - rem);
        units = p.n_whole > 0 ? max_units : (int)(rem * split);
      }
    }
  }
  if (p.split > 1 && !split_by_default<EPI>())
    e = launch<EPI, CG, can_split<EPI>()>(units, smem, mx, mw, mw2, p, status, s);
  else
    e = launch<EPI, CG, split_by_default<EPI>()>(units, smem, mx, mw, mw2, p, status, s);
  if (e != cudaSuccess) return e;
  return launched(1);
}

template <int EPI>
static cudaError_t run_cg(const CUtensorMap &mx, const CUtensorMap &mw, const CUtensorMap &mw2,
                          Params &p, int cg, int *status, cudaStream_t s) {
  return cg == 2 ? run<EPI, 2>(mx, mw, mw2, p, status, s) : run<EPI, 1>(mx, mw, mw2, p, status, s);
}

// The fused MLP: one persistent unit per SM (pair), phase 0 with the tail
// split (split tiles first), phase 1 stream-K with deferred crossings.
template <int CG>
static cudaError_t run_mlp(const CUtensorMap &mx, const CUtensorMap &mwg, const CUtensorMap &mwu,
                           const CUtensorMap &mg, const CUtensorMap &mwd, Params &p, Params &p2,
                           int *status, cudaStream_t s) {
  const int fixed = 2 * kTr + 256 + 1024;
  p.stage_bytes = p2.stage_bytes = kTileW + (p.BT / CG) * BK * 2;
  p.stages = (kSmemMax - fixed) / p.stage_bytes;
  if (p.stages > 8) p.stages = 8;
  if (p.stages < 2) return cudaErrorInvalidValue;
  p2.stages = p.stages;
  const int smem = p.stages * p.stage_bytes + fixed;
  static PerDeviceOnce once;
  cudaError_t e = once.run([](int) {
    cudaError_t r = cudaFuncSetAttribute(gemm_mlp_kernel<CG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (r == cudaSuccess && CG == 2)
      r = cudaFuncSetAttribute(gemm_mlp_kernel<CG>,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    return r;
  });
  if (e != cudaSuccess) return e;
  // same shared memory and threads as the SwiGLU kernel: the same residency
  const int units = CG == 2 ? max_pairs<EPI_SWIGLU>(kSmemMax) : num_sms();
  const int n_ft = (p.n_ft + CG - 1) / CG;
  const int64_t tiles = (int64_t)p.n_tt * n_ft;
  p.n_whole = (int)tiles;
  p.split = 1;
  p.tail_first = 1;
  const int64_t rem = tiles % units;
  const int num_kb = (p.K + BK - 1) / BK;
  int split = rem ? (int)(units / rem) : 1;
  if (split > num_kb / 8) split = num_kb / 8;       // segments of at least 8 k-blocks
  if (split > 8) split = 8;
  if (split >= 2) {
    p.split = split;
    p.n_whole = (int)(tiles - rem);
  }
  p2.stream_k = 1;
  p2.defer = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CG * units, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = CG;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = CG == 2 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_mlp_kernel<CG>, mx, mwg, mwu, mg, mwd, p, p2, status);
}

}  // namespace sab

size_t gemm_split_flags_offset() { return (size_t)tcx::num_sms() * sab::kPartFloats * sizeof(float); }
size_t gemm_mlp_flags_offset() { return gemm_split_flags_offset() + sab::kSplitFlagBytes; }
size_t gemm_split_ws_bytes() { return gemm_mlp_flags_offset() + sab::kMlpFlags * sizeof(int); }

bool gemm_mlp_fits(int M, int F, int cta_group) {
  if (M <= 0 || F <= 0 || F % 64 || (cta_group != 1 && cta_group != 2)) return false;
  const int n_tt = (M + 255) / 256;
  const int bt = ((M + n_tt - 1) / n_tt + 15) / 16 * 16;
  const int cg = bt < 32 ? 1 : cta_group;
  return (int64_t)((F / 64 + cg - 1) / cg * cg) * n_tt <= sab::kMlpFlags;
}

cudaError_t launch_gemm_mlp(const void *x, int64_t ldx, const void *w_gate, const void *w_up,
                            int64_t ldw, const void *w_down, int64_t ldwd, int M, int F, int d,
                            void *g, int64_t ldg, float *h, int64_t ldh, int *status,
                            cudaStream_t s, int cta_group, void *split_ws, int epoch) {
  using namespace sab;
  if (M == 0) return cudaSuccess;
  if (!split_ws || epoch <= 0 || !gemm_mlp_fits(M, F, cta_group)) return cudaErrorNotSupported;
  Params p{};
  p.M = M;
  p.n_tt = (M + 255) / 256;
  p.BT = ((M + p.n_tt - 1) / p.n_tt + 15) / 16 * 16;
  if (p.BT < 32) cta_group = 1;                           // keep each CTA's half >= 16 rows
  const int cg = cta_group;
  p.idesc = idesc_bf16(FM * cg, p.BT);
  Params p2 = p;
  // phase 0: gate/up, 64 SwiGLU features per CTA tile
  p.N = F;
  p.K = d;
  p.n_ft = F / 64;
  p.out = g;
  p.ldo = ldg;
  p.part = reinterpret_cast<float *>(split_ws);
  p.flag = reinterpret_cast<int *>(reinterpret_cast<char *>(split_ws) + gemm_split_flags_offset());
  // phase 1: down + residual; its k-block kb is phase 0's CTA tile kb
  p2.N = d;
  p2.K = F;
  p2.n_ft = (d + FM - 1) / FM;
  p2.out = h;
  p2.ldo = ldh;
  p.mlp_flag = p2.mlp_flag =
      reinterpret_cast<int *>(reinterpret_cast<char *>(split_ws) + gemm_mlp_flags_offset());
  p.epoch = p2.epoch = epoch;
  CUtensorMap mx, mwg, mwu, mg, mwd;
  if (!make_map(&mx, x, M, d, ldx, p.BT / cg) || !make_map(&mwg, w_gate, F, d, ldw, 64) ||
      !make_map(&mwu, w_up, F, d, ldw, 64) || !make_map(&mg, g, M, F, ldg, p.BT / cg) ||
      !make_map(&mwd, w_down, d, F, ldwd, FM))
    return cudaErrorInvalidValue;
  const cudaError_t e = cg == 2 ? run_mlp<2>(mx, mwg, mwu, mg, mwd, p, p2, status, s)
                                : run_mlp<1>(mx, mwg, mwu, mg, mwd, p, p2, status, s);
  if (e != cudaSuccess) return e;
  return launched(1);
}

// Automatic form, measured at the Llama-3-8B projection shapes for 512 to
// 4096 token rows: the CTA-pair swapped form is fastest for the SwiGLU,
// down and Q/K/V projections at every size (524 rows: 92, 45 and 22 us
// against 107, 49 and 29 us for the best single-CTA form; 4096 rows of
// SwiGLU: 2.0 PFLOP/s).  The K = 4096 residual projection (O) has few weight
// tiles; it takes the single-CTA swapped form up to 1024 rows and token rows
// on M above that.  Returns 0 (token rows on M), 1 or 2 (swapped, CTAs per
// MMA).
int gemm_auto_form(int M, int K, GemmEpi epi) {
  if (M <= 0) return 0;
  if (epi == EPI_RESID && K <= 4096) return M <= 1024 ? 1 : 0;
  return 2;
}

cudaError_t launch_gemm_sab(const void *A, int64_t lda, const void *W, const void *W2,
                            int64_t ldw, int M, int N, int K, GemmEpi epi, void *out,
                            int64_t ldo, const QkvEpi *qkv, int *status, cudaStream_t s,
                            int cta_group, void *split_ws) {
  using namespace sab;
  if (M == 0 || N == 0) return cudaSuccess;
  if (cta_group != 1 && cta_group != 2) return cudaErrorInvalidValue;
  Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.n_tt = (M + 255) / 256;
  p.BT = ((M + p.n_tt - 1) / p.n_tt + 15) / 16 * 16;
  if ((epi == EPI_QKV || epi == EPI_KDEV) && (N / 128) % 2) cta_group = 1;   // pairs take two heads
  if (p.BT < 32) cta_group = 1;                           // keep each CTA's half >= 16 rows
  const int cg = cta_group;
  p.idesc = idesc_bf16(FM * cg, p.BT);
  p.out = out;
  p.ldo = ldo;
  if (split_ws) {
    p.part = reinterpret_cast<float *>(split_ws);
    p.flag = reinterpret_cast<int *>(reinterpret_cast<char *>(split_ws) + gemm_split_flags_offset());
  }
  CUtensorMap mx, mw, mw2;
  // each CTA of a pair holds half of the token rows of B
  if (!make_map(&mx, A, M, K, lda, p.BT / cg)) return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_SWIGLU:
      p.n_ft = (N + 63) / 64;
      if (!make_map(&mw, W, N, K, ldw, 64) || !make_map(&mw2, W2, N, K, ldw, 64))
        return cudaErrorInvalidValue;
      return run_cg<EPI_SWIGLU>(mx, mw, mw2, p, cg, status, s);
    case EPI_QKV:
      if (!qkv) return cudaErrorInvalidValue;
      p.n_ft = N / 128;
      p.pos = qkv->pos;
      p.dst_row = qkv->dst_row;
      p.k_cache = qkv->k_cache;
      p.v_cache = qkv->v_cache;
      p.ld_kv = qkv->ld_kv;
      p.rope = reinterpret_cast<const float2 *>(qkv->rope);
      p.Hq = qkv->n_q_heads;
      p.Hkv = qkv->n_kv_heads;
      if (!make_map(&mw, W, N, K, ldw, FM)) return cudaErrorInvalidValue;
      return run_cg<EPI_QKV>(mx, mw, mw, p, cg, status, s);
    case EPI_KDEV:
      if (!qkv || !qkv->dev_idx || N % 128) return cudaErrorInvalidValue;
      p.n_ft = N / 128;
      p.pos = qkv->pos;
      p.dst_row = qkv->dst_row;
      p.dev_idx = qkv->dev_idx;
      p.k_cache = qkv->k_cache;
      p.ld_kv = qkv->ld_kv;
      p.rope = reinterpret_cast<const float2 *>(qkv->rope);
      p.Hq = qkv->n_q_heads;
      p.Hkv = qkv->n_kv_heads;
      if (!make_map(&mw, W, N, K, ldw, FM)) return cudaErrorInvalidValue;
      return run_cg<EPI_KDEV>(mx, mw, mw, p, cg, status, s);
    case EPI_RESID:
      p.n_ft = (N + FM - 1) / FM;
      p.stream_k = 1;
      if (!make_map(&mw, W, N, K, ldw, FM)) return cudaErrorInvalidValue;
      return run_cg<EPI_RESID>(mx, mw, mw, p, cg, status, s);
    case EPI_STORE:
      p.n_ft = (N + FM - 1) / FM;
      if (!make_map(&mw, W, N, K, ldw, FM)) return cudaErrorInvalidValue;
      return run_cg<EPI_STORE>(mx, mw, mw, p, cg, status, s);
    case EPI_STORE_F32:
      p.n_ft = (N + FM - 1) / FM;
      if (!make_map(&mw, W, N, K, ldw, FM)) return cudaErrorInvalidValue;
      return run_cg<EPI_STORE_F32>(mx, mw, mw, p, cg, status, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace cb
