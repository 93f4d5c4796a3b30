// Ring-attention backward, bf16, d = 128, on the sm_100-family tensor cores.
//
// What it computes.  The pages print no backward pass; this kernel differentiates
// the forward's definition (Module 23, "The Math: One Block at a Time";
// "3.6 Distributed Training II", section "Ring Attention").  With the forward's
// LSE the probabilities are recomputed tile by tile,
//   P = 2^(scale*log2(e) * q.k - LSE*log2(e)),   dP = dO V^T,
//   dS = P * (dP - D)   with D = rowsum(dO * O),
//   dV = P^T dO,   dK = scale * dS^T Q,   dQ = scale * dS K,
// and a key/value head's dK, dV gather the contributions of every query head of
// its group.  Two passes of one kernel template:
//   pass 0 (dK, dV): a work item is one 128-row key tile of shard r.  Its block
//     travels the ring: at step t it sits on the device of shard (r + t) mod N and
//     meets that shard's query tiles (every query head of the group in turn), so
//     the block's gradients gather where the block goes.
//   pass 1 (dQ): a work item is one 128-row query tile of shard p; it meets the
//     key blocks of shards (p - t) mod N in the forward's ring order.
// Causal: only the query tiles that see some key of the tile (pass 0), or the key
// tiles some query of the tile sees (pass 1), are visited; the rest of the mask
// is applied per element by global position (Module 23, "Exact by Construction").
//
// How (one persistent CTA per SM, 12 warps):
//   warp 0     TMA producer: pass 0's own 128-row tiles (K, V) once per item, then
//              64-row tiles of the streamed tensors (Q, dO and the tile's 64
//              LSE*log2(e) and D values in pass 0; K, V in pass 1) into a ring of
//              stages.
//   warp 1     tcgen05 issuer (converged warp, one elected lane): per streamed tile
//              two products (M = 128, N = 64) give the scores and dP -- SS in pass 0
//              (keys are the TMEM lanes), TS in pass 1 with Q and dO read from tensor
//              memory -- then TS products (M = 128, N = 128, K = 64) add P^T dO and
//              dS^T Q (pass 0) or dS K (pass 1) into accumulators, reading P and dS
//              from tensor memory and the streamed tile, still in shared memory, as
//              an MN-major operand.
//   warps 4-7 / 8-11  elementwise: one thread per TMEM lane turns scores and dP
//              into P and dS (bf16, written back into tensor memory), for the
//              even / odd streamed tiles; in pass 1 they first store the item's Q
//              (warps 4-7) and dO (8-11) rows into tensor memory; at the end of an
//              item they write the accumulators (pass 0: warps 4-7 dV, 8-11 dK;
//              pass 1: half of dQ each).
// TMEM: two tile buffers of 128 columns (scores 0-63, dP 64-127; P over 0-31 and
// dS over 64-95 once computed), so the next tile's products run while the
// elementwise warps work on the previous one; pass 0 keeps dV at 256 and dK at
// 384, pass 1 dQ at 256, Q at 384 and dO at 448.
// Every wait is bounded (~1 s); on expiry the CTA records it in the status word,
// drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bwd_internal.h"
#include "sm100_ptx.cuh"

namespace ra {
namespace {

constexpr int kThreads = 384;
constexpr uint32_t kRegsLaunch = 168;
constexpr uint32_t kRegsOther = 120;
constexpr uint32_t kRegsCompute = 192;
static_assert(128 * kRegsOther + 256 * kRegsCompute <= kThreads * kRegsLaunch, "register split");

constexpr int kFixRows = 128;                     // rows of an item's own tiles (a 128-row TMA box)
constexpr int kStreamRows = 64;                   // rows of a streamed tile
constexpr uint32_t kFixBytes = 128 * 128 * 2;     // one 128 x 128 bf16 tile
constexpr uint32_t kFixHalf = 128 * 64 * 2;       // its 128-byte swizzle column
constexpr uint32_t kStrBytes = 64 * 128 * 2;      // one 64 x 128 bf16 tile
constexpr uint32_t kStrHalf = 64 * 64 * 2;
constexpr uint32_t kLseBytes = 128 * 4;          // 64 lse2 values, then 64 D values

template <int kPass>
struct Cfg {
  static constexpr int kStages = kPass == 0 ? 4 : 6;
  static constexpr int kBufs = 2;  // score/dP buffers in tensor memory
  static constexpr uint32_t kStageBytes = kPass == 0 ? 2 * kStrBytes + 1024 : 2 * kStrBytes;
  static constexpr uint32_t kOffFix = 0;  // pass 0 only: K, V (pass 1 keeps Q, dO in tensor memory)
  static constexpr uint32_t kOffStage = kPass == 0 ? 2 * kFixBytes : 0;
  static constexpr uint32_t kOffBar = kOffStage + kStages * kStageBytes;
  static constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;  // barriers + slots, 1 KiB alignment slack
};

enum : int {
  kFixFull = 0,
  kFixEmpty = 1,
  kAccFull = 2,
  kAccEmpty = 3,
  kDone = 4,
  kSFull = 5,       // 3 (one per buffer)
  kPFull = 8,       // 3
  kItemFull = 11,   // 4
  kItemEmpty = 15,  // 4
  kStFull = 19,     // kStages
};
template <int kPass>
struct Bars {
  static constexpr int kStEmpty = kStFull + Cfg<kPass>::kStages;
  static constexpr int kNum = kStEmpty + Cfg<kPass>::kStages;
};
constexpr int kItemSlots = 4;
constexpr uint32_t kItemConsumers = 9;  // MMA warp + 8 elementwise warps

constexpr uint32_t kTmemCols = 512;
// pass 0: dV at 256, dK at 384; pass 1: dQ at 256, the item's Q at 384 and dO at 448
template <int kPass>
__device__ __forceinline__ uint32_t col_acc0() { return 256u; }
constexpr uint32_t kColAcc1 = 384;
constexpr uint32_t kColQ = 384, kColDO = 448;
__device__ __forceinline__ uint32_t col_buf(uint32_t b) { return b * 128u; }
constexpr uint32_t kColDP = 64;   // dP within a buffer; dS is written over its first 32 columns
constexpr uint32_t kIdescSS = ptx::idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdescTS = ptx::idesc_bf16_f32(128, 128, false, true);
constexpr uint64_t kWaitBudgetNs = 1000000000ull;
constexpr uint32_t kSuspendHintNs = 2000u;

struct Ctl {
  uint32_t bars;
  volatile uint32_t* abort;
  uint32_t* status;
  __device__ __forceinline__ uint32_t bar(int i) const { return bars + 8u * (uint32_t)i; }
};

__device__ __forceinline__ bool wait_bar(const Ctl& c, uint32_t bar, uint32_t parity, uint32_t who) {
  if (ptx::mbar_test(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_wait_hint(bar, parity, kSuspendHintNs)) return true;
    if ((it & 15u) == 0) {
      if (*c.abort) return false;
      if (ptx::global_timer_ns() - t0 > kWaitBudgetNs) {
        *c.abort = 1u;
        atomicOr(c.status, who);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void drain_bar(const Ctl& c, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::global_timer_ns();
  while (!ptx::mbar_test(bar, parity)) {
    if (ptx::global_timer_ns() - t0 > kWaitBudgetNs) {
      atomicOr(c.status, kStatusTimeoutTeardown);
      return;
    }
  }
}

// The bounded wait, run against a barrier that nothing completes: one warp
// initialises an mbarrier for one arrival, never arrives, and waits for its first
// phase.  The wait gives up after kWaitBudgetNs, records `who` in the status word and
// returns, as in the tensor-core kernels when a handshake never comes.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t* status, uint32_t who) {
  __shared__ __align__(8) uint64_t bar_word;
  __shared__ uint32_t abort_flag;
  const uint32_t bar = ptx::smem_addr(&bar_word);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  __syncwarp();
  Ctl c;
  c.bars = bar;
  c.abort = &abort_flag;
  c.status = status;
  wait_bar(c, bar, 0u, who);
}

// ------------------------------------------------------------------- walks --
// The streamed tiles of an item, in order.  Pass 0 (item = key tile of shard r
// whose first key sits at position kmin): ring step t puts the block on shard
// p = (r + t) mod N; every query head g of the group; query tiles it of shard p
// from the first that sees key position kmin.  Pass 1 (item = query tile of shard
// p whose last query sits at position maxq): step t meets shard r = (p - t) mod N,
// key tiles 0..last_le(r, maxq)/64.
struct Walk {
  int t, g, it, lo, hi, shard;
};

__device__ __forceinline__ int n_stream_tiles(const BwdParams& P) {
  return (int)((P.s_n + kStreamRows - 1) / kStreamRows);
}

template <int kPass>
__device__ __forceinline__ void walk_step_bounds(Walk& w, const BwdParams& P, const WorkItem& it) {
  const int N = P.n_shards;
  if (kPass == 0) {
    w.shard = (it.shard + w.t) % N;
    w.hi = n_stream_tiles(P);
    w.lo = 0;
    if (P.causal) {  // first query of the shard that sees the tile's first key, if any
      const int64_t f = first_ge(P.layout, N, P.s_n, w.shard, it.maxq);
      w.lo = f >= P.s_n ? w.hi : (int)(f / kStreamRows);
    }
  } else {
    w.shard = (it.shard - w.t + N) % N;
    w.lo = 0;
    if (P.causal) {
      const int64_t j = last_le(P.layout, N, P.s_n, w.shard, it.maxq);
      w.hi = j < 0 ? 0 : (int)(j / kStreamRows) + 1;
    } else {
      w.hi = n_stream_tiles(P);
    }
  }
}

// Advance to the next non-empty (t, g) range starting at the current one.
template <int kPass>
__device__ __forceinline__ void walk_settle(Walk& w, const BwdParams& P, const WorkItem& it) {
  const int groups = kPass == 0 ? P.group : 1;
  while (w.t < P.n_shards) {
    if (w.it < w.hi) return;
    if (++w.g < groups) {
      w.it = w.lo;
      continue;
    }
    w.g = 0;
    if (++w.t >= P.n_shards) return;
    walk_step_bounds<kPass>(w, P, it);
    w.it = w.lo;
  }
}

template <int kPass>
__device__ __forceinline__ void walk_begin(Walk& w, const BwdParams& P, const WorkItem& it) {
  w.t = 0;
  w.g = 0;
  walk_step_bounds<kPass>(w, P, it);
  w.it = w.lo;
  walk_settle<kPass>(w, P, it);
}

template <int kPass>
__device__ __forceinline__ void walk_next(Walk& w, const BwdParams& P, const WorkItem& it) {
  ++w.it;
  walk_settle<kPass>(w, P, it);
}

// Number of streamed tiles of an item (the walk's length).
template <int kPass>
__device__ __forceinline__ int item_tiles(const BwdParams& P, const WorkItem& it) {
  int n = 0;
  Walk w;
  for (w.t = 0; w.t < P.n_shards; ++w.t) {
    walk_step_bounds<kPass>(w, P, it);
    if (w.hi > w.lo) n += (w.hi - w.lo) * (kPass == 0 ? P.group : 1);
  }
  return n;
}

__device__ __forceinline__ int next_item(const Ctl& c, volatile int32_t* slots, uint32_t u, int lane) {
  const uint32_t slot = u % kItemSlots, use = u / kItemSlots;
  if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kItemFull + (int)slot), use & 1u, kStatusTimeoutSoftmax)))
    return -1;
  const int idx = slots[slot];
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(c.bar(kItemEmpty + (int)slot));
  return idx;
}

// Producer-side grid barrier for round-synchronised schedules: wait (bounded)
// until the shared counter reaches `need`.
__device__ __forceinline__ bool barrier_wait(const Ctl& c, const uint32_t* counter, uint32_t need, int lane) {
  int ok = 1;
  if (lane == 0) {
    const volatile uint32_t* ctr = counter;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 0; *ctr < need; ++it) {
      __nanosleep(128);
      if ((it & 63u) == 63u) {
        if (*c.abort) {
          ok = 0;
          break;
        }
        if (ptx::global_timer_ns() - t0 > kWaitBudgetNs) {
          *c.abort = 1u;
          atomicOr(c.status, kStatusTimeoutProducer);
          ok = 0;
          break;
        }
      }
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ---------------------------------------------------------------- producer --
struct ProducerState {
  uint32_t str_issued;  // streamed tiles issued
  uint32_t fix_issued;  // items whose own tiles were issued
};

template <int kPass>
__device__ void run_producer(const BwdParams& P, const Ctl& c, uint32_t sbase, volatile int32_t* slots,
                             const CUtensorMap* tx0, const CUtensorMap* tx1, const CUtensorMap* ty0,
                             const CUtensorMap* ty1, ProducerState& st) {
  using C = Cfg<kPass>;
  const int lane = threadIdx.x & 31;
  const uint64_t keep = ptx::l2_policy_evict_last();
  uint32_t s_it = 0;
  for (uint32_t u = 0;; ++u) {
    const uint32_t slot = u % kItemSlots, use = u / kItemSlots;
    if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kItemEmpty + (int)slot), (use & 1u) ^ 1u, kStatusTimeoutProducer)))
      break;
    int idx;
    if (P.round_sync) {
      // Round u: item u*grid + b, once every CTA has issued the loads of round u-1.
      idx = (int)(u * gridDim.x + blockIdx.x);
      if (idx >= P.n_items) idx = -1;
      if (idx >= 0 && u > 0 && !barrier_wait(c, P.item_counter, u * gridDim.x, lane)) idx = -1;
    } else {
      idx = 0;
      if (lane == 0) idx = (int)atomicAdd(P.item_counter, 1u);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      if (idx >= P.n_items) idx = -1;
    }
    if (lane == 0) slots[slot] = idx;
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(c.bar(kItemFull + (int)slot));
    if (idx < 0) break;
    RA_BOUNDS(c.status, idx < P.n_items, 20);
    const WorkItem it = P.items[idx];
    RA_BOUNDS(c.status, it.shard >= 0 && it.shard < P.n_shards && it.row0 >= 0 && it.row0 < P.s_n, 21);
    const int64_t rows_q = (int64_t)P.batch * P.heads_q * P.seq, rows_kv = (int64_t)P.batch * P.heads_kv * P.seq;
    if (kPass == 0) {
      if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kFixEmpty), (u & 1u) ^ 1u, kStatusTimeoutProducer))) break;
      // The item's own tiles: rows bh0*S + shard*s_n + row0 of K and V.  (Pass 1's own
      // Q and dO rows go to tensor memory through the elementwise warps.)
      const int32_t yf = (int32_t)((int64_t)it.bh0 * P.seq + (int64_t)it.shard * P.s_n + it.row0);
      RA_BOUNDS(c.status, yf >= 0 && yf < rows_kv, 22);
      ptx::mbar_arrive_expect_tx_warp(c.bar(kFixFull), 2 * kFixBytes);
      ptx::tma_load_2d_warp(sbase + C::kOffFix, tx0, c.bar(kFixFull), 0, yf);
      ptx::tma_load_2d_warp(sbase + C::kOffFix + kFixHalf, tx0, c.bar(kFixFull), 64, yf);
      ptx::tma_load_2d_warp(sbase + C::kOffFix + kFixBytes, tx1, c.bar(kFixFull), 0, yf);
      ptx::tma_load_2d_warp(sbase + C::kOffFix + kFixBytes + kFixHalf, tx1, c.bar(kFixFull), 64, yf);
      st.fix_issued = u + 1;
    }
    // Streamed tiles.
    int b, h_base;
    if (kPass == 0) {  // bh0 = b * Hkv + kv head; queries of heads kv*G .. kv*G + G-1
      b = it.bh0 / P.heads_kv;
      h_base = (it.bh0 % P.heads_kv) * P.group;
    } else {           // bh0 = b * Hq + h; its key/value head
      b = it.bh0 / P.heads_q;
      h_base = (it.bh0 % P.heads_q) / P.group;
    }
    Walk w;
    walk_begin<kPass>(w, P, it);
    bool ok = true;
    while (w.t < P.n_shards) {
      const int64_t head_row = kPass == 0 ? ((int64_t)b * P.heads_q + h_base + w.g) * P.seq
                                          : ((int64_t)b * P.heads_kv + h_base) * P.seq;
      const int32_t y = (int32_t)(head_row + (int64_t)w.shard * P.s_n + (int64_t)w.it * kStreamRows);
      RA_BOUNDS(c.status, w.shard >= 0 && w.shard < P.n_shards && w.it >= 0 && (int64_t)w.it * kStreamRows < P.s_n &&
                              w.g >= 0 && w.g < (kPass == 0 ? P.group : 1), 23);
      RA_BOUNDS(c.status, y >= 0 && y < (kPass == 0 ? rows_q : rows_kv), 24);
      const uint32_t s = s_it % C::kStages, phase = (s_it / C::kStages) & 1u;
      if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kStFull + C::kStages + (int)s), phase ^ 1u, kStatusTimeoutProducer))) {
        ok = false;
        break;
      }
      const uint32_t dst = sbase + C::kOffStage + s * C::kStageBytes;
      ptx::mbar_arrive_expect_tx_warp(c.bar(kStFull + (int)s), kPass == 0 ? 2 * kStrBytes + kLseBytes : 2 * kStrBytes);
      ptx::tma_load_2d_warp_hint(dst, ty0, c.bar(kStFull + (int)s), 0, y, keep);
      ptx::tma_load_2d_warp_hint(dst + kStrHalf, ty0, c.bar(kStFull + (int)s), 64, y, keep);
      ptx::tma_load_2d_warp_hint(dst + kStrBytes, ty1, c.bar(kStFull + (int)s), 0, y, keep);
      ptx::tma_load_2d_warp_hint(dst + kStrBytes + kStrHalf, ty1, c.bar(kStFull + (int)s), 64, y, keep);
      RA_BOUNDS(c.status,
                kPass != 0 || bwd_scalar_index((int64_t)b * P.heads_q + h_base + w.g, w.shard, (int64_t)w.it * kStreamRows,
                                               P.n_shards, P.n64) + 128 <=
                                  (int64_t)P.batch * P.heads_q * P.n_shards * P.n64 * 128,
                25);
      if (kPass == 0)  // the tile's 64 lse2 and 64 D values (one 512-byte block)
        ptx::bulk_load_warp(dst + 2 * kStrBytes,
                            P.lse2d + bwd_scalar_index((int64_t)b * P.heads_q + h_base + w.g, w.shard,
                                                       (int64_t)w.it * kStreamRows, P.n_shards, P.n64),
                            kLseBytes, c.bar(kStFull + (int)s));
      st.str_issued = ++s_it;
      walk_next<kPass>(w, P, it);
    }
    if (!ok) break;
    if (P.round_sync) {
      if (lane == 0) atomicAdd(P.item_counter, 1u);  // this CTA has issued its round
      __syncwarp();
    }
  }
}

// --------------------------------------------------------------------- MMA --
template <int kPass>
__device__ __forceinline__ void issue_ss(uint32_t tmem, int buf, uint32_t fix_lo, uint32_t str_lo) {
  // Scores: own tile 0 x streamed tile 0; dP: own tile 1 x streamed tile 1.  Pass 0's
  // own tiles (K, V) are in shared memory; pass 1's (Q, dO) in tensor memory, two bf16
  // of d per column, so its products read only the streamed 64-row tile from shared
  // memory.
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint32_t a0 = fix_lo + (which ? (kFixBytes >> 4) : 0u);
    const uint32_t b0 = str_lo + (which ? (kStrBytes >> 4) : 0u);
    const uint32_t d = tmem + col_buf(buf) + (which ? kColDP : 0u);
#pragma unroll
    for (uint32_t kk = 0; kk < 8; ++kk) {  // 8 steps of K = 16 over d = 128
      const uint32_t ob = ((kk >> 2) * kStrHalf + (kk & 3u) * 32u) >> 4;
      if (kPass == 0) {
        const uint32_t oa = ((kk >> 2) * kFixHalf + (kk & 3u) * 32u) >> 4;
        ptx::mma_bf16_ss_lo_warp(d, a0 + oa, b0 + ob, kIdescSS, kk > 0 ? 1u : 0u);
      } else {
        ptx::mma_bf16_ts_lo_warp(d, tmem + (which ? kColDO : kColQ) + kk * 8u, b0 + ob, kIdescSS, kk > 0 ? 1u : 0u);
      }
    }
  }
}

// acc += A[tmem, 64 K-columns as 32 words] * B[streamed 64-row tile, MN-major].
__device__ __forceinline__ void issue_ts(uint32_t d, uint32_t a_tmem, uint32_t b_lo, bool accumulate) {
#pragma unroll
  for (uint32_t kk = 0; kk < 4; ++kk)  // 4 steps of 16 rows = 8 TMEM columns of A
    ptx::mma_bf16_ts_lo_warp(d, a_tmem + kk * 8u, b_lo + ((kk * 2048u) >> 4), kIdescTS,
                             (accumulate || kk > 0) ? 1u : 0u);
}

template <int kPass>
__device__ void run_mma(const BwdParams& P, const Ctl& c, uint32_t sbase, volatile int32_t* slots, uint32_t tmem) {
  using C = Cfg<kPass>;
  constexpr uint32_t NB = (uint32_t)C::kBufs;
  const int lane = threadIdx.x & 31;
  const uint32_t fix_lo = ptx::desc_lo(sbase + C::kOffFix, 16);
  // two 128-column buffers, then the accumulators (and pass 1's Q, dO) up to column 512
  RA_BOUNDS(c.status, tmem == 0u && col_buf(C::kBufs) <= col_acc0<kPass>() && kColDO + 64u <= kTmemCols, 26);
  uint32_t s_it = 0;  // streamed tiles so far (global tile index J of this CTA)
  auto str_lo = [&](uint32_t J, uint32_t lbo) {
    return ptx::desc_lo(sbase + C::kOffStage + (J % C::kStages) * C::kStageBytes, lbo);
  };
  auto wait_stage = [&](uint32_t J) {
    return __all_sync(0xffffffffu, wait_bar(c, c.bar(kStFull + (int)(J % C::kStages)), (J / C::kStages) & 1u,
                                            kStatusTimeoutMma));
  };
  // Scores and dP of tile J into buffer J % NB.
  auto issue_tile_ss = [&](uint32_t J) {
    if (!wait_stage(J)) return false;
    issue_ss<kPass>(tmem, (int)(J % NB), fix_lo, str_lo(J, 16));
    ptx::mma_commit_warp(c.bar(kSFull + (int)(J % NB)));
    return true;
  };
  for (uint32_t u = 0;; ++u) {
    const int idx = next_item(c, slots, u, lane);
    if (idx < 0) break;
    const WorkItem it = P.items[idx];
    const uint32_t n = (uint32_t)item_tiles<kPass>(P, it);
    if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kFixFull), u & 1u, kStatusTimeoutMma))) return;
    ptx::tc_fence_after();  // pass 1: Q and dO were stored into tensor memory by other warps
    // Run NB - 1 tiles ahead: buffer (J + NB - 1) % NB was last used by tile J - 1,
    // whose TS products are issued (the tensor pipe executes in issue order).
    for (uint32_t a = 0; a + 1 < NB && a < n; ++a)
      if (!issue_tile_ss(s_it + a)) return;
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t J = s_it + i;
      if (i + NB - 1 < n && !issue_tile_ss(J + NB - 1)) return;
      if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kPFull + (int)(J % NB)), (J / NB) & 1u, kStatusTimeoutMma)))
        return;
      if (i == 0 && u > 0 &&
          !__all_sync(0xffffffffu, wait_bar(c, c.bar(kAccEmpty), (u - 1) & 1u, kStatusTimeoutMma)))
        return;
      ptx::tc_fence_after();
      // Streamed tile 0 (Q in pass 0, K in pass 1) and tile 1 (dO in pass 0) as MN-major B.
      const uint32_t y0 = str_lo(J, kStrHalf), y1 = y0 + (kStrBytes >> 4);
      const uint32_t buf = tmem + col_buf(J % NB);
      if (kPass == 0) {
        issue_ts(tmem + col_acc0<kPass>(), buf, y1, i > 0);  // dV += P^T dO
        issue_ts(tmem + kColAcc1, buf + kColDP, y0, i > 0);  // dK += dS^T Q
      } else {
        issue_ts(tmem + col_acc0<kPass>(), buf + kColDP, y0, i > 0);  // dQ += dS K
      }
      ptx::mma_commit_warp(c.bar(kStFull + C::kStages + (int)(J % C::kStages)));
    }
    if (n == 0 && u > 0 &&
        !__all_sync(0xffffffffu, wait_bar(c, c.bar(kAccEmpty), (u - 1) & 1u, kStatusTimeoutMma)))
      return;
    ptx::mma_commit_warp(c.bar(kAccFull));
    ptx::mma_commit_warp(c.bar(kFixEmpty));
    s_it += n;
  }
}

// -------------------------------------------------------------- elementwise --
// Write 64 accumulator columns [col0, col0 + 64) of this thread's row, times mul,
// as bf16 (zeros when the item met no tile).
__device__ __forceinline__ void store_row(uint32_t t_acc, uint16_t* dst_row, int col0, float mul, bool valid,
                                          bool zero) {
#pragma unroll 1
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t v[32];
    __syncwarp();
    ptx::tmem_ld32(t_acc + (uint32_t)(col0 + cc * 32), v);
    if (valid) {
      uint4* d = reinterpret_cast<uint4*>(dst_row + col0 + cc * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = zero ? 0u
                      : ptx::pack_bf16x2(__uint_as_float(v[8 * q + 2 * e]) * mul,
                                         __uint_as_float(v[8 * q + 2 * e + 1]) * mul);
        d[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// P and dS for one pair of columns (live: both unmasked).
__device__ __forceinline__ void p_ds_pair(float2 s2, float2 dp2, float2 l2, float2 d2, float2 sl2, bool live0,
                                          bool live1, uint32_t& pw, uint32_t& dw) {
  float2 x = ptx::fma2(s2, sl2, make_float2(-l2.x, -l2.y));
  x.x = live0 ? ptx::ex2_approx(x.x) : 0.f;
  x.y = live1 ? ptx::ex2_approx(x.y) : 0.f;
  const float2 ds = ptx::mul2(x, ptx::add2(dp2, make_float2(-d2.x, -d2.y)));
  pw = ptx::pack_bf16x2(x.x, x.y);
  dw = ptx::pack_bf16x2(ds.x, ds.y);
}

template <int kPass>
__device__ void run_elementwise(const BwdParams& P, const Ctl& c, const uint8_t* sgen, volatile int32_t* slots,
                                uint32_t tmem, int g, int wq, int lane) {
  using C = Cfg<kPass>;
  constexpr uint32_t NB = (uint32_t)C::kBufs;
  const int row = wq * 32 + lane;  // TMEM lane: key row (pass 0) or query row (pass 1)
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const int N = P.n_shards;
  const float2 sl2 = make_float2(P.scale_log2, P.scale_log2);
  uint32_t s_it = 0;
  for (uint32_t u = 0;; ++u) {
    const int idx = next_item(c, slots, u, lane);
    if (idx < 0) break;
    const WorkItem it = P.items[idx];
    const uint32_t n = (uint32_t)item_tiles<kPass>(P, it);
    const int64_t i_own = (int64_t)it.row0 + row;  // local row of the item's own tile
    const bool valid = i_own < P.s_n;
    const int64_t my_pos = pos_of(P.layout, N, P.s_n, it.shard, valid ? i_own : P.s_n - 1);
    const int64_t out_row = (int64_t)it.bh0 * P.seq + (int64_t)it.shard * P.s_n + i_own;
    RA_BOUNDS(c.status,
              !valid || (out_row >= 0 && out_row < (int64_t)P.batch * (kPass == 0 ? P.heads_kv : P.heads_q) * P.seq), 27);
    RA_BOUNDS(c.status, wq >= 0 && wq < 4 && (lane_off >> 16) + 32u <= 128u, 28);
    float2 own_l = make_float2(0.f, 0.f), own_d = make_float2(0.f, 0.f);  // pass 1: this row's lse2, D
    if (kPass == 1) {
      if (valid) {
        const int64_t li = bwd_scalar_index(it.bh0, it.shard, i_own, N, P.n64);
        RA_BOUNDS(c.status, li >= 0 && li + 64 < (int64_t)P.batch * P.heads_q * N * P.n64 * 128, 29);
        own_l = make_float2(P.lse2d[li], P.lse2d[li]);
        own_d = make_float2(P.lse2d[li + 64], P.lse2d[li + 64]);
      }
      // This row of Q (warps 4-7) or dO (warps 8-11) into tensor memory, once the
      // previous item's products are done with it.
      const bool okq = wait_bar(c, c.bar(kFixEmpty), (u & 1u) ^ 1u, kStatusTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, okq)) return;
      uint32_t words[64];
      const uint4* src = reinterpret_cast<const uint4*>(g ? P.dout : P.q) + (valid ? out_row * 16 : 0);
#pragma unroll
      for (int q4 = 0; q4 < 16; ++q4) {
        const uint4 v4 = valid ? src[q4] : make_uint4(0u, 0u, 0u, 0u);
        words[4 * q4] = v4.x;
        words[4 * q4 + 1] = v4.y;
        words[4 * q4 + 2] = v4.z;
        words[4 * q4 + 3] = v4.w;
      }
      ptx::tmem_st64(tmem + lane_off + (g ? kColDO : kColQ), words);
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(kFixFull));
    }

    Walk w;
    walk_begin<kPass>(w, P, it);
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t J = s_it + i;
      const int64_t tile_lo = (int64_t)w.it * kStreamRows;  // first local row of the streamed tile
      const int shard = w.shard;
      walk_next<kPass>(w, P, it);
      if ((int)(J & 1u) != g) continue;
      // Columns [c_lo, c_hi) of this tile are live for this row.
      int c_lo = 0;
      const int64_t left = P.s_n - tile_lo;
      int c_hi = left < kStreamRows ? (int)left : kStreamRows;
      if (P.causal) {
        if (kPass == 0) {  // queries of `shard` at or after this key's position
          const int64_t f = first_ge(P.layout, N, P.s_n, shard, my_pos) - tile_lo;
          c_lo = f < 0 ? 0 : (f > kStreamRows ? kStreamRows : (int)f);
        } else {           // keys of `shard` at or before this query's position
          const int64_t l = last_le(P.layout, N, P.s_n, shard, my_pos) - tile_lo + 1;
          const int lim = l < 0 ? 0 : (l > kStreamRows ? kStreamRows : (int)l);
          c_hi = lim < c_hi ? lim : c_hi;
        }
      }
      const bool ok = wait_bar(c, c.bar(kSFull + (int)(J % NB)), (J / NB) & 1u, kStatusTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, ok)) return;
      ptx::tc_fence_after();
      const uint32_t tb = tmem + lane_off + col_buf(J % NB);
      // pass 0: the tile's 64 lse2 values, then its 64 D values, in shared memory
      const float4* l4 =
          reinterpret_cast<const float4*>(sgen + C::kOffStage + (J % C::kStages) * C::kStageBytes + 2 * kStrBytes);
      uint32_t pw[32], dw[32];
      const bool full = __all_sync(0xffffffffu, c_lo == 0 && c_hi == kStreamRows);
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // columns 32*half .. 32*half + 31
        uint32_t raw[64];                       // scores in 0-31, dP in 32-63
        ptx::tmem_ld32x2(tb + 32u * half, tb + kColDP + 32u * half, raw);
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // columns c0 .. c0+3 of the tile
          const int c0 = 32 * half + 4 * q;
          float4 L, D;
          if (kPass == 0) {
            L = l4[c0 / 4];
            D = l4[16 + c0 / 4];
          } else {
            L = make_float4(own_l.x, own_l.x, own_l.x, own_l.x);
            D = make_float4(own_d.x, own_d.x, own_d.x, own_d.x);
          }
          const bool a0 = full || (c0 >= c_lo && c0 < c_hi), a1 = full || (c0 + 1 >= c_lo && c0 + 1 < c_hi);
          const bool b0 = full || (c0 + 2 >= c_lo && c0 + 2 < c_hi), b1 = full || (c0 + 3 >= c_lo && c0 + 3 < c_hi);
          const int r0 = 4 * q;
          p_ds_pair(make_float2(__uint_as_float(raw[r0]), __uint_as_float(raw[r0 + 1])),
                    make_float2(__uint_as_float(raw[32 + r0]), __uint_as_float(raw[32 + r0 + 1])),
                    make_float2(L.x, L.y), make_float2(D.x, D.y), sl2, a0, a1, pw[c0 / 2], dw[c0 / 2]);
          p_ds_pair(make_float2(__uint_as_float(raw[r0 + 2]), __uint_as_float(raw[r0 + 3])),
                    make_float2(__uint_as_float(raw[32 + r0 + 2]), __uint_as_float(raw[32 + r0 + 3])),
                    make_float2(L.z, L.w), make_float2(D.z, D.w), sl2, b0, b1, pw[c0 / 2 + 1], dw[c0 / 2 + 1]);
        }
      }
      if (kPass == 0) ptx::tmem_st32(tb, pw);  // P^T for dV (pass 1 needs only dS)
      ptx::tmem_st32(tb + kColDP, dw);
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(kPFull + (int)(J % NB)));
    }
    s_it += n;

    // Item done: write the accumulators (pass 0: dV by warps 4-7, dK by 8-11;
    // pass 1: dQ columns 0-63 by warps 4-7, 64-127 by 8-11).
    const bool ok = wait_bar(c, c.bar(kAccFull), u & 1u, kStatusTimeoutSoftmax);
    if (!__all_sync(0xffffffffu, ok)) return;
    ptx::tc_fence_after();
    if (kPass == 0) {
      uint16_t* dst = static_cast<uint16_t*>(g ? P.dk : P.dv) + out_row * 128;
      const uint32_t t_acc = tmem + lane_off + (g ? kColAcc1 : col_acc0<kPass>());
      store_row(t_acc, dst, 0, g ? P.scale : 1.0f, valid, n == 0);
      store_row(t_acc, dst, 64, g ? P.scale : 1.0f, valid, n == 0);
    } else {
      uint16_t* dst = static_cast<uint16_t*>(P.dq) + out_row * 128;
      store_row(tmem + lane_off + col_acc0<kPass>(), dst, g * 64, P.scale, valid, n == 0);
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(c.bar(kAccEmpty));
    __syncwarp();
  }
}

template <int kPass>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_bf16_kernel(const __grid_constant__ CUtensorMap tx0, const __grid_constant__ CUtensorMap tx1,
                    const __grid_constant__ CUtensorMap ty0, const __grid_constant__ CUtensorMap ty1,
                    const BwdParams P) {
  using C = Cfg<kPass>;
  using B = Bars<kPass>;
  static_assert(8 * B::kNum + 8 + 4 * kItemSlots <= 512, "barrier area");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t off_slot = C::kOffBar + 8 * B::kNum;
  Ctl c{sbase + C::kOffBar, reinterpret_cast<volatile uint32_t*>(sgen + off_slot + 4), P.status};
  volatile int32_t* slots = reinterpret_cast<volatile int32_t*>(sgen + off_slot + 8);

  if (threadIdx.x == 0) {
    ptx::mbar_init(c.bar(kFixFull), kPass == 0 ? 1 : 256);  // TMA (pass 0) or the 256 writers (pass 1)
    ptx::mbar_init(c.bar(kFixEmpty), 1);
    ptx::mbar_init(c.bar(kAccFull), 1);
    ptx::mbar_init(c.bar(kAccEmpty), 256);
    ptx::mbar_init(c.bar(kDone), 1);
    for (int b = 0; b < C::kBufs; ++b) {
      ptx::mbar_init(c.bar(kSFull + b), 1);
      ptx::mbar_init(c.bar(kPFull + b), 128);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      ptx::mbar_init(c.bar(kItemFull + s), 1);
      ptx::mbar_init(c.bar(kItemEmpty + s), kItemConsumers);
    }
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(c.bar(kStFull + s), 1);
      ptx::mbar_init(c.bar(B::kStEmpty + s), 1);
    }
    *c.abort = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tx0);
    ptx::tma_prefetch_desc(&tx1);
    ptx::tma_prefetch_desc(&ty0);
    ptx::tma_prefetch_desc(&ty1);
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + off_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + off_slot);

  ProducerState ps{0u, 0u};
  if (warp < 4) {
    ptx::regs_release<kRegsOther>();
    if (warp == 0) {
      run_producer<kPass>(P, c, sbase, slots, &tx0, &tx1, &ty0, &ty1, ps);
      __syncwarp();
    } else if (warp == 1) {
      run_mma<kPass>(P, c, sbase, slots, tmem);
      ptx::mma_commit_warp(c.bar(kDone));
      drain_bar(c, c.bar(kDone), 0);
      __syncwarp();
    }
  } else {
    ptx::regs_acquire<kRegsCompute>();
    run_elementwise<kPass>(P, c, sgen, slots, tmem, (warp - 4) >> 2, warp & 3, lane);
  }

  if (warp == 0 && lane == 0 && *c.abort) {
    // Let this CTA's own TMA loads land before its shared memory goes away.
    for (uint32_t s = 0; s < (uint32_t)C::kStages; ++s) {
      if (ps.str_issued > s) {
        const uint32_t uses = (ps.str_issued - 1 - s) / C::kStages + 1;
        drain_bar(c, c.bar(kStFull + (int)s), (uses - 1) & 1u);
      }
    }
    if (ps.fix_issued > 0) drain_bar(c, c.bar(kFixFull), (ps.fix_issued - 1) & 1u);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// [rows, 128] bf16 row-major; boxes of box_rows rows x 64 columns, 128-byte swizzle.
bool encode_bf16(CUtensorMap* map, const void* base, int64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128 * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kPass>
cudaError_t launch_pass(const BwdParams& prm, const CUtensorMap& tx0, const CUtensorMap& tx1, const CUtensorMap& ty0,
                        const CUtensorMap& ty1, int grid, cudaStream_t stream, const char** why) {
  using C = Cfg<kPass>;
  static std::atomic<int> ready[kMaxDevices];
  cudaError_t e = prepare_once(bwd_bf16_kernel<kPass>, ready, kThreads, 128 * kRegsOther + 256 * kRegsCompute,
                               (int)C::kSmemBytes, why);
  if (e != cudaSuccess) return e;
  if (prm.round_sync) {
    // The rounds wait on each other: a cooperative launch guarantees co-residency.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute coop[1];
    coop[0].id = cudaLaunchAttributeCooperative;
    coop[0].val.cooperative = 1;
    cfg.attrs = coop;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bwd_bf16_kernel<kPass>, tx0, tx1, ty0, ty1, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
  } else {
    bwd_bf16_kernel<kPass><<<grid, kThreads, C::kSmemBytes, stream>>>(tx0, tx1, ty0, ty1, prm);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) *why = "tensor-core backward launch failed";
  return e;
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t* status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, kStatusTimeoutMma);
  return cudaGetLastError();
}

cudaError_t launch_bwd_bf16(int pass, const BwdParams& prm, const void* q, const void* k, const void* v,
                            const void* dout, int grid, cudaStream_t stream, const char** why) {
  CUtensorMap a, b, y0, y1;
  const int64_t rows_q = (int64_t)prm.batch * prm.heads_q * prm.seq;
  const int64_t rows_kv = (int64_t)prm.batch * prm.heads_kv * prm.seq;
  bool ok;
  if (pass == 0)  // own tiles K, V (128 rows); streamed Q, dO (64 rows) and {lse2, D}
    ok = encode_bf16(&a, k, rows_kv, kFixRows) && encode_bf16(&b, v, rows_kv, kFixRows) &&
         encode_bf16(&y0, q, rows_q, kStreamRows) && encode_bf16(&y1, dout, rows_q, kStreamRows);
  else            // own tiles Q, dO; streamed K, V
    ok = encode_bf16(&a, q, rows_q, kFixRows) && encode_bf16(&b, dout, rows_q, kFixRows) &&
         encode_bf16(&y0, k, rows_kv, kStreamRows) && encode_bf16(&y1, v, rows_kv, kStreamRows);
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed or is unavailable";
    return cudaErrorInvalidValue;
  }
  return pass == 0 ? launch_pass<0>(prm, a, b, y0, y1, grid, stream, why)
                   : launch_pass<1>(prm, a, b, y0, y1, grid, stream, why);
}

}  // namespace ra
