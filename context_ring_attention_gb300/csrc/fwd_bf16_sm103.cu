// Ring-attention forward, bf16, d = 128, on the sm_100-family tensor cores.
//
// What it computes: for every query row of shard p, the online-softmax fold of
// Module 23, "The Math: One Block at a Time" over the key/value blocks of shards
// (p - t) mod N for ring steps t = 0..N-1 (the rotation of "3.6 Distributed
// Training II", section "Ring Attention"), finished as O = o / l; causal blocks
// strictly in the future are skipped and the rest masked by global position
// (Module 23, "Exact by Construction").  One GPU plays all N devices: the ring
// rotation is the order in which each query tile visits key tiles.
//
// How (one persistent CTA per SM, 12 warps):
//   warp 0     TMA producer: Q tiles once per work item, then K and V tiles in
//              ring order into a 5-slot shared-memory ring (128B swizzle).
//   warp 1     tcgen05 issuer: S = Q K^T into TMEM (both operands in shared
//              memory), O += P V into TMEM (P from TMEM, V from shared memory).
//   Warps 0 and 1 run converged with warp-uniform operands and one elected lane
//   issues each instruction: a single divergent lane issues MMAs too slowly to
//   keep the tensor pipe fed while the softmax warps share its scheduler.
//   warps 4-7  softmax for query tile 0, warps 8-11 for query tile 1: one thread
//              per row reads its 128 scores from TMEM in one round trip (a reducing
//              load, which also returns the row's largest score), updates
//              m and l, writes P (bf16) back into the upper half of its S columns,
//              rescales O in TMEM when m moves, and writes O / l and the LSE at the
//              end of a segment.
//   Warpgroup 0 (warps 0-3) hands registers to the softmax warpgroups (setmaxnreg).
// Two query tiles per CTA let one tile's softmax overlap the other tile's MMAs.
// TMEM: S0 cols 0-127 (P0 in 64-127), S1 128-255 (P1 in 192-255), O0 256-383,
// O1 384-511 (all 512 columns).
//
// Every mbarrier wait is bounded (~1 s).  On expiry the CTA raises an abort flag,
// records the role in the plan's status word, drains its own in-flight TMA
// loads and MMAs (bounded again), frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"
#include "sm100_ptx.cuh"

namespace ra {
namespace {

constexpr int kThreads = 384;  // 3 warpgroups: {producer, MMA, 2 idle}, softmax 0, softmax 1
// Register split (per thread): launched at kRegsLaunch; warpgroup 0 gives registers
// back so the two softmax warpgroups can hold a whole 128-score row.
// 128 * kRegsOther + 256 * kRegsSoftmax must not exceed 384 * kRegsLaunch.
constexpr uint32_t kRegsLaunch = 168;
constexpr uint32_t kRegsOther = 120;
constexpr uint32_t kRegsSoftmax = 192;
static_assert(128 * kRegsOther + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
constexpr uint32_t kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 tile
constexpr uint32_t kHalfBytes = 128 * 64 * 2;   // 128 rows x one 128-byte swizzle column
constexpr int kStages = 5;
constexpr uint32_t kOffQ = 0;                            // Q0, Q1
constexpr uint32_t kOffKV = 2 * kTileBytes;              // K/V ring
constexpr uint32_t kOffBar = kOffKV + kStages * kTileBytes;

enum : int {
  kQFull = 0,
  kQEmpty = 1,
  kKVFull = 2,
  kKVEmpty = kKVFull + kStages,
  kSFull = kKVEmpty + kStages,
  kPFull = kSFull + 2,
  kOFull = kPFull + 2,
  kDone = kOFull + 2,
  kItemFull = kDone + 1,
  kItemEmpty = kItemFull + 4,
  kNumBars = kItemEmpty + 4
};
constexpr int kItemSlots = 4;          // work-item indices handed from the producer to the other roles
constexpr uint32_t kItemConsumers = 9;  // MMA warp + 8 softmax warps
constexpr uint32_t kOffSlot = kOffBar + 8 * kNumBars;  // TMEM base written by tcgen05.alloc
constexpr uint32_t kOffAbort = kOffSlot + 4;
constexpr uint32_t kOffItems = kOffAbort + 4;  // kItemSlots int32 item indices
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + slack to align the base to 1 KiB
static_assert(8 * kNumBars + 8 + 4 * kItemSlots <= 256, "barrier area");

constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int g) { return g ? 128u : 0u; }
__device__ __forceinline__ uint32_t col_o(int g) { return g ? 384u : 256u; }
// P (bf16, two per 32-bit column) overwrites the upper half of its tile's S columns
// once the softmax has read S; the next S MMA of that tile is issued after the PV
// MMA that reads P.
constexpr uint32_t kColP = 64;

constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, 128, false, false);  // Q, K both K-major
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, 128, false, true);  // V is MN-major
constexpr uint64_t kWaitBudgetNs = 1000000000ull;
#ifndef RA_SUSPEND_HINT_NS
#define RA_SUSPEND_HINT_NS 2000u
#endif
constexpr uint32_t kSuspendHintNs = RA_SUSPEND_HINT_NS;  // a waiting thread sleeps up to this long per try
constexpr float kRescaleSlack = 8.0f;  // log2 units: keep a stale max while p <= 2^8
constexpr float kLn2 = 0.6931471805599453f;

struct Ctl {
  uint32_t bars;
  volatile uint32_t* abort;
  uint32_t* status;
  __device__ __forceinline__ uint32_t bar(int i) const { return bars + 8u * (uint32_t)i; }
};

// Bounded wait for phase `parity` of a barrier; false on abort or expiry.
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

// Teardown wait: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_bar(const Ctl& c, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::global_timer_ns();
  while (!ptx::mbar_test(bar, parity)) {
    if (ptx::global_timer_ns() - t0 > kWaitBudgetNs) {
      atomicOr(c.status, kStatusTimeoutTeardown);
      return;
    }
  }
}

// Key tiles a query tile whose largest position is maxq visits in the key block it
// meets: shard r of the ring, or (gathered) the one natural-order block of S keys.
template <bool kGathered>
__device__ __forceinline__ int kv_tiles(const FwdParams& P, int r, int64_t maxq) {
  return kGathered ? visit_tiles(RA_LAYOUT_CONTIGUOUS, 1, P.seq, P.causal, 0, maxq)
                   : visit_tiles(P.layout, P.n_shards, P.s_n, P.causal, r, maxq);
}

// Position in the virtual ring: step t, key shard r, key tile kt of nt.
struct Walk {
  int t, r, kt, nt;
};

template <bool kGathered>
__device__ __forceinline__ void walk_to_next_step(Walk& w, const FwdParams& P, int p, int64_t maxq) {
  for (++w.t; w.t < (kGathered ? P.step_lo + 1 : P.step_hi); ++w.t) {
    if (kGathered) {  // one gathered block: shard 0 of S natural-order rows
      w.r = 0;
      w.nt = visit_tiles(RA_LAYOUT_CONTIGUOUS, 1, P.seq, P.causal, 0, maxq);
    } else {
      w.r = (p - w.t + P.n_shards) % P.n_shards;
      w.nt = visit_tiles(P.layout, P.n_shards, P.s_n, P.causal, w.r, maxq);
    }
    if (w.nt > 0) {
      w.kt = 0;
      return;
    }
  }
}
template <bool kGathered>
__device__ __forceinline__ void walk_begin(Walk& w, const FwdParams& P, int p, int64_t maxq) {
  w.t = P.step_lo - 1;
  w.kt = 0;
  w.nt = 0;
  walk_to_next_step<kGathered>(w, P, p, maxq);
}
template <bool kGathered>
__device__ __forceinline__ void walk_advance(Walk& w, const FwdParams& P, int p, int64_t maxq) {
  if (++w.kt >= w.nt) walk_to_next_step<kGathered>(w, P, p, maxq);
}

// ------------------------------------------------------------- work items --
// The producer warp decides which item comes next and passes its index to the
// other roles through a small ring in shared memory.  Two schedules:
//  - dynamic: the next index of the (longest-first, key/value-head-grouped) list
//    from a global counter, so the items in flight are always neighbours in the
//    list and the grid ends evenly;
//  - round-synchronised (large problems): round u gives CTA b item u*grid + b and
//    begins only when every CTA has issued the previous round's loads.  The CTAs
//    of a round then walk the same K/V at the same pace instead of drifting apart
//    over long items, and the K/V they stream stays within L2.

// Consumer side: index of this role's u-th item, or -1 at the end / on abort.
__device__ __forceinline__ int next_item(const Ctl& c, volatile int32_t* slots, uint32_t u, int lane) {
  const uint32_t slot = u % kItemSlots, use = u / kItemSlots;
  if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kItemFull + (int)slot), use & 1u, kStatusTimeoutSoftmax)))
    return -1;
  const int idx = slots[slot];
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(c.bar(kItemEmpty + (int)slot));
  return idx;
}

// ------------------------------------------------------------------ producer --
#define TMA_Q(d, m, b, x, y) ptx::tma_load_2d_warp_hint(d, m, b, x, y, once)
#define TMA_KV(d, m, b, x, y) ptx::tma_load_2d_warp_hint(d, m, b, x, y, keep)
struct ProducerState {
  uint32_t kv_issued;
  uint32_t q_issued;
};

// Producer-side grid barrier for round-synchronised schedules: wait (bounded, like
// every wait here) until the shared counter reaches `need`.
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

template <bool kGathered>
__device__ void run_producer(const FwdParams& P, const Ctl& c, uint32_t sbase, volatile int32_t* slots,
                             const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                             ProducerState& st) {
  uint32_t kv_it = 0;
  const int lane = threadIdx.x & 31;
  const uint64_t keep = ptx::l2_policy_evict_last();   // K/V: re-read by the CTAs running together
  const uint64_t once = ptx::l2_policy_evict_first();  // Q: read once
  for (uint32_t u = 0;; ++u) {
    // Publish the next item index (or -1 at the end) to the other roles.
    const uint32_t slot = u % kItemSlots, use = u / kItemSlots;
    if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kItemEmpty + (int)slot), (use & 1u) ^ 1u, kStatusTimeoutProducer)))
      break;
    int idx;
    if (P.round_sync) {
      // Round u: item u*grid + b, once every CTA has issued the loads of round u-1
      // (all earlier rounds are full: only the last one can be short).
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
    RA_BOUNDS(c.status, idx < P.n_items, 1);
    const WorkItem it = P.items[idx];
    if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kQEmpty), (u & 1u) ^ 1u, kStatusTimeoutProducer))) break;
    const bool two = it.bh1 >= 0;
    const int64_t rows_q = (int64_t)P.batch * P.heads_q * P.seq;
    ptx::mbar_arrive_expect_tx_warp(c.bar(kQFull), (two ? 2u : 1u) * kTileBytes);
    const int32_t y0 = (int32_t)((int64_t)it.bh0 * P.seq + (int64_t)it.shard * P.s_n + it.row0);
    RA_BOUNDS(c.status, it.shard >= 0 && it.shard < P.n_shards && it.row0 >= 0 && it.row0 < P.s_n, 2);
    RA_BOUNDS(c.status, y0 >= 0 && y0 < rows_q, 3);
    TMA_Q(sbase + kOffQ, tq, c.bar(kQFull), 0, y0);
    TMA_Q(sbase + kOffQ + kHalfBytes, tq, c.bar(kQFull), 64, y0);
    if (two) {
      const int32_t y1 = (int32_t)((int64_t)it.bh1 * P.seq + (int64_t)it.shard * P.s_n + it.row1);
      RA_BOUNDS(c.status, it.row1 >= 0 && it.row1 < P.s_n && y1 >= 0 && y1 < rows_q, 3);
      TMA_Q(sbase + kOffQ + kTileBytes, tq, c.bar(kQFull), 0, y1);
      TMA_Q(sbase + kOffQ + kTileBytes + kHalfBytes, tq, c.bar(kQFull), 64, y1);
    }
    st.q_issued = u + 1;
    const int b = it.bh0 / P.heads_q;
    const int kvh = (it.bh0 % P.heads_q) / P.group;
    const int64_t kv_base = (int64_t)(b * P.heads_kv + kvh) * P.seq;
    Walk w;
    walk_begin<kGathered>(w, P, it.shard, it.maxq);
    bool ok = true;
    while (ok && w.t < P.step_hi) {
      const int slot = P.kv_rotated ? it.shard : w.r;  // where the block of step t sits
      const int32_t y = (int32_t)(kv_base + (kGathered ? 0 : (int64_t)slot * P.s_n) + (int64_t)w.kt * kTileRows);
      RA_BOUNDS(c.status, w.r >= 0 && w.r < P.n_shards && w.kt >= 0 && w.kt < w.nt &&
                              (int64_t)w.kt * kTileRows < (kGathered ? P.seq : P.s_n), 4);
      RA_BOUNDS(c.status, y >= 0 && y < (int64_t)P.batch * P.heads_kv * P.seq, 5);
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // K tile, then V tile
        const uint32_t s = kv_it % kStages, use = kv_it / kStages;
        if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kKVEmpty + s), (use & 1u) ^ 1u, kStatusTimeoutProducer))) {
          ok = false;
          break;
        }
        const uint32_t dst = sbase + kOffKV + s * kTileBytes;
        const CUtensorMap* map = which ? tv : tk;
        ptx::mbar_arrive_expect_tx_warp(c.bar(kKVFull + s), kTileBytes);
        TMA_KV(dst, map, c.bar(kKVFull + s), 0, y);
        TMA_KV(dst + kHalfBytes, map, c.bar(kKVFull + s), 64, y);
        st.kv_issued = ++kv_it;
      }
      walk_advance<kGathered>(w, P, it.shard, it.maxq);
    }
    if (!ok) break;
    if (P.round_sync) {
      if (lane == 0) atomicAdd(P.item_counter, 1u);  // this CTA has issued its round
      __syncwarp();
    }
  }
}

// ----------------------------------------------------------------------- MMA --
// Descriptor low words of the tiles the MMA thread reads (see ptx::desc_lo).
struct Descs {
  uint32_t q0;  // Q0 (K-major); Q1 follows one tile later
  uint32_t k0;  // K/V ring slot 0 as a K-major operand (K)
  uint32_t v0;  // slot 0 as an MN-major operand (V); slot s adds s tiles
};
constexpr uint32_t kTileDesc = kTileBytes >> 4;  // one tile in descriptor address units

__device__ __forceinline__ void issue_s(const Descs& dl, uint32_t tmem, int g, uint32_t ks) {
  const uint32_t a0 = dl.q0 + (uint32_t)g * kTileDesc, b0 = dl.k0 + ks * kTileDesc;
#pragma unroll
  for (uint32_t kk = 0; kk < 8; ++kk) {  // 8 steps of K = 16 over d = 128
    const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3u) * 32u) >> 4;
    ptx::mma_bf16_ss_lo_warp(tmem + col_s(g), a0 + off, b0 + off, kIdescS, kk > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ void issue_pv(const Descs& dl, uint32_t tmem, int g, uint32_t vs, bool accumulate) {
  const uint32_t a0 = tmem + col_s(g) + kColP;  // P in tensor memory
  const uint32_t b0 = dl.v0 + vs * kTileDesc;
#pragma unroll
  for (uint32_t kk = 0; kk < 8; ++kk) {  // 8 steps of 16 keys = 8 TMEM columns of P
    // V is [keys][d]: 16 keys = 2 groups of 8 rows (SBO 1 KiB); d halves 16 KiB apart (LBO).
    ptx::mma_bf16_ts_lo_warp(tmem + col_o(g), a0 + kk * 8u, b0 + ((kk * 2048u) >> 4), kIdescPV,
                        (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <bool kGathered>
__device__ void run_mma(const FwdParams& P, const Ctl& c, uint32_t sbase, volatile int32_t* slots, uint32_t tmem) {
  const bool partials = P.o_parts != nullptr;
  Descs dl;
  dl.q0 = ptx::desc_lo(sbase + kOffQ, 16);
  dl.k0 = ptx::desc_lo(sbase + kOffKV, 16);
  dl.v0 = ptx::desc_lo(sbase + kOffKV, kHalfBytes);
  uint32_t kv_it = 0, pj0 = 0, pj1 = 0;
  const int lane = threadIdx.x & 31;
  // the column map (S0, S1, O0, O1 = 0, 128, 256, 384) needs all 512 columns from 0
  RA_BOUNDS(c.status, tmem == 0u && col_o(1) + 128u <= kTmemCols, 6);
  for (uint32_t u = 0;; ++u) {
    const int idx = next_item(c, slots, u, lane);
    if (idx < 0) break;
    const WorkItem it = P.items[idx];
    const bool two = it.bh1 >= 0;
    // Waits on TMA-filled buffers need no tcgen05 fence: the mbarrier completion
    // already orders the async-proxy writes before the MMAs that read them.
    if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kQFull), u & 1u, kStatusTimeoutMma))) return;
    Walk cur;
    walk_begin<kGathered>(cur, P, it.shard, it.maxq);
    if (cur.t >= P.step_hi) {
      ptx::mma_commit_warp(c.bar(kQEmpty));
      continue;
    }
    uint32_t ks = kv_it % kStages;
    if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kKVFull + ks), (kv_it / kStages) & 1u, kStatusTimeoutMma))) return;
    issue_s(dl, tmem, 0, ks);
    ptx::mma_commit_warp(c.bar(kSFull + 0));
    if (two) {
      issue_s(dl, tmem, 1, ks);
      ptx::mma_commit_warp(c.bar(kSFull + 1));
    }
    ptx::mma_commit_warp(c.bar(kKVEmpty + ks));
    ++kv_it;
    bool first_tile = true;
    for (;;) {
      Walk nxt = cur;
      walk_advance<kGathered>(nxt, P, it.shard, it.maxq);
      const bool has_next = nxt.t < P.step_hi;
      const bool seg_first = partials ? (cur.kt == 0) : first_tile;
      const bool seg_last = partials ? (!has_next || nxt.t != cur.t) : !has_next;
      const uint32_t vs = kv_it % kStages;
      if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kKVFull + vs), (kv_it / kStages) & 1u, kStatusTimeoutMma))) return;
      ++kv_it;
      if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kPFull + 0), pj0 & 1u, kStatusTimeoutMma))) return;
      ++pj0;
      ptx::tc_fence_after();
      issue_pv(dl, tmem, 0, vs, !seg_first);
      if (seg_last) ptx::mma_commit_warp(c.bar(kOFull + 0));
      uint32_t ks2 = 0;
      if (has_next) {
        ks2 = kv_it % kStages;
        if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kKVFull + ks2), (kv_it / kStages) & 1u, kStatusTimeoutMma))) return;
        ptx::tc_fence_after();
        issue_s(dl, tmem, 0, ks2);
        ptx::mma_commit_warp(c.bar(kSFull + 0));
      }
      if (two) {
        if (!__all_sync(0xffffffffu, wait_bar(c, c.bar(kPFull + 1), pj1 & 1u, kStatusTimeoutMma))) return;
        ++pj1;
        ptx::tc_fence_after();
        issue_pv(dl, tmem, 1, vs, !seg_first);
        if (seg_last) ptx::mma_commit_warp(c.bar(kOFull + 1));
      }
      ptx::mma_commit_warp(c.bar(kKVEmpty + vs));
      if (!has_next) break;
      if (two) {
        issue_s(dl, tmem, 1, ks2);
        ptx::mma_commit_warp(c.bar(kSFull + 1));
      }
      ptx::mma_commit_warp(c.bar(kKVEmpty + ks2));
      ++kv_it;
      cur = nxt;
      first_tile = false;
    }
    ptx::mma_commit_warp(c.bar(kQEmpty));
  }
}

// ------------------------------------------------------------------- softmax --
__device__ __forceinline__ void store_segment(const FwdParams& P, uint32_t tO, float m, float l,
                                              bool valid, int64_t out_row, int t) {
  const float inv = l > 0.f ? 1.0f / l : 0.f;
  const float lse = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  const int64_t rows_all = (int64_t)P.batch * P.heads_q * P.seq;
  if (P.o_parts != nullptr) {
    float4* dst = reinterpret_cast<float4*>(P.o_parts + ((int64_t)t * rows_all + out_row) * 128);
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t v[32];
      __syncwarp();
      ptx::tmem_ld32(tO + cc * 32, v);
      if (valid) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[cc * 8 + q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                                        __uint_as_float(v[4 * q + 2]) * inv, __uint_as_float(v[4 * q + 3]) * inv);
      }
    }
    if (valid) P.lse_parts[(int64_t)t * rows_all + out_row] = lse;
  } else {
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(P.o) + out_row * 128);
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t v[32];
      __syncwarp();
      ptx::tmem_ld32(tO + cc * 32, v);
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = ptx::pack_bf16x2(__uint_as_float(v[8 * q + 2 * e]) * inv,
                                    __uint_as_float(v[8 * q + 2 * e + 1]) * inv);
          dst[cc * 4 + q] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    if (valid && P.lse != nullptr) P.lse[out_row] = lse;
  }
}

template <bool kGathered>
__device__ void run_softmax(const FwdParams& P, const Ctl& c, uint32_t sbase, volatile int32_t* slots,
                            uint32_t tmem, int g, int wq, int lane) {
  const int row = wq * 32 + lane;  // TMEM lane = query row of the tile
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = tmem + lane_off + col_s(g);
  const uint32_t tO = tmem + lane_off + col_o(g);
  RA_BOUNDS(c.status, wq >= 0 && wq < 4 && (tS & 0xFFFFu) + 128u <= kTmemCols && (tO & 0xFFFFu) + 128u <= kTmemCols &&
                          (tS & 0xFFFFu) + kColP + 64u <= kTmemCols, 7);
  const bool partials = P.o_parts != nullptr;
  const int N = P.n_shards;
  const int64_t rows_all = (int64_t)P.batch * P.heads_q * P.seq;
  const float sl2 = P.scale_log2;
  uint32_t sj = 0, oj = 0;

  for (uint32_t u = 0;; ++u) {
    const int idx = next_item(c, slots, u, lane);
    if (idx < 0) break;
    const WorkItem it = P.items[idx];
    if (g == 1 && it.bh1 < 0) continue;
    const int bh = g ? it.bh1 : it.bh0;
    const int p = it.shard;
    const int64_t i = (int64_t)(g ? it.row1 : it.row0) + row;
    const bool valid = i < P.s_n;
    const int64_t my_pos = pos_of(P.layout, N, P.s_n, p, valid ? i : P.s_n - 1);
    const int64_t out_row = (int64_t)bh * P.seq + (int64_t)p * P.s_n + i;
    RA_BOUNDS(c.status, !valid || (bh >= 0 && out_row >= 0 && out_row < rows_all), 8);
    int last_t = -1;
    const int t_end = kGathered ? P.step_lo + 1 : P.step_hi;  // gathered: one step
    for (int t = P.step_lo; t < t_end; ++t)
      if (kv_tiles<kGathered>(P, (p - t + N) % N, it.maxq) > 0) last_t = t;

    float m = -INFINITY, l = 0.f;
    bool open = false;
    for (int t = P.step_lo; t < t_end; ++t) {
      const int r = kGathered ? 0 : (p - t + N) % N;
      const int nt = kv_tiles<kGathered>(P, r, it.maxq);
      const int part = t - P.step_lo;  // index of this step's partial
      RA_BOUNDS(c.status, part >= 0 && part < P.step_hi - P.step_lo, 9);
      if (nt == 0) {
        if (partials && valid) {  // nothing of this block is causal for the tile
          float4* dst = reinterpret_cast<float4*>(P.o_parts + ((int64_t)part * rows_all + out_row) * 128);
          for (int q = 0; q < 32; ++q) dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
          P.lse_parts[(int64_t)part * rows_all + out_row] = -INFINITY;
        }
        continue;
      }
      // How many leading keys of the block met the row may see: all of its rows, or
      // (causal) those up to its last key at or before the row's position.  Rows and
      // positions fit in 32 bits (S is at most 2^31 - 1).
      const int kv_rows = (int)(kGathered ? P.seq : P.s_n);
      const int seen = !P.causal ? kv_rows
                                 : 1 + (int)(kGathered ? my_pos : last_le(P.layout, N, P.s_n, r, my_pos));
      const int keys = seen < kv_rows ? seen : kv_rows;
      for (int kt = 0; kt < nt; ++kt) {
        const bool first = partials ? (kt == 0) : !open;
        const bool last = partials ? (kt == nt - 1) : (t == last_t && kt == nt - 1);
        open = true;
        int limit = keys - kt * kTileRows;  // keys of this tile the row sees
        limit = limit < 0 ? 0 : (limit > kTileRows ? kTileRows : limit);
        RA_BOUNDS(c.status, keys >= 0 && keys <= kv_rows && (int64_t)kt * kTileRows < kv_rows, 10);

        bool ok = wait_bar(c, c.bar(kSFull + g), sj & 1u, kStatusTimeoutSoftmax);
        ++sj;
        if (!__all_sync(0xffffffffu, ok)) return;
        ptx::tc_fence_after();

        // The whole 128-column score row in registers (one TMEM round trip); the
        // reducing load also returns the largest score of each 32 columns.
        uint32_t raw[128];
        float mx4[4];
        ptx::tmem_ld128_max(tS, raw, mx4);
        float* s = reinterpret_cast<float*>(raw);
        float mx;
        if (limit < kTileRows) {
          // Causal diagonal / ragged tail: masked keys score -inf and the row max is
          // taken over the rest, with eight independent partial maxima: columns
          // a, a+8, ..., a+120 go to partial a.
#pragma unroll
          for (int e = 0; e < 128; ++e) s[e] = (e < limit) ? s[e] : -INFINITY;
          float mx8[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) mx8[a] = ptx::max3(s[a], s[a + 8], s[a + 16]);
#pragma unroll
          for (int e = 24; e + 16 <= 120; e += 16)
#pragma unroll
            for (int a = 0; a < 8; ++a) mx8[a] = ptx::max3(mx8[a], s[e + a], s[e + 8 + a]);
#pragma unroll
          for (int a = 0; a < 8; ++a) mx8[a] = fmaxf(mx8[a], s[120 + a]);
          mx = fmaxf(ptx::max3(mx8[0], mx8[1], mx8[2]),
                     fmaxf(ptx::max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        } else {
          mx = fmaxf(ptx::max3(mx4[0], mx4[1], mx4[2]), mx4[3]);
        }
        const float mt = mx * sl2;  // in log2 units; -inf stays -inf
        float m_new = m;
        bool resc = false;
        if (first) {
          m_new = mt;
          l = 0.f;
        } else if (mt > m + kRescaleSlack) {
          m_new = mt;
          resc = true;
        }
        const float alpha = resc ? ptx::ex2_approx(m - m_new) : 1.0f;
        m = m_new;
        const float mref = (m == -INFINITY) ? 0.f : m;

        // p = 2^(s*scale*log2e - m) (masked -inf -> 0), row sum, P to tensor memory as bf16.
        const float2 sc2 = make_float2(sl2, sl2);
        const float2 neg = make_float2(-mref, -mref);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        // Packed P word e overwrites register e, whose score was already consumed.
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          float2 x = ptx::fma2(make_float2(s[2 * e], s[2 * e + 1]), sc2, neg);
          x.x = ptx::ex2_approx(x.x);
          x.y = ptx::ex2_approx(x.y);
          acc[e & 3] = ptx::add2(acc[e & 3], x);
          raw[e] = ptx::pack_bf16x2(x.x, x.y);
        }
        ptx::tmem_st64(tS + kColP, *reinterpret_cast<const uint32_t(*)[64]>(raw));
        const float2 a01 = ptx::add2(acc[0], acc[1]);
        const float2 a23 = ptx::add2(acc[2], acc[3]);
        const float2 a = ptx::add2(a01, a23);
        // The PV MMA weighs each key by its bf16-rounded p while l sums the fp32 p.
        // Replace the tile's largest p by its rounded value in l as well: when one
        // key dominates a row, its rounding then cancels in o / l.
        // (computed by the same packed multiply-add as the loop's p, so that it is
        // bit for bit the p of the row's largest score)
        const float p_top = ptx::ex2_approx(ptx::fma2(make_float2(mx, mx), sc2, neg).x);
        const float p_top_bf = __uint_as_float(ptx::pack_bf16x2(p_top, 0.f) << 16);
        const float top_fix = p_top_bf - p_top;
        if (!first && __any_sync(0xffffffffu, resc)) {
          // O and l were accumulated against the old max: bring them to the new one
          // (after the scores are consumed, so their registers are free).
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            __syncwarp();
            ptx::tmem_ld32(tO + cc * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            ptx::tmem_st32(tO + cc * 32, v);
          }
          l *= alpha;
        }
        l += (a.x + a.y) + top_fix;
        ptx::tc_fence_before();
        ptx::mbar_arrive(c.bar(kPFull + g));

        if (last) {
          ok = wait_bar(c, c.bar(kOFull + g), oj & 1u, kStatusTimeoutSoftmax);
          ++oj;
          if (!__all_sync(0xffffffffu, ok)) return;
          ptx::tc_fence_after();
          store_segment(P, tO, m, l, valid, out_row, part);
          ptx::tc_fence_before();
          m = -INFINITY;
          l = 0.f;
        }
        __syncwarp();
      }
    }
  }
}

template <bool kGathered>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const FwdParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl c{sbase + kOffBar, reinterpret_cast<volatile uint32_t*>(sgen + kOffAbort), P.status};
  volatile int32_t* slots = reinterpret_cast<volatile int32_t*>(sgen + kOffItems);

  if (threadIdx.x == 0) {
    ptx::mbar_init(c.bar(kQFull), 1);
    ptx::mbar_init(c.bar(kQEmpty), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(c.bar(kKVFull + s), 1);
      ptx::mbar_init(c.bar(kKVEmpty + s), 1);
    }
    for (int g = 0; g < 2; ++g) {
      ptx::mbar_init(c.bar(kSFull + g), 1);
      ptx::mbar_init(c.bar(kPFull + g), 128);
      ptx::mbar_init(c.bar(kOFull + g), 1);
    }
    ptx::mbar_init(c.bar(kDone), 1);
    for (int s2 = 0; s2 < kItemSlots; ++s2) {
      ptx::mbar_init(c.bar(kItemFull + s2), 1);
      ptx::mbar_init(c.bar(kItemEmpty + s2), kItemConsumers);
    }
    *c.abort = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tq);
    ptx::tma_prefetch_desc(&tk);
    ptx::tma_prefetch_desc(&tv);
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + kOffSlot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + kOffSlot);

  ProducerState ps{0u, 0u};
  if (warp < 4) {
    ptx::regs_release<kRegsOther>();
    if (warp == 0) {
      run_producer<kGathered>(P, c, sbase, slots, &tq, &tk, &tv, ps);  // whole warp; one elected lane issues
      __syncwarp();
    } else if (warp == 1) {
      // The whole warp runs the MMA loop with warp-uniform values; one elected
      // lane issues each tcgen05 instruction.
      run_mma<kGathered>(P, c, sbase, slots, tmem);
      // Every MMA this warp issued must retire before TMEM is freed.
      ptx::mma_commit_warp(c.bar(kDone));
      drain_bar(c, c.bar(kDone), 0);
      __syncwarp();
    }
  } else {
    ptx::regs_acquire<kRegsSoftmax>();
    run_softmax<kGathered>(P, c, sbase, slots, tmem, (warp - 4) >> 2, warp & 3, lane);
  }

  if (warp == 0 && lane == 0 && *c.abort) {  // (every lane of warp 0 holds the same counts)
    // Let this CTA's own TMA loads land before its shared memory goes away.
    for (uint32_t s = 0; s < (uint32_t)kStages; ++s) {
      if (ps.kv_issued > s) {
        const uint32_t uses = (ps.kv_issued - 1 - s) / kStages + 1;  // loads issued to slot s
        drain_bar(c, c.bar(kKVFull + s), (uses - 1) & 1u);
      }
    }
    if (ps.q_issued > 0) drain_bar(c, c.bar(kQFull), (ps.q_issued - 1) & 1u);
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

// [rows, 128] bf16 row-major, boxes of 128 rows x 64 columns, 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128 * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kGathered>
cudaError_t launch_kernel(const FwdParams& prm, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          int grid, cudaStream_t stream, const char** why) {
  static std::atomic<int> ready[kMaxDevices];
  cudaError_t e = prepare_once(fwd_bf16_kernel<kGathered>, ready, kThreads, 128 * kRegsOther + 256 * kRegsSoftmax,
                               (int)kSmemBytes, why);
  if (e != cudaSuccess) return e;
  if (prm.round_sync) {
    // The rounds wait on each other: a cooperative launch guarantees that every CTA
    // is resident at once (it fails instead of starting otherwise).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute coop[1];
    coop[0].id = cudaLaunchAttributeCooperative;
    coop[0].val.cooperative = 1;
    cfg.attrs = coop;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fwd_bf16_kernel<kGathered>, tq, tk, tv, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
  } else {
    fwd_bf16_kernel<kGathered><<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, prm);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) *why = "tensor-core forward launch failed";
  return e;
}

}  // namespace

int fwd_bf16_smem_bytes() { return (int)kSmemBytes; }

cudaError_t launch_fwd_bf16(const FwdParams& prm, const void* q, const void* k, const void* v,
                            int grid, cudaStream_t stream, const char** why) {
  CUtensorMap tq, tk, tv;
  const int64_t rows_q = (int64_t)prm.batch * prm.heads_q * prm.seq;
  const int64_t rows_kv = (int64_t)prm.batch * prm.heads_kv * prm.seq;
  if (!encode_rows(&tq, q, rows_q) || !encode_rows(&tk, k, rows_kv) || !encode_rows(&tv, v, rows_kv)) {
    *why = "cuTensorMapEncodeTiled failed or is unavailable";
    return cudaErrorInvalidValue;
  }
  return prm.gathered ? launch_kernel<true>(prm, tq, tk, tv, grid, stream, why)
                      : launch_kernel<false>(prm, tq, tk, tv, grid, stream, why);
}

}  // namespace ra
