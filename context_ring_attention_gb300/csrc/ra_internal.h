// Internal declarations shared by the C ABI (ra_api.cu) and the kernels.
//
// Layout maps, the virtual-ring schedule and the causal tile rule live here so
// that the host planner and every kernel use one definition of each.
#pragma once

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#include "ra.h"

#ifdef __CUDACC__
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

constexpr int kTileRows = 128;  // query rows and key rows per tensor-core tile

// Natural position of local row i of shard p (see include/ra.h).
//   contiguous: p*S_N + i
//   striped:    i*N + p            (Module 23, "The Causal Imbalance -- and the
//                                   Striped Fix")
//   zigzag:     chunk p then chunk 2N-1-p, chunks of c = S_N/2 rows
RA_HD int64_t pos_of(int layout, int n_shards, int64_t s_n, int p, int64_t i) {
  if (layout == RA_LAYOUT_STRIPED) return i * n_shards + p;
  if (layout == RA_LAYOUT_ZIGZAG) {
    const int64_t c = s_n >> 1;
    return i < c ? p * c + i : (int64_t)(2 * n_shards - 1 - p) * c + (i - c);
  }
  return (int64_t)p * s_n + i;
}

// Largest local row j of shard r whose position is <= P, or -1.  Positions rise
// with the local row in every layout, so the causal keys of a query at position P
// within shard r are exactly rows 0..last_le(r, P).
RA_HD int64_t last_le(int layout, int n_shards, int64_t s_n, int r, int64_t P) {
  int64_t j;
  if (layout == RA_LAYOUT_STRIPED) {
    if (P < r) return -1;
    j = (P - r) / n_shards;
  } else if (layout == RA_LAYOUT_ZIGZAG) {
    const int64_t c = s_n >> 1;
    const int64_t lo = (int64_t)r * c;
    const int64_t hi = (int64_t)(2 * n_shards - 1 - r) * c;
    if (P < lo) return -1;
    if (P < hi) j = (P - lo < c - 1) ? P - lo : c - 1;
    else j = c + (P - hi);
  } else {
    j = P - (int64_t)r * s_n;
    if (j < 0) return -1;
  }
  return j < s_n - 1 ? j : s_n - 1;
}

// Number of key tiles of shard r a query tile whose largest position is maxq
// must visit: tiles past the last causal key are skipped (Module 23, "Exact by
// Construction": blocks strictly in the future are skipped).
RA_HD int visit_tiles(int layout, int n_shards, int64_t s_n, int causal, int r, int64_t maxq) {
  const int nk = (int)((s_n + kTileRows - 1) / kTileRows);
  if (!causal) return nk;
  const int64_t j = last_le(layout, n_shards, s_n, r, maxq);
  return j < 0 ? 0 : (int)(j / kTileRows) + 1;
}

// One unit of work for the tensor-core kernel: up to two 128-row query tiles
// that share their key/value head and their tile schedule.
struct alignas(16) WorkItem {
  int32_t bh0;    // b*Hq + h of query tile 0
  int32_t bh1;    // b*Hq + h of query tile 1, or -1 when the item has one tile
  int32_t shard;  // p
  int32_t row0;   // first local row (within shard p) of tile 0
  int32_t row1;   // first local row of tile 1
  int32_t maxq;   // largest natural position among the item's valid rows
  int32_t cost;   // key tiles visited (longest-first ordering key)
  int32_t pad;
};

// Work items of a bf16 forward per query shard: query tiles are paired per item,
// two heads of a GQA group at the same rows when Hq/Hkv is even, else two
// consecutive row tiles of one head.
inline int64_t fwd_items_per_shard(const ra_problem& pb, int64_t s_n) {
  const int64_t n_qt = (s_n + kTileRows - 1) / kTileRows;
  return ((pb.heads_q / pb.heads_kv) % 2 == 0) ? n_qt * pb.batch * (pb.heads_q / 2)
                                                : ((n_qt + 1) / 2) * pb.batch * pb.heads_q;
}

// The forward's work list in creation order: emit(item) for every item, each
// costed by the key tiles it visits over the N ring steps.  The planner and the
// plan-free entry point both build their lists here, so that both hand the
// kernel the same items in the same schedule order.
template <class Emit>
void for_each_fwd_item(const ra_problem& pb, int64_t s_n, Emit&& emit) {
  const int N = pb.n_shards;
  const int n_qt = (int)((s_n + kTileRows - 1) / kTileRows);
  const bool head_pairs = ((pb.heads_q / pb.heads_kv) % 2) == 0;
  for (int p = 0; p < N; ++p)
    for (int qt = 0; qt < n_qt; qt += head_pairs ? 1 : 2)
      for (int64_t b = 0; b < pb.batch; ++b)
        for (int h = 0; h < pb.heads_q; h += head_pairs ? 2 : 1) {
          WorkItem w{};
          w.bh0 = (int32_t)(b * pb.heads_q + h);
          w.shard = p;
          w.row0 = qt * kTileRows;
          if (head_pairs) {
            w.bh1 = w.bh0 + 1;
            w.row1 = w.row0;
          } else if (qt + 1 < n_qt) {
            w.bh1 = w.bh0;
            w.row1 = w.row0 + kTileRows;
          } else {
            w.bh1 = -1;
            w.row1 = w.row0;
          }
          const int64_t top = (w.bh1 >= 0) ? w.row1 : w.row0;
          const int64_t last = (top + kTileRows < s_n ? top + kTileRows : s_n) - 1;
          w.maxq = (int32_t)pos_of(pb.layout, N, s_n, p, last);
          int cost = 0;
          for (int t = 0; t < N; ++t) cost += visit_tiles(pb.layout, N, s_n, pb.causal, (p - t + N) % N, w.maxq);
          w.cost = cost;
          emit(w);
        }
}

// Schedule order of work items for the persistent grid, which hands items out
// round-robin: longest first (so the grid ends evenly), but items whose cost lies
// in the same bucket of ~1% of the largest cost are ordered by (batch, key/value
// head) first.  A round of items then mostly streams one key/value head, so the
// CTAs that run together read the same K/V tiles and share them through L2.
struct ScheduleKey {
  int64_t bucket, kv, cost, seq;
};
inline ScheduleKey schedule_key(const WorkItem& w, int heads_q, int group, int64_t bucket_width, int64_t seq) {
  const int64_t b = w.bh0 / heads_q, h = w.bh0 % heads_q;
  return {w.cost / bucket_width, b * (heads_q / group) + h / group, w.cost, seq};
}
inline bool schedule_before(const ScheduleKey& a, const ScheduleKey& b) {
  if (a.bucket != b.bucket) return a.bucket > b.bucket;
  if (a.kv != b.kv) return a.kv < b.kv;
  if (a.cost != b.cost) return a.cost > b.cost;
  return a.seq < b.seq;
}
inline int64_t schedule_bucket_width(int64_t max_cost) { return max_cost >= 200 ? max_cost / 100 : 1; }

// Kept at 128 bytes: a larger parameter block measurably changes the forward
// kernel's register allocation (it starts to spill).
struct FwdParams {
  int32_t batch, heads_q, heads_kv, group, head_dim, n_shards;
  int16_t layout, causal;
  // Ring steps this launch runs, [step_lo, step_hi): 0..N for a whole forward, one
  // step for a per-step launch.  Partials are indexed t - step_lo.
  int16_t step_lo, step_hi;
  int64_t seq, s_n;
  int32_t n_items;
  float scale;       // score scale
  float scale_log2;  // scale * log2(e)
  // 0: the key/value block of step t for query shard p is read in place, at the rows
  // of shard r = (p - t) mod N.  1: it is read from shard p's own rows of a receive
  // buffer that holds, in slot p, the block shard p has been passed by step t.
  int8_t kv_rotated;
  // 0: CTAs take work items from a counter as they free up.  1: round u gives CTA b
  // item u*grid + b and starts only when every CTA has issued the previous round's
  // loads (cooperative launch), so the CTAs of a round stream the same K/V in step.
  int8_t round_sync;
  // 1: K and V are one gathered block of all S keys in natural order (the
  // all-gather variant): the key side is one contiguous shard of S rows, met in a
  // single step.  0: K/V in the queries' layout, met shard by shard around the ring.
  int8_t gathered;
  int8_t pad_;
  const WorkItem* items;
  void* o;           // fused output, plan dtype
  float* lse;        // fused LSE or nullptr
  float* o_parts;    // partials mode outputs or nullptr
  float* lse_parts;
  uint32_t* status;        // device status word (bit set = a wait ran out of budget)
  uint32_t* item_counter;  // next work item, or rounds issued (round_sync); zero before each launch
};
static_assert(sizeof(FwdParams) <= 128, "FwdParams grew past 128 bytes");

// Smallest local row i of shard p whose position is >= P (s_n when none): positions
// rise with the local row, so the queries of shard p that see a key at position P
// are exactly rows first_ge(p, P)..s_n-1.
RA_HD int64_t first_ge(int layout, int n_shards, int64_t s_n, int p, int64_t P) {
  return last_le(layout, n_shards, s_n, p, P - 1) + 1;
}

// Status bits written by kernels into the plan's status word.
enum : uint32_t {
  kStatusTimeoutProducer = 1u << 0,
  kStatusTimeoutMma = 1u << 1,
  kStatusTimeoutSoftmax = 1u << 2,
  kStatusTimeoutTeardown = 1u << 3,
  kStatusTimeouts = 15u,
  kStatusBounds = 1u << 4,  // debug build: a bounds check failed; bits 8-15 hold the OR of the sites
};

// Bounds checks of the debug build (-DRA_DEBUG_BOUNDS, libra_debug.so).  A failed check
// ORs kStatusBounds and its site number (1-255, bits 8-15) into the kernel's status
// word and the kernel carries on; ra_sync_status then returns RA_ERR_BOUNDS.  The
// release build compiles the checks out.
#if defined(RA_DEBUG_BOUNDS)
#define RA_BOUNDS(status, cond, site)                                                  \
  do {                                                                                 \
    if (!(cond)) atomicOr((status), ::ra::kStatusBounds | ((uint32_t)(site) << 8));   \
  } while (0)
#else
#define RA_BOUNDS(status, cond, site) \
  do {                                \
  } while (0)
#endif

// The error a non-zero status word stands for, with its message in msg.
inline ra_status status_word_error(uint32_t word, char* msg, size_t n) {
  if (word & kStatusBounds) {
    snprintf(msg, n, "debug bounds check failed (status word 0x%x; sites OR-ed in bits 8-15: 0x%x)", word,
             (word >> 8) & 0xFFu);
    return RA_ERR_BOUNDS;
  }
  snprintf(msg, n, "device wait ran out of budget (status bits 0x%x: 1 producer, 2 mma, 4 softmax, 8 teardown)",
           word);
  return RA_ERR_TIMEOUT;
}

// Whether a bf16 problem runs its forward in synchronised rounds: when one key/value
// head's K and V (S x d x 2 bytes each) exceed 32 MiB, so that CTAs drifting apart
// over their items would stream more K/V than L2 holds, and when the longest item
// (key tiles) stays far below the kernel's wait budget.
RA_HD bool use_round_sync(int64_t seq, int head_dim, int64_t max_item_tiles) {
  return seq * head_dim * 4 > (int64_t(32) << 20) && max_item_tiles <= 131072;
}

// Launchers (each returns cudaGetLastError() of its launch).
cudaError_t launch_fwd_bf16(const FwdParams& prm, const void* q, const void* k, const void* v,
                            int grid, cudaStream_t stream, const char** why);
cudaError_t launch_fwd_f32(const FwdParams& prm, const float* q, const float* k, const float* v,
                           cudaStream_t stream);
cudaError_t launch_merge(int n_parts, int64_t rows, int d, const float* o_parts,
                         const float* lse_parts, void* o, int o_dtype, float* lse,
                         cudaStream_t stream);
cudaError_t launch_layout_perm(int layout, int64_t seq, int n_shards, int inverse,
                               int64_t rows_outer, int row_bytes, const void* src, void* dst,
                               cudaStream_t stream);
int fwd_bf16_smem_bytes();
cudaError_t launch_ulysses_a2a(int dir, int layout, int n, int batch, int heads, int64_t seq, int row_bytes,
                               const void* src, void* dst, cudaStream_t stream);

// Sets the thread-local message returned by ra_last_error().
void set_last_error(const char* msg);

// RA_OK when every non-null pointer of ptrs[0..n) is device memory of the current
// device (or managed memory) and the stream belongs to that device; otherwise
// RA_ERR_INVALID_ARG (RA_ERR_NO_DEVICE without a device), with the message set.
// The kernels run on the current device and read every buffer through it: a
// buffer of another device would be read through a mapping it may not have.
ra_status check_on_current_device(const void* const* ptrs, int n, cudaStream_t stream);

// Device ordinals below this get per-device launch state (kernel attributes set
// once per device, the plan-free entry point's scratch address).
constexpr int kMaxDevices = 64;

// Launch preparation of a warp-specialised tensor-core kernel, done once per
// device (ready[] is the kernel's own flag array): the kernel must have been
// built with at least regs_needed registers per CTA (setmaxnreg.inc waits for
// registers that exist only in the launch's allocation), and its dynamic
// shared-memory limit is raised to smem_bytes.
template <class Kernel>
cudaError_t prepare_once(Kernel kernel, std::atomic<int>* ready, uint32_t threads, uint32_t regs_needed,
                         int smem_bytes, const char** why) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *why = "cudaGetDevice failed";
    return e;
  }
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && ready[dev].load(std::memory_order_acquire)) return cudaSuccess;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kernel);
  if (e != cudaSuccess) {
    *why = "cudaFuncGetAttributes failed";
    return e;
  }
  if ((uint32_t)attr.numRegs * threads < regs_needed) {
    *why = "kernel was built with fewer launch registers than its warpgroup split needs";
    return cudaErrorInvalidConfiguration;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) {
    *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  if (cached) ready[dev].store(1, std::memory_order_release);
  return cudaSuccess;
}

}  // namespace ra
