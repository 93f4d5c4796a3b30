// C ABI of libra.so: argument checks, the ring planner and kernel dispatch.
//
// The planner turns a problem into the work list of the tensor-core kernel: one
// item per pair of 128-row query tiles that share a key/value head and a tile
// schedule (two query heads of one GQA group at the same rows, or two
// consecutive row tiles of one head), each with the number of key tiles it
// visits over the N ring steps.  Items are ordered longest first so the
// persistent grid ends evenly under a causal mask, whose per-shard work is
// uneven for contiguous shards (Module 23, "The Causal Imbalance -- and the
// Striped Fix").  For per-step launches (ra_fwd_step, ra_ring_fwd) the plan also
// holds one list per ring step, ordered by that step's cost alone.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <exception>
#include <new>
#include <vector>

#include "ra_internal.h"
#include "bwd_internal.h"

struct ra_plan_s {
  ra_problem prob;
  int64_t s_n;
  int n_qtiles, n_ktiles;
  std::vector<ra::WorkItem> items;       // whole forward: all N steps per item
  std::vector<ra::WorkItem> step_items;  // per-step lists, concatenated
  std::vector<ra::WorkItem> bwd_items;   // backward: key tiles (dK, dV), then query tiles (dQ)
  std::vector<ra::WorkItem> gather_items;  // forward over gathered (natural-order) K/V
  bool gather_round_sync = false;
  int64_t n_bwd_kv = 0;                  // how many of bwd_items are key tiles
  bool bwd_round_sync[2] = {false, false};  // per backward pass (ra::use_round_sync)
  std::vector<int64_t> step_off;         // list of step t is [step_off[t], step_off[t+1])
  std::vector<int64_t> full, partial, skip;
  int device = -1;
  ra::WorkItem* d_items = nullptr;
  ra::WorkItem* d_step_items = nullptr;
  ra::WorkItem* d_bwd_items = nullptr;
  ra::WorkItem* d_gather_items = nullptr;
  uint32_t* d_status = nullptr;
  // Stream of the plan's own allocations: its device tables are allocated and freed
  // in stream order on it (cudaMallocAsync / cudaFreeAsync), so that destroying a plan
  // never waits on the host for the device.
  cudaStream_t mem_stream = nullptr;
  cudaEvent_t ev_entry = nullptr, ev_rot = nullptr, ev_step = nullptr;  // ra_ring_fwd ordering
  bool round_sync = false;  // forward kernel schedule (ra::use_round_sync)
  int sm_count = 0;
  // One event per stream the plan's kernels were queued on, recorded after the
  // latest of them: ra_plan_destroy queues the frees of the device tables behind
  // exactly this work.  A slot whose event has completed is reused for a new stream.
  struct StreamMark {
    cudaStream_t stream;
    cudaEvent_t done;
  };
  std::vector<StreamMark> marks;
};

namespace {

thread_local char g_err[512] = "";

ra_status fail(ra_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

ra_status ok() {
  g_err[0] = '\0';
  return RA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ra_status check_layout(int32_t layout, int64_t seq, int32_t n) {
  if (layout < RA_LAYOUT_CONTIGUOUS || layout > RA_LAYOUT_ZIGZAG)
    return fail(RA_ERR_INVALID_ARG, "unknown layout %d", layout);
  if (seq < 1 || n < 1) return fail(RA_ERR_INVALID_ARG, "seq and n_shards must be >= 1");
  if (seq % n) return fail(RA_ERR_INVALID_ARG, "seq %lld is not a multiple of n_shards %d (uneven shards)", (long long)seq, n);
  if (layout == RA_LAYOUT_ZIGZAG && seq % (2 * (int64_t)n))
    return fail(RA_ERR_INVALID_ARG, "zigzag needs seq %lld to be a multiple of 2*n_shards", (long long)seq);
  if (seq > INT32_MAX) return fail(RA_ERR_UNSUPPORTED, "seq above 2^31-1");
  if (n > INT16_MAX) return fail(RA_ERR_UNSUPPORTED, "n_shards above 32767");
  return RA_OK;
}

constexpr int64_t kMaxPlanPairs = int64_t(1) << 30;
constexpr int64_t kMaxListEntries = int64_t(1) << 27;

ra_status validate(const ra_problem* p) {
  if (p->batch < 1 || p->heads_q < 1 || p->heads_kv < 1 || p->head_dim < 1)
    return fail(RA_ERR_INVALID_ARG, "batch, heads and head_dim must be >= 1");
  ra_status s = check_layout(p->layout, p->seq, p->n_shards);
  if (s != RA_OK) return s;
  if (p->heads_q % p->heads_kv) return fail(RA_ERR_INVALID_ARG, "heads_q %% heads_kv != 0");
  if (p->causal != 0 && p->causal != 1) return fail(RA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(p->scale >= 0.f) || std::isinf(p->scale)) return fail(RA_ERR_INVALID_ARG, "scale must be finite and >= 0");
  if (p->dtype == RA_DTYPE_BF16) {
    if (p->head_dim != 128) return fail(RA_ERR_UNSUPPORTED, "bf16 path needs head_dim == 128 (got %d)", p->head_dim);
  } else if (p->dtype == RA_DTYPE_F32) {
    if (p->head_dim > 128) return fail(RA_ERR_UNSUPPORTED, "f32 path needs head_dim <= 128 (got %d)", p->head_dim);
  } else {
    return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", p->dtype);
  }
  if (p->batch > INT32_MAX / p->heads_q || p->batch * (int64_t)p->heads_q * p->seq > INT32_MAX)
    return fail(RA_ERR_UNSUPPORTED, "B*Hq*S above 2^31-1 rows");
  // The planner's own work: the tile classification visits N x n_qtiles x N
  // (query tile, ring step) pairs, and the tensor-core work lists hold about
  // n_items x (N + 2) entries.  Past these limits planning alone would take
  // tens of seconds to hours and gigabytes of host memory.
  const int64_t N = p->n_shards;
  const int64_t n_qt = (p->seq / N + ra::kTileRows - 1) / ra::kTileRows;
  if (N * N * n_qt > kMaxPlanPairs)
    return fail(RA_ERR_UNSUPPORTED, "ring too large to plan: n_shards^2 x query tiles per shard above 2^30");
  if (p->dtype == RA_DTYPE_BF16) {
    const int64_t per_shard = ra::fwd_items_per_shard(*p, p->seq / N);
    if (per_shard * N * (N + 2) > kMaxListEntries)
      return fail(RA_ERR_UNSUPPORTED, "work lists too large to plan: items x (n_shards + 2) above 2^27");
  }
  return RA_OK;
}

int64_t last_row_pos(const ra_problem& pb, int64_t s_n, int p, int64_t row_start) {
  const int64_t last = std::min<int64_t>(row_start + ra::kTileRows, s_n) - 1;
  return ra::pos_of(pb.layout, pb.n_shards, s_n, p, last);
}

struct Keyed {
  ra::WorkItem w;
  int64_t order;  // creation order, the last tie-break
};

// Items in schedule order (ra::schedule_before on their current cost).
std::vector<ra::WorkItem> schedule(const std::vector<Keyed>& list, int heads_q, int group) {
  int64_t max_cost = 1;
  for (const Keyed& k : list) max_cost = std::max<int64_t>(max_cost, k.w.cost);
  const int64_t width = ra::schedule_bucket_width(max_cost);
  std::vector<ra::ScheduleKey> keys(list.size());
  for (size_t n = 0; n < list.size(); ++n) keys[n] = ra::schedule_key(list[n].w, heads_q, group, width, list[n].order);
  std::vector<size_t> idx(list.size());
  for (size_t n = 0; n < idx.size(); ++n) idx[n] = n;
  std::sort(idx.begin(), idx.end(), [&](size_t a, size_t b) { return ra::schedule_before(keys[a], keys[b]); });
  std::vector<ra::WorkItem> out(list.size());
  for (size_t n = 0; n < list.size(); ++n) out[n] = list[idx[n]].w;
  return out;
}

// Backward work lists.  dK/dV: one item per 128-row key tile (bh0 = b*Hkv + kv
// head, shard r, row0, maxq = position of the tile's first key), costed by the
// 64-row query tiles it meets over the ring (every query head of its group).
// dQ: one item per 128-row query tile (bh0 = b*Hq + h, shard p, row0, maxq =
// position of its last query), costed by the 64-row key tiles it meets.  Both in
// the forward's order rule (longest first, key/value heads grouped).
void build_bwd_schedule(ra_plan_s* pl) {
  const ra_problem& pb = pl->prob;
  const int N = pb.n_shards;
  const int64_t s_n = pl->s_n;
  const int G = pb.heads_q / pb.heads_kv;
  const int n128 = (int)((s_n + 127) / 128), n64 = (int)((s_n + 63) / 64);
  std::vector<Keyed> kv, qs;
  int64_t seqno = 0;
  for (int r = 0; r < N; ++r)
    for (int kt = 0; kt < n128; ++kt)
      for (int64_t b = 0; b < pb.batch; ++b)
        for (int hk = 0; hk < pb.heads_kv; ++hk) {
          ra::WorkItem w{};
          w.bh0 = (int32_t)(b * pb.heads_kv + hk);
          w.bh1 = -1;
          w.shard = r;
          w.row0 = kt * 128;
          w.maxq = (int32_t)ra::pos_of(pb.layout, N, s_n, r, w.row0);
          int cost = 0;
          for (int t = 0; t < N; ++t) {
            const int p = (r + t) % N;
            int lo = 0;
            if (pb.causal) {
              const int64_t f = ra::first_ge(pb.layout, N, s_n, p, w.maxq);
              lo = f >= s_n ? n64 : (int)(f / 64);
            }
            cost += (n64 - lo) * G;
          }
          w.cost = cost;
          kv.push_back({w, seqno++});
        }
  for (int p = 0; p < N; ++p)
    for (int qt = 0; qt < n128; ++qt)
      for (int64_t b = 0; b < pb.batch; ++b)
        for (int h = 0; h < pb.heads_q; ++h) {
          ra::WorkItem w{};
          w.bh0 = (int32_t)(b * pb.heads_q + h);
          w.bh1 = -1;
          w.shard = p;
          w.row0 = qt * 128;
          w.maxq = (int32_t)last_row_pos(pb, s_n, p, w.row0);
          int cost = 0;
          for (int t = 0; t < N; ++t) {
            const int r = (p - t + N) % N;
            if (!pb.causal) {
              cost += n64;
            } else {
              const int64_t j = ra::last_le(pb.layout, N, s_n, r, w.maxq);
              cost += j < 0 ? 0 : (int)(j / 64) + 1;
            }
          }
          w.cost = cost;
          qs.push_back({w, seqno++});
        }
  // schedule_key groups by key/value head from bh0 / heads_q: give the key-tile
  // items a query-head index of their group so that they group the same way.
  std::vector<Keyed> kv_keyed = kv;
  for (Keyed& k : kv_keyed) {
    const int64_t b = k.w.bh0 / pb.heads_kv, hk = k.w.bh0 % pb.heads_kv;
    k.w.bh0 = (int32_t)(b * pb.heads_q + hk * G);
  }
  std::vector<ra::WorkItem> kv_sorted = schedule(kv_keyed, pb.heads_q, G);
  for (ra::WorkItem& w : kv_sorted) {
    const int64_t b = w.bh0 / pb.heads_q, hk = (w.bh0 % pb.heads_q) / G;
    w.bh0 = (int32_t)(b * pb.heads_kv + hk);
  }
  const std::vector<ra::WorkItem> q_sorted = schedule(qs, pb.heads_q, G);
  // Round sync when the streamed data of a head exceeds L2's reach and the longest
  // item (in 64-row tiles, counted as half of a 128-row tile) stays short.
  int64_t max_kv = 0, max_q = 0;
  for (const Keyed& k : kv) max_kv = std::max<int64_t>(max_kv, k.w.cost);
  for (const Keyed& k : qs) max_q = std::max<int64_t>(max_q, k.w.cost);
  pl->bwd_round_sync[0] = ra::use_round_sync(pb.seq, pb.head_dim, max_kv / 2);
  pl->bwd_round_sync[1] = ra::use_round_sync(pb.seq, pb.head_dim, max_q / 2);
  pl->bwd_items = kv_sorted;
  pl->bwd_items.insert(pl->bwd_items.end(), q_sorted.begin(), q_sorted.end());
  pl->n_bwd_kv = (int64_t)kv_sorted.size();
}

void build_schedule(ra_plan_s* pl) {
  const ra_problem& pb = pl->prob;
  const int N = pb.n_shards;
  const int64_t s_n = pl->s_n;
  pl->n_qtiles = (int)((s_n + ra::kTileRows - 1) / ra::kTileRows);
  pl->n_ktiles = pl->n_qtiles;

  // Per-shard tile classification of one 128-row query tile against every key
  // tile it meets over the ring (FULL / PARTIAL / SKIP).
  pl->full.assign(N, 0);
  pl->partial.assign(N, 0);
  pl->skip.assign(N, 0);
  for (int p = 0; p < N; ++p) {
    for (int qt = 0; qt < pl->n_qtiles; ++qt) {
      const int64_t i0 = (int64_t)qt * ra::kTileRows;
      const int64_t qmin = ra::pos_of(pb.layout, N, s_n, p, i0);
      const int64_t qmax = last_row_pos(pb, s_n, p, i0);
      for (int t = 0; t < N; ++t) {
        const int r = (p - t + N) % N;
        if (!pb.causal) {
          pl->full[p] += pl->n_ktiles;
          continue;
        }
        const int visit = ra::visit_tiles(pb.layout, N, s_n, 1, r, qmax);
        const int64_t jmin = ra::last_le(pb.layout, N, s_n, r, qmin);
        // a key tile is FULL when its last key is causal for the tile's first query
        int64_t nfull = 0;
        if (jmin >= s_n - 1) nfull = pl->n_ktiles;
        else if (jmin >= 0) nfull = (jmin + 1) / ra::kTileRows;
        pl->full[p] += nfull;
        pl->partial[p] += visit - nfull;
        pl->skip[p] += pl->n_ktiles - visit;
      }
    }
  }

  if (pb.dtype != RA_DTYPE_BF16) return;  // the SIMT kernel walks rows, not items

  const int G = pb.heads_q / pb.heads_kv;
  std::vector<Keyed> list;
  int64_t seqno = 0;
  ra::for_each_fwd_item(pb, s_n, [&](const ra::WorkItem& w) { list.push_back({w, seqno++}); });
  pl->items = schedule(list, pb.heads_q, G);
  int64_t max_cost = 0;
  for (const Keyed& k : list) max_cost = std::max<int64_t>(max_cost, k.w.cost);
  pl->round_sync = ra::use_round_sync(pb.seq, pb.head_dim, max_cost);

  build_bwd_schedule(pl);

  // The all-gather variant: the same items, each meeting one natural-order block of
  // all S keys (the keys at or before its last query, when causal).
  {
    std::vector<Keyed> g = list;
    int64_t gmax = 0;
    for (Keyed& k : g) {
      k.w.cost = ra::visit_tiles(RA_LAYOUT_CONTIGUOUS, 1, pb.seq, pb.causal, 0, k.w.maxq);
      gmax = std::max<int64_t>(gmax, k.w.cost);
    }
    pl->gather_items = schedule(g, pb.heads_q, G);
    pl->gather_round_sync = ra::use_round_sync(pb.seq, pb.head_dim, gmax);
  }

  // One list per ring step: the same items, costed by that step's key tiles alone.
  // Items with no causal key in the step stay in the list (they write the empty
  // partial: O_t = 0, LSE_t = -inf).
  pl->step_items.clear();
  pl->step_off.assign(1, 0);
  for (int t = 0; t < N; ++t) {
    std::vector<Keyed> step = list;
    for (Keyed& k : step)
      k.w.cost = ra::visit_tiles(pb.layout, N, s_n, pb.causal, (k.w.shard - t + N) % N, k.w.maxq);
    const std::vector<ra::WorkItem> ordered = schedule(step, pb.heads_q, G);
    pl->step_items.insert(pl->step_items.end(), ordered.begin(), ordered.end());
    pl->step_off.push_back((int64_t)pl->step_items.size());
  }
}

ra_status upload(ra_plan_s* pl) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    pl->device = -1;
    return RA_OK;  // host-only plan
  }
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    pl->device = -1;
    return RA_OK;
  }
  pl->device = dev;
  cudaDeviceGetAttribute(&pl->sm_count, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = cudaStreamCreateWithFlags(&pl->mem_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    pl->mem_stream = nullptr;
    return fail(RA_ERR_CUDA, "plan stream: %s", cudaGetErrorString(e));
  }
  cudaStream_t ms = pl->mem_stream;
  e = cudaMallocAsync(reinterpret_cast<void**>(&pl->d_status), 256, ms);
  if (e == cudaSuccess) e = cudaMemsetAsync(pl->d_status, 0, 256, ms);
  auto put = [&](const std::vector<ra::WorkItem>& host, ra::WorkItem** dev) {
    if (e != cudaSuccess || host.empty()) return;
    const size_t bytes = host.size() * sizeof(ra::WorkItem);
    e = cudaMallocAsync(reinterpret_cast<void**>(dev), bytes, ms);
    if (e == cudaSuccess) e = cudaMemcpyAsync(*dev, host.data(), bytes, cudaMemcpyHostToDevice, ms);
  };
  put(pl->items, &pl->d_items);
  put(pl->step_items, &pl->d_step_items);
  put(pl->bwd_items, &pl->d_bwd_items);
  put(pl->gather_items, &pl->d_gather_items);
  // the tables are in place before any launch on another stream reads them
  if (e == cudaSuccess) e = cudaStreamSynchronize(ms);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pl->ev_entry, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pl->ev_rot, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pl->ev_step, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "plan upload failed: %s", cudaGetErrorString(e));
  return RA_OK;
}


// Kernel parameters common to every forward launch of a plan: the whole ring, K/V
// read in place; callers set items, outputs and, for per-step launches, the range.
ra::FwdParams fwd_params(const ra_plan_s* plan) {
  const ra_problem& pb = plan->prob;
  ra::FwdParams prm{};
  prm.batch = (int32_t)pb.batch;
  prm.heads_q = pb.heads_q;
  prm.heads_kv = pb.heads_kv;
  prm.group = pb.heads_q / pb.heads_kv;
  prm.head_dim = pb.head_dim;
  prm.n_shards = pb.n_shards;
  prm.layout = (int16_t)pb.layout;
  prm.causal = (int16_t)pb.causal;
  prm.seq = pb.seq;
  prm.s_n = plan->s_n;
  prm.scale = pb.scale;
  prm.scale_log2 = pb.scale * 1.4426950408889634f;
  prm.status = plan->d_status;
  prm.item_counter = plan->d_status + 1;
  prm.step_lo = 0;
  prm.step_hi = (int16_t)pb.n_shards;
  prm.kv_rotated = 0;
  prm.round_sync = plan->round_sync ? 1 : 0;
  prm.gathered = 0;
  return prm;
}

ra_status mark_use(ra_plan_s* plan, cudaStream_t st);

// Launch the plan's forward kernel (tensor-core for bf16, SIMT for f32) on stream.
ra_status launch(ra_plan_s* plan, const ra::FwdParams& prm, const void* q, const void* k,
                 const void* v, cudaStream_t st) {
  cudaError_t e;
  if (plan->prob.dtype == RA_DTYPE_BF16) {
    if (prm.n_items == 0) return ok();
    const int grid = std::min(prm.n_items, plan->sm_count > 0 ? plan->sm_count : 148);
    const char* why = "";
    // The kernel hands out work items from a counter that starts at zero.
    e = cudaMemsetAsync(prm.item_counter, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "counter reset: %s", cudaGetErrorString(e));
    e = ra::launch_fwd_bf16(prm, q, k, v, grid, st, &why);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
      // Not every CTA can be resident (the GPU is shared): the dynamic schedule
      // needs no co-residency and computes the same result.
      cudaGetLastError();
      ra::FwdParams dyn = prm;
      dyn.round_sync = 0;
      e = ra::launch_fwd_bf16(dyn, q, k, v, grid, st, &why);
    }
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "%s: %s", why, cudaGetErrorString(e));
  } else {
    e = ra::launch_fwd_f32(prm, static_cast<const float*>(q), static_cast<const float*>(k),
                           static_cast<const float*>(v), st);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "f32 forward launch failed: %s", cudaGetErrorString(e));
  }
  const ra_status s = mark_use(plan, st);
  return s != RA_OK ? s : ok();
}

ra_status check_device(const ra_plan_s* plan) {
  if (plan->device < 0) return fail(RA_ERR_NO_DEVICE, "plan was built without a CUDA device");
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device)
    return fail(RA_ERR_INVALID_ARG, "current device %d differs from the plan's device %d", cur, plan->device);
  return RA_OK;
}

// Record, on `st`, that the plan's device tables are in use by the work queued there
// so far (ra_plan_destroy queues its frees behind it).
ra_status mark_use(ra_plan_s* plan, cudaStream_t st) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) cudaGetLastError();
  if (cap != cudaStreamCaptureStatusNone) return RA_OK;  // queued into a graph, not run yet
  ra_plan_s::StreamMark* slot = nullptr;
  for (ra_plan_s::StreamMark& m : plan->marks)
    if (m.stream == st) slot = &m;
  if (slot == nullptr)
    for (ra_plan_s::StreamMark& m : plan->marks)
      if (cudaEventQuery(m.done) == cudaSuccess) {  // that stream's use has ended
        m.stream = st;
        slot = &m;
        break;
      }
  cudaGetLastError();  // a not-ready query is not an error
  if (slot == nullptr) {
    cudaEvent_t ev = nullptr;
    const cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "plan use event: %s", cudaGetErrorString(e));
    plan->marks.push_back({st, ev});
    slot = &plan->marks.back();
  }
  const cudaError_t e = cudaEventRecord(slot->done, st);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "plan use event record: %s", cudaGetErrorString(e));
  return RA_OK;
}

size_t elem_bytes(const ra_problem& pb) { return pb.dtype == RA_DTYPE_BF16 ? 2 : 4; }

bool overlap(const void* a, const void* b, size_t bytes) {
  const char* x = static_cast<const char*>(a);
  const char* y = static_cast<const char*>(b);
  return x < y + bytes && y < x + bytes;
}

// The exchange: dst slot (p + 1) mod N <- src slot p for every [S, d] matrix of a
// [B, Hkv, S, d] tensor.  Two strided copy-engine transfers: slots 0..N-2 move up
// by one shard, slot N-1 wraps to slot 0.
cudaError_t rotate_one(const ra_plan_s* plan, const void* src, void* dst, cudaStream_t st) {
  const ra_problem& pb = plan->prob;
  const size_t row = (size_t)pb.head_dim * elem_bytes(pb);
  const size_t pitch = (size_t)pb.seq * row;
  const size_t shard = (size_t)plan->s_n * row;
  const size_t height = (size_t)pb.batch * pb.heads_kv;
  const int N = pb.n_shards;
  const char* s = static_cast<const char*>(src);
  char* d = static_cast<char*>(dst);
  if (N == 1) return cudaMemcpyAsync(d, s, pitch * height, cudaMemcpyDeviceToDevice, st);
  cudaError_t e = cudaMemcpy2DAsync(d + shard, pitch, s, pitch, (size_t)(N - 1) * shard, height,
                                    cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return e;
  return cudaMemcpy2DAsync(d, pitch, s + (size_t)(N - 1) * shard, pitch, shard, height,
                           cudaMemcpyDeviceToDevice, st);
}

}  // namespace

void ra::set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

ra_status ra::check_on_current_device(const void* const* ptrs, int n, cudaStream_t stream) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_NO_DEVICE, "no CUDA device");
  }
  for (int i = 0; i < n; ++i) {
    if (ptrs[i] == nullptr) continue;
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, ptrs[i]);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(RA_ERR_INVALID_ARG, "pointer %p: %s", ptrs[i], cudaGetErrorString(e));
    }
    if (a.type == cudaMemoryTypeDevice) {
      if (a.device != cur)
        return fail(RA_ERR_INVALID_ARG, "pointer %p is memory of device %d, the current device is %d", ptrs[i],
                    a.device, cur);
    } else if (a.type != cudaMemoryTypeManaged) {
      return fail(RA_ERR_INVALID_ARG, "pointer %p is not device memory", ptrs[i]);
    }
  }
  int sd = -1;
  const cudaError_t e = cudaStreamGetDevice(stream, &sd);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_INVALID_ARG, "stream: %s", cudaGetErrorString(e));
  }
  if (sd != cur) return fail(RA_ERR_INVALID_ARG, "the stream belongs to device %d, the current device is %d", sd, cur);
  return RA_OK;
}

extern "C" {

ra_status ra_plan(const ra_problem* prob, ra_plan_t* out) {
  if (prob == nullptr || out == nullptr) return fail(RA_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  ra_status s = validate(prob);
  if (s != RA_OK) return s;
  ra_plan_s* pl = new (std::nothrow) ra_plan_s();
  if (pl == nullptr) return fail(RA_ERR_UNSUPPORTED, "out of host memory");
  pl->prob = *prob;
  if (pl->prob.scale == 0.f) pl->prob.scale = 1.0f / std::sqrt((float)prob->head_dim);
  pl->s_n = prob->seq / prob->n_shards;
  try {
    build_schedule(pl);
  } catch (const std::exception& ex) {  // host allocation of the work lists failed
    delete pl;
    return fail(RA_ERR_UNSUPPORTED, "planning failed on the host: %s", ex.what());
  }
  s = upload(pl);
  if (s != RA_OK) {
    ra_plan_destroy(pl);
    return s;
  }
  *out = pl;
  return ok();
}

ra_status ra_plan_destroy(ra_plan_t plan) {
  if (plan == nullptr) return ok();
  if (plan->device >= 0) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != plan->device) cudaSetDevice(plan->device);
    // Kernels of this plan queued earlier may still read its work tables or its
    // status word: the frees are queued behind them (and only them), in stream
    // order, and the host does not wait.
    if (plan->mem_stream != nullptr) {
      for (const ra_plan_s::StreamMark& m : plan->marks) cudaStreamWaitEvent(plan->mem_stream, m.done, 0);
      void* mem[] = {plan->d_items, plan->d_step_items, plan->d_bwd_items, plan->d_gather_items, plan->d_status};
      for (void* p : mem)
        if (p != nullptr) cudaFreeAsync(p, plan->mem_stream);
      cudaStreamDestroy(plan->mem_stream);  // released once its queued frees have run
    }
    for (const ra_plan_s::StreamMark& m : plan->marks) cudaEventDestroy(m.done);
    cudaGetLastError();
    if (plan->ev_entry) cudaEventDestroy(plan->ev_entry);
    if (plan->ev_rot) cudaEventDestroy(plan->ev_rot);
    if (plan->ev_step) cudaEventDestroy(plan->ev_step);
    if (cur >= 0 && cur != plan->device) cudaSetDevice(cur);
  }
  delete plan;
  return ok();
}

ra_status ra_plan_tile_counts(ra_plan_t plan, int64_t* full, int64_t* partial, int64_t* skip) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  const size_t n = (size_t)plan->prob.n_shards;
  if (full) std::memcpy(full, plan->full.data(), n * sizeof(int64_t));
  if (partial) std::memcpy(partial, plan->partial.data(), n * sizeof(int64_t));
  if (skip) std::memcpy(skip, plan->skip.data(), n * sizeof(int64_t));
  return ok();
}

ra_status ra_fwd(ra_plan_t plan, const void* q, const void* k, const void* v, void* o, float* lse,
                 float* o_parts, float* lse_parts, void* stream) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  if (q == nullptr || k == nullptr || v == nullptr) return fail(RA_ERR_INVALID_ARG, "null q/k/v");
  const bool partials = o_parts != nullptr || lse_parts != nullptr;
  if (partials) {
    if (o_parts == nullptr || lse_parts == nullptr)
      return fail(RA_ERR_INVALID_ARG, "partials mode needs both o_parts and lse_parts");
    if (o != nullptr || lse != nullptr)
      return fail(RA_ERR_INVALID_ARG, "pass either o/lse (fused) or o_parts/lse_parts (partials), not both");
  } else if (o == nullptr) {
    return fail(RA_ERR_INVALID_ARG, "null o");
  }
  const void* ptrs[] = {q, k, v, o, lse, o_parts, lse_parts};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return fail(RA_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
  ra_status s = check_device(plan);
  if (s == RA_OK) s = ra::check_on_current_device(ptrs, 7, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  ra::FwdParams prm = fwd_params(plan);
  prm.items = plan->d_items;
  prm.n_items = (int32_t)plan->items.size();
  prm.o = o;
  prm.lse = lse;
  prm.o_parts = o_parts;
  prm.lse_parts = lse_parts;
  return launch(plan, prm, q, k, v, static_cast<cudaStream_t>(stream));
}

ra_status ra_merge_partials(int32_t n_parts, int64_t rows, int32_t d, const float* o_parts,
                            const float* lse_parts, void* o, int32_t o_dtype, float* lse, void* stream) {
  if (n_parts < 1 || rows < 1 || d < 1 || d > 1024)
    return fail(RA_ERR_INVALID_ARG, "n_parts, rows >= 1 and 1 <= d <= 1024 required");
  if (o_dtype != RA_DTYPE_F32 && o_dtype != RA_DTYPE_BF16) return fail(RA_ERR_INVALID_ARG, "bad o_dtype");
  if (o_parts == nullptr || lse_parts == nullptr || o == nullptr)
    return fail(RA_ERR_INVALID_ARG, "null pointer");
  const void* ptrs[] = {o_parts, lse_parts, o, lse};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return fail(RA_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
  const ra_status s = ra::check_on_current_device(ptrs, 4, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  cudaError_t e = ra::launch_merge(n_parts, rows, d, o_parts, lse_parts, o, o_dtype, lse,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "merge launch failed: %s", cudaGetErrorString(e));
  return ok();
}

ra_status ra_layout_perm(int32_t layout, int64_t seq, int32_t n_shards, int32_t inverse,
                         int64_t rows_outer, int32_t row_bytes, const void* src, void* dst, void* stream) {
  ra_status s = check_layout(layout, seq, n_shards);
  if (s != RA_OK) return s;
  if (rows_outer < 1 || row_bytes < 4 || row_bytes % 4)
    return fail(RA_ERR_INVALID_ARG, "rows_outer >= 1 and row_bytes a positive multiple of 4 required");
  if (rows_outer > INT64_MAX / seq / row_bytes) return fail(RA_ERR_UNSUPPORTED, "tensor above 2^63-1 bytes");
  if (src == nullptr || dst == nullptr) return fail(RA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(src) || !aligned16(dst)) return fail(RA_ERR_INVALID_ARG, "src/dst must be 16-byte aligned");
  const int64_t bytes = rows_outer * seq * (int64_t)row_bytes;
  const char* a = static_cast<const char*>(src);
  const char* b = static_cast<const char*>(dst);
  if (a < b + bytes && b < a + bytes) return fail(RA_ERR_INVALID_ARG, "src and dst overlap");
  const void* ptrs[] = {src, dst};
  s = ra::check_on_current_device(ptrs, 2, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  cudaError_t e = ra::launch_layout_perm(layout, seq, n_shards, inverse ? 1 : 0, rows_outer, row_bytes,
                                         src, dst, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "layout permute launch failed: %s", cudaGetErrorString(e));
  return ok();
}

ra_status ra_layout_index(int32_t layout, int64_t seq, int32_t n_shards, int64_t* pos_out) {
  ra_status s = check_layout(layout, seq, n_shards);
  if (s != RA_OK) return s;
  if (pos_out == nullptr) return fail(RA_ERR_INVALID_ARG, "null pos_out");
  const int64_t s_n = seq / n_shards;
  for (int p = 0; p < n_shards; ++p)
    for (int64_t i = 0; i < s_n; ++i) pos_out[p * s_n + i] = ra::pos_of(layout, n_shards, s_n, p, i);
  return ok();
}

ra_status ra_fwd_step(ra_plan_t plan, int32_t step, const void* q, const void* k_blk, const void* v_blk,
                      float* o_part, float* lse_part, void* stream) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  const ra_problem& pb = plan->prob;
  if (step < 0 || step >= pb.n_shards)
    return fail(RA_ERR_INVALID_ARG, "step %d outside 0..%d", step, pb.n_shards - 1);
  if (q == nullptr || k_blk == nullptr || v_blk == nullptr || o_part == nullptr || lse_part == nullptr)
    return fail(RA_ERR_INVALID_ARG, "null pointer");
  const void* ptrs[] = {q, k_blk, v_blk, o_part, lse_part};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(RA_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
  ra_status s = check_device(plan);
  if (s == RA_OK) s = ra::check_on_current_device(ptrs, 5, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  ra::FwdParams prm = fwd_params(plan);
  prm.step_lo = (int16_t)step;
  prm.step_hi = (int16_t)(step + 1);
  prm.kv_rotated = 1;
  if (!plan->step_off.empty()) {
    prm.items = plan->d_step_items + plan->step_off[step];
    prm.n_items = (int32_t)(plan->step_off[step + 1] - plan->step_off[step]);
  }
  prm.o_parts = o_part;
  prm.lse_parts = lse_part;
  return launch(plan, prm, q, k_blk, v_blk, static_cast<cudaStream_t>(stream));
}

ra_status ra_ring_rotate(ra_plan_t plan, const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                         void* stream) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  if (k_src == nullptr || v_src == nullptr || k_dst == nullptr || v_dst == nullptr)
    return fail(RA_ERR_INVALID_ARG, "null pointer");
  const ra_problem& pb = plan->prob;
  const size_t bytes = (size_t)pb.batch * pb.heads_kv * pb.seq * pb.head_dim * elem_bytes(pb);
  if (overlap(k_src, k_dst, bytes) || overlap(v_src, v_dst, bytes) || overlap(k_dst, v_dst, bytes))
    return fail(RA_ERR_INVALID_ARG, "a destination overlaps its source or the other destination");
  ra_status s = check_device(plan);
  const void* ptrs[] = {k_src, v_src, k_dst, v_dst};
  if (s == RA_OK) s = ra::check_on_current_device(ptrs, 4, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = rotate_one(plan, k_src, k_dst, st);
  if (e == cudaSuccess) e = rotate_one(plan, v_src, v_dst, st);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "rotation copy failed: %s", cudaGetErrorString(e));
  return ok();
}

ra_status ra_ring_fwd(ra_plan_t plan, const void* q, const void* k, const void* v, void* o, float* lse,
                      void* k_buf, void* v_buf, float* o_parts, float* lse_parts, void* stream,
                      void* comm_stream) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  const ra_problem& pb = plan->prob;
  const int N = pb.n_shards;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || o_parts == nullptr ||
      lse_parts == nullptr || (N > 1 && (k_buf == nullptr || v_buf == nullptr)))
    return fail(RA_ERR_INVALID_ARG, "null pointer");
  const void* ptrs[] = {q, k, v, o, lse, k_buf, v_buf, o_parts, lse_parts};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return fail(RA_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
  const size_t kv_bytes = (size_t)pb.batch * pb.heads_kv * pb.seq * pb.head_dim * elem_bytes(pb);
  if (N > 1 && (overlap(k_buf, v_buf, 2 * kv_bytes) || overlap(k_buf, k, kv_bytes) ||
                overlap(k_buf, v, kv_bytes) || overlap(v_buf, k, kv_bytes) || overlap(v_buf, v, kv_bytes)))
    return fail(RA_ERR_INVALID_ARG, "receive buffers overlap each other or K/V");
  ra_status s = check_device(plan);
  if (s == RA_OK) s = ra::check_on_current_device(ptrs, 9, static_cast<cudaStream_t>(stream));
  if (s == RA_OK) s = ra::check_on_current_device(nullptr, 0, static_cast<cudaStream_t>(comm_stream));
  if (s != RA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = static_cast<cudaStream_t>(comm_stream);
  const int64_t rows = pb.batch * (int64_t)pb.heads_q * pb.seq;
  char* kb = static_cast<char*>(k_buf);
  char* vb = static_cast<char*>(v_buf);
  cudaError_t e = cudaSuccess;
  auto cuda_fail = [&](const char* what) { return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e)); };

  // The communication stream starts after everything already queued on stream
  // (the caller's writes of K and V, earlier users of the receive buffers).
  if ((e = cudaEventRecord(plan->ev_entry, st)) != cudaSuccess) return cuda_fail("event record");
  if ((e = cudaStreamWaitEvent(cs, plan->ev_entry, 0)) != cudaSuccess) return cuda_fail("stream wait");
  for (int t = 0; t < N; ++t) {
    // Block held at step t: K/V themselves at step 0, then receive buffer (t - 1) % 2.
    const void* kt = t == 0 ? k : kb + (size_t)((t - 1) % 2) * kv_bytes;
    const void* vt = t == 0 ? v : vb + (size_t)((t - 1) % 2) * kv_bytes;
    if (t >= 1 && (e = cudaStreamWaitEvent(st, plan->ev_rot, 0)) != cudaSuccess) return cuda_fail("stream wait");
    if (t + 1 < N) {
      // Pass the block on while step t computes.  Its destination was last read
      // by step t - 1.
      if (t >= 2 && (e = cudaStreamWaitEvent(cs, plan->ev_step, 0)) != cudaSuccess) return cuda_fail("stream wait");
      s = ra_ring_rotate(plan, kt, vt, kb + (size_t)(t % 2) * kv_bytes, vb + (size_t)(t % 2) * kv_bytes, cs);
      if (s != RA_OK) return s;
      if ((e = cudaEventRecord(plan->ev_rot, cs)) != cudaSuccess) return cuda_fail("event record");
    }
    s = ra_fwd_step(plan, t, q, kt, vt, o_parts + (size_t)t * rows * pb.head_dim, lse_parts + (size_t)t * rows, st);
    if (s != RA_OK) return s;
    if ((e = cudaEventRecord(plan->ev_step, st)) != cudaSuccess) return cuda_fail("event record");
  }
  return ra_merge_partials(N, rows, pb.head_dim, o_parts, lse_parts, o, pb.dtype, lse, st);
}

ra_status ra_bwd_scratch_size(ra_plan_t plan, int64_t* bytes) {
  if (plan == nullptr || bytes == nullptr) return fail(RA_ERR_INVALID_ARG, "null argument");
  const ra_problem& pb = plan->prob;
  const int64_t n64 = (plan->s_n + 63) / 64;
  *bytes = pb.batch * (int64_t)pb.heads_q * pb.n_shards * n64 * 128 * (int64_t)sizeof(float);
  return ok();
}

ra_status ra_bwd(ra_plan_t plan, const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, float* scratch, void* stream) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  const ra_problem& pb = plan->prob;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv, scratch};
  for (const void* p : ptrs) {
    if (p == nullptr) return fail(RA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(p)) return fail(RA_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
  }
  ra_status s = check_device(plan);
  if (s == RA_OK) s = ra::check_on_current_device(ptrs, 10, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t n64 = (plan->s_n + 63) / 64;
  cudaError_t e = ra::launch_bwd_prep(pb.dtype, pb.batch * (int64_t)pb.heads_q, pb.seq, pb.n_shards, pb.head_dim, o,
                                      dout, lse, scratch, st);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "backward preparation launch failed: %s", cudaGetErrorString(e));

  ra::BwdParams prm{};
  prm.batch = (int32_t)pb.batch;
  prm.heads_q = pb.heads_q;
  prm.heads_kv = pb.heads_kv;
  prm.group = pb.heads_q / pb.heads_kv;
  prm.head_dim = pb.head_dim;
  prm.n_shards = pb.n_shards;
  prm.layout = (int16_t)pb.layout;
  prm.causal = (int16_t)pb.causal;
  prm.seq = pb.seq;
  prm.s_n = plan->s_n;
  prm.scale = pb.scale;
  prm.scale_log2 = pb.scale * 1.4426950408889634f;
  prm.lse2d = scratch;
  prm.n64 = n64;
  prm.dq = dq;
  prm.dk = dk;
  prm.dv = dv;
  prm.q = q;
  prm.dout = dout;
  prm.status = plan->d_status;
  prm.item_counter = plan->d_status + 1;
  if (pb.dtype != RA_DTYPE_BF16) {
    e = ra::launch_bwd_f32(prm, static_cast<const float*>(q), static_cast<const float*>(k),
                           static_cast<const float*>(v), static_cast<const float*>(dout), st);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "f32 backward launch failed: %s", cudaGetErrorString(e));
    s = mark_use(plan, st);
    return s != RA_OK ? s : ok();
  }
  const int sms = plan->sm_count > 0 ? plan->sm_count : 148;
  for (int pass = 0; pass < 2; ++pass) {
    const int64_t n = pass == 0 ? plan->n_bwd_kv : (int64_t)plan->bwd_items.size() - plan->n_bwd_kv;
    prm.items = plan->d_bwd_items + (pass == 0 ? 0 : plan->n_bwd_kv);
    prm.n_items = (int32_t)n;
    if (n == 0) continue;
    // each pass hands out work items from a counter that starts at zero
    e = cudaMemsetAsync(prm.item_counter, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "counter reset: %s", cudaGetErrorString(e));
    const char* why = "";
    prm.round_sync = plan->bwd_round_sync[pass] ? 1 : 0;
    e = ra::launch_bwd_bf16(pass, prm, q, k, v, dout, (int)std::min<int64_t>(n, sms), st, &why);
    if (e == cudaErrorCooperativeLaunchTooLarge) {  // not every CTA resident: dynamic schedule
      cudaGetLastError();
      prm.round_sync = 0;
      e = ra::launch_bwd_bf16(pass, prm, q, k, v, dout, (int)std::min<int64_t>(n, sms), st, &why);
    }
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "%s: %s", why, cudaGetErrorString(e));
  }
  s = mark_use(plan, st);
  return s != RA_OK ? s : ok();
}

ra_status ra_allgather_kv(ra_plan_t plan, const void* k, const void* v, void* k_all, void* v_all, void* stream) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  const ra_problem& pb = plan->prob;
  const void* ptrs[] = {k, v, k_all, v_all};
  for (const void* p : ptrs) {
    if (p == nullptr) return fail(RA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(p)) return fail(RA_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
  }
  const size_t bytes = (size_t)pb.batch * pb.heads_kv * pb.seq * pb.head_dim * elem_bytes(pb);
  if (overlap(k, k_all, bytes) || overlap(v, v_all, bytes) || overlap(k_all, v_all, bytes))
    return fail(RA_ERR_INVALID_ARG, "a destination overlaps its source or the other destination");
  ra_status s = check_device(plan);
  if (s == RA_OK) s = ra::check_on_current_device(ptrs, 4, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int row_bytes = pb.head_dim * (int)elem_bytes(pb);
  const int64_t outer = pb.batch * (int64_t)pb.heads_kv;
  // layout order -> natural order: every shard's rows land at their positions
  cudaError_t e = ra::launch_layout_perm(pb.layout, pb.seq, pb.n_shards, 1, outer, row_bytes, k, k_all, st);
  if (e == cudaSuccess) e = ra::launch_layout_perm(pb.layout, pb.seq, pb.n_shards, 1, outer, row_bytes, v, v_all, st);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "gather launch failed: %s", cudaGetErrorString(e));
  return ok();
}

ra_status ra_fwd_gathered(ra_plan_t plan, const void* q, const void* k_all, const void* v_all, void* o, float* lse,
                          void* stream) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  if (q == nullptr || k_all == nullptr || v_all == nullptr || o == nullptr)
    return fail(RA_ERR_INVALID_ARG, "null pointer");
  const void* ptrs[] = {q, k_all, v_all, o, lse};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return fail(RA_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
  ra_status s = check_device(plan);
  if (s == RA_OK) s = ra::check_on_current_device(ptrs, 5, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  ra::FwdParams prm = fwd_params(plan);
  prm.gathered = 1;
  prm.step_lo = 0;
  prm.step_hi = 1;
  prm.items = plan->d_gather_items;
  prm.n_items = (int32_t)plan->gather_items.size();
  prm.round_sync = plan->gather_round_sync ? 1 : 0;
  prm.o = o;
  prm.lse = lse;
  return launch(plan, prm, q, k_all, v_all, static_cast<cudaStream_t>(stream));
}

ra_status ra_ulysses_a2a(int32_t direction, int32_t layout, int64_t seq, int32_t n_shards, int64_t batch,
                          int32_t heads, int32_t row_bytes, const void* src, void* dst, void* stream) {
  ra_status s = check_layout(layout, seq, n_shards);
  if (s != RA_OK) return s;
  if (direction != 0 && direction != 1) return fail(RA_ERR_INVALID_ARG, "direction must be 0 or 1");
  if (batch < 1 || heads < 1 || heads % n_shards)
    return fail(RA_ERR_INVALID_ARG, "batch >= 1 and heads a positive multiple of n_shards required");
  if (row_bytes != 256 && row_bytes != 4)
    return fail(RA_ERR_UNSUPPORTED, "row_bytes must be 256 (d = 128 bf16) or 4 (one float)");
  if (batch > INT32_MAX || batch * (int64_t)heads * seq > INT32_MAX)
    return fail(RA_ERR_UNSUPPORTED, "B*H*S above 2^31-1 rows");
  if (src == nullptr || dst == nullptr) return fail(RA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(src) || !aligned16(dst)) return fail(RA_ERR_INVALID_ARG, "src/dst must be 16-byte aligned");
  if (overlap(src, dst, (size_t)(batch * heads * seq) * row_bytes))
    return fail(RA_ERR_INVALID_ARG, "src and dst overlap");
  const void* ptrs[] = {src, dst};
  s = ra::check_on_current_device(ptrs, 2, static_cast<cudaStream_t>(stream));
  if (s != RA_OK) return s;
  cudaError_t e = ra::launch_ulysses_a2a(direction, layout, n_shards, (int)batch, heads, seq, row_bytes, src, dst,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "exchange launch failed: %s", cudaGetErrorString(e));
  return ok();
}

ra_status ra_wait_selftest(uint32_t* status_out) {
  if (status_out == nullptr) return fail(RA_ERR_INVALID_ARG, "null status_out");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_NO_DEVICE, "no CUDA device");
  }
  uint32_t* d_word = nullptr;
  cudaError_t e = cudaMalloc(&d_word, sizeof(uint32_t));
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
  e = cudaMemset(d_word, 0, sizeof(uint32_t));
  if (e == cudaSuccess) e = ra::launch_wait_selftest(d_word, nullptr);
  if (e == cudaSuccess) e = cudaMemcpy(status_out, d_word, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  cudaFree(d_word);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "wait self-test: %s", cudaGetErrorString(e));
  return ok();
}

ra_status ra_sync_status(ra_plan_t plan, void* stream) {
  if (plan == nullptr) return fail(RA_ERR_INVALID_ARG, "null plan");
  if (plan->device < 0) return fail(RA_ERR_NO_DEVICE, "plan was built without a CUDA device");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  uint32_t word = 0;
  e = cudaMemcpy(&word, plan->d_status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (word != 0) {
    cudaMemset(plan->d_status, 0, sizeof(word));
    char msg[200];
    const ra_status code = ra::status_word_error(word, msg, sizeof(msg));
    return fail(code, "%s", msg);
  }
  return ok();
}

const char* ra_last_error(void) { return g_err; }

}  // extern "C"
