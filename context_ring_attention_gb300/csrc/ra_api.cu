// C ABI of libra.so: argument checks, the ring planner and kernel dispatch.
//
// The planner turns a problem into the work list of the tensor-core kernel: one
// item per pair of 128-row query tiles that share a key/value head and a tile
// schedule (two query heads of one GQA group at the same rows, or two
// consecutive row tiles of one head), each with the number of key tiles it
// visits over the N ring steps.  Items are ordered longest first so the
// persistent grid ends evenly under a causal mask, whose per-shard work is
// uneven for contiguous shards (Module 23, "The Causal Imbalance -- and the
// Striped Fix").
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "ra_internal.h"

struct ra_plan_s {
  ra_problem prob;
  int64_t s_n;
  int n_qtiles, n_ktiles;
  std::vector<ra::WorkItem> items;
  std::vector<int64_t> full, partial, skip;
  int device = -1;
  ra::WorkItem* d_items = nullptr;
  uint32_t* d_status = nullptr;
  int sm_count = 0;
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
  return RA_OK;
}

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
  const int64_t rows = p->batch * (int64_t)p->heads_q * p->seq;
  if (p->batch > INT32_MAX / p->heads_q || rows > INT32_MAX)
    return fail(RA_ERR_UNSUPPORTED, "B*Hq*S above 2^31-1 rows");
  return RA_OK;
}

int64_t last_row_pos(const ra_problem& pb, int64_t s_n, int p, int64_t row_start) {
  const int64_t last = std::min<int64_t>(row_start + ra::kTileRows, s_n) - 1;
  return ra::pos_of(pb.layout, pb.n_shards, s_n, p, last);
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
  const bool head_pairs = (G % 2) == 0;
  struct Keyed {
    ra::WorkItem w;
    int64_t order;
  };
  std::vector<Keyed> list;
  int64_t seqno = 0;
  for (int p = 0; p < N; ++p) {
    for (int qt = 0; qt < pl->n_qtiles; qt += head_pairs ? 1 : 2) {
      for (int64_t b = 0; b < pb.batch; ++b) {
        for (int h = 0; h < pb.heads_q; h += head_pairs ? 2 : 1) {
          ra::WorkItem w{};
          w.bh0 = (int32_t)(b * pb.heads_q + h);
          w.shard = p;
          w.row0 = qt * ra::kTileRows;
          if (head_pairs) {
            w.bh1 = w.bh0 + 1;
            w.row1 = w.row0;
          } else if (qt + 1 < pl->n_qtiles) {
            w.bh1 = w.bh0;
            w.row1 = w.row0 + ra::kTileRows;
          } else {
            w.bh1 = -1;
            w.row1 = w.row0;
          }
          const int64_t top_row = (w.bh1 >= 0) ? w.row1 : w.row0;
          w.maxq = (int32_t)last_row_pos(pb, s_n, p, top_row);
          int cost = 0;
          for (int t = 0; t < N; ++t)
            cost += ra::visit_tiles(pb.layout, N, s_n, pb.causal, (p - t + N) % N, w.maxq);
          w.cost = cost;
          list.push_back({w, seqno++});
        }
      }
    }
  }
  int64_t max_cost = 1;
  for (const Keyed& k : list) max_cost = std::max<int64_t>(max_cost, k.w.cost);
  const int64_t width = ra::schedule_bucket_width(max_cost);
  std::vector<ra::ScheduleKey> keys(list.size());
  for (size_t n = 0; n < list.size(); ++n)
    keys[n] = ra::schedule_key(list[n].w, pb.heads_q, G, width, list[n].order);
  std::vector<size_t> idx(list.size());
  for (size_t n = 0; n < idx.size(); ++n) idx[n] = n;
  std::sort(idx.begin(), idx.end(), [&](size_t a, size_t b) { return ra::schedule_before(keys[a], keys[b]); });
  pl->items.resize(list.size());
  for (size_t n = 0; n < list.size(); ++n) pl->items[n] = list[idx[n]].w;
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
  cudaError_t e = cudaMalloc(&pl->d_status, 256);
  if (e == cudaSuccess) e = cudaMemset(pl->d_status, 0, 256);
  if (e == cudaSuccess && !pl->items.empty()) {
    e = cudaMalloc(&pl->d_items, pl->items.size() * sizeof(ra::WorkItem));
    if (e == cudaSuccess)
      e = cudaMemcpy(pl->d_items, pl->items.data(), pl->items.size() * sizeof(ra::WorkItem),
                     cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "plan upload failed: %s", cudaGetErrorString(e));
  return RA_OK;
}

}  // namespace

void ra::set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

extern "C" {

ra_status ra_plan(const ra_problem* prob, ra_plan_t* out) {
  if (prob == nullptr || out == nullptr) return fail(RA_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  ra_status s = validate(prob);
  if (s != RA_OK) return s;
  ra_plan_s* pl = new (std::nothrow) ra_plan_s();
  if (pl == nullptr) return fail(RA_ERR_INVALID_ARG, "out of host memory");
  pl->prob = *prob;
  if (pl->prob.scale == 0.f) pl->prob.scale = 1.0f / std::sqrt((float)prob->head_dim);
  pl->s_n = prob->seq / prob->n_shards;
  build_schedule(pl);
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
    cudaFree(plan->d_items);
    cudaFree(plan->d_status);
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
  const ra_problem& pb = plan->prob;
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
  if (plan->device < 0) return fail(RA_ERR_NO_DEVICE, "plan was built without a CUDA device");
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device)
    return fail(RA_ERR_INVALID_ARG, "current device %d differs from the plan's device %d", cur, plan->device);

  ra::FwdParams prm{};
  prm.batch = (int32_t)pb.batch;
  prm.heads_q = pb.heads_q;
  prm.heads_kv = pb.heads_kv;
  prm.group = pb.heads_q / pb.heads_kv;
  prm.head_dim = pb.head_dim;
  prm.n_shards = pb.n_shards;
  prm.layout = pb.layout;
  prm.causal = pb.causal;
  prm.seq = pb.seq;
  prm.s_n = plan->s_n;
  prm.n_items = (int32_t)plan->items.size();
  prm.scale = pb.scale;
  prm.scale_log2 = pb.scale * 1.4426950408889634f;
  prm.items = plan->d_items;
  prm.o = o;
  prm.lse = lse;
  prm.o_parts = o_parts;
  prm.lse_parts = lse_parts;
  prm.status = plan->d_status;
  prm.item_counter = plan->d_status + 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (pb.dtype == RA_DTYPE_BF16) {
    if (prm.n_items == 0) return ok();
    const int grid = std::min(prm.n_items, plan->sm_count > 0 ? plan->sm_count : 148);
    const char* why = "";
    // The kernel hands out work items from a counter that starts at zero.
    e = cudaMemsetAsync(prm.item_counter, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "counter reset: %s", cudaGetErrorString(e));
    e = ra::launch_fwd_bf16(prm, q, k, v, grid, st, &why);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "%s: %s", why, cudaGetErrorString(e));
  } else {
    e = ra::launch_fwd_f32(prm, static_cast<const float*>(q), static_cast<const float*>(k),
                           static_cast<const float*>(v), st);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "f32 forward launch failed: %s", cudaGetErrorString(e));
  }
  return ok();
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
  if (src == nullptr || dst == nullptr) return fail(RA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(src) || !aligned16(dst)) return fail(RA_ERR_INVALID_ARG, "src/dst must be 16-byte aligned");
  const int64_t bytes = rows_outer * seq * (int64_t)row_bytes;
  const char* a = static_cast<const char*>(src);
  const char* b = static_cast<const char*>(dst);
  if (a < b + bytes && b < a + bytes) return fail(RA_ERR_INVALID_ARG, "src and dst overlap");
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
    return fail(RA_ERR_TIMEOUT, "device wait ran out of budget (status bits 0x%x: 1 producer, 2 mma, 4 softmax, 8 teardown)", word);
  }
  return ok();
}

const char* ra_last_error(void) { return g_err; }

}  // extern "C"
