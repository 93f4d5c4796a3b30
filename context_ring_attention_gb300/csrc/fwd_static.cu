// ra_fwd_static: the bf16 ring forward for callers that cannot allocate memory.
//
// Some callers cannot call cudaMalloc at run time -- code that runs under a
// memory pool or allocator it must not bypass, or that has to fix its whole
// device footprint at load time -- and so cannot create a plan (ra_plan
// allocates the work table and status word).  This entry point needs no plan:
// the work table and the status word live in one file-scope device array of
// fixed size, which every GPU that loads this library holds until the process
// exits.  Nothing here calls cudaMalloc, cudaFree or any allocating routine;
// the host-side work list is built in a static host buffer.
//
// The device array is shared by every call: calls whose kernels overlap on the
// GPU (other streams, other host threads) race on it.  Calls from several host
// threads are serialised on the host while the work list is built and copied.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "ra_internal.h"

namespace {

constexpr int kMaxItems = 131072;           // work items: e.g. 1M tokens x 32 query heads
constexpr size_t kStatusBytes = 256;        // status word at the start of the array
constexpr size_t kScratchBytes = kStatusBytes + (size_t)kMaxItems * sizeof(ra::WorkItem);  // 4 MiB + 256 B
constexpr int kMaxDevices = ra::kMaxDevices;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct Keyed {
  ra::WorkItem w;
  int64_t order;
};
Keyed g_host_items[kMaxItems];  // host staging for the work list
std::mutex g_mutex;
void* g_dev_addr[kMaxDevices] = {};  // device address of g_scratch, per device
int g_dev_sms[kMaxDevices] = {};

ra_status fail(ra_status s, const char* msg) {
  char buf[256];
  snprintf(buf, sizeof(buf), "ra_fwd_static: %s", msg);
  ra::set_last_error(buf);
  return s;
}

ra_status check_problem(const ra_problem* p) {
  if (p == nullptr) return fail(RA_ERR_INVALID_ARG, "null problem");
  if (p->batch < 1 || p->heads_q < 1 || p->heads_kv < 1 || p->n_shards < 1 || p->seq < 1)
    return fail(RA_ERR_INVALID_ARG, "sizes must be >= 1");
  if (p->layout < RA_LAYOUT_CONTIGUOUS || p->layout > RA_LAYOUT_ZIGZAG) return fail(RA_ERR_INVALID_ARG, "bad layout");
  if (p->seq % p->n_shards) return fail(RA_ERR_INVALID_ARG, "seq is not a multiple of n_shards");
  if (p->layout == RA_LAYOUT_ZIGZAG && p->seq % (2 * (int64_t)p->n_shards))
    return fail(RA_ERR_INVALID_ARG, "zigzag needs seq to be a multiple of 2*n_shards");
  if (p->heads_q % p->heads_kv) return fail(RA_ERR_INVALID_ARG, "heads_q is not a multiple of heads_kv");
  if (p->causal != 0 && p->causal != 1) return fail(RA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(p->scale >= 0.f) || std::isinf(p->scale)) return fail(RA_ERR_INVALID_ARG, "scale must be finite and >= 0");
  if (p->dtype != RA_DTYPE_BF16 || p->head_dim != 128)
    return fail(RA_ERR_UNSUPPORTED, "only bf16 with head_dim 128 is supported");
  if (p->n_shards > INT16_MAX) return fail(RA_ERR_UNSUPPORTED, "n_shards above 32767");
  if (p->seq > INT32_MAX || p->batch > INT32_MAX / p->heads_q || p->batch * (int64_t)p->heads_q * p->seq > INT32_MAX)
    return fail(RA_ERR_UNSUPPORTED, "more than 2^31-1 rows");
  return RA_OK;
}

// Whether the problem's work list fits the static arrays (and its costing, every
// item against every ring step, stays short).
bool fits(const ra_problem& pb) {
  const int64_t N = pb.n_shards;
  const int64_t items = ra::fwd_items_per_shard(pb, pb.seq / N) * N;
  return items <= kMaxItems && items * N <= (int64_t(1) << 30);
}

// The planner's work list (ra::for_each_fwd_item, sorted by the same schedule
// rule), written into the static host buffer.  Returns the item count, or -1 when
// it would not fit; *max_cost receives the longest item's key-tile count.
int64_t build_items(const ra_problem& pb, int64_t* max_cost_out) {
  const int N = pb.n_shards;
  const int64_t s_n = pb.seq / N;
  if (!fits(pb)) return -1;
  int64_t n = 0;
  ra::for_each_fwd_item(pb, s_n, [&](const ra::WorkItem& w) {
    g_host_items[n] = {w, n};
    ++n;
  });
  int64_t max_cost = 1;
  for (int64_t i = 0; i < n; ++i) max_cost = std::max<int64_t>(max_cost, g_host_items[i].w.cost);
  *max_cost_out = max_cost;
  const int64_t width = ra::schedule_bucket_width(max_cost);
  const int G = pb.heads_q / pb.heads_kv;
  std::sort(g_host_items, g_host_items + n, [&](const Keyed& a, const Keyed& b) {
    return ra::schedule_before(ra::schedule_key(a.w, pb.heads_q, G, width, a.order),
                               ra::schedule_key(b.w, pb.heads_q, G, width, b.order));
  });
  return n;
}

}  // namespace

extern "C" ra_status ra_fwd_static(const ra_problem* prob, const void* q, const void* k, const void* v,
                                   void* o, float* lse, void* stream) {
  ra_status s = check_problem(prob);
  if (s != RA_OK) return s;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return fail(RA_ERR_INVALID_ARG, "null pointer");
  const void* ptrs[] = {q, k, v, o, lse};
  for (const void* p : ptrs)
    if (p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u)) return fail(RA_ERR_INVALID_ARG, "pointer not 16-byte aligned");

  if (!fits(*prob))
    return fail(RA_ERR_UNSUPPORTED, "work list exceeds the static maximum of 131072 items (or 2^30 item-steps)");
  const ra_status dev_ok = ra::check_on_current_device(ptrs, 5, static_cast<cudaStream_t>(stream));
  if (dev_ok != RA_OK) return dev_ok;

  std::lock_guard<std::mutex> lock(g_mutex);
  int64_t max_cost = 0;
  const int64_t n_items = build_items(*prob, &max_cost);

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_NO_DEVICE, "no CUDA device");
  }
  if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_UNSUPPORTED, "device ordinal above 63");
  if (g_dev_addr[dev] == nullptr) {
    // First call on this device (which is current): look up the array's device address.
    void* addr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&addr, g_scratch);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, cudaGetErrorString(e));
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, cudaGetErrorString(e));
    g_dev_sms[dev] = sms;
    g_dev_addr[dev] = addr;
  }
  unsigned char* base = static_cast<unsigned char*>(g_dev_addr[dev]);
  ra::WorkItem* d_items = reinterpret_cast<ra::WorkItem*>(base + kStatusBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // The sorted items without their sort keys, contiguous for the copy.
  static ra::WorkItem packed[kMaxItems];
  for (int64_t i = 0; i < n_items; ++i) packed[i] = g_host_items[i].w;
  // Pageable-source async copies return once the source has been staged, so the
  // static host buffer may be reused by the next call.
  cudaError_t e = cudaMemcpyAsync(d_items, packed, (size_t)n_items * sizeof(ra::WorkItem), cudaMemcpyHostToDevice, st);
  // status word and work-item counter start at zero
  if (e == cudaSuccess) e = cudaMemsetAsync(base, 0, 2 * sizeof(uint32_t), st);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, cudaGetErrorString(e));

  ra::FwdParams prm{};
  prm.batch = (int32_t)prob->batch;
  prm.heads_q = prob->heads_q;
  prm.heads_kv = prob->heads_kv;
  prm.group = prob->heads_q / prob->heads_kv;
  prm.head_dim = prob->head_dim;
  prm.n_shards = prob->n_shards;
  prm.layout = (int16_t)prob->layout;
  prm.causal = (int16_t)prob->causal;
  prm.seq = prob->seq;
  prm.s_n = prob->seq / prob->n_shards;
  prm.n_items = (int32_t)n_items;
  prm.scale = prob->scale > 0.f ? prob->scale : 1.0f / std::sqrt(128.0f);
  prm.scale_log2 = prm.scale * 1.4426950408889634f;
  prm.items = d_items;
  prm.o = o;
  prm.lse = lse;
  prm.o_parts = nullptr;
  prm.lse_parts = nullptr;
  prm.status = reinterpret_cast<uint32_t*>(base);
  prm.item_counter = reinterpret_cast<uint32_t*>(base) + 1;
  prm.step_lo = 0;
  prm.step_hi = (int16_t)prob->n_shards;
  prm.kv_rotated = 0;
  prm.round_sync = ra::use_round_sync(prob->seq, prob->head_dim, max_cost) ? 1 : 0;
  prm.gathered = 0;
  if (n_items == 0) return RA_OK;
  const int grid = (int)std::min<int64_t>(n_items, g_dev_sms[dev] > 0 ? g_dev_sms[dev] : 148);
  const char* why = "";
  e = ra::launch_fwd_bf16(prm, q, k, v, grid, st, &why);
  if (e == cudaErrorCooperativeLaunchTooLarge) {  // not every CTA resident: dynamic schedule
    cudaGetLastError();
    prm.round_sync = 0;
    e = ra::launch_fwd_bf16(prm, q, k, v, grid, st, &why);
  }
  if (e != cudaSuccess) {
    char msg[200];
    snprintf(msg, sizeof(msg), "%s: %s", why, cudaGetErrorString(e));
    return fail(RA_ERR_CUDA, msg);
  }
  ra::set_last_error("");
  return RA_OK;
}

extern "C" ra_status ra_fwd_static_status(void* stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_NO_DEVICE, "no CUDA device");
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (dev < 0 || dev >= kMaxDevices || g_dev_addr[dev] == nullptr) {  // no call on this device yet
    ra::set_last_error("");
    return RA_OK;
  }
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  uint32_t word = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&word, g_dev_addr[dev], sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word != 0) e = cudaMemset(g_dev_addr[dev], 0, sizeof(word));
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, cudaGetErrorString(e));
  if (word != 0) {
    char msg[200];
    const ra_status code = ra::status_word_error(word, msg, sizeof(msg));
    return fail(code, msg);
  }
  ra::set_last_error("");
  return RA_OK;
}
