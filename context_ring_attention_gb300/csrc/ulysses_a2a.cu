// DeepSpeed-Ulysses' exchange (named on the Q&A page "Explain ring attention ...",
// section "Related approaches": a split by attention heads with an all-to-all
// instead of a ring), for N devices:
//   seq -> head:  [B, H, S, row] in layout order (device p: rows p*S/N.. of every
//                 head) -> [N, B, H/N, S, row] (device p': heads p'H/N.., all
//                 tokens by position)
//   head -> seq:  the inverse.
// Each device then attends over the whole sequence for its heads (an ordinary
// forward with batch N*B, H/N heads, one shard), and the exchange back returns
// O and the LSE to the sequence shards.  HBM-bound row moves: a block row
// (device, batch, head) decodes its indices once; the row's position <-> (shard,
// local row) map is the layout's; 256-byte rows move as 16 x 16 B by a half-warp.
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerThread = 4;
constexpr int kRowsPerPass = kThreads / 16;
constexpr int kRowsPerBlock = kRowsPerPass * kRowsPerThread;  // 64 rows of 256 B per block

// (shard, local row) holding natural position s.
__device__ __forceinline__ void shard_of(int layout, int n, int s_n, int s, int& p, int& i) {
  if (layout == RA_LAYOUT_STRIPED) {
    p = s % n;
    i = s / n;
  } else if (layout == RA_LAYOUT_ZIGZAG) {
    const int c = s_n >> 1, chunk = s / c, off = s - chunk * c;
    p = chunk < n ? chunk : 2 * n - 1 - chunk;
    i = chunk < n ? off : c + off;
  } else {
    p = s / s_n;
    i = s - p * s_n;
  }
}

// Row gather for both directions.  dir 0 (dst [N, B, hl, S]): dst row (p', b, h', s)
// <- src row (b, p'*hl + h', p*s_n + i) of the layout-ordered [B, H, S], where shard p
// row i holds position s.  dir 1 (dst [B, H, S] layout order, walked as (b, h, p, i)):
// dst row (b, h, p*s_n + i) <- src row (h / hl, b, h % hl, pos(p, i)).
// `outer` indexes all dst dims but the innermost row index.
template <typename Vec, int kLanes>
__global__ void __launch_bounds__(kThreads)
    a2a_kernel(int dir, int layout, int n, int batch, int heads, int seq, int64_t outer_count,
               const Vec* __restrict__ src, Vec* __restrict__ dst) {
  const int s_n = seq / n, hl = heads / n;
  const int lane = threadIdx.x % kLanes, sub = threadIdx.x / kLanes;
  constexpr int kPass = kThreads / kLanes;
  const int inner = dir == 0 ? seq : s_n;  // dst rows per outer index
  const int j0 = blockIdx.x * (kPass * kRowsPerThread);
  for (int64_t o = blockIdx.y; o < outer_count; o += gridDim.y) {
    int64_t src_base;
    int p = 0;
    if (dir == 0) {    // o = (p' * B + b) * hl + h'
      const int hh = (int)(o % hl);
      const int b = (int)((o / hl) % batch);
      const int pq = (int)(o / ((int64_t)hl * batch));
      src_base = ((int64_t)b * heads + (int64_t)pq * hl + hh) * seq;  // + p * s_n + i
    } else {           // o = ((b * H) + h) * N + p
      p = (int)(o % n);
      const int h = (int)((o / n) % heads);
      const int b = (int)(o / ((int64_t)n * heads));
      src_base = (((int64_t)(h / hl) * batch + b) * hl + (h % hl)) * seq;  // + pos(p, i)
    }
    Vec v[kRowsPerThread];
    int64_t to[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
      const int j = j0 + r * kPass + sub;
      to[r] = -1;
      if (j < inner) {
        int64_t from;
        if (dir == 0) {
          int ps, i;
          shard_of(layout, n, s_n, j, ps, i);
          from = src_base + (int64_t)ps * s_n + i;
        } else {
          from = src_base + pos_of(layout, n, s_n, p, j);
        }
        to[r] = o * inner + j;
        v[r] = src[from * kLanes + lane];
      }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r)
      if (to[r] >= 0) dst[to[r] * kLanes + lane] = v[r];
  }
}

}  // namespace

cudaError_t launch_ulysses_a2a(int dir, int layout, int n, int batch, int heads, int64_t seq, int row_bytes,
                               const void* src, void* dst, cudaStream_t stream) {
  const int64_t s_n = seq / n;
  const int64_t outer = (int64_t)n * batch * (dir == 0 ? heads / n : heads);  // dst rows / inner
  const int64_t inner = dir == 0 ? seq : s_n;
  const int64_t gy = outer < 65535 ? outer : 65535;
  if (row_bytes == 256) {
    dim3 grid((unsigned)((inner + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)gy);
    a2a_kernel<uint4, 16><<<grid, kThreads, 0, stream>>>(dir, layout, n, batch, heads, (int)seq, outer,
                                                          static_cast<const uint4*>(src), static_cast<uint4*>(dst));
  } else if (row_bytes == 4) {  // one float (the LSE) per row
    constexpr int kRows = kThreads * kRowsPerThread;
    dim3 grid((unsigned)((inner + kRows - 1) / kRows), (unsigned)gy);
    a2a_kernel<uint32_t, 1><<<grid, kThreads, 0, stream>>>(dir, layout, n, batch, heads, (int)seq, outer,
                                                            static_cast<const uint32_t*>(src),
                                                            static_cast<uint32_t*>(dst));
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ra
