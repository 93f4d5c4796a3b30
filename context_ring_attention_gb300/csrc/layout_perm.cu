// Row gather/scatter between natural order and a ring layout (contiguous;
// striped, Module 23 "The Causal Imbalance -- and the Striped Fix"; zigzag).
// HBM-bound copy: whole rows move, 16-byte vectors when the row allows it.
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kThreads = 256;

// Each block copies rows of one outer index; blockIdx.y walks the outer rows.
template <typename Vec>
__global__ void __launch_bounds__(kThreads)
    perm_kernel(int layout, int n_shards, int64_t seq, int64_t s_n, int inverse, int64_t rows_outer,
                int vecs_per_row, const Vec* __restrict__ src, Vec* __restrict__ dst) {
  const int64_t per_outer = seq * vecs_per_row;
  for (int64_t o = blockIdx.y; o < rows_outer; o += gridDim.y) {
    const Vec* s = src + o * per_outer;
    Vec* d = dst + o * per_outer;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < per_outer;
         e += (int64_t)gridDim.x * kThreads) {
      const int64_t j = e / vecs_per_row;
      const int c = (int)(e - j * vecs_per_row);
      const int p = (int)(j / s_n);
      const int64_t pj = pos_of(layout, n_shards, s_n, p, j - (int64_t)p * s_n);
      if (inverse)
        d[pj * vecs_per_row + c] = s[e];
      else
        d[e] = s[pj * vecs_per_row + c];
    }
  }
}

// 256-byte rows (128 bf16 values, the attention case): a half-warp moves one
// row as 16 x 16 B; each thread keeps kRowsPerThread rows in flight (all loads,
// then all stores); row positions use 32-bit arithmetic once per row.
constexpr int kRowsPerThread = 4;
constexpr int kRowsPerPass = kThreads / 16;                      // 16 rows per block pass
constexpr int kRowsPerBlock = kRowsPerPass * kRowsPerThread;     // 64 rows per block

__global__ void __launch_bounds__(kThreads)
    perm256_kernel(int layout, int n_shards, int seq, int s_n, int inverse, int64_t rows_outer,
                   const uint4* __restrict__ src, uint4* __restrict__ dst) {
  const int lane16 = threadIdx.x & 15;
  const int sub = threadIdx.x >> 4;
  const int j0 = blockIdx.x * kRowsPerBlock;
  for (int64_t o = blockIdx.y; o < rows_outer; o += gridDim.y) {
    const uint4* s = src + o * (int64_t)seq * 16;
    uint4* d = dst + o * (int64_t)seq * 16;
    uint4 v[kRowsPerThread];
    int to[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
      const int j = j0 + r * kRowsPerPass + sub;
      to[r] = -1;
      if (j < seq) {
        const int p = j / s_n;
        const int pj = (int)pos_of(layout, n_shards, s_n, p, j - p * s_n);
        const int from = inverse ? j : pj;
        to[r] = inverse ? pj : j;
        v[r] = s[(int64_t)from * 16 + lane16];
      }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r)
      if (to[r] >= 0) d[(int64_t)to[r] * 16 + lane16] = v[r];
  }
}

}  // namespace

cudaError_t launch_layout_perm(int layout, int64_t seq, int n_shards, int inverse,
                               int64_t rows_outer, int row_bytes, const void* src, void* dst,
                               cudaStream_t stream) {
  const int64_t s_n = seq / n_shards;
  if (row_bytes == 256) {
    const int64_t gy = rows_outer < 65535 ? rows_outer : 65535;
    dim3 grid((unsigned)((seq + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)gy);
    perm256_kernel<<<grid, kThreads, 0, stream>>>(layout, n_shards, (int)seq, (int)s_n, inverse, rows_outer,
                                                 static_cast<const uint4*>(src), static_cast<uint4*>(dst));
    return cudaGetLastError();
  }
  const bool v16 = (row_bytes % 16) == 0;
  const int vpr = v16 ? row_bytes / 16 : row_bytes / 4;
  const int64_t per_outer = seq * vpr;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (per_outer + kThreads - 1) / kThreads;
  const int64_t total_cap = (int64_t)sms * 8;  // ~8 resident blocks per SM in flight
  const int64_t gy = rows_outer < 65535 ? rows_outer : 65535;
  int64_t gx = (total_cap + gy - 1) / gy;
  if (gx > want) gx = want;
  if (gx < 1) gx = 1;
  dim3 grid((unsigned)gx, (unsigned)gy);
  if (v16)
    perm_kernel<uint4><<<grid, kThreads, 0, stream>>>(layout, n_shards, seq, s_n, inverse, rows_outer, vpr,
                                                     static_cast<const uint4*>(src), static_cast<uint4*>(dst));
  else
    perm_kernel<uint32_t><<<grid, kThreads, 0, stream>>>(layout, n_shards, seq, s_n, inverse, rows_outer, vpr,
                                                         static_cast<const uint32_t*>(src),
                                                         static_cast<uint32_t*>(dst));
  return cudaGetLastError();
}

}  // namespace ra
