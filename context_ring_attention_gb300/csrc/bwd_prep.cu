// Backward pass, preparation: per query row, the two scalars every gradient
// kernel needs.
//
//   lse2[row] = LSE[row] * log2(e)       (P = 2^(scale*log2(e)*q.k - lse2))
//   D[row]    = sum_c dO[row, c] O[row, c]
//
// D is the row sum of P * dP that the softmax Jacobian subtracts:
// dS = P * (dP - D).  The forward's LSE makes P recomputable without the row
// maximum.  HBM-bound: one warp per row reads dO and O once.  The output is laid
// out in blocks of 64 rows of one (batch, query head, shard) -- 64 lse2 values,
// then 64 D values, zeros past the shard's end -- so that a gradient kernel
// fetches a 64-row tile's scalars with one bulk copy and reads four columns per
// shared-memory load.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bwd_internal.h"

namespace ra {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Row sum of dO * O for one row, by one warp.
template <typename T>
__device__ __forceinline__ float row_dot(const T* a, const T* b, int d, int lane) {
  float acc = 0.f;
  if (sizeof(T) == 2 && d == 128) {  // bf16, d = 128: 8 bytes per lane
    const uint2 x = reinterpret_cast<const uint2*>(a)[lane], y = reinterpret_cast<const uint2*>(b)[lane];
    const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
    const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
    const float2 y0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y.x));
    const float2 y1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y.y));
    acc = x0.x * y0.x;
    acc = fmaf(x0.y, y0.y, acc);
    acc = fmaf(x1.x, y1.x, acc);
    acc = fmaf(x1.y, y1.y, acc);
  } else {
    for (int c = lane; c < d; c += 32) acc = fmaf(to_f(a[c]), to_f(b[c]), acc);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  return acc;
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
    bwd_prep_kernel(int64_t padded_rows, int64_t seq, int n_shards, int64_t n64, int d, const T* __restrict__ o,
                    const T* __restrict__ dout, const float* __restrict__ lse, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t s_n = seq / n_shards;
  for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < padded_rows;
       r += (int64_t)gridDim.x * kWarps) {
    // padded row r: block r / 64 = (bh * N + p) * n64 + tile, row c = r % 64 of the tile
    const int64_t blk = r >> 6, c = r & 63;
    const int64_t tile = blk % n64, bp = blk / n64;
    const int p = (int)(bp % n_shards);
    const int64_t bh = bp / n_shards;
    const int64_t i = tile * 64 + c;
    float l2 = 0.f, dd = 0.f;
    if (i < s_n) {
      const int64_t row = bh * seq + (int64_t)p * s_n + i;
      dd = row_dot(o + row * d, dout + row * d, d, lane);
      l2 = lse[row] * kLog2e;
    }
    if (lane == 0) {
      out[blk * 128 + c] = l2;
      out[blk * 128 + 64 + c] = dd;
    }
  }
}

}  // namespace

cudaError_t launch_bwd_prep(int dtype, int64_t bh_count, int64_t seq, int n_shards, int d, const void* o,
                            const void* dout, const float* lse, float* out, cudaStream_t stream) {
  const int64_t s_n = seq / n_shards;
  const int64_t n64 = (s_n + 63) / 64;
  const int64_t padded = bh_count * n_shards * n64 * 64;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (padded + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sms * 16;
  const unsigned grid = (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
  if (dtype == RA_DTYPE_BF16)
    bwd_prep_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, stream>>>(
        padded, seq, n_shards, n64, d, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
        lse, out);
  else
    bwd_prep_kernel<float><<<grid, kWarps * 32, 0, stream>>>(padded, seq, n_shards, n64, d,
                                                             static_cast<const float*>(o),
                                                             static_cast<const float*>(dout), lse, out);
  return cudaGetLastError();
}

}  // namespace ra
