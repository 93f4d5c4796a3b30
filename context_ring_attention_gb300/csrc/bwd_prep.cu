// Backward pass, preparation: per query row, the two scalars every gradient
// kernel needs.
//
//   lse2[row] = LSE[row] * log2(e)       (P = 2^(scale*log2(e)*q.k - lse2))
//   D[row]    = sum_c dO[row, c] O[row, c]
//
// D is the row sum of P * dP that the softmax Jacobian subtracts:
// dS = P * (dP - D).  The forward's LSE makes P recomputable without the row
// maximum.  HBM-bound: one warp per row reads dO and O once; rows are written as
// float4 {lse2, D, 0, 0} so that the gradient kernels can fetch 64 consecutive
// rows with one TMA box.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"

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

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
    bwd_prep_kernel(int64_t rows, int d, const T* __restrict__ o, const T* __restrict__ dout,
                    const float* __restrict__ lse, float4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); row < rows;
       row += (int64_t)gridDim.x * kWarps) {
    const T* a = o + row * d;
    const T* b = dout + row * d;
    float acc = 0.f;
    for (int c = lane; c < d; c += 32) acc = fmaf(to_f(a[c]), to_f(b[c]), acc);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) out[row] = make_float4(lse[row] * kLog2e, acc, 0.f, 0.f);
  }
}

// d = 128 bf16: a lane reads 4 consecutive elements (8 bytes) of each row.
__global__ void __launch_bounds__(kWarps * 32)
    bwd_prep_bf16_d128(int64_t rows, const uint2* __restrict__ o, const uint2* __restrict__ dout,
                       const float* __restrict__ lse, float4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); row < rows;
       row += (int64_t)gridDim.x * kWarps) {
    const uint2 x = o[row * 32 + lane], y = dout[row * 32 + lane];
    const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
    const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
    const float2 y0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y.x));
    const float2 y1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y.y));
    float acc = x0.x * y0.x;
    acc = fmaf(x0.y, y0.y, acc);
    acc = fmaf(x1.x, y1.x, acc);
    acc = fmaf(x1.y, y1.y, acc);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) out[row] = make_float4(lse[row] * kLog2e, acc, 0.f, 0.f);
  }
}

}  // namespace

cudaError_t launch_bwd_prep(int dtype, int64_t rows, int d, const void* o, const void* dout, const float* lse,
                            float4* out, cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (rows + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sms * 16;
  const unsigned grid = (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
  if (dtype == RA_DTYPE_BF16 && d == 128)
    bwd_prep_bf16_d128<<<grid, kWarps * 32, 0, stream>>>(rows, static_cast<const uint2*>(o),
                                                         static_cast<const uint2*>(dout), lse, out);
  else if (dtype == RA_DTYPE_BF16)
    bwd_prep_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, stream>>>(
        rows, d, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, out);
  else
    bwd_prep_kernel<float><<<grid, kWarps * 32, 0, stream>>>(rows, d, static_cast<const float*>(o),
                                                             static_cast<const float*>(dout), lse, out);
  return cudaGetLastError();
}

}  // namespace ra
