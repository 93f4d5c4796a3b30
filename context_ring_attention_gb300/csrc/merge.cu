// Exact merge of partial attention results (order independence of the
// online-softmax fold, Module 23, "The Math: One Block at a Time"):
//   LSE = ln sum_t e^(LSE_t),   O = sum_t e^(LSE_t - LSE) O_t.
// HBM-bound: one warp per row, 16-byte loads along d.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <bool kBf16Out>
__global__ void __launch_bounds__(kWarps * 32)
    merge_kernel(int n_parts, int64_t rows, int d, const float* __restrict__ o_parts,
                 const float* __restrict__ lse_parts, void* __restrict__ o, float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); row < rows; row += stride) {
    float top = -INFINITY;
    for (int t = lane; t < n_parts; t += 32) top = fmaxf(top, lse_parts[(int64_t)t * rows + row]);
    top = warp_max(top);
    float z = 0.f;
    if (top != -INFINITY)
      for (int t = lane; t < n_parts; t += 32) z += expf(lse_parts[(int64_t)t * rows + row] - top);
    z = warp_sum(z);
    const float big = (top != -INFINITY) ? top + logf(z) : -INFINITY;
    if (lane == 0 && lse != nullptr) lse[row] = big;

    const bool vec = (d % 4) == 0;
    for (int c0 = (vec ? lane * 4 : lane); c0 < d; c0 += (vec ? 128 : 32)) {
      float a[4] = {0.f, 0.f, 0.f, 0.f};
      const int w = vec ? 4 : 1;
      if (big != -INFINITY) {
        for (int t = 0; t < n_parts; ++t) {
          const float lt = lse_parts[(int64_t)t * rows + row];
          if (lt == -INFINITY) continue;
          const float wt = expf(lt - big);
          const float* src = o_parts + ((int64_t)t * rows + row) * d + c0;
          if (vec) {
            const float4 x = *reinterpret_cast<const float4*>(src);
            a[0] = fmaf(wt, x.x, a[0]);
            a[1] = fmaf(wt, x.y, a[1]);
            a[2] = fmaf(wt, x.z, a[2]);
            a[3] = fmaf(wt, x.w, a[3]);
          } else {
            a[0] = fmaf(wt, src[0], a[0]);
          }
        }
      }
      if (kBf16Out) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(o) + row * d + c0;
        for (int e = 0; e < w; ++e) dst[e] = __float2bfloat16_rn(a[e]);
      } else {
        float* dst = static_cast<float*>(o) + row * d + c0;
        if (vec)
          *reinterpret_cast<float4*>(dst) = make_float4(a[0], a[1], a[2], a[3]);
        else
          dst[0] = a[0];
      }
    }
  }
}

}  // namespace

cudaError_t launch_merge(int n_parts, int64_t rows, int d, const float* o_parts,
                         const float* lse_parts, void* o, int o_dtype, float* lse,
                         cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (rows + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  if (o_dtype == RA_DTYPE_BF16)
    merge_kernel<true><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(n_parts, rows, d, o_parts, lse_parts, o, lse);
  else
    merge_kernel<false><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(n_parts, rows, d, o_parts, lse_parts, o, lse);
  return cudaGetLastError();
}

}  // namespace ra
