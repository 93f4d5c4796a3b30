// Exact merge of partial attention results (order independence of the
// online-softmax fold, Module 23, "The Math: One Block at a Time"):
//   LSE = ln sum_t e^(LSE_t),   O = sum_t e^(LSE_t - LSE) O_t.
// HBM-bound: one warp per row, 16-byte loads along d.  For d = 128 (the attention
// case) a lane owns 4 columns and the part weights are computed once per row by the
// lanes t < n_parts and broadcast.  Up to 8 parts (a ring of up to 8 devices), a
// warp takes two rows at a time and issues every load of both rows -- 16 blocks of
// 512 bytes and the LSEs -- before any arithmetic, so that enough bytes are in
// flight per SM to cover the HBM latency.
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

__device__ __forceinline__ void store_row(void* o, int64_t row, int lane, float4 a, bool bf16_out) {
  if (bf16_out) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(o)[row * 32 + lane] = pk;
  } else {
    reinterpret_cast<float4*>(o)[row * 32 + lane] = a;
  }
}

// d = 128 and n_parts <= kFewParts: kRowsPerWarp rows per warp at a time, all loads first.
constexpr int kFewParts = 8;
constexpr int kRowsPerWarp = 2;
template <bool kBf16Out>
__global__ void __launch_bounds__(kWarps * 32)
    merge_d128_few_kernel(int n_parts, int64_t rows, const float4* __restrict__ o_parts,
                          const float* __restrict__ lse_parts, void* __restrict__ o, float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t first = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRowsPerWarp;
  const int64_t stride = (int64_t)gridDim.x * kWarps * kRowsPerWarp;
  for (int64_t r0 = first; r0 < rows; r0 += stride) {
    float lt[kRowsPerWarp];
    float4 x[kRowsPerWarp][kFewParts];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int64_t row = r0 + r;
      const bool in = row < rows;
      lt[r] = (in && lane < n_parts) ? lse_parts[(int64_t)lane * rows + row] : -INFINITY;
#pragma unroll
      for (int b = 0; b < kFewParts; ++b)
        x[r][b] = (in && b < n_parts) ? o_parts[((int64_t)b * rows + row) * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int64_t row = r0 + r;
      if (row >= rows) break;  // warp-uniform
      const float top = warp_max(lt[r]);
      const float e = (top != -INFINITY && lt[r] != -INFINITY) ? expf(lt[r] - top) : 0.f;
      const float z = warp_sum(e);
      const float big = (top != -INFINITY) ? top + logf(z) : -INFINITY;
      const float w_lane = (big != -INFINITY && lt[r] != -INFINITY) ? expf(lt[r] - big) : 0.f;
      if (lane == 0 && lse != nullptr) lse[row] = big;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int b = 0; b < kFewParts; ++b) {
        const float w = __shfl_sync(0xffffffffu, w_lane, b);
        if (b < n_parts && w != 0.f) {  // a part with LSE = -inf adds nothing (its O may be anything)
          a.x = fmaf(w, x[r][b].x, a.x);
          a.y = fmaf(w, x[r][b].y, a.y);
          a.z = fmaf(w, x[r][b].z, a.z);
          a.w = fmaf(w, x[r][b].w, a.w);
        }
      }
      store_row(o, row, lane, a, kBf16Out);
    }
  }
}

// d = 128, more parts: lane owns columns 4*lane .. 4*lane + 3 of every part.
template <bool kBf16Out>
__global__ void __launch_bounds__(kWarps * 32)
    merge_d128_kernel(int n_parts, int64_t rows, const float4* __restrict__ o_parts,
                      const float* __restrict__ lse_parts, void* __restrict__ o, float* __restrict__ lse) {
  constexpr int kBatch = 8;  // parts whose loads are in flight together
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); row < rows; row += stride) {
    // lane t < n_parts (t < 32 here; more parts go through the generic kernel) holds LSE_t
    const float lt = lane < n_parts ? lse_parts[(int64_t)lane * rows + row] : -INFINITY;
    const float top = warp_max(lt);
    const float e = (top != -INFINITY && lt != -INFINITY) ? expf(lt - top) : 0.f;
    const float z = warp_sum(e);
    const float big = (top != -INFINITY) ? top + logf(z) : -INFINITY;
    const float w_lane = (big != -INFINITY && lt != -INFINITY) ? expf(lt - big) : 0.f;  // this lane's part weight
    if (lane == 0 && lse != nullptr) lse[row] = big;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t0 = 0; t0 < n_parts; t0 += kBatch) {
      float4 x[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        if (t0 + b < n_parts) x[b] = o_parts[((int64_t)(t0 + b) * rows + row) * 32 + lane];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const float w = __shfl_sync(0xffffffffu, w_lane, (t0 + b) & 31);
        if (t0 + b < n_parts && w != 0.f) {
          a.x = fmaf(w, x[b].x, a.x);
          a.y = fmaf(w, x[b].y, a.y);
          a.z = fmaf(w, x[b].z, a.z);
          a.w = fmaf(w, x[b].w, a.w);
        }
      }
    }
    store_row(o, row, lane, a, kBf16Out);
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
  if (d == 128 && n_parts <= kFewParts) {
    int64_t few_blocks = (rows + kWarps * kRowsPerWarp - 1) / (kWarps * kRowsPerWarp);
    if (few_blocks > cap) few_blocks = cap;
    if (o_dtype == RA_DTYPE_BF16)
      merge_d128_few_kernel<true><<<(unsigned)few_blocks, kWarps * 32, 0, stream>>>(
          n_parts, rows, reinterpret_cast<const float4*>(o_parts), lse_parts, o, lse);
    else
      merge_d128_few_kernel<false><<<(unsigned)few_blocks, kWarps * 32, 0, stream>>>(
          n_parts, rows, reinterpret_cast<const float4*>(o_parts), lse_parts, o, lse);
    return cudaGetLastError();
  }
  if (d == 128 && n_parts <= 32) {
    if (o_dtype == RA_DTYPE_BF16)
      merge_d128_kernel<true><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(
          n_parts, rows, reinterpret_cast<const float4*>(o_parts), lse_parts, o, lse);
    else
      merge_d128_kernel<false><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(
          n_parts, rows, reinterpret_cast<const float4*>(o_parts), lse_parts, o, lse);
    return cudaGetLastError();
  }
  if (o_dtype == RA_DTYPE_BF16)
    merge_kernel<true><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(n_parts, rows, d, o_parts, lse_parts, o, lse);
  else
    merge_kernel<false><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(n_parts, rows, d, o_parts, lse_parts, o, lse);
  return cudaGetLastError();
}

}  // namespace ra
