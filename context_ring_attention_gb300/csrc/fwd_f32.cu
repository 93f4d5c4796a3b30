// Ring-attention forward in float32 on CUDA cores (any d <= 128).
//
// The same fold as the tensor-core kernel -- Module 23, "The Math: One Block at
// a Time", visited in the ring order of "3.6 Distributed Training II", section
// "Ring Attention" -- kept in fp32 with the accurate expf/logf for the small
// float32 problems (the Q&A page's 4-device toy, 96-token examples).  One warp
// owns one query row: each lane scores one key of a 32-key chunk, the warp
// updates (m, l) together, and each lane accumulates d/32 output columns.
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxD = 128;

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

__global__ void __launch_bounds__(kWarps * 32)
    fwd_f32_kernel(const FwdParams P, const float* __restrict__ q, const float* __restrict__ k,
                   const float* __restrict__ v) {
  __shared__ float qs[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows_all = (int64_t)P.batch * P.heads_q * P.seq;
  const int64_t grow = (int64_t)blockIdx.x * kWarps + warp;  // global query row
  if (grow >= rows_all) return;
  const int d = P.head_dim, N = P.n_shards;
  const int64_t bh = grow / P.seq, srow = grow % P.seq;
  const int p = (int)(srow / P.s_n);
  const int64_t i = srow % P.s_n;
  const int b = (int)(bh / P.heads_q), h = (int)(bh % P.heads_q);
  const int64_t kv_base = ((int64_t)b * P.heads_kv + h / P.group) * P.seq;
  const int64_t my_pos = pos_of(P.layout, N, P.s_n, p, i);

  for (int c = lane; c < d; c += 32) qs[warp][c] = q[grow * d + c];
  __syncwarp();

  const bool partials = P.o_parts != nullptr;
  float m = -INFINITY, l = 0.f;
  float acc[kMaxD / 32];
#pragma unroll
  for (int x = 0; x < kMaxD / 32; ++x) acc[x] = 0.f;

  for (int t = P.step_lo; t < P.step_hi; ++t) {
    const int r = (p - t + N) % N;
    // Keys of shard r with position <= my_pos are rows 0..J (positions rise with the row);
    // gathered K/V is one natural-order block of S keys: rows 0..my_pos.
    const int64_t kv_rows = P.gathered ? P.seq : P.s_n;
    const int64_t nkeys = !P.causal ? kv_rows : (P.gathered ? my_pos + 1 : last_le(P.layout, N, P.s_n, r, my_pos) + 1);
    const int slot = P.gathered ? 0 : (P.kv_rotated ? p : r);  // where the block of step t sits
    const float* kb = k + (kv_base + (int64_t)slot * P.s_n) * d;
    const float* vb = v + (kv_base + (int64_t)slot * P.s_n) * d;
    RA_BOUNDS(P.status, nkeys >= 0 && nkeys <= kv_rows && slot >= 0 && slot < N &&
                            kv_base + (int64_t)slot * P.s_n + nkeys <= (int64_t)P.batch * P.heads_kv * P.seq, 40);
    for (int64_t j0 = 0; j0 < nkeys; j0 += 32) {
      const int64_t j = j0 + lane;
      float s = -INFINITY;
      if (j < nkeys) {
        const float* kr = kb + j * d;
        float dot = 0.f;
        for (int c = 0; c < d; ++c) dot = fmaf(qs[warp][c], kr[c], dot);
        s = dot * P.scale;
      }
      const float m_new = fmaxf(m, warp_max(s));           // finite: key j0 is allowed
      const float corr = expf(m - m_new);                  // 0 when m was -inf
      const float pj = (j < nkeys) ? expf(s - m_new) : 0.f;
      l = l * corr + warp_sum(pj);
#pragma unroll
      for (int x = 0; x < kMaxD / 32; ++x) acc[x] *= corr;
      const int nj = (nkeys - j0 < 32) ? (int)(nkeys - j0) : 32;
      for (int jj = 0; jj < nj; ++jj) {
        const float pb = __shfl_sync(0xffffffffu, pj, jj);
        const float* vr = vb + (j0 + jj) * d;
#pragma unroll
        for (int x = 0; x < kMaxD / 32; ++x) {
          const int col = lane + 32 * x;
          if (col < d) acc[x] = fmaf(pb, vr[col], acc[x]);
        }
      }
      m = m_new;
    }
    if (partials) {  // this step's block alone, then start afresh
      float* dst = P.o_parts + ((int64_t)(t - P.step_lo) * rows_all + grow) * d;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int x = 0; x < kMaxD / 32; ++x) {
        const int col = lane + 32 * x;
        if (col < d) dst[col] = acc[x] * inv;
        acc[x] = 0.f;
      }
      if (lane == 0) P.lse_parts[(int64_t)(t - P.step_lo) * rows_all + grow] = l > 0.f ? m + logf(l) : -INFINITY;
      m = -INFINITY;
      l = 0.f;
    }
  }
  if (!partials) {
    float* dst = static_cast<float*>(P.o) + grow * d;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int x = 0; x < kMaxD / 32; ++x) {
      const int col = lane + 32 * x;
      if (col < d) dst[col] = acc[x] * inv;
    }
    if (lane == 0 && P.lse != nullptr) P.lse[grow] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdParams& prm, const float* q, const float* k, const float* v,
                           cudaStream_t stream) {
  const int64_t rows = (int64_t)prm.batch * prm.heads_q * prm.seq;
  const int64_t blocks = (rows + kWarps - 1) / kWarps;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  fwd_f32_kernel<<<(unsigned)blocks, kWarps * 32, 0, stream>>>(prm, q, k, v);
  return cudaGetLastError();
}

}  // namespace ra
