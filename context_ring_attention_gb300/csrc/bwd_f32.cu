// Ring-attention backward in float32 on CUDA cores (any d <= 128), for the small
// float32 problems.  It differentiates the forward's definition: with
// P = exp(scale q.k - LSE) recomputed from the forward's LSE,
//   dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO,
// D = rowsum(dO * O) (from the preparation kernel).
//   dQ:     one warp per query row; it meets the key blocks in the forward's ring
//           order, shard (p - t) mod N at step t ("3.6 Distributed Training II",
//           section "Ring Attention").
//   dK, dV: one warp per key row of shard r; the row's block travels the ring and
//           meets the queries of shard (r + t) mod N at step t, every query head
//           of its group in turn, so the gradients gather where the block goes.
// Lanes span 32 keys (or queries) at a time; each lane keeps d/32 output columns.
#include <cuda_runtime.h>

#include <cstdint>

#include "bwd_internal.h"

namespace ra {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxD = 128;

__device__ __forceinline__ float dot_row(const float* a, const float* b, int d) {
  float acc = 0.f;
  for (int c = 0; c < d; ++c) acc = fmaf(a[c], b[c], acc);
  return acc;
}

__global__ void __launch_bounds__(kWarps * 32)
    bwd_f32_dq_kernel(const BwdParams P, const float* __restrict__ q, const float* __restrict__ k,
                      const float* __restrict__ v, const float* __restrict__ dout) {
  __shared__ float qs[kWarps][kMaxD], dos[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows_all = (int64_t)P.batch * P.heads_q * P.seq;
  const int64_t grow = (int64_t)blockIdx.x * kWarps + warp;
  if (grow >= rows_all) return;
  const int d = P.head_dim, N = P.n_shards;
  const int64_t bh = grow / P.seq, srow = grow % P.seq;
  const int p = (int)(srow / P.s_n);
  const int64_t i = srow % P.s_n;
  const int b = (int)(bh / P.heads_q), h = (int)(bh % P.heads_q);
  const int64_t kv_base = ((int64_t)b * P.heads_kv + h / P.group) * P.seq;
  const int64_t my_pos = pos_of(P.layout, N, P.s_n, p, i);
  for (int c = lane; c < d; c += 32) {
    qs[warp][c] = q[grow * d + c];
    dos[warp][c] = dout[grow * d + c];
  }
  __syncwarp();
  const int64_t li = bwd_scalar_index(bh, p, i, N, P.n64);
  RA_BOUNDS(P.status, li >= 0 && li + 64 < (int64_t)P.batch * P.heads_q * N * P.n64 * 128, 41);
  const float2 ld = make_float2(P.lse2d[li], P.lse2d[li + 64]);
  float acc[kMaxD / 32];
#pragma unroll
  for (int x = 0; x < kMaxD / 32; ++x) acc[x] = 0.f;
  for (int t = 0; t < N; ++t) {
    const int r = (p - t + N) % N;
    const int64_t nkeys = P.causal ? last_le(P.layout, N, P.s_n, r, my_pos) + 1 : P.s_n;
    const float* kb = k + (kv_base + (int64_t)r * P.s_n) * d;
    const float* vb = v + (kv_base + (int64_t)r * P.s_n) * d;
    for (int64_t j0 = 0; j0 < nkeys; j0 += 32) {
      const int64_t j = j0 + lane;
      float ds = 0.f;
      if (j < nkeys) {
        const float pj = exp2f(fmaf(dot_row(qs[warp], kb + j * d, d), P.scale_log2, -ld.x));
        ds = pj * (dot_row(dos[warp], vb + j * d, d) - ld.y);
      }
      const int nj = (nkeys - j0 < 32) ? (int)(nkeys - j0) : 32;
      for (int jj = 0; jj < nj; ++jj) {
        const float dsb = __shfl_sync(0xffffffffu, ds, jj);
        const float* kr = kb + (j0 + jj) * d;
#pragma unroll
        for (int x = 0; x < kMaxD / 32; ++x) {
          const int col = lane + 32 * x;
          if (col < d) acc[x] = fmaf(dsb, kr[col], acc[x]);
        }
      }
    }
  }
  float* dst = static_cast<float*>(P.dq) + grow * d;
#pragma unroll
  for (int x = 0; x < kMaxD / 32; ++x) {
    const int col = lane + 32 * x;
    if (col < d) dst[col] = acc[x] * P.scale;
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    bwd_f32_dkdv_kernel(const BwdParams P, const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, const float* __restrict__ dout) {
  __shared__ float ks[kWarps][kMaxD], vs[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows_all = (int64_t)P.batch * P.heads_kv * P.seq;
  const int64_t grow = (int64_t)blockIdx.x * kWarps + warp;  // key row
  if (grow >= rows_all) return;
  const int d = P.head_dim, N = P.n_shards;
  const int64_t bk = grow / P.seq, srow = grow % P.seq;
  const int r = (int)(srow / P.s_n);
  const int64_t j = srow % P.s_n;
  const int b = (int)(bk / P.heads_kv), hk = (int)(bk % P.heads_kv);
  const int64_t key_pos = pos_of(P.layout, N, P.s_n, r, j);
  for (int c = lane; c < d; c += 32) {
    ks[warp][c] = k[grow * d + c];
    vs[warp][c] = v[grow * d + c];
  }
  __syncwarp();
  float dk[kMaxD / 32], dv[kMaxD / 32];
#pragma unroll
  for (int x = 0; x < kMaxD / 32; ++x) dk[x] = dv[x] = 0.f;
  for (int t = 0; t < N; ++t) {
    const int p = (r + t) % N;  // the device this block sits on at step t
    const int64_t i_lo = P.causal ? first_ge(P.layout, N, P.s_n, p, key_pos) : 0;
    for (int g = 0; g < P.group; ++g) {
      const int64_t qrow0 = ((int64_t)b * P.heads_q + (int64_t)hk * P.group + g) * P.seq + (int64_t)p * P.s_n;
      for (int64_t i0 = i_lo; i0 < P.s_n; i0 += 32) {
        const int64_t i = i0 + lane;
        float pi = 0.f, ds = 0.f;
        if (i < P.s_n) {
          const int64_t row = qrow0 + i;
          const int64_t li = bwd_scalar_index((int64_t)b * P.heads_q + (int64_t)hk * P.group + g, p, i, N, P.n64);
          RA_BOUNDS(P.status, row >= 0 && row < (int64_t)P.batch * P.heads_q * P.seq && li >= 0 &&
                                  li + 64 < (int64_t)P.batch * P.heads_q * N * P.n64 * 128, 42);
          const float2 ld = make_float2(P.lse2d[li], P.lse2d[li + 64]);
          pi = exp2f(fmaf(dot_row(q + row * d, ks[warp], d), P.scale_log2, -ld.x));
          ds = pi * (dot_row(dout + row * d, vs[warp], d) - ld.y);
        }
        const int ni = (P.s_n - i0 < 32) ? (int)(P.s_n - i0) : 32;
        for (int ii = 0; ii < ni; ++ii) {
          const float pb = __shfl_sync(0xffffffffu, pi, ii);
          const float db = __shfl_sync(0xffffffffu, ds, ii);
          const float* qr = q + (qrow0 + i0 + ii) * d;
          const float* dor = dout + (qrow0 + i0 + ii) * d;
#pragma unroll
          for (int x = 0; x < kMaxD / 32; ++x) {
            const int col = lane + 32 * x;
            if (col < d) {
              dv[x] = fmaf(pb, dor[col], dv[x]);
              dk[x] = fmaf(db, qr[col], dk[x]);
            }
          }
        }
      }
    }
  }
  float* dkd = static_cast<float*>(P.dk) + grow * d;
  float* dvd = static_cast<float*>(P.dv) + grow * d;
#pragma unroll
  for (int x = 0; x < kMaxD / 32; ++x) {
    const int col = lane + 32 * x;
    if (col < d) {
      dkd[col] = dk[x] * P.scale;
      dvd[col] = dv[x];
    }
  }
}

}  // namespace

cudaError_t launch_bwd_f32(const BwdParams& prm, const float* q, const float* k, const float* v,
                           const float* dout, cudaStream_t stream) {
  const int64_t rows_q = (int64_t)prm.batch * prm.heads_q * prm.seq;
  const int64_t rows_kv = (int64_t)prm.batch * prm.heads_kv * prm.seq;
  const int64_t bq = (rows_q + kWarps - 1) / kWarps, bk = (rows_kv + kWarps - 1) / kWarps;
  if (bq > 0x7fffffff || bk > 0x7fffffff) return cudaErrorInvalidConfiguration;
  bwd_f32_dq_kernel<<<(unsigned)bq, kWarps * 32, 0, stream>>>(prm, q, k, v, dout);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_f32_dkdv_kernel<<<(unsigned)bk, kWarps * 32, 0, stream>>>(prm, q, k, v, dout);
  return cudaGetLastError();
}

}  // namespace ra
