// Declarations of the backward pass (bwd_prep.cu, bwd_f32.cu, bwd_bf16_sm103.cu and
// ra_bwd in ra_api.cu), kept apart from the forward's so that the two evolve
// independently.
#pragma once

#include "ra_internal.h"

namespace ra {

// Backward pass: per query row the scalars lse2 = LSE * log2(e) and
// D = rowsum(dO * O), stored in blocks of 64 rows of one (batch, query head, shard):
// block ((b*Hq + h) * N + p) * n64 + i/64 holds 64 lse2 values, then 64 D values
// (zeros past the shard's last row).  Returns the float index of row i's lse2; its
// D is 64 floats further.
RA_HD int64_t bwd_scalar_index(int64_t bh, int p, int64_t i, int n_shards, int64_t n64) {
  return (((bh * n_shards + p) * n64) + i / 64) * 128 + (i % 64);
}

// Backward-pass kernels (dQ, dK, dV from dO, with the forward's LSE).
struct BwdParams {
  int32_t batch, heads_q, heads_kv, group, head_dim, n_shards;
  int16_t layout, causal;
  int32_t n_items;  // tensor-core kernels: work items of this pass
  int64_t seq, s_n;
  float scale;       // score scale
  float scale_log2;  // scale * log2(e)
  const float* lse2d;   // per query row lse2 and D, in 64-row blocks (bwd_scalar_index)
  int64_t n64;          // 64-row blocks per shard
  int32_t round_sync;   // hand out items in synchronised rounds (as FwdParams::round_sync)
  void* dq;             // [B, Hq, S, d], plan dtype
  void* dk;             // [B, Hkv, S, d]
  void* dv;
  const void* q;        // pass 1 reads its own query rows of Q and dO directly
  const void* dout;
  const WorkItem* items;
  uint32_t* status;
  uint32_t* item_counter;
};

// Launchers (each returns cudaGetLastError() of its launch).
cudaError_t launch_bwd_prep(int dtype, int64_t bh_count, int64_t seq, int n_shards, int d, const void* o,
                            const void* dout, const float* lse, float* out, cudaStream_t stream);
cudaError_t launch_bwd_f32(const BwdParams& prm, const float* q, const float* k, const float* v,
                           const float* dout, cudaStream_t stream);
// pass 0: dK and dV (items are key tiles); pass 1: dQ (items are query tiles).
cudaError_t launch_bwd_bf16(int pass, const BwdParams& prm, const void* q, const void* k, const void* v,
                            const void* dout, int grid, cudaStream_t stream, const char** why);
// The tensor-core kernels' bounded wait on a barrier nothing completes (about 1 s);
// it records kStatusTimeoutMma in *status.
cudaError_t launch_wait_selftest(uint32_t* status, cudaStream_t stream);


}  // namespace ra
