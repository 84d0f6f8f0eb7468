// Merge of split-KV partial results (Flash-Decoding's final step,
// "04 Transformers, Attention, and FlashAttention", Flash-Decoding: the K/V
// sequence is cut into chunks, each chunk is attended to on its own, and the
// chunk results are combined).
//
// Split s of a row holds O_s (normalised over that split's keys) and
// LSE_s = log sum over those keys of exp(scale * q.k).  The row's result is
//   LSE = log sum_s exp(LSE_s)           (computed as M + log sum exp(LSE_s - M))
//   O   = sum_s exp(LSE_s - LSE) * O_s
// which is exact: exp(LSE_s - LSE) is the share of the softmax mass that
// split s holds.  An empty split has LSE_s = -inf and weight 0.
//
// One warp per row; each lane owns D/32 consecutive output columns, so every
// split's row is read with one coalesced D*4-byte access.  The kernel is
// bound by HBM: per row it reads n_splits * (4*D + 4) bytes and writes
// 2*D + 4.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "pdl.cuh"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int MERGE_WARPS = 8;

template <int D>
__global__ void __launch_bounds__(MERGE_WARPS * 32)
    fa_merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                    uint16_t* __restrict__ o, float* __restrict__ lse, int64_t rows,
                    int n_splits) {
  constexpr int PER_LANE = D / 32;
  pdl_wait();  // the partials come from the split pass (programmatic launch)
  const int64_t row = static_cast<int64_t>(blockIdx.x) * MERGE_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;

  float mx = -INFINITY;
  for (int s = lane; s < n_splits; s += 32) mx = fmaxf(mx, lse_part[s * rows + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sum = 0.f;
  if (mx != -INFINITY)
    for (int s = lane; s < n_splits; s += 32) {
      const float ls = lse_part[s * rows + row];
      if (ls != -INFINITY) sum += expf(ls - mx);
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float lse_row = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);

  float acc[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;
  if (lse_row != -INFINITY)
    for (int s = 0; s < n_splits; ++s) {
      const float ls = lse_part[s * rows + row];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - lse_row);
      const float* src = o_part + (s * rows + row) * D + lane * PER_LANE;
      if constexpr (PER_LANE == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
  uint16_t* dst = o + row * D + lane * PER_LANE;
  if constexpr (PER_LANE == 4) {
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0], acc[1]);
  }
  if (lane == 0) lse[row] = lse_row;
}

}  // namespace fa
