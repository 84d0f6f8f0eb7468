// FP8 (E4M3) block quantisation of Q or K for the FP8 forward.
//
// "FlashAttention 深度解析", third part, section 2.3 (FP8 与块量化): the tensor
// is split into blocks, each block gets the scale s = max(|block|) / FP8_MAX
// and is stored as Quantize(block / s).  A block is 128 consecutive rows of
// one head (the forward kernel's tile), all d columns; FP8_MAX = 448, the
// largest finite E4M3 value.  A block of zeros gets the scale 1.
//
// One CTA per block: a pass for the block's amax, then a pass that divides
// (correctly rounded fp32 division) and converts pairs with
// cvt.rn.satfinite.e4m3x2 (round to nearest even, saturating).  The block
// (at most 32 KB of bf16) is read twice, the second time from L2.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int QUANT_THREADS = 256;

template <int D>
__global__ void __launch_bounds__(QUANT_THREADS) fa_quantize_fp8_kernel(const uint16_t* __restrict__ x,
                                                                        uint8_t* __restrict__ codes,
                                                                        float* __restrict__ scales,
                                                                        int L, int n_blocks) {
  __shared__ float warp_max[QUANT_THREADS / 32];
  const int blk = static_cast<int>(blockIdx.x % static_cast<unsigned>(n_blocks));
  const long long bh = blockIdx.x / static_cast<unsigned>(n_blocks);
  const int row0 = blk * 128;
  const int rows = min(128, L - row0);
  const size_t base = (static_cast<size_t>(bh) * L + row0) * D;
  const int n = rows * D;  // a multiple of 8 (D is 64 or 128)

  float amax = 0.f;
  for (int i = threadIdx.x * 8; i < n; i += QUANT_THREADS * 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(x + base + i);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      amax = fmax3(amax, fabsf(__uint_as_float(ws[k] << 16)),
                   fabsf(__uint_as_float(ws[k] & 0xffff0000u)));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int k = 1; k < QUANT_THREADS / 32; ++k) amax = fmaxf(amax, warp_max[k]);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (threadIdx.x == 0) scales[bh * n_blocks + blk] = s;

  for (int i = threadIdx.x * 8; i < n; i += QUANT_THREADS * 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(x + base + i);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint16_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      c[k] = pack_e4m3x2(__fdiv_rn(__uint_as_float(ws[k] << 16), s),
                         __fdiv_rn(__uint_as_float(ws[k] & 0xffff0000u), s));
    *reinterpret_cast<uint2*>(codes + base + i) =
        make_uint2(static_cast<uint32_t>(c[0]) | (static_cast<uint32_t>(c[1]) << 16),
                   static_cast<uint32_t>(c[2]) | (static_cast<uint32_t>(c[3]) << 16));
  }
}

}  // namespace fa
