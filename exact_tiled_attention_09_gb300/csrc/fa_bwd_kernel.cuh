// Exact attention backward for sm_103a: recomputation of P from Q, K and the
// forward log-sum-exp, TMA + tcgen05 + TMEM, fp32 gradients accumulated on
// chip.
//
// The gradients are those of "FlashAttention 深度解析", first part, section
// 4.1 (dV = P^T dO, dP = dO V^T, dS = P (.) (dP - rowsum(dP (.) P))) with the
// chain rule through the scaled scores S = scale * Q K^T (dQ = scale * dS K,
// dK = scale * dS^T Q); P is recomputed block by block from the stored
// per-row log-sum-exp instead of being read back (section 4.2, 重计算策略).
// The row sum rowsum(dP (.) P)_i equals <dO_i, O_i> (dP = dO V^T and O = P V),
// which a pre-pass computes once per query row from O and dO.
//
// Work unit: one block j of 128 keys of one (batch, head).  Its CTA keeps
// K_j and V_j in shared memory and dK_j, dV_j in tensor memory, and walks
// the query blocks i (all of them, or i >= j with the causal mask).  The
// grid is persistent, one CTA per SM: a CTA starts with the unit of its
// own index and then claims the next unclaimed unit from a counter (zeroed
// by the pre-pass), so the set-up, the tensor-memory allocation and the
// launch of a CTA are paid once per SM, and the next unit's first copies
// and products start while the last one's dK and dV leave.  Per query block
// a unit computes, transposed so that its own keys are the TMEM lanes:
//
//   S^T  = K_j Q_i^T                (SS MMA, M = keys, N = queries, K = d)
//   dP^T = V_j dO_i^T               (SS MMA)
//   P^T  = exp2(S^T * scale*log2e - lse_i*log2e)     (gradient warps)
//   dV_j += P^T dO_i                (TS MMA: P^T from TMEM, bf16 over S^T)
//   dS^T = scale * P^T (.) (dP^T - D_i)               (gradient warps, bf16
//                                                      into shared memory)
//   dK_j += dS^T Q_i                (SS MMA, dS^T K-major)
//   dQ_i  = dS K_j                  (SS MMA, the same dS tile read MN-major,
//                                    into the dP^T columns)
//
// and dQ_i is added into an fp32 accumulator in global memory (tensor
// reduce-adds; every key block of the head contributes to every dQ_i).
// Post-pass: dQ = bf16(accumulator).
//
// Warp roles (576 threads; 704 at d = 64):
//   warp 0      MMA issuer, owner of the tensor memory (whole warp polls,
//               one elected lane issues)
//   warp 1      TMA producer: K_j, V_j per unit; Q_i and dO_i into a ring
//               of stages (two at d = 128, three at d = 64), continued
//               across units; issues the dQ reduce-adds; claims units and
//               publishes each in one of two shared-memory slots (full /
//               free barriers) that the other roles read
//   warps 2..17 gradient warps: warp w handles TMEM lanes 32*(w%4)..+31
//               (its keys) and query columns 32*h..32*h+31, h = (w-2)/4
//   warps 18..21 d = 64 only: dQ warps, one per TMEM lane quarter: copy dQ_i
//               out of tensor memory and stage it (phase C below)
//
// Tensor memory (512 columns): [0,128) S^T, then P^T as packed bf16 (group
// h's 32 queries in columns 32h..32h+15); [128,256) dP^T, then dQ_i
// (d = 128; at d = 64 dQ_i has [384,448) of its own, so dP_{i+1} need not
// wait for dQ_i to be copied out); [256,256+D) dV_j; [256+D,256+2D) dK_j.
//
// Order of the MMAs per query block (tcgen05 operations of one thread
// complete in issue order, which the hand-offs rely on):
//   d = 128: dP_i | wait P ready: dV_i | wait dS ready: dK_i, dQ_i (two
//            column halves) | S_{i+1}
//   d = 64:  dP_i | wait P ready: dV_i, S_{i+1} | wait dS ready: dK_i, dQ_i
// and the gradient warps work on phases A (P), B (dS), C (dQ out) as
// A(i) B(i) C(i) at d = 128 and A(0), then B(i) A(i+1) at d = 64, where the
// MMA work per block is half as large, P of the next block is computed
// while dK_i and dQ_i run, and the dQ warps run C(i).  S_{i+1} overwrites
// P^T_i only after dV_i has read it; dP_{i+1} is issued after dK_i and dQ_i
// (at d = 128 also after dQ_i has left its columns), so its commit proves
// dK_i and dQ_i have read the dS tile before the gradient warps write
// dS_{i+1}.  After a unit's last block the MMA warp commits once more
// (fin): the producer waits for it before copying the next unit's K and V
// over the last ones, and so does the epilogue when the dQ warps, not the
// gradient warps, track dq_full.  Blocks are numbered across the CTA's
// units, so each once-per-block barrier simply continues its phases from
// one unit to the next; the next unit's dV and dK products (which start
// their accumulators afresh) wait for its first P, which the gradient warps
// write only after reading the previous dV and dK out.
//
// Copies and the dQ path.  Q_i (with its per-query terms) and dO_i have
// separate full barriers.  dQ_i leaves through the producer warp: the
// gradient warps stage it in block i's Q and dO buffers (free once dQ_i is
// final: every MMA that read them is complete) and arrive on dq_staged; the
// producer issues the tensor reduce-adds as two groups, columns 0..d/2-1
// (staged in the Q buffer) first, and refills the Q buffer (Q_{i+2}, needed
// first) as soon as that group has been read, the dO buffer after the
// second.  At d = 128 dQ_i is computed as two 64-column halves with a
// commit each: the first half is staged, reduced and the Q buffer refilled
// while the tensor core computes the second, and the Q copy enters the
// copy engine before the second half's reduce.  dK_j and dV_j leave at the
// end of a unit as bf16 from the gradient warps; at d = 128 each warp
// passes its part through its own bytes of the dS tile first, so that its
// global stores are row-contiguous.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "pdl.cuh"
#include "sm103_ptx.cuh"

namespace fa {

// Gradient warps: BWD_GRAD_GROUPS per TMEM lane quarter, each taking
// 128 / BWD_GRAD_GROUPS query columns of S^T and dP^T and D / BWD_GRAD_GROUPS
// columns of dQ, dK and dV.  Four groups (16 warps) keep four warps per
// sub-partition on the element-wise phases, whose per-warp chains of
// tensor-memory loads, exponentials and shared-memory stores are
// latency-bound with two.
constexpr int BWD_GRAD_GROUPS = 4;
constexpr int BWD_GRAD_WARPS = 4 * BWD_GRAD_GROUPS;
constexpr int BWD_FIRST_GRAD_WARP = 2;
constexpr int BWD_DS_BYTES = 128 * 128 * 2;  // dS^T tile, two 128 x 64 boxes

// Wait sites of the backward kernel (bit index in the device status word).
enum : uint32_t {
  SITE_B_KV = 8,
  SITE_B_FULL = 9,
  SITE_B_DQST = 10,

  SITE_B_S = 11,
  SITE_B_DP = 12,
  SITE_B_P = 13,
  SITE_B_DS = 14,
  SITE_B_DQ = 15,
  SITE_B_DQFREE = 16,
  SITE_B_ALIGN = 17,  // not a wait: the shared-memory base left too little slack
  SITE_B_UNIT = 18,   // a unit slot (published or taken by every reader)
  SITE_B_FIN = 19,    // the producer's wait for the previous unit's MMAs
};

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dimension must be 64 or 128");
  static constexpr int BOXES = D / 64;
  static constexpr int TILE_BYTES = 128 * D * 2;
  // Q/dO stages.  At d = 64 there is room for three, and the pipeline runs
  // S_{i+1} right behind dV_i so that P of the next block is computed while
  // dK_i and dQ_i run (EARLY_S); the third stage gives the copy of Q_{i+1}
  // the time that the dQ reduce of the stage's previous block takes.  At
  // d = 128 two stages fill shared memory and S_{i+1} follows dQ_i.
  static constexpr int STAGES = (D == 64) ? 3 : 2;
  static constexpr bool EARLY_S = (D == 64);
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE_BYTES;
  // stage s: Q at +0, dO at +TILE, -lse*log2e [128] at +2*TILE, -scale*D
  // [128] at +2*TILE+512.
  static constexpr int STAGE_OFF = 2 * TILE_BYTES;
  static constexpr int ROWTERM_OFF = 2 * TILE_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES + 1024;
  static constexpr int DS_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = DS_OFF + BWD_DS_BYTES;
  // kv_full, fullQ[S], fulldO[S], dq_staged[S], s_full, dp_full, p_ready,
  // ds_ready, dq_full, dq_free, drain, dq_full2, dq_staged2[S], fin,
  // unit_full[2], unit_free[2]
  static constexpr int NBAR = 1 + 3 * STAGES + 7 + 1 + STAGES + 1 + 4;
  // then the TMEM address, the abort flag and the two unit slots (unit
  // index and its query-block count, 8 B each)
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  // The tiles need a 1024-byte aligned base; the launch adds as much slack
  // as the 227 KB budget leaves (up to 1024 bytes) and the kernel checks the
  // slack it actually needs.
  static constexpr int USED_BYTES = MISC_OFF + 24;
  static constexpr int SLACK = (232448 - USED_BYTES) < 1024 ? (232448 - USED_BYTES) / 16 * 16 : 1024;
  static constexpr int SMEM_BYTES = USED_BYTES + SLACK;
  static_assert(SLACK >= 0 && SMEM_BYTES <= 232448, "shared memory budget");
  // dQ staging: 8 * D/64 boxes of 4 KB fill the Q and dO buffers exactly,
  // the first half in the Q buffer
  static constexpr int DQ_BOXES = 8 * BOXES;
  // Packed bf16 P^T of gradient group h (queries CQ*h.., CQ = 128 / groups)
  // lies in columns CQ*h..CQ*h + CQ/2 - 1 (over its own S^T columns): the
  // 16 queries of MMA k-step kk start at this column.
  __host__ __device__ static constexpr uint32_t p_col(int kk) {
    return (128 / BWD_GRAD_GROUPS) * (16 * kk / (128 / BWD_GRAD_GROUPS)) +
           (16 * kk % (128 / BWD_GRAD_GROUPS)) / 2;
  }
  static_assert(DQ_BOXES * 4096 == 2 * TILE_BYTES, "dQ staging fills the Q/dO buffers");
  static constexpr uint32_t S_COL = 0;
  static constexpr uint32_t DP_COL = 128;
  static constexpr uint32_t DV_COL = 256;
  static constexpr uint32_t DK_COL = 256 + D;
  // d = 64 leaves 128 tensor-memory columns free: dQ_i gets its own 64, so
  // dP_{i+1} need not wait until dQ_i has been copied out (at d = 128 dQ_i
  // reuses dP_i's columns).
  static constexpr bool SPLIT_DQ = (D == 64);
  // d = 128: dQ_i is computed as two 64-column halves with a commit each.
  // The first half is staged (into the Q buffer) and its reduce started
  // while the tensor core still computes the second, which brings the
  // refill of the Q buffer for block i+2 forward.
  static constexpr bool DQ_HALVES = (D == 128);
  // d = 64: four more warps (one per TMEM lane quarter, after the gradient
  // warps) copy dQ_i out of tensor memory and stage it, so that the
  // gradient warps go from dS_i straight to P of the next block.
  static constexpr int DQ_WARPS = (D == 64) ? 4 : 0;
  static constexpr int FIRST_DQ_WARP = BWD_FIRST_GRAD_WARP + BWD_GRAD_WARPS;
  static constexpr int THREADS = 32 * (FIRST_DQ_WARP + DQ_WARPS);
  // arrivals on dq_free and dq_staged: the warps that copy dQ out
  static constexpr int DQ_COPIERS = DQ_WARPS ? DQ_WARPS : BWD_GRAD_WARPS;
  // warps that read every published unit: the MMA, gradient and dQ warps
  static constexpr int UNIT_READERS = 1 + BWD_GRAD_WARPS + DQ_WARPS;
  static constexpr uint32_t DQ_COL = SPLIT_DQ ? 256 + 2 * D : DP_COL;
  static_assert(!SPLIT_DQ || DQ_COL + D <= 512, "tensor memory budget");
};

struct BwdArgs {
  uint16_t* dk;            // bf16 [BH, L, D]
  uint16_t* dv;            // bf16 [BH, L, D]
  float* dq_acc;           // fp32 [BH, L, D], zeroed by the pre-pass
  const float* nlse2;      // fp32 [BH, Lp]: -lse * log2(e); -inf past L
  const float* nds;        // fp32 [BH, Lp]: -scale * <dO_i, O_i>; 0 past L
  int L;
  int Lp;                  // L rounded up to a multiple of 128
  int n_kv;                // key blocks per head = Lp / 128
  int bh;                  // B * H
  int group_heads;         // heads per scheduling group (see the CTA order)
  float scale_log2;        // scale * log2(e)
  float scale;
  unsigned int* status;
  unsigned long long timeout_ns;
  int test_withhold_kv;    // test hook: skip the K/V copies so the first wait runs out
  unsigned int* sched;     // units claimed after the first wave, zeroed by the pre-pass
  int n_units;             // B * H * n_kv
};

// Pre-pass arguments: per query row, the two per-row terms the main kernel
// needs, and the zeroed dQ accumulator.
struct BwdPreArgs {
  const uint16_t* o;       // bf16 [BH, L, D]
  const uint16_t* dout;    // bf16 [BH, L, D]
  const float* lse;        // fp32 [BH, L]
  float* nlse2;            // fp32 [BH, Lp]
  float* nds;              // fp32 [BH, Lp]
  float* dq_acc;           // fp32 [BH, L, D]
  unsigned int* sched;     // the main kernel's unit counter
  int L;
  int Lp;
  long long rows;          // BH * Lp
  float scale;
};

// Tensor-memory moves of N consecutive 32-bit columns per lane in one
// instruction (one wide access costs less than several narrow ones).
__device__ __forceinline__ void bwd_tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
template <int N>
__device__ __forceinline__ void bwd_tmem_ld(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32 || N == 64, "16, 32 or 64 columns");
  if constexpr (N == 64)
    tmem_ld64(taddr, r);
  else if constexpr (N == 32)
    tmem_ld32(taddr, r);
  else
    bwd_tmem_ld16(taddr, r);
}
template <int N>
__device__ __forceinline__ void bwd_tmem_st(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32)
    tmem_st32(taddr, r);
  else
    tmem_st16(taddr, r);
}
// Registers written by a tensor-memory load are not read before the wait.
template <int N>
__device__ __forceinline__ void reg_fence_n(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

constexpr int BWD_AUX_WARPS = 8;  // warps per block of the pre-pass
constexpr int BWD_PRE_ROWS = 4;   // rows per warp of the pre-pass

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Pre-pass, one warp per BWD_PRE_ROWS consecutive rows of [BH, Lp]:
// D_i = <dO_i, O_i> (fp32, bf16 inputs), stored as -scale * D_i, and
// -lse_i * log2(e); rows past L get the values that make them vanish in the
// main kernel (P = 0, dS = 0).  It also zeroes the dQ accumulator rows, and
// block 0 the main kernel's unit counter.  The loads of all the warp's rows
// are issued before any is used (more bytes in flight per warp: the kernel
// is bound by HBM).  The main kernel is its
// programmatic dependant: it is launched as the last blocks of this grid
// exit (no early trigger: a gradient CTA resident early would take the
// registers that blocks of this pass need on its SM).
template <int D>
__global__ void __launch_bounds__(BWD_AUX_WARPS * 32) fa_bwd_pre_kernel(const BwdPreArgs a) {
  using Vec = typename std::conditional<D == 64, uint32_t, uint2>::type;
  const long long row0 =
      (static_cast<long long>(blockIdx.x) * BWD_AUX_WARPS + (threadIdx.x >> 5)) * BWD_PRE_ROWS;
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.sched = 0u;
  Vec ow[BWD_PRE_ROWS], dw[BWD_PRE_ROWS];
  bool live[BWD_PRE_ROWS];
#pragma unroll
  for (int k = 0; k < BWD_PRE_ROWS; ++k) {
    const long long row = row0 + k;
    const long long bh = row / a.Lp;
    const int q = static_cast<int>(row - bh * a.Lp);
    live[k] = row < a.rows && q < a.L;
    if (live[k]) {
      const size_t src = (static_cast<size_t>(bh) * a.L + q) * D;
      ow[k] = reinterpret_cast<const Vec*>(a.o + src)[lane];
      dw[k] = reinterpret_cast<const Vec*>(a.dout + src)[lane];
      if constexpr (D == 64)
        reinterpret_cast<float2*>(a.dq_acc + src)[lane] = make_float2(0.f, 0.f);
      else
        reinterpret_cast<float4*>(a.dq_acc + src)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int k = 0; k < BWD_PRE_ROWS; ++k) {
    const long long row = row0 + k;
    if (row >= a.rows) break;
    float acc = 0.f;
    if (live[k]) {
      if constexpr (D == 64) {
        const uint32_t o1 = ow[k], d1 = dw[k];
        acc = fmaf(bf16_hi(o1), bf16_hi(d1), bf16_lo(o1) * bf16_lo(d1));
      } else {
        const uint2 o2 = ow[k], d2 = dw[k];
        acc = bf16_lo(o2.x) * bf16_lo(d2.x);
        acc = fmaf(bf16_hi(o2.x), bf16_hi(d2.x), acc);
        acc = fmaf(bf16_lo(o2.y), bf16_lo(d2.y), acc);
        acc = fmaf(bf16_hi(o2.y), bf16_hi(d2.y), acc);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const long long bh = row / a.Lp;
      const int q = static_cast<int>(row - bh * a.Lp);
      if (live[k]) {
        a.nlse2[row] = -a.lse[static_cast<size_t>(bh) * a.L + q] * 1.4426950408889634f;
        a.nds[row] = -a.scale * acc;
      } else {
        a.nlse2[row] = -INFINITY;
        a.nds[row] = 0.f;
      }
    }
  }
}

// Post-pass: dQ = bf16(accumulator), four elements per thread and step,
// BWD_POST_UNROLL steps' loads issued together.  Launched as a dependant of
// the main kernel: it waits for that grid before reading the accumulator.
constexpr int BWD_POST_UNROLL = 4;
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const float* __restrict__ acc,
                                                          uint16_t* __restrict__ dq,
                                                          long long n4) {
  pdl_wait();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n4;
       i0 += stride * BWD_POST_UNROLL) {
    float4 v[BWD_POST_UNROLL];
#pragma unroll
    for (int u = 0; u < BWD_POST_UNROLL; ++u) {
      const long long i = i0 + u * stride;
      if (i < n4) v[u] = reinterpret_cast<const float4*>(acc)[i];
    }
#pragma unroll
    for (int u = 0; u < BWD_POST_UNROLL; ++u) {
      const long long i = i0 + u * stride;
      if (i < n4)
        reinterpret_cast<uint2*>(dq)[i] =
            make_uint2(pack_bf16x2(v[u].x, v[u].y), pack_bf16x2(v[u].z, v[u].w));
    }
  }
}

// Main backward kernel: persistent, one CTA per SM, each taking work units
// (head, key block) in turn; see the file comment.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const BwdArgs args) {
  using C = BwdCfg<D>;
  constexpr uint32_t BOX = 128 * 64 * 2;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  if (base - raw > static_cast<uint32_t>(C::SLACK)) {
    // Not enough room to align the tiles: report and leave before any
    // barrier, copy or tensor-memory allocation (uniform across the CTA).
    if (threadIdx.x == 0) atomicOr(args.status, 1u << SITE_B_ALIGN);
    return;
  }

  const uint32_t sK = base + C::K_OFF;
  const uint32_t sV = base + C::V_OFF;
  auto sQ = [&](int st) { return base + C::STAGE_OFF + st * C::STAGE_BYTES; };
  auto sdO = [&](int st) { return base + C::STAGE_OFF + st * C::STAGE_BYTES + C::TILE_BYTES; };
  // per-query terms of stage st: -lse*log2e at +0, -scale*D at +512 (bytes)
  auto rowterms = [&](int st) {
    return base_ptr + C::STAGE_OFF + st * C::STAGE_BYTES + C::ROWTERM_OFF;
  };
  const uint32_t sDS = base + C::DS_OFF;
  uint8_t* const ds_ptr = base_ptr + C::DS_OFF;
  // dQ staging: 32-row x 32-float pieces at 4 KB steps from the Q buffer
  // on; piece 4*c + q holds dQ columns 32c..32c+31 of query rows 32q..32q+31,
  // so the four pieces of a column strip c form one 128-row box of the
  // reduce (16 KB), and columns 0..D/2-1 fill the Q buffer.
  auto dq_box = [&](int st, int b) -> uint32_t { return sQ(st) + b * 4096; };
  const uint32_t bars = base + C::BAR_OFF;
  const uint32_t bar_kv = bars;
  auto bar_fullq = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_fulldo = [&](int s) { return bars + 8u * (1 + C::STAGES + s); };
  // dq_staged of stage s completes once per use of the stage, so it can
  // never run a phase ahead of the producer: staging block k+2 needs block
  // k+2 loaded, which the producer does only after consuming block k's phase.
  auto bar_dqst = [&](int s) { return bars + 8u * (1 + 2 * C::STAGES + s); };
  const uint32_t bar_s = bars + 8u * (1 + 3 * C::STAGES);
  const uint32_t bar_dp = bar_s + 8;
  const uint32_t bar_p = bar_s + 16;
  const uint32_t bar_ds = bar_s + 24;
  const uint32_t bar_dq = bar_s + 32;
  const uint32_t bar_dqfree = bar_s + 40;
  const uint32_t bar_drain = bar_s + 48;
  const uint32_t bar_dq2 = bar_s + 56;  // second half of dQ_i (DQ_HALVES)
  // dq_staged2 of stage s: the second half of the stage's dQ (DQ_HALVES)
  auto bar_dqst2 = [&](int s) { return bar_s + 64 + 8u * s; };
  // every MMA of the current unit has completed (one commit after its last
  // block)
  const uint32_t bar_fin = bar_s + 64 + 8u * C::STAGES;
  // unit slot s: written by the producer (unit_full), read by every reader
  // warp (unit_free)
  auto bar_ufull = [&](int s) { return bar_fin + 8u + 8u * s; };
  auto bar_ufree = [&](int s) { return bar_fin + 24u + 8u * s; };
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);
  volatile int* const unit_slot = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 8);

  const int warp = warp_index_uniform();
  const int lane = threadIdx.x & 31;
  const int L = args.L;
  const int n_kv = args.n_kv;

  // Work units in claim order.  Heads go in groups of `group_heads` whose Q,
  // dO and dQ accumulator fit comfortably in L2 (every key block of a head
  // re-reads them).  Non-causal units all cost the same and go head-major;
  // causal key block j visits n_kv - j query blocks, so within a group block
  // 0 of every head goes first (longest first).  A CTA starts with unit
  // blockIdx.x and then claims the next unclaimed one from a counter in the
  // workspace, as the hardware would hand out CTAs.
  struct Unit {
    int bh, jblk, q_first, n_i;
  };
  auto decode = [&](int idx) {
    const int BH = args.bh;
    const int G = args.group_heads;
    const int g0 = (idx / (G * n_kv)) * G;
    const int gsz = min(G, BH - g0);
    const int rk = idx - g0 * n_kv;
    Unit u;
    u.bh = CAUSAL ? g0 + rk % gsz : g0 + rk / n_kv;
    u.jblk = CAUSAL ? rk / gsz : rk % n_kv;
    u.q_first = CAUSAL ? u.jblk : 0;
    u.n_i = n_kv - u.q_first;  // query blocks visited, >= 1
    return u;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_fullq(s), 1);
      mbar_init(bar_fulldo(s), 1);
      mbar_init(bar_dqst(s), C::DQ_COPIERS);  // one arrival per copying warp: dQ staged
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, BWD_GRAD_WARPS);  // one arrival per gradient warp
    mbar_init(bar_ds, BWD_GRAD_WARPS);
    mbar_init(bar_dq, 1);
    mbar_init(bar_dqfree, C::DQ_COPIERS);
    mbar_init(bar_drain, 1);
    mbar_init(bar_dq2, 1);
    mbar_init(bar_fin, 1);
    for (int s = 0; s < C::STAGES; ++s) mbar_init(bar_dqst2(s), C::DQ_COPIERS);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_ufull(s), 1);
      mbar_init(bar_ufree(s), C::UNIT_READERS);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmdQ);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, args.status, args.timeout_ns};
  auto warp_wait = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
    const bool w = mbar_wait(bar, parity, ctl, site);
    return __all_sync(0xffffffffu, w);
  };
  // Blocks are counted over all the CTA's units: block b uses stage
  // b % STAGES, the stage's (b / STAGES)-th phase, and phase b of each
  // once-per-block barrier.  All three depend on b modulo BM = 2 * STAGES
  // only, which is what every role keeps (no overflow however many units a
  // CTA takes).
  constexpr int BM = 2 * C::STAGES;
  auto stage_of = [](int b) { return b % C::STAGES; };
  auto use_parity = [](int b) { return static_cast<uint32_t>(b / C::STAGES) & 1u; };
  auto par = [](int b) { return static_cast<uint32_t>(b) & 1u; };
  // Unit k of this CTA (k = 0, 1, ...), for a reader warp: its index (and
  // its query-block count in n_i), -1 after the last one, or -2 if the wait
  // gave up.
  auto read_unit = [&](int k, int& n_i) -> int {
    const int s = k & 1;
    if (!warp_wait(bar_ufull(s), static_cast<uint32_t>(k >> 1) & 1u, SITE_B_UNIT)) return -2;
    const int u = unit_slot[2 * s];
    n_i = unit_slot[2 * s + 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_ufree(s));
    return u;
  };

  if (warp == 1) {
    // ------------------------------------------------------------ producer
    Unit u = decode(static_cast<int>(blockIdx.x));
    if (lane == 0) {
      unit_slot[0] = static_cast<int>(blockIdx.x);
      unit_slot[1] = u.n_i;
      mbar_arrive(bar_ufull(0));
    }
    __syncwarp();
    auto load_kv = [&](const Unit& w) {
      if (!args.test_withhold_kv && elect_one()) {
        mbar_arrive_expect_tx(bar_kv, 2 * C::TILE_BYTES);
        for (int c = 0; c < C::BOXES; ++c) {
          tma_load_3d(sK + c * BOX, &tmK, bar_kv, c * 64, w.jblk * 128, w.bh);
          tma_load_3d(sV + c * BOX, &tmV, bar_kv, c * 64, w.jblk * 128, w.bh);
        }
      }
      __syncwarp();
    };
    load_kv(u);
    uint32_t kv_par = 0;  // phase parity of the last K/V load
    // The per-query terms, the zeroed dQ accumulator and the zeroed unit
    // counter come from the pre-pass, which may still be running
    // (programmatic launch).
    pdl_wait();
    // (head, query block) of the block each stage holds, for its reduce
    int st_bh[C::STAGES], st_qb[C::STAGES];
#pragma unroll
    for (int t = 0; t < C::STAGES; ++t) st_bh[t] = st_qb[t] = 0;
    // per stage: loaded at all (bit s), the phase parity of its last Q / dO
    // load (for the drain after an abort)
    uint32_t q_used = 0, q_par = 0, do_used = 0, do_par = 0;
    auto load_q = [&](int blk, int b, int qb) {
      const int st = stage_of(blk);
      q_used |= 1u << st;
      q_par = (q_par & ~(1u << st)) | (use_parity(blk) << st);
      if (elect_one()) {
        mbar_arrive_expect_tx(bar_fullq(st), C::TILE_BYTES + 1024);
        const int row = qb * 128;
        for (int c = 0; c < C::BOXES; ++c)
          tma_load_3d(sQ(st) + c * BOX, &tmQ, bar_fullq(st), c * 64, row, b);
        const size_t term = static_cast<size_t>(b) * args.Lp + row;
        const uint32_t terms = smem_u32(rowterms(st));
        bulk_load_1d(terms, args.nlse2 + term, 512, bar_fullq(st));
        bulk_load_1d(terms + 512, args.nds + term, 512, bar_fullq(st));
      }
      __syncwarp();
    };
    auto load_do = [&](int blk, int b, int qb) {
      const int st = stage_of(blk);
      do_used |= 1u << st;
      do_par = (do_par & ~(1u << st)) | (use_parity(blk) << st);
      if (elect_one()) {
        mbar_arrive_expect_tx(bar_fulldo(st), C::TILE_BYTES);
        for (int c = 0; c < C::BOXES; ++c)
          tma_load_3d(sdO(st) + c * BOX, &tmdO, bar_fulldo(st), c * 64, qb * 128, b);
      }
      __syncwarp();
#pragma unroll
      for (int t = 0; t < C::STAGES; ++t)
        if (t == st) {
          st_bh[t] = b;
          st_qb[t] = qb;
        }
    };
    // dQ of block blk is staged: add it into the accumulator (one reduce per
    // box, 32 rows x 32 floats each) in two groups, the boxes in the Q
    // buffer first.  Returns once the Q buffer has been read; the caller
    // waits for the rest (bulk_wait_group_read0) before reusing the dO
    // buffer.  The stage's coordinates are those of blk until load_do
    // refills it.
    auto reduce_half = [&](int blk, int half) {
      const int st = stage_of(blk);
      int b = 0, qb = 0;
#pragma unroll
      for (int t = 0; t < C::STAGES; ++t)
        if (t == st) {
          b = st_bh[t];
          qb = st_qb[t];
        }
      if (elect_one()) {
        for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c)
          tma_reduce_add_3d(&tmdQ, dq_box(st, 4 * c), 32 * c, qb * 128, b);
        bulk_commit_group();
      }
      __syncwarp();
    };
    auto reduce_block = [&](int blk) -> bool {
      const int st = stage_of(blk);
      if (!warp_wait(bar_dqst(st), use_parity(blk), SITE_B_DQST)) return false;
      reduce_half(blk, 0);
      if (C::DQ_HALVES && !warp_wait(bar_dqst2(st), use_parity(blk), SITE_B_DQST)) return false;
      reduce_half(blk, 1);
      if (elect_one()) bulk_wait_group_read1();
      __syncwarp();
      return true;
    };
    // Block g reuses the stage of block g - STAGES: Q_g once the first reduce
    // group of that block has been read, dO_g once the second has.  At d = 128 the
    // second group is issued only after the Q_g copy (measured: Q_g arrives
    // sooner and the wait for S_g shrinks; at d = 64 the other order is
    // faster).  The K/V copy of a unit after the first follows the Q and dO
    // copies of its first block, once every MMA of the previous unit (the
    // last readers of K and V) has completed.
    // Blocks modulo BM: the next to load and the next to reduce; pending
    // blocks are loaded and not yet reduced (at most STAGES).
    int gm = 0, rm = 0, pending = 0;
    bool ok = true;
    for (int k = 0;;) {
      for (int i = 0; i < u.n_i && ok; ++i) {
        const int qb = u.q_first + i;
        const bool reuse = pending == C::STAGES;  // the stage holds block rm
        if (reuse) {
          if constexpr (C::DQ_HALVES) {
            // the first half's reduce, then Q into the Q buffer it frees,
            // ahead of the second half's reduce in the copy engine
            ok = warp_wait(bar_dqst(stage_of(rm)), use_parity(rm), SITE_B_DQST);
            if (!ok) break;
            reduce_half(rm, 0);
            if (elect_one()) bulk_wait_group_read0();
            __syncwarp();
          } else {
            ok = reduce_block(rm);
            if (!ok) break;
            rm = (rm + 1) % BM;
            --pending;
          }
        }
        load_q(gm, u.bh, qb);
        if (reuse) {
          if constexpr (C::DQ_HALVES) {
            ok = warp_wait(bar_dqst2(stage_of(rm)), use_parity(rm), SITE_B_DQST);
            if (!ok) break;
            reduce_half(rm, 1);
            rm = (rm + 1) % BM;
            --pending;
          }
          if (elect_one()) bulk_wait_group_read0();
          __syncwarp();
        }
        load_do(gm, u.bh, qb);
        ++pending;
        gm = (gm + 1) % BM;
        if (i == 0 && k > 0) {
          ok = warp_wait(bar_fin, static_cast<uint32_t>(k - 1) & 1u, SITE_B_FIN);
          if (!ok) break;
          load_kv(u);
          kv_par ^= 1u;
        }
      }
      if (!ok) break;
      // Claim the next unit and publish it (or the end, -1) in slot k % 2
      // once every reader has taken the unit that slot held.
      int next = -1;
      if (lane == 0) {
        const long long t = static_cast<long long>(gridDim.x) + atomicAdd(args.sched, 1u);
        next = t < args.n_units ? static_cast<int>(t) : -1;
      }
      next = __shfl_sync(0xffffffffu, next, 0);
      if (next >= 0) {
        u = decode(next);
      }
      ++k;
      if (k >= 2) {
        ok = warp_wait(bar_ufree(k & 1), static_cast<uint32_t>((k >> 1) - 1) & 1u, SITE_B_UNIT);
        if (!ok) break;
      }
      if (lane == 0) {
        unit_slot[2 * (k & 1)] = next;
        unit_slot[2 * (k & 1) + 1] = next >= 0 ? u.n_i : 0;
        mbar_arrive(bar_ufull(k & 1));
      }
      __syncwarp();
      if (next < 0) break;
    }
    for (; ok && pending > 0; --pending, rm = (rm + 1) % BM) ok = reduce_block(rm);
    if (elect_one()) {
      if (!ok) {
        // Let every copy already issued land before the CTA exits.
        if (!args.test_withhold_kv) mbar_wait_drain(bar_kv, kv_par, args.timeout_ns);
        for (int s = 0; s < C::STAGES; ++s) {
          if ((q_used >> s) & 1u) mbar_wait_drain(bar_fullq(s), (q_par >> s) & 1u, args.timeout_ns);
          if ((do_used >> s) & 1u) mbar_wait_drain(bar_fulldo(s), (do_par >> s) & 1u, args.timeout_ns);
        }
      }
      // The reduces must have read the staged dQ before the shared memory
      // goes; their writes complete with the grid, before the dependent
      // conversion pass reads the accumulator.
      bulk_wait_group_read0();
    }
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t ID_S = idesc_bf16_f32_ab(128, 128, false, false);
    constexpr uint32_t ID_DV = idesc_bf16_f32_ab(128, D, false, true);
    constexpr uint32_t ID_DK = idesc_bf16_f32_ab(128, D, false, true);
    constexpr uint32_t ID_DQ = idesc_bf16_f32_ab(128, D, true, true);
    constexpr uint32_t ID_DQH = idesc_bf16_f32_ab(128, 64, true, true);
    // scores-like products: A and B K-major tiles of this CTA, K = d
    auto issue_kmajor = [&](uint32_t dcol, uint32_t a, uint32_t b, uint32_t bar) {
      if (elect_one()) {
        // descriptors built once; a step moves the start-address field by
        // off / 16 (no carry out of the field inside shared memory)
        const uint64_t ad = sdesc_sw128(a, 16, 1024);
        const uint64_t bd = sdesc_sw128(b, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BOX + (kk & 3) * 32;
          mma_ss(tmem + dcol, ad + (off >> 4), bd + (off >> 4), ID_S, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar);
      }
      __syncwarp();
    };
    auto issue_next_s = [&](int blk) -> bool {
      const int st2 = stage_of(blk);
      if (!warp_wait(bar_fullq(st2), use_parity(blk), SITE_B_FULL)) return false;
      tc_fence_after();
      issue_kmajor(C::S_COL, sK, sQ(st2), bar_s);
      return true;
    };
    bool ok = true;
    int g = 0;  // first block of the current unit, modulo BM
    for (int k = 0; ok; ++k) {
      int n_i = 0;
      const int unit = read_unit(k, n_i);
      if (unit < 0) {
        ok = unit == -1;
        break;
      }
      // K_j, V_j of this unit, then S of its first block
      ok = warp_wait(bar_kv, static_cast<uint32_t>(k) & 1u, SITE_B_KV);
      if (ok) ok = issue_next_s(g);
      for (int i = 0; i < n_i && ok; ++i) {
        const int b = (g + i) % BM;
        const int st = stage_of(b);
        if ((k > 0 || i > 0) && !C::SPLIT_DQ) {
          // dP_b goes into the columns dQ_{b-1} occupies until copied out
          ok = warp_wait(bar_dqfree, par(b + 1), SITE_B_DQFREE);
          if (!ok) break;
        }
        ok = warp_wait(bar_fulldo(st), use_parity(b), SITE_B_FULL);
        if (!ok) break;
        tc_fence_after();
        issue_kmajor(C::DP_COL, sV, sdO(st), bar_dp);
        // dV += P^T dO_b once the gradient warps have written P^T (for the
        // first block of a unit this also says that they have read the
        // previous unit's dV and dK out).
        ok = warp_wait(bar_p, par(b), SITE_B_P);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t dod = sdesc_sw128(sdO(st), BOX, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::DV_COL, tmem + C::S_COL + C::p_col(kk), dod + kk * (2048 >> 4), ID_DV,
                   (i > 0 || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
        if (C::EARLY_S && i + 1 < n_i) {
          ok = issue_next_s((b + 1) % BM);  // S_{b+1} behind dV_b, which has read P^T_b
          if (!ok) break;
        }
        // dK += dS^T Q_b and dQ_b = dS K_j once dS^T is in shared memory.
        ok = warp_wait(bar_ds, par(b), SITE_B_DS);
        if (!ok) break;
        if (C::SPLIT_DQ && (k > 0 || i > 0)) {
          // dQ_b goes into the columns of dQ_{b-1}: copied out by now?
          ok = warp_wait(bar_dqfree, par(b + 1), SITE_B_DQFREE);
          if (!ok) break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t dsk = sdesc_sw128(sDS, 16, 1024);     // dS^T, K-major
          const uint64_t dsm = sdesc_sw128(sDS, BOX, 1024);    // the same tile, MN-major
          const uint64_t qmn = sdesc_sw128(sQ(st), BOX, 1024);
          const uint64_t kmn = sdesc_sw128(sK, BOX, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::DK_COL, dsk + (((kk >> 2) * BOX + (kk & 3) * 32) >> 4),
                   qmn + kk * (2048 >> 4), ID_DK, (i > 0 || kk > 0) ? 1u : 0u);
          if constexpr (C::DQ_HALVES) {
            // columns 64h..64h+63 of dQ_b from box h of K (MN-major, N = 64)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint64_t kh = sdesc_sw128(sK + hh * BOX, BOX, 1024);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss(tmem + C::DQ_COL + 64 * hh, dsm + kk * (2048 >> 4), kh + kk * (2048 >> 4),
                       ID_DQH, kk > 0 ? 1u : 0u);
              mma_commit(hh == 0 ? bar_dq : bar_dq2);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::DQ_COL, dsm + kk * (2048 >> 4), kmn + kk * (2048 >> 4), ID_DQ,
                     kk > 0 ? 1u : 0u);
            mma_commit(bar_dq);
          }
        }
        __syncwarp();
        if (!C::EARLY_S && i + 1 < n_i) {
          ok = issue_next_s((b + 1) % BM);
          if (!ok) break;
        }
      }
      if (!ok) break;
      // every MMA of the unit: dV_j and dK_j final, K_j and V_j free
      if (elect_one()) mma_commit(bar_fin);
      __syncwarp();
      g = (g + n_i) % BM;
    }
    if (!ok) {
      // Every MMA already issued must finish before the tensor memory is freed.
      if (elect_one()) {
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0, args.timeout_ns);
      }
      __syncwarp();
    }
  } else if (C::DQ_WARPS > 0 && warp >= C::FIRST_DQ_WARP) {
    // ------------------------------------------------------------ dQ warps
    // Warp q (TMEM lanes 32q..32q+31 = query rows of dQ_b): per block, dQ_b
    // out of tensor memory, 32 columns at a time, then into the staging
    // pieces of the block's Q/dO buffers (every MMA that read Q_b and dO_b is
    // complete: the dq_full arrival follows them).
    const int quarter = warp & 3;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true;
    int b = 0;  // modulo BM
    for (int k = 0; ok; ++k) {
      int n_i = 0;
      const int unit = read_unit(k, n_i);
      if (unit < 0) {
        ok = unit == -1;
        break;
      }
      for (int i = 0; i < n_i && ok; ++i, b = (b + 1) % BM) {
        const int st = stage_of(b);
        ok = __all_sync(0xffffffffu, mbar_wait(bar_dq, par(b), ctl, SITE_B_DQ));
        if (!ok) break;
        tc_fence_after();
        uint32_t qv[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(lane_base + C::DQ_COL + 32 * c, qv[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) reg_fence32(qv[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dqfree);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint8_t* const row_ptr = base_ptr + (dq_box(st, c * 4 + quarter) - base) + lane * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(row_ptr + ((u ^ (lane & 7)) * 16)) =
                make_uint4(qv[c][4 * u], qv[c][4 * u + 1], qv[c][4 * u + 2], qv[c][4 * u + 3]);
        }
        fence_proxy_async_smem();  // the producer's reduce reads the stage via the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dqst(st));
      }
    }
  } else {
    // ------------------------------------------------------------ gradient warps
    // Warp (quarter, h): TMEM lanes 32*quarter..+31 (its keys, or its queries
    // for dQ), query columns CQ*h..CQ*h+CQ-1 of S^T and dP^T, and columns
    // CW*h..CW*h+CW-1 of dQ_i, dK and dV.
    constexpr int CQ = 128 / BWD_GRAD_GROUPS;
    constexpr int CW = D / BWD_GRAD_GROUPS;
    const int h = (warp - BWD_FIRST_GRAD_WARP) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // the current unit
    Unit w{};
    int g0 = 0;  // its first block, modulo BM
    // this lane's key is w.jblk * 128 + r; the unit's block has keys past L
    // only if it is the last one of a ragged L
    auto key_ok = [&] { return w.jblk * 128 + r < L; };
    auto tail_blk = [&] { return (w.jblk + 1) * 128 > L; };
    const uint64_t sl2x2 = f2_pack(args.scale_log2, args.scale_log2);
    const uint64_t scale2 = f2_pack(args.scale, args.scale);
    auto terms_of = [&](int b) {
      return reinterpret_cast<const float*>(rowterms(stage_of(b))) + CQ * h;
    };
    float p[CQ];  // P^T of this warp's queries, block of the last phase A

    // Phase A of block i: P^T = exp2(S^T * scale*log2e - lse*log2e), kept in
    // fp32 for dS and written to TMEM as bf16 (the A operand of
    // dV += P^T dO) over the first CQ/2 of the warp's own S^T columns.  The
    // masks apply only on the causal diagonal block and in the last key
    // block of a ragged L (both uniform across the CTA); elsewhere the
    // per-element selects are compiled out.
    // b: the block modulo BM; i: its index in the unit
    auto phase_a = [&](int b, int i) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(bar_s, par(b), ctl, SITE_B_S))) return false;
      tc_fence_after();
      const int qb = w.q_first + i;
      const bool diag = CAUSAL && qb == w.jblk;
      const float* const terms = terms_of(b);
      uint32_t sr[CQ];
      bwd_tmem_ld<CQ>(lane_base + C::S_COL + CQ * h, sr);
      tmem_wait_ld();
      reg_fence_n(sr);
      auto compute = [&](auto mask_tag) {
        constexpr bool MASK = decltype(mask_tag)::value;
        uint32_t pk[CQ / 2];
        const float4* nl = reinterpret_cast<const float4*>(terms);
#pragma unroll
        for (int e = 0; e < CQ; e += 4) {
          const float4 a = nl[e >> 2];
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2x2,
                           f2_pack(a.x, a.y)),
                    x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), sl2x2,
                           f2_pack(a.z, a.w)),
                    x2, x3);
          float pe[4] = {ex2_approx(x0), ex2_approx(x1), ex2_approx(x2), ex2_approx(x3)};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            // causal: key r > query (CQ*h + e + u) of the same block;
            // keys past L (zero rows of K) never contribute.
            if constexpr (MASK)
              if ((diag && r > CQ * h + e + u) || !key_ok()) pe[u] = 0.f;
            p[e + u] = pe[u];
          }
          pk[e >> 1] = pack_bf16x2(pe[0], pe[1]);
          pk[(e >> 1) + 1] = pack_bf16x2(pe[2], pe[3]);
        }
        bwd_tmem_st<CQ / 2>(lane_base + C::S_COL + CQ * h, pk);
      };
      if (diag || tail_blk())
        compute(std::true_type{});
      else
        compute(std::false_type{});
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);
      return true;
    };

    // Phase B of block i: dS^T = P^T (.) (scale * dP^T - scale * D), bf16
    // into the 128B-swizzled dS tile: row = key, box b holds queries
    // 64b..64b+63, 16-byte unit u of row r at unit u ^ (r % 8).
    auto phase_b = [&](int b) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(bar_dp, par(b), ctl, SITE_B_DP))) return false;
      tc_fence_after();
      const float* const terms = terms_of(b);
      uint32_t dr[CQ];
      bwd_tmem_ld<CQ>(lane_base + C::DP_COL + CQ * h, dr);
      tmem_wait_ld();
      reg_fence_n(dr);
      const float4* nd = reinterpret_cast<const float4*>(terms + 128);
      uint8_t* const row_ptr = ds_ptr + ((CQ * h) >> 6) * BOX + r * 128;
      const int unit0 = ((CQ * h) & 63) >> 3;
#pragma unroll
      for (int e = 0; e < CQ; e += 8) {
        uint32_t pk[4];
#pragma unroll
        for (int g = 0; g < 8; g += 4) {
          const float4 b = nd[(e + g) >> 2];
          float d0, d1, d2, d3;
          f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(dr[e + g]), __uint_as_float(dr[e + g + 1])),
                                  scale2, f2_pack(b.x, b.y)),
                           f2_pack(p[e + g], p[e + g + 1])),
                    d0, d1);
          f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(dr[e + g + 2]),
                                          __uint_as_float(dr[e + g + 3])),
                                  scale2, f2_pack(b.z, b.w)),
                           f2_pack(p[e + g + 2], p[e + g + 3])),
                    d2, d3);
          pk[g >> 1] = pack_bf16x2(d0, d1);
          pk[(g >> 1) + 1] = pack_bf16x2(d2, d3);
        }
        const int unit = (unit0 + (e >> 3)) ^ (r & 7);
        *reinterpret_cast<uint4*>(row_ptr + unit * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
      return true;
    };

    // Phase C of block i: copy this warp's columns of dQ_i out of TMEM and
    // release them, then stage them in block i's Q/dO buffers (every MMA
    // that read Q_i and dO_i is complete: the dq_full arrival follows them)
    // for the producer's reduce into the fp32 accumulator.  Pieces are 32
    // rows x 32 floats, 128-byte swizzled (16-byte unit u of row r at unit
    // u ^ (r % 8)); rows past L are skipped by the reduce.  With DQ_HALVES
    // the two column halves are copied and staged one after the other, each
    // as soon as its product has completed (half 0 lands in the Q buffer).
    auto stage_dq = [&](int st, const uint32_t* qv, int col0, int ncols) {
#pragma unroll 4
      for (int u = 0; u < ncols / 4; ++u) {
        const int col = col0 + 4 * u;
        uint8_t* const row_ptr =
            base_ptr + (dq_box(st, (col >> 5) * 4 + quarter) - base) + lane * 128;
        *reinterpret_cast<uint4*>(row_ptr + ((((col & 31) >> 2) ^ (lane & 7)) * 16)) =
            make_uint4(qv[4 * u], qv[4 * u + 1], qv[4 * u + 2], qv[4 * u + 3]);
      }
      fence_proxy_async_smem();  // the producer's reduce reads the stage via the async proxy
      __syncwarp();
    };
    auto phase_c = [&](int b) -> bool {
      const int st = stage_of(b);
      if constexpr (C::DQ_HALVES) {
        constexpr int HW = 64 / BWD_GRAD_GROUPS;  // columns per warp and half
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (!__all_sync(0xffffffffu, mbar_wait(hh == 0 ? bar_dq : bar_dq2, par(b), ctl, SITE_B_DQ)))
            return false;
          tc_fence_after();
          uint32_t qv[HW];
          bwd_tmem_ld<HW>(lane_base + C::DQ_COL + 64 * hh + HW * h, qv);
          tmem_wait_ld();
          reg_fence_n(qv);
          if (hh == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_dqfree);
          }
          stage_dq(st, qv, 64 * hh + HW * h, HW);
          if (lane == 0) mbar_arrive(hh == 0 ? bar_dqst(st) : bar_dqst2(st));
        }
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(bar_dq, par(b), ctl, SITE_B_DQ))) return false;
        tc_fence_after();
        uint32_t qv[CW];
        bwd_tmem_ld<CW>(lane_base + C::DQ_COL + CW * h, qv);
        tmem_wait_ld();
        reg_fence_n(qv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dqfree);
        stage_dq(st, qv, CW * h, CW);
        if (lane == 0) mbar_arrive(bar_dqst(st));
      }
      return true;
    };

    bool ok = true;
    for (int k = 0; ok; ++k) {
      int n_i = 0;
      const int unit = read_unit(k, n_i);
      if (unit < 0) {
        ok = unit == -1;
        break;
      }
      w = decode(unit);
      if constexpr (C::EARLY_S) {
        // A(0); then per block B(i), A(i+1), C(i): P of the next block is
        // computed while dK_i and dQ_i run on the tensor core.
        ok = phase_a(g0, 0);
        for (int i = 0; i < w.n_i && ok; ++i) {
          const int b = (g0 + i) % BM;
          ok = phase_b(b);
          if (ok && i + 1 < w.n_i) ok = phase_a((b + 1) % BM, i + 1);
          if (C::DQ_WARPS == 0 && ok) ok = phase_c(b);
        }
      } else {
        for (int i = 0; i < w.n_i && ok; ++i) {
          const int b = (g0 + i) % BM;
          ok = phase_a(b, i);
          if (ok) ok = phase_b(b);
          if (ok) ok = phase_c(b);
        }
      }

      // Epilogue: dV_j and dK_j are final once every MMA of the unit has
      // completed.  With phase C on these warps the unit's last dq_full
      // arrival says so; when the dQ warps copy dQ out, these warps wait
      // for the MMA warp's commit after the unit (fin: one phase per unit;
      // they observe none of dq_full's, and a parity wait on a barrier
      // several phases behind would alias).  bf16 (round to nearest even),
      // rows < L.  The next unit's dV and dK products start only after
      // these warps' next P-ready arrival, which follows these loads.
      if (C::DQ_WARPS > 0 && ok) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar_fin, static_cast<uint32_t>(k) & 1u, ctl, SITE_B_DQ));
        if (ok) tc_fence_after();
      }
      if (!ok) break;
      if constexpr (D == 128) {
        // The stores are made row-contiguous through the warp's own bytes of
        // the dS tile (the bytes it writes in phase B: rows 32*quarter..+31,
        // 64 bytes each, 128-byte swizzled).  No other warp touches them, no
        // product reads the tile before the next unit's dS-ready arrivals,
        // and every product that read it has completed.  Each lane writes its
        // own row's 64 bytes of dV (then dK); read back, four neighbouring
        // lanes hold one row's, so a store instruction covers 8 rows in
        // 64-byte pieces instead of 32 rows in 16-byte pieces (measured: the
        // 16-byte stores of 16 warps held the epilogue for about 8,000
        // cycles and delayed the next unit's first product).
        uint8_t* const mine = ds_ptr + ((CQ * h) >> 6) * BOX + quarter * 32 * 128;
        const int pu0 = ((CQ * h) & 63) >> 3;  // the warp's first unit in a row
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {  // dV, then dK
          uint32_t v[CW];
          bwd_tmem_ld<CW>(lane_base + (which == 0 ? C::DV_COL : C::DK_COL) + CW * h, v);
          tmem_wait_ld();
          reg_fence_n(v);
#pragma unroll
          for (int u = 0; u < CW / 8; ++u)
            *reinterpret_cast<uint4*>(mine + lane * 128 + (((pu0 + u) ^ (lane & 7)) * 16)) =
                make_uint4(pack_bf16x2(__uint_as_float(v[8 * u]), __uint_as_float(v[8 * u + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7])));
          __syncwarp();
          uint16_t* const out = which == 0 ? args.dv : args.dk;
          const int q = lane & 3;  // unit within the row
#pragma unroll 1
          for (int s = 0; s < 4; ++s) {
            const int rr = s * 8 + (lane >> 2);  // row within the warp's 32
            const uint4 val = *reinterpret_cast<const uint4*>(
                mine + rr * 128 + (((pu0 + q) ^ (rr & 7)) * 16));
            const int key = w.jblk * 128 + quarter * 32 + rr;
            if (key < L)
              *reinterpret_cast<uint4*>(out + (static_cast<size_t>(w.bh) * L + key) * D + CW * h +
                                        q * 8) = val;
          }
          __syncwarp();
        }
      } else {
        // d = 64: each lane stores its own row's 32 bytes (measured: the
        // route through the dS tile gained nothing here)
        const size_t row = static_cast<size_t>(w.bh) * L + w.jblk * 128 + r;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t col0 = (which == 0 ? C::DV_COL : C::DK_COL) + CW * h;
          uint16_t* const out = which == 0 ? args.dv : args.dk;
          uint32_t v[CW];
          bwd_tmem_ld<CW>(lane_base + col0, v);
          tmem_wait_ld();
          reg_fence_n(v);
          if (key_ok()) {
            uint4* dst = reinterpret_cast<uint4*>(out + row * D + CW * h);
#pragma unroll
            for (int u = 0; u < CW / 8; ++u)
              dst[u] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * u]), __uint_as_float(v[8 * u + 1])),
                                  pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3])),
                                  pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5])),
                                  pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7])));
          }
        }
      }
      g0 = (g0 + w.n_i) % BM;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
