// Exact attention forward for sm_103a: TMA + tcgen05 + TMEM, online softmax.
//
// One CTA owns one tile of BLOCK_M = 128 query rows of one (batch, head) and
// walks the K/V blocks of BLOCK_N = 128 keys in order, as in the
// FlashAttention-2 forward ("04 Transformers, Attention, and FlashAttention",
// Algorithm 1: Q split into row blocks, the K/V loop inside, running max m,
// running sum l and unnormalised O on chip, O / l and m + log l at the end).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: loads Q once, then streams K_j and V_j tiles
//               through a ring of shared-memory slots (full/empty mbarriers).
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into a TMEM buffer
//               (two buffers, so S_{j+1} is computed while the softmax works
//               on S_j), then O += P_j V_j with P_j read from TMEM.  The
//               whole warp allocates and frees the tensor memory.
//   warps 2..5  softmax: thread r owns query row r (TMEM lane r).  Per block
//               it reads its 128 scores, applies the masks, updates the
//               running max, writes P = exp2(scale*log2e*S - m) as bf16 over
//               the scores it came from, and rescales O (and l) by
//               exp2(m_old - m_new) whenever the running max grew; a warp
//               skips the O pass when no row in it saw a larger max (the
//               correction is then exactly 1).  At the end it writes O / l
//               (bf16) and the log-sum-exp (fp32).
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128)    S buffer 0 (P_j packed bf16 in its first 64 columns)
//   [128,256)  S buffer 1
//   [256,256+D) O accumulator
//
// Shared memory (1024-byte aligned): NSLOT ring slots of one 128 x D tile
// each, then the Q tile, then the mbarriers.  A tile is stored as D/64
// boxes of 128 rows x 64 columns with the 128-byte swizzle, the layout the
// tensor map writes and the MMA descriptors read.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int BLOCK_M = 128;
constexpr int BLOCK_N = 128;
constexpr int NUM_THREADS = 192;
// Rescale threshold (log2 units).  Zero keeps the exact running max of the
// recurrence, so the largest P~ of a row is exp2(0) = 1, exact in bf16.  A
// positive threshold (keeping a stale max while it is within TAU) saves
// rescale passes but rounds the dominant weight of peaked rows to bf16,
// which costs up to 2^-9 relative on O.
constexpr float RESCALE_TAU = 0.0f;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;        // buffer b at S_COL + 128 * b
constexpr uint32_t O_COL = 256;
constexpr int BOX_BYTES = 128 * 64 * 2;  // one 128-row x 64-column bf16 box

// Wait sites (bit index in the device status word).
enum : uint32_t {
  SITE_Q = 1,
  SITE_EMPTY = 2,
  SITE_FULL = 3,
  SITE_S = 4,
  SITE_P = 5,
  SITE_O = 6,
  SITE_DRAIN = 7,
};

template <int D>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dimension must be 64 or 128");
  static constexpr int BOXES = D / 64;
  static constexpr int TILE_BYTES = BLOCK_N * D * 2;
  static constexpr int NSLOT = (D == 64) ? 8 : 5;
  static constexpr int Q_OFF = NSLOT * TILE_BYTES;
  static constexpr int BAR_OFF = Q_OFF + TILE_BYTES;
  // q_full, full[NSLOT], empty[NSLOT], s_full[2], p_full[2], o_ready, drain
  static constexpr int NBAR = 1 + 2 * NSLOT + 2 + 2 + 1 + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct FwdArgs {
  uint16_t* o;        // bf16 [BH, L, D]
  float* lse;         // fp32 [BH, L]
  int L;
  int n_qtiles;       // ceil(L / BLOCK_M)
  float scale_log2;   // scale * log2(e)
  unsigned int* status;
  unsigned long long timeout_ns;
};

// Wait that ignores the CTA abort flag (used while draining after an abort).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity,
                                                unsigned long long timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);

  const uint32_t ring = base;
  const uint32_t sQ = base + C::Q_OFF;
  const uint32_t bars = base + C::BAR_OFF;
  const uint32_t bar_q = bars;
  auto bar_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bars + 8u * (1 + C::NSLOT + s); };
  auto bar_s = [&](int b) { return bars + 8u * (1 + 2 * C::NSLOT + b); };
  auto bar_p = [&](int b) { return bars + 8u * (3 + 2 * C::NSLOT + b); };
  const uint32_t bar_o = bars + 8u * (5 + 2 * C::NSLOT);
  const uint32_t bar_drain = bars + 8u * (6 + 2 * C::NSLOT);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int L = args.L;
  const int n_qt = args.n_qtiles;

  // Tile order: head-major, so the CTAs resident at one time share the K/V
  // of a few heads in L2.  Causal: heaviest (last) query tile of a head first.
  const int bh = static_cast<int>(blockIdx.x) / n_qt;
  const int qt_raw = static_cast<int>(blockIdx.x) % n_qt;
  const int qt = CAUSAL ? (n_qt - 1 - qt_raw) : qt_raw;
  const int n_kv_all = (L + BLOCK_N - 1) / BLOCK_N;
  // Causal: blocks wholly above the diagonal (first key > last query) skipped.
  const int n_kv = CAUSAL ? min(n_kv_all, (qt * BLOCK_M + BLOCK_M - 1) / BLOCK_N + 1) : n_kv_all;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s(b), 1);
      mbar_init(bar_p(b), 4 * 32);
    }
    mbar_init(bar_o, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, args.status, args.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, C::TILE_BYTES);
      for (int c = 0; c < C::BOXES; ++c)
        tma_load_3d(sQ + c * BOX_BYTES, &tmQ, bar_q, c * 64, qt * BLOCK_M, bh);
      int cnt = 0;
      bool ok = true;
      auto load = [&](const CUtensorMap* map, int j) -> bool {
        const int s = cnt % C::NSLOT;
        const uint32_t use = static_cast<uint32_t>(cnt / C::NSLOT);
        if (!mbar_wait(bar_empty(s), (use & 1u) ^ 1u, ctl, SITE_EMPTY)) return false;
        mbar_arrive_expect_tx(bar_full(s), C::TILE_BYTES);
        const uint32_t dst = ring + s * C::TILE_BYTES;
        for (int c = 0; c < C::BOXES; ++c)
          tma_load_3d(dst + c * BOX_BYTES, map, bar_full(s), c * 64, j * BLOCK_N, bh);
        ++cnt;
        return true;
      };
      // Same order the MMA warp consumes: K_0, K_1, V_0, K_2, V_1, ..., V_last.
      for (int j = 0; j < n_kv && ok; ++j) {
        ok = load(&tmK, j);
        if (ok && j > 0) ok = load(&tmV, j - 1);
      }
      if (ok) ok = load(&tmV, n_kv - 1);
      if (!ok) {
        // Let every copy already issued land before the CTA exits.
        mbar_wait_drain(bar_q, 0, args.timeout_ns);
        for (int s = 0; s < C::NSLOT; ++s) {
          const int issued = cnt > s ? (cnt - 1 - s) / C::NSLOT + 1 : 0;
          if (issued > 0) mbar_wait_drain(bar_full(s), (issued - 1) & 1, args.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(BLOCK_M, BLOCK_N, false);
      constexpr uint32_t IDESC_O = idesc_bf16_f32(BLOCK_M, D, true);
      int cnt = 0;
      bool ok = mbar_wait(bar_q, 0, ctl, SITE_Q);
      tc_fence_after();
      auto take = [&](uint32_t& addr, int& s) -> bool {
        s = cnt % C::NSLOT;
        const uint32_t use = static_cast<uint32_t>(cnt / C::NSLOT);
        if (!mbar_wait(bar_full(s), use & 1u, ctl, SITE_FULL)) return false;
        tc_fence_after();
        addr = ring + s * C::TILE_BYTES;
        ++cnt;
        return true;
      };
      auto issue_s = [&](int j) -> bool {
        uint32_t kaddr;
        int s;
        if (!take(kaddr, s)) return false;
        const uint32_t d_tmem = tmem + S_COL + 128u * (j & 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
          mma_ss(d_tmem, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kaddr + off, 16, 1024),
                 IDESC_S, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_empty(s));
        mma_commit(bar_s(j & 1));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait(bar_p(j & 1), (j >> 1) & 1, ctl, SITE_P)) return false;
        tc_fence_after();
        uint32_t vaddr;
        int s;
        if (!take(vaddr, s)) return false;
        const uint32_t p_tmem = tmem + S_COL + 128u * (j & 1);
#pragma unroll
        for (int kk = 0; kk < BLOCK_N / 16; ++kk) {
          mma_ts(tmem + O_COL, p_tmem + kk * 8, sdesc_sw128(vaddr + kk * 2048, BOX_BYTES, 1024),
                 IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_empty(s));
        mma_commit(bar_o);
        return true;
      };
      for (int j = 0; j < n_kv && ok; ++j) {
        ok = issue_s(j);
        if (ok && j > 0) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(n_kv - 1);
      if (!ok) {
        // Every MMA already issued must finish before the tensor memory is freed.
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0, args.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int q_row = qt * BLOCK_M + row;
    const float sl2 = args.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    float m = -INFINITY;  // running max of scale*log2e*s (or the stale reference)
    float l = 0.f;        // running sum of P~ in that reference
    bool ok = true;

    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      const bool w = mbar_wait(bar_s(b), (j >> 1) & 1, ctl, SITE_S);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + S_COL + 128u * b + 32u * c, sr[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(sr[c]);

      // Masks: keys past the end of the sequence; causal keys after the query.
      const int k0 = j * BLOCK_N;
      const bool need_mask = (k0 + BLOCK_N > L) || (CAUSAL && k0 + BLOCK_N - 1 > qt * BLOCK_M);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int key = k0 + c * 32 + e;
            const bool masked = key >= L || (CAUSAL && key > q_row);
            if (masked) sr[c][e] = __float_as_uint(-INFINITY);
          }
      }

      // Row max in scaled log2 units.
      float mx[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mx[t] = -INFINITY;
      if (pos_scale) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(sr[c][e]));
      } else {
        // scale <= 0: work on x = scale*log2e*s directly (masked stays -inf).
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float s = __uint_as_float(sr[c][e]);
            const float x = (s == -INFINITY) ? -INFINITY : s * sl2;
            sr[c][e] = __float_as_uint(x);
            mx[e & 7] = fmaxf(mx[e & 7], x);
          }
      }
      float blk = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                        fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      if (pos_scale) blk *= sl2;
      const float m_new = fmaxf(m, blk);

      float corr = 1.f;
      bool rescale = false;
      if (j == 0) {
        m = m_new;
      } else if (m_new - m > RESCALE_TAU) {
        corr = ex2_approx(m - m_new);
        m = m_new;
        rescale = true;
      }
      // P~ = exp2(x - m); x = s*sl2 (fused) or the precomputed x.
      const float mul = pos_scale ? sl2 : 1.f;
      const float neg_m = -m;
      float sum[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) sum[t] = 0.f;
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c][e]), mul, neg_m));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c][e + 1]), mul, neg_m));
          sum[e & 7] += p0;
          sum[(e + 1) & 7] += p1;
          const int col = c * 32 + e;  // key within the block
          pk[col >> 6][(col & 63) >> 1] = pack_bf16x2(p0, p1);
        }
      tmem_st32(lane_base + S_COL + 128u * b, pk[0]);
      tmem_st32(lane_base + S_COL + 128u * b + 32u, pk[1]);
      const float rowsum =
          ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
      l = (j == 0) ? rowsum : fmaf(corr, l, rowsum);

      if (__any_sync(0xffffffffu, rescale)) {
        // O holds P_0..P_{j-1} contributions once PV_{j-1} (the j-th commit) is done.
        const bool wo = mbar_wait(bar_o, (j - 1) & 1, ctl, SITE_O);
        if (!__all_sync(0xffffffffu, wo)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_base + O_COL + 32u * c, ov);
          tmem_wait_ld();
          reg_fence32(ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr);
          tmem_st32(lane_base + O_COL + 32u * c, ov);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p(b));
    }

    if (ok) {
      // Epilogue: wait for the last PV (commit number n_kv), then O / l and LSE.
      const bool w = mbar_wait(bar_o, (n_kv - 1) & 1, ctl, SITE_O);
      if (__all_sync(0xffffffffu, w)) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const bool store = q_row < L;
        const size_t row_off = (static_cast<size_t>(bh) * L + q_row) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_base + O_COL + 32u * c, ov);
          tmem_wait_ld();
          reg_fence32(ov);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l,
                                __uint_as_float(ov[2 * e + 1]) * inv_l);
          if (store) {
            uint4* dst = reinterpret_cast<uint4*>(args.o + row_off + c * 32);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              dst[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
          }
        }
        if (store)
          args.lse[static_cast<size_t>(bh) * L + q_row] = (m + log2f(l)) * 0.69314718055994531f;
      }
    }
    tmem_wait_st();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace fa
