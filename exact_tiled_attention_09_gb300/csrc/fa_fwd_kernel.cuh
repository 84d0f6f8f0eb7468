// Exact attention forward for sm_103a: TMA + tcgen05 + TMEM, online softmax.
//
// Work unit: one CTA owns 2 x 128 query rows (two Q tiles) of one
// (batch, head) and walks the K/V blocks of 128 keys in order, as in the
// FlashAttention-2 forward ("04 Transformers, Attention, and FlashAttention",
// Algorithm 1: Q split into row blocks, the K/V loop inside, running max m,
// running sum l and unnormalised O kept on chip, O / l and m + log l written
// at the end).  Two Q tiles per CTA let the tensor core work on one tile
// while the softmax of the other runs (the overlap of matmul and softmax that
// "FlashAttention 深度解析", third part, section 2.2 describes for Hopper,
// re-targeted here to tcgen05 and tensor memory).
//
// Warp roles (320 threads; 352 at d = 64):
//   warp 0      MMA issuer and owner of the tensor memory: all 32 lanes run
//               the loop and poll the barriers, one elected lane issues
//               (d = 64: the products of Q tile 0 only)
//   warp 1      TMA producer (same scheme): loads Q0 and Q1 once, then K_j
//               and V_j tiles into a ring of shared-memory slots (full/empty
//               mbarriers)
//   warps 2..5  softmax of Q tile 0 (row r = TMEM lane r; warp w may only
//               touch lanes 32*(w%4) .. 32*(w%4)+31, so the four warps of a
//               group cover quarters 2, 3, 0, 1)
//   warps 6..9  softmax of Q tile 1
//   warp 10     d = 64 only: MMA issuer of Q tile 1
//
// d = 128, MMA order per K/V block j (each S_t buffer holds P_t after the
// softmax, so S_t of block j+1 is issued only after O_t += P_t V_j):
//   PV0_j, S0_{j+1}, PV1_j, S1_{j+1}
// The tensor core therefore computes PV1_j and S1_{j+1} while softmax 0
// works on S0_{j+1}, and the other way round.  Because tcgen05 operations of
// one thread complete in issue order, the arrival that publishes S_t of
// block j+1 also proves O_t += P_t V_j finished, so the softmax may rescale
// O_t right away.
//
// d = 64 differs: P_t has tensor-memory columns of its own, so S_t of block
// j+1 is issued as soon as the softmax has read S_t of block j (s_free), and
// each tile has its own MMA warp, so neither tile's products wait behind the
// other's barriers.  The softmax computes block j's exponentials in
// registers, then waits for O_t += P_t V_{j-1} (o_done, committed after
// every PV at d = 64) before writing P_t and rescaling O_t; the tile runs
// from block to block without waiting for the tensor core.  Both MMA warps
// release every ring slot (empty barriers count 2).
//
// Softmax per block (per row): scores s -> mask -> m_new = max(m, rowmax)
// (in units of scale*log2(e)) -> P~ = exp2(s*scale*log2e - m_new) written as
// bf16 over the first 64 columns of its S buffer (d = 64: into P_t's own
// columns) -> l = c*l + rowsum(P~) and
// O *= c with c = exp2(m - m_new) whenever the max grew (a warp skips the O
// pass when no row of it changed: c is then exactly 1).
//
// Tensor memory (512 columns x 128 lanes of 32 bits):
//   [0,128) S0/P0   [128,256) S1/P1   [256,256+D) O0   [256+D,256+2D) O1
//   d = 64: P0 at [384,448) and P1 at [448,512) instead (bf16, two per column)
//
// Shared memory (1024-byte aligned): NSLOT ring slots, then Q0 and Q1, then
// the mbarriers.  Every tile is stored as D/64 boxes of 128 rows x 64 columns
// with the 128-byte swizzle, the layout the tensor map writes and the MMA
// descriptors read.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int BLOCK_M = 128;          // rows per Q tile (one TMEM lane each)
constexpr int BLOCK_N = 128;          // keys per K/V block
constexpr int TILES_PER_CTA = 2;
constexpr int ROWS_PER_CTA = BLOCK_M * TILES_PER_CTA;
constexpr int MMA_WARP = 0;
constexpr int PRODUCER_WARP = 1;
constexpr int FIRST_SOFTMAX_WARP = 2;
constexpr uint32_t TMEM_COLS = 512;
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

template <int D, bool FP8 = false>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dimension must be 64 or 128");
  static constexpr int BOXES = D / 64;
  static constexpr int TILE_BYTES = BLOCK_N * D * 2;  // a bf16 tile (V; Q, K unless FP8)
  static constexpr int NSLOT = (D == 64) ? 8 : 4;
  // Q and K tiles: bf16 as D/64 boxes of 64 columns, or with FP8 one box of
  // 128 rows x D bytes (E4M3 codes; 128-byte swizzle at D = 128, 64-byte at
  // D = 64).
  static constexpr int QK_BOXES = FP8 ? 1 : BOXES;
  static constexpr int QK_BOX_BYTES = FP8 ? BLOCK_N * D : BOX_BYTES;
  static constexpr int QK_BOX_COLS = FP8 ? D : 64;
  static constexpr int QK_TILE_BYTES = FP8 ? BLOCK_N * D : TILE_BYTES;
  // d = 64: P_t gets tensor-memory columns of its own, S_t is free as soon
  // as the softmax has read it, and each Q tile has its own MMA warp.
  static constexpr bool SPLIT_P = (D == 64);
  static constexpr int WARPS_PER_TILE = 4;  // softmax warps: one per TMEM lane quarter
  static constexpr int SOFTMAX_WARPS = TILES_PER_CTA * WARPS_PER_TILE;
  static constexpr int MMA_WARP_T1 = FIRST_SOFTMAX_WARP + SOFTMAX_WARPS;  // d = 64 only
  static constexpr int THREADS = 32 * (FIRST_SOFTMAX_WARP + SOFTMAX_WARPS + (SPLIT_P ? 1 : 0));
  static constexpr int Q_OFF = NSLOT * TILE_BYTES;
  static constexpr int BAR_OFF = Q_OFF + TILES_PER_CTA * QK_TILE_BYTES;
  // q_full, full[NSLOT], empty[NSLOT], s_full[2], p_full[2], o_done[2],
  // drain[2] (one per MMA warp), s_free[2]
  static constexpr int NBAR = 1 + 2 * NSLOT + 2 + 2 + 2 + 2 + 2;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  __host__ __device__ static constexpr uint32_t S_COL(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t O_COL(int t) {
    return 256u + static_cast<uint32_t>(D) * t;
  }
  __host__ __device__ static constexpr uint32_t P_COL(int t) {
    return SPLIT_P ? 384u + 64u * t : S_COL(t);
  }
  static_assert(!SPLIT_P || 384 + 2 * 64 <= 512, "tensor memory budget");
};

struct FwdArgs {
  uint16_t* o;        // bf16 [BH, L, D]
  float* lse;         // fp32 [BH, L]
  // Split-KV only: K/V blocks per split, and the per-split results
  // (normalised over the split's keys) the merge kernel combines.
  int blocks_per_split;
  float* o_part;      // fp32 [n_splits, BH, L, D]
  float* lse_part;    // fp32 [n_splits, BH, L]
  int L;
  int n_ctiles;       // ceil(L / ROWS_PER_CTA)
  int bh;             // B * H
  int group_heads;    // heads per scheduling group (see the CTA order)
  float scale_log2;   // scale * log2(e)
  // FP8 only: fp32 scales of the 128-row blocks of Q and K, [BH, n_blocks]
  const float* q_scale;
  const float* k_scale;
  int n_blocks;       // ceil(L / 128)
  unsigned int* status;
  unsigned long long timeout_ns;
  int test_withhold_q;  // test hook: skip the Q copy so the first MMA wait runs out
};

// N chunks of 32 consecutive tensor-memory columns moved with one wide
// instruction (measured: one x128 load of a score row instead of four x32
// loads lifts the d = 64 forward by 4%).
template <int N>
__device__ __forceinline__ void tmem_ld_chunks(uint32_t taddr, uint32_t (&r)[N][32]) {
  using W = uint32_t[N * 32];
  if constexpr (N == 4)
    tmem_ld128(taddr, reinterpret_cast<W&>(r));
  else if constexpr (N == 2)
    tmem_ld64(taddr, reinterpret_cast<W&>(r));
  else
    tmem_ld32(taddr, r[0]);
}
template <int N>
__device__ __forceinline__ void tmem_st_chunks(uint32_t taddr, uint32_t (&r)[N][32]) {
  using W = uint32_t[N * 32];
  if constexpr (N == 4)
    tmem_st128(taddr, reinterpret_cast<W&>(r));
  else if constexpr (N == 2)
    tmem_st64(taddr, reinterpret_cast<W&>(r));
  else
    tmem_st32(taddr, r[0]);
}
// N chunks of 16 columns (packed bf16 P of 32 keys each).
template <int N>
__device__ __forceinline__ void tmem_st_pchunks(uint32_t taddr, uint32_t (&r)[N][16]) {
  using W = uint32_t[N * 16];
  if constexpr (N == 4)
    tmem_st64(taddr, reinterpret_cast<W&>(r));
  else if constexpr (N == 2)
    tmem_st32(taddr, reinterpret_cast<W&>(r));
  else
    tmem_st16(taddr, r[0]);
}

// Number of K/V blocks Q tile t of this CTA needs (0 if the tile lies wholly
// past the end of the sequence).  Causal: blocks whose first key exceeds the
// tile's last query are skipped.
template <bool CAUSAL>
__device__ __forceinline__ int blocks_for_tile(int row0, int L) {
  if (row0 >= L) return 0;
  const int all = (L + BLOCK_N - 1) / BLOCK_N;
  return CAUSAL ? min(all, (row0 + BLOCK_M - 1) / BLOCK_N + 1) : all;
}

// SPLIT: the CTA covers only K/V blocks [split * blocks_per_split,
// (split + 1) * blocks_per_split) of its rows and writes fp32 partial results
// (Flash-Decoding's per-chunk pass, "04 Transformers, Attention, and
// FlashAttention", Flash-Decoding); the merge kernel finishes them.
//
// FP8: Q and K are E4M3 codes with one fp32 scale per 128-row block ("FlashAttention
// 深度解析", third part, section 2.3: Q_FP8 = Quantize(Q_block / s_q), S =
// Q_FP8 K_FP8^T * s_q * s_k); S comes from a kind::f8f6f4 MMA, and s_q * s_k
// joins the softmax multiplier of each block.  P and V stay bf16.
template <int D, bool CAUSAL, bool SPLIT, bool FP8 = false>
__global__ void __launch_bounds__(FwdCfg<D, FP8>::THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using C = FwdCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);

  const uint32_t ring = base;
  const uint32_t sQ = base + C::Q_OFF;  // tile t at sQ + t * QK_TILE_BYTES
  const uint32_t bars = base + C::BAR_OFF;
  const uint32_t bar_q = bars;
  auto bar_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bars + 8u * (1 + C::NSLOT + s); };
  auto bar_s = [&](int t) { return bars + 8u * (1 + 2 * C::NSLOT + t); };
  auto bar_p = [&](int t) { return bars + 8u * (3 + 2 * C::NSLOT + t); };
  auto bar_o = [&](int t) { return bars + 8u * (5 + 2 * C::NSLOT + t); };
  auto bar_drain = [&](int t) { return bars + 8u * (7 + 2 * C::NSLOT + t); };
  auto bar_sfree = [&](int t) { return bars + 8u * (9 + 2 * C::NSLOT + t); };
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);

  const int warp = warp_index_uniform();
  const int lane = threadIdx.x & 31;
  const int L = args.L;
  const int n_ct = args.n_ctiles;

  // CTA order.  Heads are taken in groups of `group_heads` whose K and V
  // together fit comfortably in L2, so the CTAs resident at one time re-read
  // K/V from L2, not HBM.  Non-causal CTAs all cost the same and go
  // head-major.  Causal CTAs cost in proportion to their row index, so
  // within a group the longest go first across all of the group's heads
  // (longest-processing-time order), which keeps the tail of the launch
  // short.
  const int BH = args.bh;
  const int G = args.group_heads;
  const int n_units = BH * n_ct;                   // CTAs per split
  const int split = SPLIT ? static_cast<int>(blockIdx.x) / n_units : 0;
  const int idx = static_cast<int>(blockIdx.x) - split * n_units;
  const int g0 = (idx / (G * n_ct)) * G;           // first head of the group
  const int gsz = min(G, BH - g0);                 // heads in this group
  const int r = idx - g0 * n_ct;                   // rank within the group
  const int bh = CAUSAL ? g0 + r % gsz : g0 + r / n_ct;
  const int ct = CAUSAL ? n_ct - 1 - r / gsz : r % n_ct;
  const int row_base = ct * ROWS_PER_CTA;
  // Block range of this CTA: [jb, jb + n_blk); every loop below counts
  // blocks from jb (barrier phases and ring positions use the local count).
  int nb0 = blocks_for_tile<CAUSAL>(row_base, L);
  int nb1 = blocks_for_tile<CAUSAL>(row_base + BLOCK_M, L);
  int jb = 0;
  if (SPLIT) {
    jb = split * args.blocks_per_split;
    const int je = jb + args.blocks_per_split;
    nb0 = max(0, min(nb0, je) - jb);
    nb1 = max(0, min(nb1, je) - jb);
  }
  const int n_blk0 = nb0;
  const int n_blk1 = nb1;
  const int n_blk = max(n_blk0, n_blk1);  // K/V blocks loaded

  // d = 64: the producer lane sets up the barriers and sends Q and the first
  // K/V block on their way before the CTA-wide setup (tensor-memory
  // allocation, the block barrier); on short launches the first loads are
  // the critical path (measured: +3% at L = 1024, while d = 128 lost 2% with
  // the same change, so it keeps the setup below).
  constexpr bool EARLY = C::SPLIT_P;
  const bool early_kv = EARLY && n_blk > 0;
  if (threadIdx.x == (EARLY ? PRODUCER_WARP * 32 : 0)) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), C::SPLIT_P ? 2 : 1);  // d = 64: both MMA warps release
    }
    for (int t = 0; t < TILES_PER_CTA; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_p(t), C::WARPS_PER_TILE);  // one arrival per softmax warp
      mbar_init(bar_o(t), 1);
    }
    for (int t = 0; t < TILES_PER_CTA; ++t) {
      mbar_init(bar_drain(t), 1);
      mbar_init(bar_sfree(t), C::WARPS_PER_TILE);  // one arrival per softmax warp
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (EARLY && !args.test_withhold_q) {
      mbar_arrive_expect_tx(bar_q, TILES_PER_CTA * C::QK_TILE_BYTES);
      for (int t = 0; t < TILES_PER_CTA; ++t)
        for (int c = 0; c < C::QK_BOXES; ++c)
          tma_load_3d(sQ + t * C::QK_TILE_BYTES + c * C::QK_BOX_BYTES, &tmQ, bar_q,
                      c * C::QK_BOX_COLS, row_base + t * BLOCK_M, bh);
    }
    if (early_kv) {
      // ring positions 0 (K_0) and 1 (V_0): fresh slots, nothing to wait for
      mbar_arrive_expect_tx(bar_full(0), C::QK_TILE_BYTES);
      for (int c = 0; c < C::QK_BOXES; ++c)
        tma_load_3d(ring + c * C::QK_BOX_BYTES, &tmK, bar_full(0), c * C::QK_BOX_COLS,
                    jb * BLOCK_N, bh);
      mbar_arrive_expect_tx(bar_full(1), C::TILE_BYTES);
      for (int c = 0; c < C::BOXES; ++c)
        tma_load_3d(ring + C::TILE_BYTES + c * BOX_BYTES, &tmV, bar_full(1), c * 64,
                    jb * BLOCK_N, bh);
    }
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, args.status, args.timeout_ns};

  // The producer and MMA warps run their loops with all 32 lanes (uniform
  // control flow, so loop state stays in uniform registers); every lane
  // polls the barriers and one elected lane issues the copies, MMAs and
  // commits (always the same lane, so its commits track its own MMAs).
  auto warp_wait = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
    const bool w = mbar_wait(bar, parity, ctl, site);
    return __all_sync(0xffffffffu, w);
  };

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (!EARLY && !args.test_withhold_q && elect_one()) {
      mbar_arrive_expect_tx(bar_q, TILES_PER_CTA * C::QK_TILE_BYTES);
      for (int t = 0; t < TILES_PER_CTA; ++t)
        for (int c = 0; c < C::QK_BOXES; ++c)
          tma_load_3d(sQ + t * C::QK_TILE_BYTES + c * C::QK_BOX_BYTES, &tmQ, bar_q,
                      c * C::QK_BOX_COLS, row_base + t * BLOCK_M, bh);
    }
    __syncwarp();
    // d = 64: Q, K_0 and V_0 were sent before the CTA-wide setup.
    int cnt = early_kv ? 2 : 0;
    bool ok = true;
    auto load = [&](const CUtensorMap* map, int j, bool is_k) -> bool {
      const int s = cnt % C::NSLOT;
      const uint32_t use = static_cast<uint32_t>(cnt / C::NSLOT);
      if (!warp_wait(bar_empty(s), (use & 1u) ^ 1u, SITE_EMPTY)) return false;
      if (elect_one()) {
        const int boxes = is_k ? C::QK_BOXES : C::BOXES;
        const int box_bytes = is_k ? C::QK_BOX_BYTES : BOX_BYTES;
        const int box_cols = is_k ? C::QK_BOX_COLS : 64;
        mbar_arrive_expect_tx(bar_full(s), is_k ? C::QK_TILE_BYTES : C::TILE_BYTES);
        const uint32_t dst = ring + s * C::TILE_BYTES;
        for (int c = 0; c < boxes; ++c)
          tma_load_3d(dst + c * box_bytes, map, bar_full(s), c * box_cols, (jb + j) * BLOCK_N,
                      bh);
      }
      __syncwarp();
      ++cnt;
      return true;
    };
    // Ring positions: K_j at 2j, V_j at 2j + 1 (the MMA warp's first uses
    // come in this order).
    // Q and block 0 go out first; the rest of the ring waits until Q has
    // landed, so that on a short, cold launch (every CTA loading from DRAM
    // at once) the first score products are not queued behind K/V blocks
    // needed later.
    for (int j = early_kv ? 1 : 0; j < n_blk && ok; ++j) {
      if (j == 1 && !args.test_withhold_q) ok = warp_wait(bar_q, 0, SITE_Q);
      if (ok) ok = load(&tmK, j, true);
      if (ok) ok = load(&tmV, j, false);
    }
    if (!ok && lane == 0) {
      // Let every copy already issued land before the CTA exits.
      if (!args.test_withhold_q) mbar_wait_drain(bar_q, 0, args.timeout_ns);
      for (int s = 0; s < C::NSLOT; ++s) {
        const int issued = cnt > s ? (cnt - 1 - s) / C::NSLOT + 1 : 0;
        if (issued > 0) mbar_wait_drain(bar_full(s), (issued - 1) & 1, args.timeout_ns);
      }
    }
  } else if (warp == MMA_WARP || (C::SPLIT_P && warp == C::MMA_WARP_T1)) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t IDESC_S = idesc_bf16_f32(BLOCK_M, BLOCK_N, false);
    constexpr uint32_t IDESC_O = idesc_bf16_f32(BLOCK_M, D, true);
    auto n_t = [&](int t) { return t == 0 ? n_blk0 : n_blk1; };
    bool ok = warp_wait(bar_q, 0, SITE_Q);
    tc_fence_after();
    // Wait for ring position `pos` to be filled; returns its slot address.
    auto acquire = [&](int pos, uint32_t& addr) -> bool {
      const int s = pos % C::NSLOT;
      const uint32_t use = static_cast<uint32_t>(pos / C::NSLOT);
      if (!warp_wait(bar_full(s), use & 1u, SITE_FULL)) return false;
      tc_fence_after();
      addr = ring + s * C::TILE_BYTES;
      return true;
    };
    auto release = [&](int pos) {
      if (elect_one()) mma_commit(bar_empty(pos % C::NSLOT));
      __syncwarp();
    };
    auto issue_s = [&](int t, uint32_t kaddr) {
      const uint32_t q = sQ + t * C::QK_TILE_BYTES;
      if (elect_one()) {
        if constexpr (FP8) {
          // 32 codes (32 bytes) per step along rows of D bytes
          constexpr uint32_t IDESC_S8 = idesc_e4m3_f32(BLOCK_M, BLOCK_N);
          constexpr uint32_t SWZ = (D == 128) ? 2u : 4u;     // 128- or 64-byte rows
          constexpr uint32_t SBO = (D == 128) ? 1024u : 512u;  // 8-row atom
          const uint64_t qd = sdesc_swz(q, 16, SBO, SWZ);
          const uint64_t kd = sdesc_swz(kaddr, 16, SBO, SWZ);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_ss_f8(tmem + C::S_COL(t), qd + kk * (32 >> 4), kd + kk * (32 >> 4), IDESC_S8,
                      kk > 0 ? 1u : 0u);
        } else {
          // Descriptors built once; a k-step moves the start-address field
          // (address / 16, bits 0-13) by off / 16, which never carries out
          // of the field inside shared memory.
          const uint64_t qd = sdesc_sw128(q, 16, 1024);
          const uint64_t kd = sdesc_sw128(kaddr, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
            mma_ss(tmem + C::S_COL(t), qd + (off >> 4), kd + (off >> 4), IDESC_S,
                   kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar_s(t));
      }
      __syncwarp();
    };
    auto issue_pv = [&](int t, int j, uint32_t vaddr) -> bool {
      if (!warp_wait(bar_p(t), j & 1, SITE_P)) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t vd = sdesc_sw128(vaddr, BOX_BYTES, 1024);
#pragma unroll
        for (int kk = 0; kk < BLOCK_N / 16; ++kk) {
          mma_ts(tmem + C::O_COL(t), tmem + C::P_COL(t) + kk * 8, vd + kk * (2048 >> 4), IDESC_O,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        // With its own P columns the softmax waits for every PV (it rewrites
        // P_t and may rescale O_t next block); otherwise only the epilogue.
        if (C::SPLIT_P || j == n_t(t) - 1) mma_commit(bar_o(t));
      }
      __syncwarp();
      return true;
    };

    uint32_t kaddr = 0, vaddr = 0;
    if constexpr (C::SPLIT_P) {
      // d = 64: this warp issues only tile t's products.  Per block j:
      // S_t of block j+1 as soon as the softmax has read S_t of block j
      // (s_free), then O_t += P_t V_j when P_t is ready.  Every ring position
      // is released by both MMA warps (count 2): a commit where this warp's
      // MMAs read the slot, a plain arrival where tile t had no use for it,
      // always after the slot was seen full.
      const int t = warp == MMA_WARP ? 0 : 1;
      const int n_mine = n_t(t);
      auto release_t = [&](int pos, bool used) {
        if (elect_one()) {
          if (used)
            mma_commit(bar_empty(pos % C::NSLOT));
          else
            mbar_arrive(bar_empty(pos % C::NSLOT));
        }
        __syncwarp();
      };
      if (ok && n_blk > 0) {
        ok = acquire(0, kaddr);
        if (ok) {
          if (n_mine > 0) issue_s(t, kaddr);
          release_t(0, n_mine > 0);
        }
      }
      for (int j = 0; j < n_blk && ok; ++j) {
        if (j + 1 < n_blk) {
          ok = acquire(2 * j + 2, kaddr);
          const bool use_k = j + 1 < n_mine;
          if (ok && use_k) {
            ok = warp_wait(bar_sfree(t), j & 1, SITE_S);
            if (ok) {
              tc_fence_after();
              issue_s(t, kaddr);
            }
          }
          if (ok) release_t(2 * j + 2, use_k);
        }
        if (ok) ok = acquire(2 * j + 1, vaddr);
        const bool use_v = j < n_mine;
        if (ok && use_v) ok = issue_pv(t, j, vaddr);
        if (ok) release_t(2 * j + 1, use_v);
      }
      if (!ok) {
        // Every MMA this warp issued must finish before the tensor memory is freed.
        if (elect_one()) {
          mma_commit(bar_drain(t));
          mbar_wait_drain(bar_drain(t), 0, args.timeout_ns);
        }
        __syncwarp();
      }
    } else {
    if (ok && n_blk > 0) {
      ok = acquire(0, kaddr);
      if (ok) {
        for (int t = 0; t < TILES_PER_CTA; ++t)
          if (n_t(t) > 0) issue_s(t, kaddr);
        release(0);
      }
    }
    for (int j = 0; j < n_blk && ok; ++j) {
      ok = acquire(2 * j + 1, vaddr);
      // K_{j+1} is taken just before its first use, so PV0_j never waits
      // for it.  Some tile uses K_{j+1} whenever j + 1 < n_blk.
      bool k_next = false;
      for (int t = 0; t < TILES_PER_CTA && ok; ++t) {
        if (j < n_t(t)) ok = issue_pv(t, j, vaddr);
        if (ok && j + 1 < n_t(t)) {
          if (!k_next) ok = acquire(2 * j + 2, kaddr);
          k_next = true;
          if (ok) issue_s(t, kaddr);
        }
      }
      if (ok) {
        release(2 * j + 1);
        if (k_next) release(2 * j + 2);
      }
    }
    if (!ok) {
      // Every MMA already issued must finish before the tensor memory is freed.
      if (elect_one()) {
        mma_commit(bar_drain(0));
        mbar_wait_drain(bar_drain(0), 0, args.timeout_ns);
      }
      __syncwarp();
    }
    }  // one MMA warp for both tiles (d = 128)
  } else {
    // ------------------------------------------------------------ softmax
    // Warp (t, quarter): Q tile t, rows 32*quarter .. +31 (its TMEM lanes),
    // all 128 key columns of every block.
    constexpr int NCH = BLOCK_N / 32;  // 32-column score chunks
    constexpr int OCH = D / 32;        // 32-column O chunks
    const int sidx = warp - FIRST_SOFTMAX_WARP;
    const int t = sidx >> 2;           // Q tile of this warp
    const int quarter = warp & 3;     // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = C::S_COL(t);
    const uint32_t p_col = C::P_COL(t);
    const uint32_t o_col = C::O_COL(t);
    const int tile_row0 = row_base + t * BLOCK_M;
    const int q_row = tile_row0 + row;
    const int n_my = t == 0 ? n_blk0 : n_blk1;
    float sl2 = args.scale_log2;  // FP8: times s_q * s_k of the block, set per block
    const bool pos_scale = args.scale_log2 > 0.f;  // the block scales are positive
    float m = -INFINITY;  // running max of scale*log2e*s
    float l = 0.f;        // running sum of P~ relative to m
    bool ok = true;
    float sq = 1.f;
    float ks = 1.f;  // FP8: the scale of the next K block, loaded a block ahead
    if constexpr (FP8)
      if (n_my > 0) {
        sq = args.q_scale[static_cast<size_t>(bh) * args.n_blocks + tile_row0 / BLOCK_M];
        ks = args.k_scale[static_cast<size_t>(bh) * args.n_blocks + jb];
      }
    for (int j = 0; j < n_my; ++j) {
      if constexpr (FP8) {
        sl2 = args.scale_log2 * sq * ks;
        if (j + 1 < n_my) ks = args.k_scale[static_cast<size_t>(bh) * args.n_blocks + jb + j + 1];
      }
      const bool w = mbar_wait(bar_s(t), j & 1, ctl, SITE_S);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[NCH][32];
      tmem_ld_chunks<NCH>(lane_base + s_col, sr);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < NCH; ++c) reg_fence32(sr[c]);
      if constexpr (C::SPLIT_P) {
        // The scores are in registers: S_t may take the next block's product.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfree(t));
      }

      // Masks: keys past the end of the sequence; causal keys after the query.
      const int k0 = (jb + j) * BLOCK_N;
      const bool need_mask = (k0 + BLOCK_N > L) || (CAUSAL && k0 + BLOCK_N - 1 > tile_row0);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int key = k0 + c * 32 + e;
            const bool masked = key >= L || (CAUSAL && key > q_row);
            if (masked) sr[c][e] = __float_as_uint(-INFINITY);
          }
      }

      // Row max in units of scale*log2(e).
      float blk;
      if (pos_scale) {
        // eight independent chains of three-way maxima (short latency)
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              mx[i] = fmax3(mx[i], __uint_as_float(sr[c][e + 2 * i]),
                            __uint_as_float(sr[c][e + 2 * i + 1]));
        blk = fmaxf(fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), mx[6]), mx[7]) *
              sl2;
      } else {
        // scale <= 0: work on x = scale*log2e*s directly (masked stays -inf).
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float s = __uint_as_float(sr[c][e]);
            const float x = (s == -INFINITY) ? -INFINITY : s * sl2;
            sr[c][e] = __float_as_uint(x);
            mx[e & 3] = fmaxf(mx[e & 3], x);
          }
        blk = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);
      }
      const float m_new = fmaxf(m, blk);
      // Every row sees at least one unmasked key in every block it visits,
      // so m_new is finite here.
      float corr = 1.f;
      const bool grew = j > 0 && m_new > m;
      if (grew) corr = ex2_approx(m - m_new);
      m = m_new;

      // P~ = exp2(x - m) with x = s*sl2 (fused, two lanes per instruction) or
      // the precomputed x; the row sum accumulates in four packed pairs.
      const float mul = pos_scale ? sl2 : 1.f;
      const uint64_t mul2 = f2_pack(mul, mul);
      const uint64_t negm2 = f2_pack(-m, -m);
      uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
      // Keys 32c..32c+31 pack into columns 16c..16c+15 of the P columns.
      // With separate P columns the stores (one wide store of all 64
      // columns) wait until O_t += P_t V_{j-1} has completed (it reads the
      // same columns); the exponentials run first, so that wait overlaps
      // them.
      uint32_t pk[NCH][16];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), mul2,
                           negm2),
                    x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          sum2[(e >> 1) & 3] = f2_add(sum2[(e >> 1) & 3], f2_pack(p0, p1));
          pk[c][e >> 1] = pack_bf16x2(p0, p1);
        }
        if constexpr (!C::SPLIT_P) tmem_st16(lane_base + p_col + 16u * c, pk[c]);
      }
      if constexpr (C::SPLIT_P) {
        if (j > 0) {
          // P_t and O_t are free once O_t += P_t V_{j-1} has completed.
          const bool wo = mbar_wait(bar_o(t), (j - 1) & 1, ctl, SITE_O);
          if (!__all_sync(0xffffffffu, wo)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st_pchunks<NCH>(lane_base + p_col, pk);
      }
      float s_lo, s_hi;
      f2_unpack(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), s_lo, s_hi);
      const float rowsum = s_lo + s_hi;
      l = (j == 0) ? rowsum : fmaf(corr, l, rowsum);

      // O_t is quiescent here: O_t += P_t V_{j-1} has completed (with separate
      // P columns the o_done wait above says so; otherwise the arrival on
      // s_full for this block came after it), and the next PV waits for p_full.
      if (__any_sync(0xffffffffu, grew)) {
        // All of this warp's O_t columns in one round trip: issue every load,
        // wait once, scale in packed pairs, store back.
        // (64 columns: one wide load and store; 128 columns: per-chunk
        // stores after one round of loads, measured faster on the
        // rescale-heavy d = 128 causal workload)
        constexpr bool WIDE_O = OCH <= 2;
        uint32_t ov[OCH][32];
        if constexpr (WIDE_O) {
          tmem_ld_chunks<OCH>(lane_base + o_col, ov);
        } else {
#pragma unroll
          for (int c = 0; c < OCH; ++c) tmem_ld32(lane_base + o_col + 32u * c, ov[c]);
        }
        tmem_wait_ld();
        const uint64_t corr2 = f2_pack(corr, corr);
#pragma unroll
        for (int c = 0; c < OCH; ++c) {
          reg_fence32(ov[c]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float a, b;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(ov[c][e]), __uint_as_float(ov[c][e + 1])),
                             corr2),
                      a, b);
            ov[c][e] = __float_as_uint(a);
            ov[c][e + 1] = __float_as_uint(b);
          }
          if constexpr (!WIDE_O) tmem_st32(lane_base + o_col + 32u * c, ov[c]);
        }
        if constexpr (WIDE_O) tmem_st_chunks<OCH>(lane_base + o_col, ov);
      }
      // One arrival per warp: every lane's tensor-memory stores are complete
      // (wait::st) and ordered (fence) before the warp syncs and lane 0
      // arrives.  128 separate arrivals on one barrier word serialise.
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p(t));
    }

    const bool store = q_row < L;
    if (ok && n_my > 0) {
      // Epilogue: wait for the last O_t += P_t V, then O / l and LSE.
      const bool w = mbar_wait(bar_o(t), C::SPLIT_P ? (n_my - 1) & 1 : 0, ctl, SITE_O);
      if (__all_sync(0xffffffffu, w)) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const float lse_row = (m + log2f(l)) * 0.69314718055994531f;
        const size_t row = static_cast<size_t>(bh) * L + q_row;
        constexpr bool WIDE_EPI = OCH <= 2;  // as for the rescale
        uint32_t oall[WIDE_EPI ? OCH : 1][32];
        if constexpr (WIDE_EPI) {
          tmem_ld_chunks<OCH>(lane_base + o_col, oall);
          tmem_wait_ld();
        }
#pragma unroll
        for (int c = 0; c < OCH; ++c) {
          uint32_t (&ov)[32] = oall[WIDE_EPI ? c : 0];
          if constexpr (!WIDE_EPI) {
            tmem_ld32(lane_base + o_col + 32u * c, ov);
            tmem_wait_ld();
          }
          reg_fence32(ov);
          if constexpr (SPLIT) {
            // fp32 partial, normalised over this split's keys.
            if (store) {
              float4* dst = reinterpret_cast<float4*>(
                  args.o_part + (static_cast<size_t>(split) * args.bh * L + row) * D + c * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(__uint_as_float(ov[4 * i]) * inv_l,
                                     __uint_as_float(ov[4 * i + 1]) * inv_l,
                                     __uint_as_float(ov[4 * i + 2]) * inv_l,
                                     __uint_as_float(ov[4 * i + 3]) * inv_l);
            }
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l,
                                  __uint_as_float(ov[2 * e + 1]) * inv_l);
            if (store) {
              uint4* dst = reinterpret_cast<uint4*>(args.o + row * D + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        }
        if (store) {
          if constexpr (SPLIT)
            args.lse_part[static_cast<size_t>(split) * args.bh * L + row] = lse_row;
          else
            args.lse[row] = lse_row;
        }
      }
    } else if (SPLIT && ok && store) {
      // No key of this split is visible to this tile (causal): an empty
      // partial, weight exp(-inf) = 0 in the merge.
      const size_t row = static_cast<size_t>(bh) * L + q_row;
      float4* dst = reinterpret_cast<float4*>(
          args.o_part + (static_cast<size_t>(split) * args.bh * L + row) * D);
#pragma unroll
      for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      args.lse_part[static_cast<size_t>(split) * args.bh * L + row] = -INFINITY;
    }
    tmem_wait_st();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace fa
