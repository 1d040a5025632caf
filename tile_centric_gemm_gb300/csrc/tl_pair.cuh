// tl_pair.cuh -- the CTA-pair (cta_group::2) GEMM core shared by the kernels:
// a 256 x 256 output tile per cluster of two CTAs on two SMs.  Each CTA stages
// its own 128 rows of A and its own 128 columns of B per 64-deep k-block; the
// leader CTA issues tcgen05.mma.cta_group::2 (M=256, N=256), which reads both
// CTAs' shared memory and accumulates rows 0-127 in the leader's TMEM and rows
// 128-255 in the peer's.  Compared with one CTA per 128 x 256 tile this moves a
// third less operand data from L2 per flop and halves the B staging per CTA.
#pragma once

#include "tl_common.cuh"

namespace tl {
namespace pair {

constexpr int BM = 256;  // pair tile rows (128 per CTA)
constexpr int BN = 256;  // pair tile columns (B staged as 128 columns per CTA)
constexpr int BK = 64;
constexpr int HM = 128;
constexpr int HN = 128;
constexpr int STAGES = 6;
constexpr uint32_t A_STAGE = HM * BK * 2;            // 16 KB
constexpr uint32_t B_STAGE = BK * HN * 2;            // 16 KB = 2 boxes of 64 x 64
constexpr uint32_t CTA_STAGE_TX = A_STAGE + B_STAGE;  // bytes one CTA loads per stage
constexpr uint32_t PAIR_STAGE_TX = 2 * CTA_STAGE_TX;  // bytes the leader's full barrier expects
// A narrow tile (at most HN columns left, N = 128): each CTA stages one 64-column box of B.
constexpr uint32_t PAIR_STAGE_TX_NARROW = 2 * (A_STAGE + B_BOX_BYTES);
constexpr uint32_t SMEM_A = 0;
constexpr uint32_t SMEM_B = SMEM_A + STAGES * A_STAGE;
constexpr uint32_t SMEM_END = SMEM_B + STAGES * B_STAGE;  // 192 KB
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, true);
constexpr uint32_t IDESC_NARROW = idesc_bf16_f32(BM, BN / 2, true);

struct __align__(8) Bars {
  uint64_t full[STAGES];     // leader: both CTAs' TMA bytes of a stage
  uint64_t empty[STAGES];    // both CTAs: stage consumed (multicast commit)
  uint64_t tmem_full[2];     // both CTAs: accumulator ready (multicast commit)
  uint64_t tmem_empty[2];    // leader: the epilogue warps of the pair drained it
  uint64_t copy[COPY_NBUF];  // copy-warp staging
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t splitk_ok;        // split-K: every split of this CTA's half-tile arrived
};

// Four UMMA_K steps of one k-block from stage s; issued by the leader only.  A narrow tile
// (IDESC_NARROW) reads only the first B box of each CTA.
__device__ __forceinline__ void mma_kblock(uint8_t* smem, int s, uint32_t d_tmem, bool first,
                                           uint32_t idesc = IDESC) {
  const uint32_t a0 = smem_u32(smem + SMEM_A + s * A_STAGE);
  const uint32_t b0 = smem_u32(smem + SMEM_B + s * B_STAGE);
#pragma unroll
  for (int kk = 0; kk < BK / UMMA_K; ++kk) {
    const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
    const uint64_t bd = sdesc_sw128(b0 + kk * 2048, B_BOX_BYTES, 1024);
    tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (first && kk == 0) ? 0u : 1u);
  }
}

// Initialise the pair's barriers (thread 0 of each CTA) and allocate TMEM
// (warp kWarpMma of each CTA), then synchronise the cluster so that no CTA
// signals a barrier of its peer before the peer has initialised it.
// epi_arrivals: arrivals that free an accumulator (by default one per epilogue warp of
// both CTAs).
__device__ __forceinline__ uint32_t setup(Bars* bars, int warp, uint32_t epi_arrivals = 2 * kNumEpiWarps) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tmem_full[a], 1);
      mbar_init(&bars->tmem_empty[a], epi_arrivals);
    }
    for (int b = 0; b < COPY_NBUF; ++b) mbar_init(&bars->copy[b], 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  return bars->tmem_base;
}

// End of the kernel: every thread of both CTAs is done with TMEM and with the
// peer's barriers before the pair frees TMEM and exits.
__device__ __forceinline__ void teardown(Bars* bars, int warp, uint32_t tmem_base) {
  tc_fence_before();
  __syncthreads();
  if (bars->abort) {
    const uint64_t t0 = now_ns();
    while (now_ns() - t0 < 50000) {
    }
  }
  cluster_sync();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// The epilogue warps of either CTA release an accumulator to the leader's MMA issuer.
__device__ __forceinline__ void release_accumulator(Bars* bars, int acc, uint32_t rank) {
  if (rank == 0) mbar_arrive(&bars->tmem_empty[acc]);
  else mbar_arrive_cluster(map_to_rank(&bars->tmem_empty[acc], 0));
}

struct NeverNarrow {
  __device__ __forceinline__ bool operator()(int) const { return false; }
};

// MMA issuer loop of the leader: `ntiles` tiles of `kb` k-blocks each, ring state in (s, ph);
// narrow(j) says whether this pair's j-th tile is a narrow one (N = 128).
template <class Narrow = NeverNarrow>
__device__ __forceinline__ void mma_loop(uint8_t* smem, Bars* bars, uint32_t tmem_base, int ntiles, int KB,
                                         volatile uint32_t* abort, uint32_t* status, uint64_t pipe_timeout,
                                         Narrow narrow = Narrow()) {
  int s = 0;
  uint32_t ph = 0;
  for (int j = 0; j < ntiles && !*abort; ++j) {
    const int acc = j & 1;
    const uint32_t acc_ph = uint32_t(j >> 1) & 1u;
    if (!mbar_wait(&bars->tmem_empty[acc], acc_ph ^ 1u, abort, status, pipe_timeout, 2)) return;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
    const uint32_t idesc = narrow(j) ? IDESC_NARROW : IDESC;
    for (int kb = 0; kb < KB; ++kb) {
      if (!mbar_wait(&bars->full[s], ph, abort, status, pipe_timeout, 3)) return;
      tc_fence_after();
      mma_kblock(smem, s, d_tmem, kb == 0, idesc);
      tc_commit_pair(&bars->empty[s], 0x3);
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
    tc_commit_pair(&bars->tmem_full[acc], 0x3);
  }
}

// Producer: load one k-block of this CTA's halves of A and B into stage s,
// completing on the leader's full barrier.  Returns false if the pipeline aborted.
struct Producer {
  int s = 0;
  uint32_t ph = 0;
  // narrow: a narrow tile, one 64-column box of B from b_x (the CTA's half of 128 columns).
  __device__ __forceinline__ bool load(uint8_t* smem, Bars* bars, uint32_t rank, const CUtensorMap* ma, int a_x,
                                       int a_y, const CUtensorMap* mb, int b_x, int b_y, volatile uint32_t* abort,
                                       uint32_t* status, uint64_t pipe_timeout, bool narrow = false) {
    if (!mbar_wait(&bars->empty[s], ph ^ 1u, abort, status, pipe_timeout, 1)) return false;
    if (rank == 0) mbar_arrive_expect_tx(&bars->full[s], narrow ? PAIR_STAGE_TX_NARROW : PAIR_STAGE_TX);
    const uint32_t full = map_to_rank(&bars->full[s], 0);
    tma_load_2d_pair(smem + SMEM_A + s * A_STAGE, ma, full, a_x, a_y);
    uint8_t* b_dst = smem + SMEM_B + s * B_STAGE;
    tma_load_2d_pair(b_dst, mb, full, b_x, b_y);
    if (!narrow) tma_load_2d_pair(b_dst + B_BOX_BYTES, mb, full, b_x + 64, b_y);
    if (++s == STAGES) {
      s = 0;
      ph ^= 1u;
    }
    return true;
  }
  // The same with L2 eviction-priority policies on the operand lines (pol_a for A, pol_b for B).
  __device__ __forceinline__ bool load_hint(uint8_t* smem, Bars* bars, uint32_t rank, const CUtensorMap* ma, int a_x,
                                            int a_y, const CUtensorMap* mb, int b_x, int b_y, uint64_t pol_a,
                                            uint64_t pol_b, volatile uint32_t* abort, uint32_t* status,
                                            uint64_t pipe_timeout) {
    if (!mbar_wait(&bars->empty[s], ph ^ 1u, abort, status, pipe_timeout, 1)) return false;
    if (rank == 0) mbar_arrive_expect_tx(&bars->full[s], PAIR_STAGE_TX);
    const uint32_t full = map_to_rank(&bars->full[s], 0);
    tma_load_2d_pair_hint(smem + SMEM_A + s * A_STAGE, ma, full, a_x, a_y, pol_a);
    uint8_t* b_dst = smem + SMEM_B + s * B_STAGE;
    tma_load_2d_pair_hint(b_dst, mb, full, b_x, b_y, pol_b);
    tma_load_2d_pair_hint(b_dst + B_BOX_BYTES, mb, full, b_x + 64, b_y, pol_b);
    if (++s == STAGES) {
      s = 0;
      ph ^= 1u;
    }
    return true;
  }
  __device__ __forceinline__ bool load_hint(uint8_t* smem, Bars* bars, uint32_t rank, const CUtensorMap* ma, int a_x,
                                            int a_y, const CUtensorMap* mb, int b_x, int b_y, uint64_t pol,
                                            volatile uint32_t* abort, uint32_t* status, uint64_t pipe_timeout) {
    return load_hint(smem, bars, rank, ma, a_x, a_y, mb, b_x, b_y, pol, pol, abort, status, pipe_timeout);
  }
};

}  // namespace pair
}  // namespace tl
