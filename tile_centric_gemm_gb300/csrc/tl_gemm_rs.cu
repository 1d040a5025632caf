// tl_gemm_rs.cu -- GEMM -> ReduceScatter fused at tile granularity in one launch.
//
// TileLink talk summary ("TileLink: Generating Efficient Compute-Communication
// Overlapping Kernels using Tile-Centric Primitives"):
//  * Key Findings / Experimental Setup & Results -- GEMM-ReduceScatter.
//  * Technical Deep Dive, persistent kernels -- the GEMM is a plain persistent
//    GEMM plus one produce_tile_notify per finished tile; the reduce stage
//    waits on its own tile and its peers' tiles (consume_tile_wait,
//    peer_tile_wait) and receives partials in push mode.
//
// Work items: output tile tau = (dest d, m tile, n tile) of 256 x 256, in
// destination order, within a destination n tile by n tile with the m tiles
// innermost (neighbouring tiles share B columns and the destination's A rows,
// which stay in L2); its R partial tiles P_r = A_r[rows of tau] . B_r[:, cols
// of tau] are items tau*R + j, rank r = (d + 1 + tau + j) mod R (the rotation
// spreads the destination rank's own item over the CTAs).  Items go
// round-robin over CTA pairs (clusters of two, tcgen05.mma.cta_group::2); CTA
// h of a pair owns rows h*128 .. h*128+127 of every tile it works on.
//
// Receive slots form a ring of 3 * pairs items (two 128-row halves each): item
// i pushes half h into half-slot 2 * (i mod ring) + h, after the R reducers of
// half h of the tile that used the slot before have released their "reduced"
// flags.  The ring is about 57 MB for 76 pairs.  Deadlock freedom:
// a push of tile tau waits only on earlier tiles (slot-free flags, its own
// pair's earlier accumulator) and a reduce of tau only on pushes of tau and
// its own earlier reduces, so by induction on tau every tile completes.
//
// Per CTA: warp 0 TMA producer (its halves of A_r, B_r), warp 1 tcgen05 MMA
// issuer (leader only), warps 2-5 pushers, warps 6-13 reducers.  For item
// (tau, j) and half h:
//   push:   TMEM -> registers -> fp32 receive slot of the item; release the
//           arrival flag tau*R + r (produce_tile_notify).  Before reusing a ring
//           slot the pushers acquire the "reduced" flags of the tile that last
//           used it (the slot-free barrier of the pull protocol).
//   reduce: acquire the R arrival flags of tau (consume_tile_wait on its own
//           partial, peer_tile_wait on the others), sum row slice j of the tile
//           over the R slots in rank order 0..R-1 in fp32, store bf16 rows of
//           out[d], then release the "reduced" flag of (tau, j).
// Pushers never wait on peers' partials and reducers never hold TMEM, so the
// tensor pipe is not stalled by the reduction.  Flags: [0, 2*items) arrival
// flags indexed 2*(tau*R + r) + h; [2*items, 4*items) reduced flags indexed
// 2*(tau*R + j) + h.
//
// Chain schedule (tl_gemm_rs, every option).  The same sum, accumulated on the
// way instead of at the destination, like the partial sums of a ring reduce
// travelling from rank to rank: the destinations are taken in groups of
// kChainGroup, and within a group items run pass by pass (pass j: every tile's
// partial of the j-th rank of the summation order -- rank j, or rank d+1+j mod
// R in ring order).  The chain launches 11 warps: eight drain each accumulator
// (warps 2-9, one per TMEM lane quarter and column half, each freeing the
// accumulator after its last read of it; warp 10 releases a pass's flags once
// all eight have stored their share); those of (tau, j) wait for pass j-1's
// arrival flag of the tile (peer_tile_wait), add their partial (rounded to bf16 first with
// bf16 partials) to the tile's fp32 running sum S_tau in the workspace (the
// next chunk's sums loaded while the current one is added) and release the
// flags of (tau, j); pass R-1 writes bf16(S_tau) to out[d] instead.  The
// push-and-reduce schedule above runs for the no-allocation entry point, whose
// fixed scratch holds a ring of slots but not a running sum per tile.  A group's running sums (17 MB per
// destination at 1024 x 4096) stay in L2 from rank to rank, each rank's B_r is
// read once per group and A_r about once, and no partial is read back from a
// ring slot.  The results are the same bits as the push-and-reduce
// schedule's.  Deadlock freedom: (tau, r) waits only on (tau, r-1), an item
// with a lower index, and every pair takes its items in increasing index
// order.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "tl_internal.h"
#include "tl_pair.cuh"

namespace tl {
namespace {

constexpr int RS_MAX_RANKS = 32;
constexpr int kWarpRed0 = kWarpEpi0 + kNumEpiWarps;  // first reducer warp
constexpr int kNumRedWarps = 8;
constexpr int kNumRedThreads = kNumRedWarps * 32;
constexpr int RS_THREADS = (kWarpRed0 + kNumRedWarps) * 32;
constexpr uint32_t RS_SMEM_BARS = pair::SMEM_END;
// chain schedule, per accumulator: the epilogue threads' stores are done (stored[a], one
// arrival per chain epilogue thread) and the notifier has released the pass (notified[a])
struct ChainBars {
  uint64_t stored[2];
  uint64_t notified[2];
};
constexpr uint32_t RS_SMEM_CHAIN = RS_SMEM_BARS + (uint32_t(sizeof(pair::Bars)) + 7u) / 8u * 8u;
constexpr uint32_t RS_SMEM_BYTES = RS_SMEM_CHAIN + sizeof(ChainBars) + 1024;
constexpr int RB = 8;                             // ranks loaded per batch in the reduce
constexpr int QU = 2;                             // float4 elements per thread per round in the reduce
// chain schedule: destinations whose running sums stay in L2 while their R ranks pass
constexpr int kChainGroup = 2;
// The chain schedule's epilogue: two groups of four warps, each adding half of the columns.
constexpr int kChainParts = 2;
constexpr int kChainEpiWarps = kNumEpiWarps * kChainParts;
constexpr int kChainEpiThreads = kChainEpiWarps * 32;
constexpr int kWarpChainNotify = kWarpEpi0 + kChainEpiWarps;  // releases each pass's flags
constexpr int RS_CHAIN_THREADS = (kWarpChainNotify + 1) * 32;  // the chain launches no reducer warps
constexpr int kChainChunks = pair::BN / 32 / kChainParts;

struct RsParams {
  CUtensorMap map_a[RS_MAX_RANKS];  // A_r [M, K_r], box 128 rows
  CUtensorMap map_b[RS_MAX_RANKS];  // B_r [K_r, N], box 64 x 64
  uint16_t* out[RS_MAX_RANKS];      // out[d] [Md, N] bf16
  float* slots;                     // [ring_items][2][half_floats] fp32 receive half-slots
  uint32_t* flags;                  // [2][items][2]: arrival, then reduced
  uint32_t* status;
  int32_t* trace;                   // optional: tile and rank of each item
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int32_t R, M, Md, K, N;
  int32_t Mt_d, Nt, KB, num_tiles, num_items, slice_rows, ring_items, half_floats;
  int32_t ring_order;  // destination d sums ranks d+1, ..., d instead of 0, ..., R-1
  uint32_t epoch;
};

struct Item {
  int tau, d, mt, nt, r, j;
};

template <bool kChain>
__device__ __forceinline__ Item item_of(const RsParams& p, int i) {
  Item it;
  if (kChain) {
    // groups of kChainGroup destinations; within a group rank by rank, the group's
    // tiles in order; j = r names the item's flags
    const int tpg = min(p.num_tiles, kChainGroup * p.Mt_d * p.Nt);
    const int g = i / (p.R * tpg), rem = i - g * (p.R * tpg);
    const int gt = min(tpg, p.num_tiles - g * tpg);  // tiles of this (perhaps last, smaller) group
    it.j = rem / gt;                                 // the pass: position in the summation order
    it.tau = g * tpg + (rem - it.j * gt);
  } else {
    it.tau = i / p.R;
    it.j = i % p.R;
  }
  const int per_d = p.Mt_d * p.Nt;
  it.d = it.tau / per_d;
  const int rem = it.tau % per_d;
  it.mt = rem % p.Mt_d;
  it.nt = rem / p.Mt_d;
  if (!kChain) it.r = (it.d + 1 + it.tau + it.j) % p.R;
  // chain: pass j adds rank j, or rank d+1+j (mod R) in ring order
  else it.r = p.ring_order ? (it.d + 1 + it.j) % p.R : it.j;
  return it;
}

// kBf16: partials rounded to bf16 (TL_RS_BF16_PARTIALS); kChain: the chain schedule
// (every option), else push and reduce (the no-allocation entry point).
template <bool kBf16, bool kChain>
__global__ void __launch_bounds__(kChain ? RS_CHAIN_THREADS : RS_THREADS, 1)
    gemm_rs_kernel(const __grid_constant__ RsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  pair::Bars* bars = reinterpret_cast<pair::Bars*>(smem + RS_SMEM_BARS);
  ChainBars* cb = reinterpret_cast<ChainBars*>(smem + RS_SMEM_CHAIN);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const uint32_t rank = cluster_ctarank();
  const int h = int(rank);
  const int pair_id = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  if (kChain && threadIdx.x == 0) {
    for (int a = 0; a < 2; ++a) {
      mbar_init(&cb->stored[a], kChainEpiThreads);
      mbar_init(&cb->notified[a], 1);
    }
  }
  // chain: every chain epilogue warp of both CTAs frees the accumulator after its last read
  const uint32_t tmem_base = pair::setup(bars, warp, kChain ? 2 * kChainEpiWarps : 2 * kNumEpiWarps);
  volatile uint32_t* abort = &bars->abort;
  const int my_items = pair_id < p.num_items ? (p.num_items - 1 - pair_id) / npairs + 1 : 0;
  uint32_t* arrived = p.flags;                         // 2*(tau*R + r) + h
  uint32_t* reduced = p.flags + 2 * size_t(p.num_items);  // 2*(tau*R + j) + h

  if (warp == kWarpTma) {
    // ---------------------------------------------------------------- TMA producer (this CTA's halves)
    if (lane == 0) {
      pair::Producer prod;
      // operands stay in L2 ahead of the streamed partials: A rows are reused across a
      // destination's n tiles and B columns across its m tiles
      const uint64_t keep = l2_policy_evict_last();
      for (int i = pair_id; i < p.num_items && !*abort; i += npairs) {
        const Item it = item_of<kChain>(p, i);
        if (p.trace && rank == 0) p.trace[i] = ((it.d * p.Mt_d + it.mt) * p.Nt + it.nt) * p.R + it.r;
        const int row0 = it.d * p.Md + it.mt * pair::BM + h * pair::HM;
        for (int kb = 0; kb < p.KB; ++kb)
          if (!prod.load_hint(smem, bars, rank, &p.map_a[it.r], kb * pair::BK, row0, &p.map_b[it.r],
                              it.nt * pair::BN + h * pair::HN, kb * pair::BK, keep, abort, p.status,
                              p.pipe_timeout_ns))
            break;
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && rank == 0)
      pair::mma_loop(smem, bars, tmem_base, my_items, p.KB, abort, p.status, p.pipe_timeout_ns);
    __syncwarp();
  } else if (kChain && warp == kWarpChainNotify) {
    // ---------------------------------------------------------------- chain notifier
    // produce_tile_notify for each pass, off the epilogue's path: once every epilogue thread
    // has stored its share of the item (their arrivals order their writes before this
    // thread's release), release the pass's arrival and "reduced" flags
    if (lane == 0) {
      int jj = 0;
      for (int i = pair_id; i < p.num_items; i += npairs, ++jj) {
        const Item it = item_of<true>(p, i);
        const int acc = jj & 1;
        if (!mbar_wait(&cb->stored[acc], uint32_t(jj >> 1) & 1u, abort, p.status, p.pipe_timeout_ns, 6)) break;
        st_release(arrived + 2 * (it.tau * p.R + it.j) + h, p.epoch);
        st_release(reduced + 2 * (it.tau * p.R + it.j) + h, p.epoch);
        mbar_arrive(&cb->notified[acc]);
      }
    }
    __syncwarp();
  } else if (kChain && warp < kWarpEpi0 + kChainEpiWarps) {
    // ---------------------------------------------------------------- pushers: chain accumulation
    // Two groups of four warps (the pushers and the first four reducer warps, which the
    // chain does not need), one warp per TMEM lane quarter in each; group q adds columns
    // [q, q+1) * 128 of every accumulator.
    const int wq = warp & 3;
    const int part = (warp - kWarpEpi0) / kNumEpiWarps;
    const int row_in_half = wq * 32 + lane;
    // S_tau in the half-slot layout [slice][col/4][row in slice][4] of the push schedule
    const int my_slice = row_in_half / p.slice_rows, my_row = row_in_half % p.slice_rows;
    const size_t my_base = (size_t(my_slice) * 64 * p.slice_rows + my_row) * 4;
    int jj = 0;
    for (int i = pair_id; i < p.num_items; i += npairs, ++jj) {
      const Item it = item_of<true>(p, i);
      const int acc = jj & 1;
      const uint32_t acc_ph = uint32_t(jj >> 1) & 1u;
      // peer_tile_wait: the previous pass's partial is in S_tau (it ran a whole pass of the
      // group's tiles earlier)
      if (it.j > 0 && lane == 0) {
        const int f = 2 * (it.tau * p.R + it.j - 1) + h;
        wait_flag(arrived + f, p.epoch, p.status, p.timeout_ns, uint32_t(f), TL_ERR_TIMEOUT);
      }
      __syncwarp();
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      if (!named_bar_and(1, kChainEpiThreads, ok)) break;
      tc_fence_after();
      float* S = p.slots + (size_t(it.tau) * 2 + h) * p.half_floats + my_base;
      const bool first = it.j == 0, last = it.j == p.R - 1;
      const int orow = it.mt * pair::BM + h * pair::HM + row_in_half;  // row of out[d]
      uint16_t* orowp = p.out[it.d] + size_t(orow) * p.N;
      const uint64_t keep = l2_policy_evict_last();  // S_tau is read again by the next rank
      const int nch = min(pair::BN / 32, (p.N - it.nt * pair::BN + 31) / 32);
      // this warp's share of the columns; the next chunk's running sums loaded one chunk ahead
      const int c_lo = part * kChainChunks, c_hi = min(nch, c_lo + kChainChunks);
      float4 sn[8];
      if (!first && c_lo < c_hi) {
#pragma unroll
        for (int g = 0; g < 8; ++g) sn[g] = ld_global_cg_v4f_hint(S + size_t(c_lo * 8 + g) * p.slice_rows * 4, keep);
      }
      for (int c = c_lo; c < c_hi; ++c) {
        const int col0 = it.nt * pair::BN + c * 32;
        float4 sv[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) sv[g] = sn[g];
        if (!first && c + 1 < c_hi) {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            sn[g] = ld_global_cg_v4f_hint(S + size_t((c + 1) * 8 + g) * p.slice_rows * 4, keep);
        }
        uint32_t v[32];
        tmem_ld_32cols(tmem_base + (uint32_t(wq * 32) << 16) + uint32_t(acc * pair::BN + c * 32), v);
        tmem_ld_wait();
        if (c == c_hi - 1) {
          // this warp's last read of the accumulator: hand it back before the adds and stores
          tc_fence_before();
          __syncwarp();
          if (lane == 0) pair::release_accumulator(bars, acc, rank);
        }
        float* f = reinterpret_cast<float*>(v);
        if (kBf16) {
          // the partial rounded to bf16 (RNE) before it joins the sum
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const uint32_t w = pack_bf16x2(f[2 * q], f[2 * q + 1]);  // low half: f[2q]
            f[2 * q] = __uint_as_float(w << 16);
            f[2 * q + 1] = __uint_as_float(w & 0xFFFF0000u);
          }
        }
        float* sc = S + size_t(c * 8) * p.slice_rows * 4;
        if (!first) {
          // ((P_a + P_b) + ...) + P_r in fp32, one rounding per pass
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            f[g * 4 + 0] = __fadd_rn(sv[g].x, f[g * 4 + 0]);
            f[g * 4 + 1] = __fadd_rn(sv[g].y, f[g * 4 + 1]);
            f[g * 4 + 2] = __fadd_rn(sv[g].z, f[g * 4 + 2]);
            f[g * 4 + 3] = __fadd_rn(sv[g].w, f[g * 4 + 3]);
          }
        }
        if (!last) {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            st_global_cg_v4f_hint(sc + size_t(g) * p.slice_rows * 4, f[g * 4], f[g * 4 + 1], f[g * 4 + 2],
                                  f[g * 4 + 3], keep);
        } else if (orow < p.Md) {
          // the destination's row shard: bf16 of the complete sum
#pragma unroll
          for (int g = 0; g < 4; ++g)
            if (col0 + g * 8 < p.N)
              st_global_v4(orowp + col0 + g * 8, pack_bf16x2(f[g * 8], f[g * 8 + 1]),
                           pack_bf16x2(f[g * 8 + 2], f[g * 8 + 3]), pack_bf16x2(f[g * 8 + 4], f[g * 8 + 5]),
                           pack_bf16x2(f[g * 8 + 6], f[g * 8 + 7]));
        }
      }
      if (c_lo >= c_hi) {
        // no columns for this warp (a narrow last column tile): nothing to read
        tc_fence_before();
        __syncwarp();
        if (lane == 0) pair::release_accumulator(bars, acc, rank);
      }
      // this thread's writes of the item are done: the notifier releases the pass once all
      // have arrived (it has handled the item two back, which used the same barrier)
      if (jj >= 2 && !mbar_wait(&cb->notified[acc], (uint32_t(jj >> 1) & 1u) ^ 1u, abort, p.status,
                                p.pipe_timeout_ns, 7))
        break;
      mbar_arrive(&cb->stored[acc]);
    }
  } else if (!kChain && warp < kWarpRed0) {
    // ---------------------------------------------------------------- pushers
    const int wq = warp & 3;                         // TMEM lane quarter of this warp
    const int et = (warp - kWarpEpi0) * 32 + lane;  // 0..127 among pusher threads
    const int row_in_half = wq * 32 + lane;
    // half-slot layout [slice][col/4][row in slice][4]: every slice is one contiguous block,
    // and a warp's store covers runs of slice_rows * 16 contiguous bytes
    const int my_slice = row_in_half / p.slice_rows, my_row = row_in_half % p.slice_rows;
    const size_t my_base = (size_t(my_slice) * 64 * p.slice_rows + my_row) * 4;
    int jj = 0;
    for (int i = pair_id; i < p.num_items; i += npairs, ++jj) {
      const Item it = item_of<false>(p, i);
      const int acc = jj & 1;
      const uint32_t acc_ph = uint32_t(jj >> 1) & 1u;
      // slot free: the R reducers of this half of the tile that last used the slot are done with it
      if (i >= p.ring_items && lane == 0) {
        const int prev_tau = (i - p.ring_items) / p.R;
        for (int j = 0; j < p.R; ++j) {
          const int f = 2 * (prev_tau * p.R + j) + h;
          wait_flag(reduced + f, p.epoch, p.status, p.timeout_ns, uint32_t(2 * p.num_items + f), TL_ERR_TIMEOUT);
        }
      }
      __syncwarp();
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      // all four pusher warps leave together (they meet at a named barrier below)
      if (!named_bar_and(1, kNumEpiThreads, ok)) break;
      tc_fence_after();
      // element offset of this thread's first value in its half-slot (4-byte floats, or
      // 2-byte bf16 values in half the bytes)
      const size_t slot_el = (size_t(i % p.ring_items) * 2 + h) * p.half_floats + my_base;
      const uint64_t stream = l2_policy_evict_first();  // partial lines: written once, read once
      for (int c = 0; c < pair::BN / 32; ++c) {
        if (it.nt * pair::BN + c * 32 >= p.N) break;
        uint32_t v[32];
        tmem_ld_32cols(tmem_base + (uint32_t(wq * 32) << 16) + uint32_t(acc * pair::BN + c * 32), v);
        tmem_ld_wait();
        if (kBf16) {
          uint16_t* slot16 = reinterpret_cast<uint16_t*>(p.slots) + slot_el;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float* f = reinterpret_cast<const float*>(v + g * 4);
            st_global_cg_v2u_hint(slot16 + size_t(c * 8 + g) * p.slice_rows * 4, pack_bf16x2(f[0], f[1]),
                                  pack_bf16x2(f[2], f[3]), stream);
          }
        } else {
          float* slot = p.slots + slot_el;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float* f = reinterpret_cast<const float*>(v + g * 4);
            st_global_cg_v4f_hint(slot + size_t(c * 8 + g) * p.slice_rows * 4, f[0], f[1], f[2], f[3], stream);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) pair::release_accumulator(bars, acc, rank);
      // produce_tile_notify: the barrier orders every pusher thread's writes before
      // thread 0's gpu-scope release, which makes them visible to its acquirers
      named_bar_sync(1, kNumEpiThreads);
      if (et == 0) st_release(arrived + 2 * (it.tau * p.R + it.r) + h, p.epoch);
    }
  } else if (!kChain) {
    // ---------------------------------------------------------------- reducers (this CTA's half)
    const int et = (warp - kWarpRed0) * 32 + lane;  // 0..127 among reducer threads
    for (int i = pair_id; i < p.num_items; i += npairs) {
      const Item it = item_of<false>(p, i);
      // consume_tile_wait / peer_tile_wait: all R partials of this half have arrived
      if (lane == 0) {
        for (int r = 0; r < p.R; ++r) {
          const int f = 2 * (it.tau * p.R + r) + h;
          wait_flag(arrived + f, p.epoch, p.status, p.timeout_ns, uint32_t(f), TL_ERR_TIMEOUT);
        }
      }
      __syncwarp();
      const int s0 = it.j * p.slice_rows;
      const int s_rows = max(0, min(p.slice_rows, pair::HM - s0));
      const int n_cols = min(pair::BN, p.N - it.nt * pair::BN);  // valid columns (multiple of 8)
      const int total = s_rows * (n_cols / 4);                   // float4 elements of the slice
      // rank r's partial was pushed by item tau*R + j(r), j(r) = (r - d - 1 - tau) mod R,
      // into half-slot 2 * ((tau*R + j(r)) mod ring_items) + h
      const uint64_t drop = l2_policy_evict_first();  // each partial line is read once, here
      const int jbase = ((-(it.d + 1 + it.tau)) % p.R + p.R) % p.R;
      const int ring_base = int((size_t(it.tau) * p.R) % size_t(p.ring_items));
      uint16_t* out = p.out[it.d];
      const int orow_base = it.mt * pair::BM + h * pair::HM + s0;
      for (int e0 = et; e0 < total; e0 += kNumRedThreads * QU) {
        int off[QU];  // float offset of each element inside a half-slot, -1 when past the slice
        int orow[QU];
        int ocol[QU];
#pragma unroll
        for (int u = 0; u < QU; ++u) {
          const int e = e0 + u * kNumRedThreads;
          const int c4 = e / s_rows, sr = e - c4 * s_rows;
          off[u] = e < total ? ((it.j * 64 + c4) * p.slice_rows + sr) * 4 : -1;
          orow[u] = orow_base + sr;
          ocol[u] = it.nt * pair::BN + c4 * 4;
        }
        float4 acc4[QU];
        for (int rb = 0; rb < p.R; rb += RB) {
          float4 v[RB][QU];
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) {
            if (rb + rr < p.R) {
              // position rb + rr of the summation order: rank rb + rr, or d + 1 + rb + rr around the ring
              int rank_r = rb + rr;
              if (p.ring_order) {
                rank_r += it.d + 1;
                rank_r -= rank_r >= p.R ? p.R : 0;
                rank_r -= rank_r >= p.R ? p.R : 0;
              }
              int j = jbase + rank_r;
              j -= j >= p.R ? p.R : 0;
              int slot = ring_base + j;
              slot -= slot >= p.ring_items ? p.ring_items : 0;
              const size_t base_el = (size_t(slot) * 2 + h) * p.half_floats;
              if (kBf16) {
                // raw words now, widened below, so every load of the batch is in flight together
                const uint16_t* src16 = reinterpret_cast<const uint16_t*>(p.slots) + base_el;
#pragma unroll
                for (int u = 0; u < QU; ++u)
                  if (off[u] >= 0) {
                    const uint2 w = ld_global_cg_v2u_hint(src16 + off[u], drop);
                    v[rr][u] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), 0.f, 0.f);
                  }
              } else {
                const float* src = p.slots + base_el;
#pragma unroll
                for (int u = 0; u < QU; ++u)
                  if (off[u] >= 0) v[rr][u] = ld_global_cg_v4f_hint(src + off[u], drop);
              }
            }
          }
          if (kBf16) {
#pragma unroll
            for (int rr = 0; rr < RB; ++rr)
#pragma unroll
              for (int u = 0; u < QU; ++u)
                v[rr][u] = unpack_bf16x4(make_uint2(__float_as_uint(v[rr][u].x), __float_as_uint(v[rr][u].y)));
          }
          // fixed order (rank order, or ring order): acc = ((P_a + P_b) + P_c) + ...
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) {
            if (rb + rr < p.R) {
#pragma unroll
              for (int u = 0; u < QU; ++u) {
                if (rb + rr == 0) {
                  acc4[u] = v[rr][u];
                } else {
                  acc4[u].x = __fadd_rn(acc4[u].x, v[rr][u].x);
                  acc4[u].y = __fadd_rn(acc4[u].y, v[rr][u].y);
                  acc4[u].z = __fadd_rn(acc4[u].z, v[rr][u].z);
                  acc4[u].w = __fadd_rn(acc4[u].w, v[rr][u].w);
                }
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < QU; ++u) {
          if (off[u] >= 0 && orow[u] < p.Md) {
            uint2 pk;
            pk.x = pack_bf16x2(acc4[u].x, acc4[u].y);
            pk.y = pack_bf16x2(acc4[u].z, acc4[u].w);
            *reinterpret_cast<uint2*>(out + size_t(orow[u]) * p.N + ocol[u]) = pk;
          }
        }
      }
      // slice j of this half of tile tau is read: release its "reduced" flag (slot-free barrier)
      named_bar_sync(2, kNumRedThreads);
      if (et == 0) st_release(reduced + 2 * (it.tau * p.R + it.j) + h, p.epoch);
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
    }
  }
  pair::teardown(bars, warp, tmem_base);
}

int rs_num_tiles(int R, int M, int N) {
  const int Md = M / R;
  return cdiv(Md, pair::BM) * cdiv(N, pair::BN) * R;
}

// CTA pairs of a launch: at most half the SMs, at most one per item.
int rs_pairs(int num_items, int sm_count) { return std::max(1, std::min(sm_count / 2, num_items)); }

// Items in the ring of receive slots: three waves of pairs, or every item when fewer.
int rs_ring_items(int num_items, int pairs) { return std::min(num_items, 3 * pairs); }

int current_sm_count() {
  DeviceInfo di{};
  return device_info(&di) == TL_OK ? di.sm_count : 0;
}

// floats of one half-slot: R slices of ceil(128/R) rows x 256 columns
int rs_half_floats(int R) { return R * cdiv(pair::HM, R) * pair::BN; }

size_t rs_slots_bytes(int ring_items, int R) { return size_t(ring_items) * 2 * rs_half_floats(R) * sizeof(float); }

// Validate the arguments shared by both entry points.
tl_status rs_check(const tl_gemm_rs_args* a, const char* who) {
  if (!a) return fail(TL_ERR_INVALID, "%s: NULL args", who);
  if (a->R < 1 || a->R > RS_MAX_RANKS)
    return fail(a->R > RS_MAX_RANKS ? TL_ERR_UNSUPPORTED : TL_ERR_INVALID, "%s: R=%d outside 1..%d", who, a->R,
                RS_MAX_RANKS);
  if (a->M < a->R || a->M % a->R) return fail(TL_ERR_INVALID, "%s: M=%d must be a positive multiple of R", who, a->M);
  if (a->K_r < 1 || a->N < 1) return fail(TL_ERR_INVALID, "%s: empty shape", who);
  if (a->K_r % 8 || a->N % 8)
    return fail(TL_ERR_UNSUPPORTED, "%s: K_r (%d) and N (%d) must be multiples of 8", who, a->K_r, a->N);
  if (!a->A || !a->B || !a->out) return fail(TL_ERR_INVALID, "%s: NULL pointer argument", who);
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "%s: epoch must be nonzero", who);
  if (a->options & ~(TL_RS_BF16_PARTIALS | TL_RS_RING_ORDER))
    return fail(TL_ERR_INVALID, "%s: unknown options 0x%x", who, a->options);
  for (int r = 0; r < a->R; ++r) {
    if (!a->A[r] || !a->B[r] || !a->out[r] || !aligned16(a->A[r]) || !aligned16(a->B[r]) || !aligned16(a->out[r]))
      return fail(TL_ERR_INVALID, "%s: rank %d pointer NULL or not 16-byte aligned", who, r);
  }
  if ((long long)rs_num_tiles(a->R, a->M, a->N) * a->R * 4 > (1ll << 30))
    return fail(TL_ERR_UNSUPPORTED, "%s: too many tiles", who);
  return TL_OK;
}

// bytes of the chain schedule's running sums: one fp32 tile per output tile
size_t rs_chain_bytes(int R, int M, int N) { return size_t(rs_num_tiles(R, M, N)) * 2 * rs_half_floats(R) * sizeof(float); }

// Fill the kernel parameters and launch.  chain: the chain schedule (the workspace
// holds rs_chain_bytes), else push and reduce through a ring of receive slots.
tl_status rs_launch(RsParams* p, const tl_gemm_rs_args* a, float* slots, uint32_t* flags, uint32_t* status,
                    int sm_count, cudaStream_t st, bool chain) {
  for (int r = 0; r < a->R; ++r) {
    if (tl_status s = make_map_bf16(&p->map_a[r], a->A[r], a->M, a->K_r, size_t(a->K_r) * 2, pair::HM, pair::BK))
      return s;
    if (tl_status s = make_map_bf16(&p->map_b[r], a->B[r], a->K_r, a->N, size_t(a->N) * 2, pair::BK, 64)) return s;
    p->out[r] = static_cast<uint16_t*>(a->out[r]);
  }
  p->slots = slots;
  p->flags = flags;
  p->status = status;
  p->trace = a->trace;
  p->timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
  p->pipe_timeout_ns = 2 * p->timeout_ns + 1000000000ull;
  p->R = a->R;
  p->M = a->M;
  p->Md = a->M / a->R;
  p->K = a->K_r;
  p->N = a->N;
  p->Mt_d = cdiv(p->Md, pair::BM);
  p->Nt = cdiv(a->N, pair::BN);
  p->KB = cdiv(a->K_r, pair::BK);
  p->num_tiles = rs_num_tiles(a->R, a->M, a->N);
  p->num_items = p->num_tiles * a->R;
  p->slice_rows = cdiv(pair::HM, a->R);
  p->half_floats = rs_half_floats(a->R);
  p->epoch = a->epoch;
  p->ring_order = (a->options & TL_RS_RING_ORDER) ? 1 : 0;
  const int pairs = rs_pairs(p->num_items, sm_count);
  p->ring_items = rs_ring_items(p->num_items, pairs);
  void* args[] = {p};
  const bool bf16 = (a->options & TL_RS_BF16_PARTIALS) != 0;
  const void* kernel = chain ? (bf16 ? reinterpret_cast<const void*>(&gemm_rs_kernel<true, true>)
                                     : reinterpret_cast<const void*>(&gemm_rs_kernel<false, true>))
                             : (bf16 ? reinterpret_cast<const void*>(&gemm_rs_kernel<true, false>)
                                     : reinterpret_cast<const void*>(&gemm_rs_kernel<false, false>));
  return launch_coop(kernel, 2 * pairs, chain ? RS_CHAIN_THREADS : RS_THREADS, RS_SMEM_BYTES, st, args, 2);
}

}  // namespace
}  // namespace tl

extern "C" size_t tl_gemm_rs_workspace_size(int R, int M, int N) {
  if (R < 1 || M < R || N < 1 || M % R) return 0;
  const int items = tl::rs_num_tiles(R, M, N) * R;
  const int sms = tl::current_sm_count();
  // without a usable device, size for every item (always enough)
  const int ring = sms >= 2 ? tl::rs_ring_items(items, tl::rs_pairs(items, sms)) : items;
  return std::max(tl::rs_slots_bytes(ring, R), tl::rs_chain_bytes(R, M, N));
}

extern "C" int tl_gemm_rs_num_flags(int R, int M, int N) {
  if (R < 1 || M < R || N < 1 || M % R) return -1;
  return 4 * tl::rs_num_tiles(R, M, N) * R;  // arrival and reduced flags for both halves
}

extern "C" tl_status tl_gemm_rs(const tl_gemm_rs_args* a, void* stream) {
  using namespace tl;
  if (tl_status s = rs_check(a, "tl_gemm_rs")) return s;
  if (!a->workspace || !a->signals) return fail(TL_ERR_INVALID, "tl_gemm_rs: NULL workspace or signals");
  if (!aligned16(a->workspace)) return fail(TL_ERR_INVALID, "tl_gemm_rs: workspace not 16-byte aligned");
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  const size_t need = tl_gemm_rs_workspace_size(a->R, a->M, a->N);
  if (a->workspace_bytes < need)
    return fail(TL_ERR_INVALID, "tl_gemm_rs: workspace %zu bytes, need %zu", a->workspace_bytes, need);
  const int nflags = tl_gemm_rs_num_flags(a->R, a->M, a->N);
  if (a->signals->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_gemm_rs: signals hold %d flags, need %d", a->signals->num_flags, nflags);
  if (a->signals->device != di.device) return fail(TL_ERR_INVALID, "tl_gemm_rs: signals belong to another device");
  RsParams* p = new (std::nothrow) RsParams;
  if (!p) return fail(TL_ERR_INTERNAL, "out of host memory");
  std::memset(p, 0, sizeof(RsParams));
  const tl_status st = rs_launch(p, a, static_cast<float*>(a->workspace), a->signals->flags, a->signals->status,
                                 di.sm_count, (cudaStream_t)stream, true);
  delete p;
  return st;
}

// ---------------------------------------------------------------- GEMM-RS without allocation
// Some callers cannot allocate device memory: code that runs while a custom
// allocator owns the device, inside a runtime that forbids cudaMalloc on its
// hot path, or before any allocator exists.  tl_gemm_rs_noalloc serves them
// with the GEMM-RS kernel above, taking its scratch (flags, status word and
// fp32 receive slots) from a fixed file-scope device array instead of a
// caller-provided workspace and a tl_signals object.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // TL_GEMM_RS_NOALLOC_MAX_BYTES
constexpr size_t kNoAllocHeader = 256;                       // status words, then flags

static_assert(kNoAllocScratchBytes == size_t(TL_GEMM_RS_NOALLOC_MAX_BYTES), "header and library disagree");

// Held by every GPU that loads this library, until the process exits.
static __device__ __align__(256) uint8_t g_rs_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array, looked up once per device with that
// device current.  In host code the array's name is only a host-side stand-in.
// The address is kept until the process exits; a cudaDeviceReset reloads the
// module and makes it stale, which the header rules out.
tl_status noalloc_scratch(int dev, uint8_t** out) {
  static std::mutex mu;
  static uint8_t* addr[64] = {};
  if (dev < 0 || dev >= 64) return tl::fail(TL_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_rs_noalloc_scratch);
    if (e != cudaSuccess) return tl::cuda_ok(e, "cudaGetSymbolAddress(GEMM-RS scratch)");
    addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = addr[dev];
  return TL_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

namespace {
size_t noalloc_scratch_needed(int R, int M, int N, int sm_count);
}  // namespace

extern "C" tl_status tl_gemm_rs_noalloc(const tl_gemm_rs_args* a, uint32_t* dev_status, void* stream) {
  using namespace tl;
  if (tl_status s = rs_check(a, "tl_gemm_rs_noalloc")) return s;
  if (a->workspace || a->workspace_bytes || a->signals)
    return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: workspace and signals must be NULL (the scratch is static)");
  if (dev_status && !aligned16(dev_status)) return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: dev_status alignment");
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  const size_t need = noalloc_scratch_needed(a->R, a->M, a->N, di.sm_count);
  if (need == 0 || need > kNoAllocScratchBytes)
    return fail(TL_ERR_UNSUPPORTED,
                "tl_gemm_rs_noalloc: R=%d M=%d N=%d needs %zu bytes of scratch; the static scratch holds %zu "
                "(use tl_gemm_rs with a caller-allocated workspace)",
                a->R, a->M, a->N, need, kNoAllocScratchBytes);
  uint8_t* scratch = nullptr;
  if (tl_status s = noalloc_scratch(di.device, &scratch)) return s;

  const int nflags = tl_gemm_rs_num_flags(a->R, a->M, a->N);
  uint32_t* status = reinterpret_cast<uint32_t*>(scratch);
  uint32_t* flags = reinterpret_cast<uint32_t*>(scratch + kNoAllocHeader);
  float* slots = reinterpret_cast<float*>(scratch + align_up(kNoAllocHeader + size_t(nflags) * 4, 256));
  cudaStream_t st = (cudaStream_t)stream;
  // the array keeps the previous call's flags: clear them (and the internal status word)
  if (tl_status s = cuda_ok(cudaMemsetAsync(scratch, 0, kNoAllocHeader + size_t(nflags) * 4, st),
                            "cudaMemsetAsync(GEMM-RS scratch flags)"))
    return s;
  RsParams p;  // on the stack: no heap allocation on this path
  std::memset(&p, 0, sizeof(RsParams));
  // the fixed scratch holds a ring of receive slots: the push-and-reduce schedule (the same bits)
  return rs_launch(&p, a, slots, flags, dev_status ? dev_status : status, di.sm_count, st, false);
}

namespace {
size_t noalloc_scratch_needed(int R, int M, int N, int sm_count) {
  if (R < 1 || M < R || N < 1 || M % R || sm_count < 2) return 0;
  const int nitems = tl::rs_num_tiles(R, M, N) * R;
  const size_t nflags = 4 * size_t(nitems);
  const int ring = tl::rs_ring_items(nitems, tl::rs_pairs(nitems, sm_count));
  return align_up(kNoAllocHeader + nflags * 4, 256) + tl::rs_slots_bytes(ring, R);
}
}  // namespace
