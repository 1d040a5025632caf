// tl_moe.cu -- AllGather + grouped MoE GEMM at tile granularity.
//
// TileLink talk summary ("TileLink: Generating Efficient Compute-Communication
// Overlapping Kernels using Tile-Centric Primitives"):
//  * Key Findings / Experimental Setup & Results -- the MoE layer overlaps an
//    AllGather of tokens with a GroupGEMM over experts (this file covers that
//    part; ReduceScatter, TopK-reduce and scatter of the layer are not here).
//  * Technical Deep Dive -- for dynamic workloads the tile -> rank/barrier
//    dependencies come from lookup tables built from the routing and passed
//    to the kernel.
//
// Two stream-ordered launches, the second with programmatic dependent launch (its
// launch is set up while the first runs, and it waits for the first to finish
// before it reads the tables):
//  1. moe_route_kernel (a cluster of 8 CTAs): histogram of topk_ids over experts,
//     exclusive scan, stable counting sort of the (token, slot) pairs by expert
//     (perm and its inverse), then the tile table -- per 256-row tile its
//     expert, first sorted row, rows, lowest and highest producer barrier and
//     source-rank mask -- and the consumer tile order.
//  2. moe_gemm_kernel (persistent CTA pairs, one CTA per SM): copy warps move
//     the token rows into `sorted_tokens` with bulk TMA copies -- pull mode
//     (default): chunks of rows_per_barrier sorted rows in sorted order, each row
//     fetched from its token's shard, one flag per chunk; push mode: each
//     shard's tokens, in the order self, self+1, ..., scattered to their k sorted
//     positions, one flag per chunk of a shard's tokens.  The TMA warps of each
//     256-row expert tile acquire the flags of its barrier range, then a
//     tcgen05.mma.cta_group::2 grouped GEMM multiplies the tile's sorted rows by
//     its expert's weight.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "tl_epilogue.cuh"
#include "tl_internal.h"
#include "tl_moe_ws.cuh"
#include "tl_pair.cuh"

namespace tl {
namespace {

constexpr int MOE_MAX_E = 64;
constexpr int MOE_MAX_R = 32;
constexpr int MOE_MAX_TILES = 8192;
constexpr int ROUTE_THREADS = 1024;
constexpr uint32_t ROUTE_CTAS = 8;  // the routing kernel's cluster
constexpr int ROUTE_WARPS = ROUTE_THREADS / 32;
constexpr int kWarpCopy = 6;
constexpr int MOE_THREADS = 7 * 32;
constexpr int TM = pair::BM;  // rows of an expert tile
// shared memory: the pipeline stages, the copy warp's staging (three buffers),
// then one 32 x 32 Y box per epilogue warp for the TMA-store epilogue
constexpr int MOE_COPY_NBUF = 3;
constexpr uint32_t MOE_SMEM_COPY = pair::SMEM_END;
constexpr uint32_t MOE_SMEM_CSTAGE = MOE_SMEM_COPY + MOE_COPY_NBUF * COPY_CHUNK;
constexpr uint32_t MOE_SMEM_BARS = MOE_SMEM_CSTAGE + kNumEpiWarps * C_BOX_BYTES;
// the copy warp's tables: the shard pointers, and the tokens of the next MOE_TOKB sorted rows
constexpr int MOE_TOKB = 16;
constexpr uint32_t MOE_SMEM_XS = (MOE_SMEM_BARS + uint32_t(sizeof(pair::Bars)) + 15u) / 16u * 16u;
constexpr uint32_t MOE_SMEM_BYTES = MOE_SMEM_XS + MOE_MAX_R * 8 + MOE_TOKB * 4 + 1024;

static_assert(TM == MOE_TILE_ROWS, "expert tiles are CTA-pair tiles");


struct RouteParams {
  const int32_t* topk;    // [T, k]
  int32_t* perm;          // [P] sorted position -> token*k + slot
  int32_t* offsets;       // [E+1]
  int32_t* ws;            // workspace
  uint32_t* status;
  int32_t T, k, E, R, T_r, rpb, bpr, self, max_tiles, pull;
  int32_t k_shift;  // log2(k) when k is a power of two, else -1
};

// Lanes of `am` whose expert equals this lane's (e < 64): one ballot per bit of e.
__device__ __forceinline__ unsigned same_expert_lanes(unsigned am, int e) {
  unsigned peers = am;
#pragma unroll
  for (int b = 0; b < 6; ++b) {
    const bool bit = (e >> b) & 1;
    const unsigned bb = __ballot_sync(am, bit);
    peers &= bit ? bb : ~bb;
  }
  return peers;
}

// Routing on a cluster of ROUTE_CTAS CTAs: CTA c owns the c-th contiguous range
// of the P = T*k (token, slot) pairs, and its warps own consecutive sub-ranges
// (the experts of a warp's first ROUTE_CACHE rounds of 32 pairs stay in registers
// between the two passes over them).
//  1. per-warp expert counts over the warp's pairs;
//  2. (cluster barrier) every CTA reads every CTA's per-expert totals from
//     distributed shared memory: expert offsets (exclusive scan), tile offsets
//     and, for a stable sort, the base of each of its warps per expert = offset +
//     the counts of every lower CTA and every lower warp of this CTA; stable
//     scatter of the pairs (perm and its inverse, in global memory), each pair
//     also marking its tile's source rank and token barrier in shared memory;
//  3. (cluster barrier) the tile table, one tile per warp across the cluster,
//     the masks and barrier ranges combined from every CTA's shared memory,
//     the tile keys gathered in CTA 0's shared memory;
//  4. (cluster barrier) CTA 0 ranks the tiles by (key, index): the consumer order.
constexpr int ROUTE_CACHE = 4;

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

__global__ void __launch_bounds__(ROUTE_THREADS, 1) moe_route_kernel(const RouteParams p) {
  extern __shared__ int32_t sm[];
  const int E = p.E;
  int32_t* cnt = sm;                       // [ROUTE_WARPS][E] per-warp counts, then per-warp bases
  int32_t* ctot = cnt + ROUTE_WARPS * E;   // [E] this CTA's per-expert totals (read by the cluster)
  int32_t* s_off = ctot + E;               // [E+1] expert offsets
  int32_t* s_toff = s_off + (E + 1);       // [E+1] first tile of each expert
  int32_t* s_below = s_toff + (E + 1);     // [E] pairs of each expert in the lower CTAs of the cluster
  int32_t* s_key = s_below + E;            // [max_tiles] tile keys (CTA 0)
  // per tile, over this CTA's pairs: source-rank mask, lowest and highest token barrier
  int32_t* s_mask = s_key + p.max_tiles;
  int32_t* s_blo = s_mask + p.max_tiles;
  int32_t* s_bhi = s_blo + p.max_tiles;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank();
  // the grouped GEMM's launch may proceed now; it waits for this kernel before reading the tables
  pdl_launch_dependents();
  const int P = p.T * p.k;
  const int per_cta = ((P + ROUTE_CTAS - 1) / ROUTE_CTAS + 31) / 32 * 32;
  const int c0 = min(P, int(crank) * per_cta), c1 = min(P, c0 + per_cta);
  const int per_warp = ((c1 - c0 + ROUTE_WARPS - 1) / ROUTE_WARPS + 31) / 32 * 32;
  const int q0 = min(c1, c0 + warp * per_warp), q1 = min(c1, q0 + per_warp);
  int32_t* tiles = p.ws + ws_tiles(p.max_tiles);
  int32_t* order = p.ws + ws_order(p.max_tiles);
  int32_t* inv = p.ws + ws_inv(p.max_tiles);

  // the experts of the warp's first rounds, every load in flight together
  int ecache[ROUTE_CACHE];
#pragma unroll
  for (int i = 0; i < ROUTE_CACHE; ++i) {
    const int q = q0 + i * 32 + lane;
    ecache[i] = q < q1 ? p.topk[q] : 0;
  }
  for (int i = tid; i < ROUTE_WARPS * E; i += ROUTE_THREADS) cnt[i] = 0;
  for (int t = tid; t < p.max_tiles; t += ROUTE_THREADS) {
    s_mask[t] = 0;
    s_blo[t] = 0x7fffffff;
    s_bhi[t] = -1;
  }
  __syncthreads();
  // 1. per-warp histograms over contiguous ranges of pairs
  auto count = [&](int e, int base) {
    const int q = base + lane;
    const bool act = q < q1;
    if (act && (e < 0 || e >= E)) {
      record_error(p.status, TL_ERR_INVALID, uint32_t(q), uint32_t(e), uint32_t(E));
      e = min(max(e, 0), E - 1);
    }
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const unsigned peers = same_expert_lanes(am, e);
      if (lane == __ffs(peers) - 1) cnt[warp * E + e] += __popc(peers);
    }
    __syncwarp();
  };
#pragma unroll
  for (int i = 0; i < ROUTE_CACHE; ++i)
    if (q0 + i * 32 < q1) count(ecache[i], q0 + i * 32);
  for (int base = q0 + ROUTE_CACHE * 32; base < q1; base += 32)
    count(base + lane < q1 ? p.topk[base + lane] : 0, base);
  __syncthreads();
  for (int e = tid; e < E; e += ROUTE_THREADS) {
    int c = 0;
    for (int w = 0; w < ROUTE_WARPS; ++w) c += cnt[w * E + e];
    ctot[e] = c;
  }
  cluster_sync();
  // 2. expert totals and offsets from every CTA's totals, then the tile offsets
  if (warp == 0) {
    // one lane per expert (E <= 64 in two rounds): totals, then a warp scan for the offsets
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int tot = 0, below = 0;
      if (e < E) {
        for (uint32_t c = 0; c < ROUTE_CTAS; ++c) {
          const int v = int(ld_shared_cluster_u32(map_to_rank(&ctot[e], c)));
          tot += v;
          below += c < crank ? v : 0;
        }
      }
      const int incl = warp_incl_scan(tot, lane);
      if (e < E) {
        s_off[e] = carry + incl - tot;
        s_below[e] = below;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_off[E] = carry;
  }
  __syncthreads();
  // the base of each warp per expert: the expert's offset, then the counts of the lower
  // CTAs, then those of the lower warps of this CTA
  for (int e = tid; e < E; e += ROUTE_THREADS) {
    int run = s_off[e] + s_below[e];
    for (int w = 0; w < ROUTE_WARPS; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
  }
  // tiles per expert and their offsets (every CTA, from the same totals)
  if (tid == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_toff[e] = acc;
      acc += (s_off[e + 1] - s_off[e] + TM - 1) / TM;
    }
    s_toff[E] = acc;
    if (crank == 0) {
      p.ws[0] = min(acc, p.max_tiles);
      if (acc > p.max_tiles)
        record_error(p.status, TL_ERR_INTERNAL, 0xFFFE0000u, uint32_t(acc), uint32_t(p.max_tiles));
    }
  }
  __syncthreads();
  // stable scatter: pairs keep their (token, slot) order inside an expert; each pair also
  // marks its tile's source rank and token barrier range (this CTA's share of the table)
  auto scatter = [&](int e_raw, int base) {
    const int q = base + lane;
    const bool act = q < q1;
    const int e = act ? min(max(e_raw, 0), E - 1) : 0;
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const unsigned peers = same_expert_lanes(am, e);
      const int pos = cnt[warp * E + e] + __popc(peers & ((1u << lane) - 1u));
      p.perm[pos] = q;
      inv[q] = pos;
      const int tok = p.k_shift >= 0 ? (q >> p.k_shift) : q / p.k;
      const int r = tok / p.T_r;
      const int b = r * p.bpr + (tok - r * p.T_r) / p.rpb;
      const int t = s_toff[e] + (pos - s_off[e]) / TM;
      if (t < p.max_tiles) {
        atomicOr(reinterpret_cast<unsigned*>(&s_mask[t]), 1u << r);
        atomicMin(&s_blo[t], b);
        atomicMax(&s_bhi[t], b);
      }
      __syncwarp(am);
      if (lane == __ffs(peers) - 1) cnt[warp * E + e] += __popc(peers);
    }
    __syncwarp();
  };
#pragma unroll
  for (int i = 0; i < ROUTE_CACHE; ++i)
    if (q0 + i * 32 < q1) scatter(ecache[i], q0 + i * 32);
  for (int base = q0 + ROUTE_CACHE * 32; base < q1; base += 32)
    scatter(base + lane < q1 ? p.topk[base + lane] : 0, base);
  if (crank == 0)
    for (int e = tid; e <= E; e += ROUTE_THREADS) p.offsets[e] = s_off[e];
  // every CTA's share of the per-tile masks and barrier ranges is complete
  cluster_sync();
  // 3. the tile table, one warp per tile across the cluster: rows of a tile are one
  //    expert's, tokens ascending
  const int ntiles = min(s_toff[E], p.max_tiles);
  for (int t = int(crank) * ROUTE_WARPS + warp; t < ntiles; t += ROUTE_CTAS * ROUTE_WARPS) {
    int lo_e = 0, hi_e = E - 1;  // last expert whose first tile <= t (empty experts are skipped over)
    while (lo_e < hi_e) {
      const int mid = (lo_e + hi_e + 1) >> 1;
      if (s_toff[mid] <= t) lo_e = mid; else hi_e = mid - 1;
    }
    const int e = lo_e;
    const int row0 = s_off[e] + (t - s_toff[e]) * TM;
    const int rows = min(TM, s_off[e + 1] - row0);
    // the tile's source ranks and barrier range: every CTA's share, through distributed
    // shared memory (lane c reads CTA c's)
    uint32_t mask = 0;
    int blo = 0x7fffffff, bhi = -1;
    if (lane < int(ROUTE_CTAS)) {
      mask = ld_shared_cluster_u32(map_to_rank(&s_mask[t], uint32_t(lane)));
      blo = int(ld_shared_cluster_u32(map_to_rank(&s_blo[t], uint32_t(lane))));
      bhi = int(ld_shared_cluster_u32(map_to_rank(&s_bhi[t], uint32_t(lane))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mask |= __shfl_xor_sync(0xffffffffu, mask, o);
      blo = min(blo, __shfl_xor_sync(0xffffffffu, blo, o));
      bhi = max(bhi, __shfl_xor_sync(0xffffffffu, bhi, o));
    }
    if (lane == 0) {
      int key = 0;
      if (p.pull) {
        // pull: the tile's own chunks of sorted rows; chunks arrive in sorted order
        blo = row0 / p.rpb;
        bhi = (row0 + rows - 1) / p.rpb;
        key = bhi;
      } else {
        // push: latest arrival position among the source barriers in [blo, bhi];
        // barrier (r, c) arrives at ((r - self) mod R) * bpr + c
        for (int r = blo / p.bpr; r <= bhi / p.bpr; ++r) {
          const int c_hi = (r == bhi / p.bpr) ? bhi % p.bpr : p.bpr - 1;
          key = max(key, ((r - p.self + p.R) % p.R) * p.bpr + c_hi);
        }
      }
      int32_t* tr = tiles + 6 * t;
      tr[0] = e;
      tr[1] = row0;
      tr[2] = rows;
      tr[3] = blo;
      tr[4] = bhi;
      tr[5] = int32_t(mask);
      st_shared_cluster_u32(map_to_rank(&s_key[t], 0), uint32_t(key));
    }
  }
  cluster_sync();
  // 4. consumer order: tiles by (key, index)
  if (crank == 0) {
    for (int t = tid; t < ntiles; t += ROUTE_THREADS) {
      const int kt = s_key[t];
      int rank = 0;
      for (int u = 0; u < ntiles; ++u) {
        const int ku = s_key[u];
        rank += (ku < kt) || (ku == kt && u < t);
      }
      order[rank] = t;
    }
  }
}

struct MoeParams {
  CUtensorMap map_a;               // sorted tokens [P, H]
  CUtensorMap map_y;               // Y [P, N], box 32 x 32, 64-byte swizzle (TMA stores)
  CUtensorMap map_w[MOE_MAX_E];    // W_e [H, N]
  const uint8_t* x[MOE_MAX_R];     // shards [T_r, H]
  uint8_t* sorted;
  uint16_t* Y;
  const int32_t* ws;
  uint32_t* flags;
  uint32_t* status;
  int32_t* trace;
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int32_t R, self, T_r, H, N, E, k, rpb, bpr, Nt, KB, num_items, max_tiles, pull, P;
  uint32_t epoch;
  const int32_t* perm;
  int32_t hold_first, hold_count;  // chunks the copy warps move last (tl_test_hold_chunks)
  uint64_t hold_ns;
};

// Work item q of the grouped GEMM: unit q in consumer order (expert tile order[q / Nt],
// 256-column tile q % Nt).  A last column tile of at most 128 columns runs as an N = 128
// product (narrow).
struct MoeWork {
  int t, n, col0;
  bool narrow;
};

__device__ __forceinline__ MoeWork moe_work(const MoeParams& p, const int32_t* order, int q) {
  MoeWork w;
  w.t = order[q / p.Nt];
  w.n = q % p.Nt;
  w.col0 = w.n * pair::BN;
  w.narrow = p.N - w.col0 <= pair::HN;
  return w;
}

__global__ void __launch_bounds__(MOE_THREADS, 1) moe_gemm_kernel(const __grid_constant__ MoeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  pair::Bars* bars = reinterpret_cast<pair::Bars*>(smem + MOE_SMEM_BARS);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const uint32_t rank = cluster_ctarank();
  const int h = int(rank);
  const int pair_id = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  const int32_t* tiles = p.ws + ws_tiles(p.max_tiles);
  const int32_t* order = p.ws + ws_order(p.max_tiles);
  const int32_t* inv = p.ws + ws_inv(p.max_tiles);
  const uint32_t tmem_base = pair::setup(bars, warp);
  // programmatic dependent launch: the routing kernel's tables are complete and visible
  // only after this
  pdl_wait_previous();
  const int num_work = p.ws[0] * p.Nt;
  volatile uint32_t* abort = &bars->abort;
  const int my_work = pair_id < num_work ? (num_work - 1 - pair_id) / npairs + 1 : 0;

  if (warp == kWarpTma) {
    // ---------------------------------------------------------------- TMA producer (this CTA's 128 rows)
    pair::Producer prod;
    int last_t = -1;
    for (int q = pair_id; q < num_work; q += npairs) {
      const MoeWork w = moe_work(p, order, q);
      const int t = w.t;
      const int32_t* tr = tiles + 6 * t;
      const int e = tr[0], row0 = tr[1];
      if (t != last_t) {
        // consume_tile_wait through the lookup table: every barrier in [lo, hi]
        for (int id = tr[3] + lane; id <= tr[4]; id += 32)
          wait_flag(p.flags + id, p.epoch, p.status, p.timeout_ns, uint32_t(id), TL_ERR_TIMEOUT);
      }
      last_t = t;
      __syncwarp();
      if (lane == 0) {
        if (p.trace && rank == 0) p.trace[q] = t * p.Nt + w.n;
        fence_proxy_async_global();
        const int b_x = w.col0 + h * (w.narrow ? pair::HN / 2 : pair::HN);
        for (int kb = 0; kb < p.KB; ++kb)
          if (!prod.load(smem, bars, rank, &p.map_a, kb * pair::BK, row0 + h * pair::HM, &p.map_w[e], b_x,
                         kb * pair::BK, abort, p.status, p.pipe_timeout_ns, w.narrow))
            break;
      }
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      pair::mma_loop(smem, bars, tmem_base, my_work, p.KB, abort, p.status, p.pipe_timeout_ns,
                     [&](int j) { return moe_work(p, order, pair_id + j * npairs).narrow; });
    }
    __syncwarp();
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kNumEpiWarps) {
    // ---------------------------------------------------------------- epilogue: rows of this expert only
    const int wq = warp & 3;
    uint8_t* cbox = smem + MOE_SMEM_CSTAGE + uint32_t(wq) * C_BOX_BYTES;
    int j = 0;
    for (int q = pair_id; q < num_work; q += npairs, ++j) {
      const int acc = j & 1;
      const uint32_t acc_ph = uint32_t(j >> 1) & 1u;
      const MoeWork w = moe_work(p, order, q);
      const int32_t* tr = tiles + 6 * w.t;
      const int row0 = tr[1], rows = tr[2];
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int lr = h * pair::HM + wq * 32 + lane;
      const bool row_ok = lr < rows;
      // this warp's 32 rows: all of this expert's (one TMA store per 32 x 32 box), some of them
      // (plain stores: the rows after them belong to the next tile), or none
      const int box_r0 = h * pair::HM + wq * 32;
      const bool whole = box_r0 + 32 <= rows;
      const int nchunks = (w.narrow ? pair::HN : pair::BN) / 32;
      for (int c = 0; c < nchunks; ++c) {
        const int col0 = w.col0 + c * 32;
        if (col0 >= p.N) break;
        uint32_t v[32];
        tmem_ld_32cols(tmem_base + (uint32_t(wq * 32) << 16) + uint32_t(acc * pair::BN + c * 32), v);
        tmem_ld_wait();
        if (whole) {
          store_box_bf16(&p.map_y, cbox, 1, lane, v, col0, row0 + box_r0);
        } else if (row_ok) {
          uint16_t* yrow = p.Y + size_t(row0 + lr) * p.N + col0;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (col0 + g * 8 < p.N) {
              const float* f = reinterpret_cast<const float*>(v + g * 8);
              st_global_v4(yrow + g * 8, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                           pack_bf16x2(f[6], f[7]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) pair::release_accumulator(bars, acc, rank);
    }
    if (lane == 0) bulk_wait<0>();  // every store of this warp is complete
    __syncwarp();
  } else if (warp == kWarpCopy) {
    // ---------------------------------------------------------------- AllGather + local scatter
    // shard pointers in shared memory (a parameter array read with a varying index is slow)
    const uint8_t** xs = reinterpret_cast<const uint8_t**>(smem + MOE_SMEM_XS);
    int32_t* stok = reinterpret_cast<int32_t*>(smem + MOE_SMEM_XS + MOE_MAX_R * 8);
    if (lane < p.R) xs[lane] = p.x[lane];
    __syncwarp();
    if (lane == 0) {
      uint8_t* stage = smem + MOE_SMEM_COPY;
      int tb_base = 0, tb_end = 0;  // pull: sorted rows whose tokens are in stok
      const uint32_t row_bytes = uint32_t(p.H) * 2u;
      const int pieces = int((row_bytes + COPY_CHUNK - 1) / COPY_CHUNK);
      uint32_t seq = 0;  // pieces loaded by this CTA: buffer seq % NBUF, parity (seq / NBUF) & 1
      const uint64_t pol_keep = l2_policy_evict_last();
      bool dead = false;
      const uint64_t t0 = now_ns();
      // the flag an item releases; held items (a test facility) go after the others
      auto flag_of = [&](int it) { return p.pull ? it : ((p.self + it / p.bpr) % p.R) * p.bpr + it % p.bpr; };
      auto held = [&](int it) {
        return p.hold_count > 0 && flag_of(it) >= p.hold_first && flag_of(it) < p.hold_first + p.hold_count;
      };
      bool any_held = false;
      for (int pass = 0; pass < 2 && !dead; ++pass) {
        if (pass == 1) {
          if (!any_held) break;
          while (now_ns() - t0 < p.hold_ns && !*abort && ld_volatile(p.status) == 0u) __nanosleep(1000);
        }
        for (int it = blockIdx.x; it < p.num_items && !dead; it += gridDim.x) {
          if (held(it) != (pass == 1)) {
            any_held = any_held || held(it);
            continue;
          }
          // push: item = (shard r, chunk c of its tokens), each token scattered to its k sorted rows;
          // pull: item = chunk of rpb sorted rows, each gathered from its token's shard
          const int jj = it / p.bpr, c = it % p.bpr;
          const int r = (p.self + jj) % p.R;  // push: shards self, self+1, ...
          const int t0 = p.pull ? it * p.rpb : c * p.rpb;
          const int t1 = p.pull ? min(p.P, t0 + p.rpb) : min(p.T_r, t0 + p.rpb);
          const int nunits = (t1 - t0) * pieces;
          int issued = 0, stored = 0;
          while (stored < nunits) {
            while (issued < nunits && issued - stored < MOE_COPY_NBUF) {
              const uint32_t q = seq + uint32_t(issued);
              const int buf = int(q % MOE_COPY_NBUF);
              bulk_wait_read_dyn(stored - issued + MOE_COPY_NBUF - 1);
              const int tl = t0 + issued / pieces, pc = issued % pieces;
              const uint32_t off = uint32_t(pc) * COPY_CHUNK;
              const uint32_t sz = min(COPY_CHUNK, row_bytes - off);
              const uint8_t* src;
              if (p.pull) {
                if (tl >= tb_end || tl < tb_base) {
                  // the tokens of the next MOE_TOKB rows of the item, their loads in flight together
                  tb_base = tl;
                  tb_end = min(t1, tl + MOE_TOKB);
                  int v[MOE_TOKB];
#pragma unroll
                  for (int i = 0; i < MOE_TOKB; ++i) v[i] = tb_base + i < tb_end ? p.perm[tb_base + i] : 0;
#pragma unroll
                  for (int i = 0; i < MOE_TOKB; ++i) stok[i] = v[i] / p.k;
                }
                const int tok = stok[tl - tb_base];
                src = xs[tok / p.T_r] + size_t(tok % p.T_r) * row_bytes + off;
              } else {
                src = xs[r] + size_t(tl) * row_bytes + off;
              }
              mbar_arrive_expect_tx(&bars->copy[buf], sz);
              bulk_g2s(stage + buf * COPY_CHUNK, src, sz, &bars->copy[buf]);
              ++issued;
            }
            const uint32_t q = seq + uint32_t(stored);
            const int buf = int(q % MOE_COPY_NBUF);
            if (!mbar_wait(&bars->copy[buf], (q / MOE_COPY_NBUF) & 1u, abort, p.status, p.pipe_timeout_ns, 5)) {
              dead = true;
              break;
            }
            const int tl = t0 + stored / pieces, pc = stored % pieces;
            const uint32_t off = uint32_t(pc) * COPY_CHUNK;
            const uint32_t sz = min(COPY_CHUNK, row_bytes - off);
            if (p.pull) {
              // evict-last: the grouped GEMM reads these rows soon, once per column tile
              bulk_s2g_hint(p.sorted + size_t(tl) * row_bytes + off, stage + buf * COPY_CHUNK, sz, pol_keep);
            } else {
              const int tok = r * p.T_r + tl;
              for (int sl = 0; sl < p.k; ++sl) {
                const int pos = inv[tok * p.k + sl];
                bulk_s2g(p.sorted + size_t(pos) * row_bytes + off, stage + buf * COPY_CHUNK, sz);
              }
            }
            bulk_commit();
            ++stored;
          }
          seq += uint32_t(nunits);
          bulk_wait<0>();
          if (dead) break;
          fence_proxy_async_global();
          st_release(p.flags + (p.pull ? it : r * p.bpr + c), p.epoch);
        }
      }
      bulk_wait<0>();
    }
    __syncwarp();
  }
  pair::teardown(bars, warp, tmem_base);
}


// push: tokens of a shard per flag (about 128 KB of source rows); pull: sorted rows per flag (about 64 KB)
int moe_default_rpb(int mode, int H, int T_r, long long P) {
  if (mode == TL_MODE_PULL) return int(std::min<long long>(P, std::max(1, int(65536 / (size_t(H) * 2)))));
  return std::min(T_r, std::max(1, int(131072 / (size_t(H) * 2))));
}

}  // namespace
}  // namespace tl

extern "C" size_t tl_moe_workspace_size(int R, int T_r, int E, int topk) {
  if (R < 1 || T_r < 1 || E < 1 || topk < 1) return 0;
  const long long P = (long long)R * T_r * topk;
  if (P > (1ll << 30)) return 0;
  const int mt = tl::moe_max_tiles(int(P), E);
  return size_t(tl::ws_inv(mt) + P) * sizeof(int32_t);
}

extern "C" int tl_moe_num_flags(int mode, int R, int T_r, int H, int topk, int rows_per_barrier, int* effective_rpb) {
  if (R < 1 || T_r < 1 || H < 1 || topk < 1 || (mode != TL_MODE_PULL && mode != TL_MODE_PUSH)) return -1;
  const long long P = (long long)R * T_r * topk;
  if (P > (1ll << 30)) return -1;
  const int lim = mode == TL_MODE_PULL ? int(P) : T_r;
  const int rpb = rows_per_barrier > 0 ? std::min(rows_per_barrier, lim) : tl::moe_default_rpb(mode, H, T_r, P);
  if (effective_rpb) *effective_rpb = rpb;
  return mode == TL_MODE_PULL ? tl::cdiv(int(P), rpb) : R * tl::cdiv(T_r, rpb);
}

extern "C" tl_status tl_moe_ag_gemm(const tl_moe_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: NULL args");
  if (a->R < 1 || a->R > MOE_MAX_R)
    return fail(a->R > MOE_MAX_R ? TL_ERR_UNSUPPORTED : TL_ERR_INVALID, "tl_moe_ag_gemm: R=%d outside 1..%d", a->R,
                MOE_MAX_R);
  if (a->E < 1 || a->E > MOE_MAX_E)
    return fail(a->E > MOE_MAX_E ? TL_ERR_UNSUPPORTED : TL_ERR_INVALID, "tl_moe_ag_gemm: E=%d outside 1..%d", a->E,
                MOE_MAX_E);
  if (a->self_rank < 0 || a->self_rank >= a->R) return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: self_rank");
  if (a->T_r < 1 || a->H < 1 || a->N < 1 || a->topk < 1 || a->topk > a->E)
    return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: bad shape (T_r=%d H=%d N=%d topk=%d E=%d)", a->T_r, a->H, a->N,
                a->topk, a->E);
  if (a->H % 8 || a->N % 8)
    return fail(TL_ERR_UNSUPPORTED, "tl_moe_ag_gemm: H (%d) and N (%d) must be multiples of 8", a->H, a->N);
  if (!a->X || !a->topk_ids || !a->W || !a->sorted_tokens || !a->Y || !a->perm || !a->expert_offsets ||
      !a->workspace || !a->signals)
    return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: NULL pointer argument");
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: epoch must be nonzero");
  for (int r = 0; r < a->R; ++r)
    if (!a->X[r] || !aligned16(a->X[r])) return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: shard %d pointer", r);
  for (int e = 0; e < a->E; ++e)
    if (!a->W[e] || !aligned16(a->W[e])) return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: weight %d pointer", e);
  if (!aligned16(a->sorted_tokens) || !aligned16(a->Y) || !aligned16(a->workspace) ||
      (reinterpret_cast<uintptr_t>(a->topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(a->perm) & 3u) ||
      (reinterpret_cast<uintptr_t>(a->expert_offsets) & 3u))
    return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: pointer alignment");
  const long long T = (long long)a->R * a->T_r;
  const long long P = T * a->topk;
  if (P > (1ll << 30)) return fail(TL_ERR_UNSUPPORTED, "tl_moe_ag_gemm: too many routed rows");
  const int max_tiles = moe_max_tiles(int(P), a->E);
  if (max_tiles > MOE_MAX_TILES)
    return fail(TL_ERR_UNSUPPORTED, "tl_moe_ag_gemm: %d row tiles exceed %d", max_tiles, MOE_MAX_TILES);
  const size_t need = tl_moe_workspace_size(a->R, a->T_r, a->E, a->topk);
  if (a->workspace_bytes < need)
    return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: workspace %zu bytes, need %zu", a->workspace_bytes, need);
  if (a->mode != TL_MODE_PULL && a->mode != TL_MODE_PUSH) return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: mode %d", a->mode);
  const bool pull = a->mode == TL_MODE_PULL;
  int rpb = 0;
  const int nflags = tl_moe_num_flags(a->mode, a->R, a->T_r, a->H, a->topk, a->rows_per_barrier, &rpb);
  if (a->signals->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: signals hold %d flags, need %d", a->signals->num_flags, nflags);
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  if (a->signals->device != di.device) return fail(TL_ERR_INVALID, "tl_moe_ag_gemm: signals belong to another device");
  {
    // the token shards are moved with bulk TMA copies: device memory only
    const uint8_t* xdev[TL_MAX_RANKS];
    uint64_t host_mask = 0;
    if (tl_status s = classify_shards("tl_moe_ag_gemm", a->X, a->R, di.device, xdev, &host_mask)) return s;
    if (host_mask) return fail(TL_ERR_UNSUPPORTED, "tl_moe_ag_gemm: token shards must be device memory");
  }
  cudaStream_t st = (cudaStream_t)stream;

  // 1. routing and lookup tables
  RouteParams rp{};
  rp.topk = a->topk_ids;
  rp.perm = a->perm;
  rp.offsets = a->expert_offsets;
  rp.ws = static_cast<int32_t*>(a->workspace);
  rp.status = a->signals->status;
  rp.T = int(T);
  rp.k = a->topk;
  rp.E = a->E;
  rp.R = a->R;
  rp.T_r = a->T_r;
  rp.rpb = rpb;
  rp.bpr = cdiv(a->T_r, rpb);
  rp.self = a->self_rank;
  rp.max_tiles = max_tiles;
  rp.pull = pull ? 1 : 0;
  rp.k_shift = (a->topk & (a->topk - 1)) == 0 ? __builtin_ctz(unsigned(a->topk)) : -1;
  const size_t route_smem = (size_t(ROUTE_WARPS) * a->E + 2 * a->E + 2 * (a->E + 1) + 4 * size_t(max_tiles)) * sizeof(int32_t);
  if (route_smem > size_t(di.max_smem_optin))
    return fail(TL_ERR_UNSUPPORTED, "tl_moe_ag_gemm: routing needs %zu bytes of shared memory", route_smem);
  {
    void* rargs[] = {&rp};
    if (tl_status s = launch_coop(reinterpret_cast<const void*>(&moe_route_kernel), int(ROUTE_CTAS), ROUTE_THREADS,
                                  route_smem, st, rargs, int(ROUTE_CTAS)))
      return s;
  }

  // 2. AllGather + scatter and grouped GEMM
  MoeParams* p = new (std::nothrow) MoeParams;
  if (!p) return fail(TL_ERR_INTERNAL, "out of host memory");
  std::memset(p, 0, sizeof(MoeParams));
  tl_status res = TL_OK;
  do {
    if ((res = make_map_bf16(&p->map_a, a->sorted_tokens, P, a->H, size_t(a->H) * 2, pair::HM, pair::BK))) break;
    if ((res = make_map_bf16(&p->map_y, a->Y, P, a->N, size_t(a->N) * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))) break;
    for (int e = 0; e < a->E && !res; ++e)
      res = make_map_bf16(&p->map_w[e], a->W[e], a->H, a->N, size_t(a->N) * 2, pair::BK, 64);
    if (res) break;
    for (int r = 0; r < a->R; ++r) p->x[r] = static_cast<const uint8_t*>(a->X[r]);
    p->sorted = static_cast<uint8_t*>(a->sorted_tokens);
    p->Y = static_cast<uint16_t*>(a->Y);
    p->ws = static_cast<const int32_t*>(a->workspace);
    p->flags = a->signals->flags;
    p->status = a->signals->status;
    p->trace = a->trace;
    p->timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
    p->pipe_timeout_ns = 2 * p->timeout_ns + 1000000000ull;
    p->R = a->R;
    p->self = a->self_rank;
    p->T_r = a->T_r;
    p->H = a->H;
    p->N = a->N;
    p->E = a->E;
    p->k = a->topk;
    p->rpb = rpb;
    p->bpr = cdiv(a->T_r, rpb);
    p->Nt = cdiv(a->N, pair::BN);
    p->KB = cdiv(a->H, pair::BK);
    p->num_items = pull ? nflags : a->R * p->bpr;
    p->max_tiles = max_tiles;
    p->pull = pull ? 1 : 0;
    p->P = int(P);
    p->perm = a->perm;
    p->epoch = a->epoch;
    if ((res = test_hold("tl_moe_ag_gemm", p->timeout_ns, &p->hold_first, &p->hold_count, &p->hold_ns))) break;
    const int pairs = std::max(1, std::min(di.sm_count / 2, std::max(max_tiles * p->Nt, (p->num_items + 1) / 2)));
    void* args[] = {p};
    res = launch_coop(reinterpret_cast<const void*>(&moe_gemm_kernel), 2 * pairs, MOE_THREADS, MOE_SMEM_BYTES, st,
                      args, 2, /*early_start=*/true);
  } while (false);
  delete p;
  return res;
}
