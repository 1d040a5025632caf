// tl_moe_down.cu -- the down-projection side of the MoE layer: a grouped GEMM
// whose per-rank partials are reduce-scattered at tile granularity, then the
// TopK-reduce that combines each token's expert outputs with its gate weights
// and scatters them back to the token's own rank.
//
// TileLink talk summary ("TileLink: Generating Efficient Compute-Communication
// Overlapping Kernels using Tile-Centric Primitives"):
//  * Key Findings / Experimental Setup & Results -- the MoE layer overlaps
//    GroupGEMM, ReduceScatter, TopK-reduce and a local scatter (this file; the
//    AllGather + GroupGEMM part is tl_moe.cu).
//  * Technical Deep Dive -- the reduce stage of a persistent GEMM waits on its
//    own and its peers' tiles (as in tl_gemm_rs.cu); for dynamic workloads the
//    tiles come from a lookup table built from the routing.
//
// Launch 1, moe_down_kernel (CTA pairs, tcgen05.mma.cta_group::2): output tile
// tau = (expert tile t of the routing's tile table, 256-column tile n), column
// tiles in groups of four with the tiles inside a group (weight panel reuse);
// its R partials P_r = H_r[rows of t] . W2_r[expert slice, cols of n] are items
// tau*R + j, rank r = (tau + j) mod R, taken round-robin by the CTA pairs.
// Per CTA: warp 0 TMA producer, warp 1 MMA issuer (leader), warps 2-5 pushers
// (the fp32 partial half-tile into a ring slot, then the arrival flag), warps
// 6-13 reducers (acquire the R arrival flags of their half, sum their row slice
// in rank order into Y, and release the "reduced" flag that frees the slot).
// Both move only the rows of the tile's expert: the padding rows of an expert's
// last tile are computed by the MMAs but neither pushed nor read.  The K loop runs over I_r; columns of
// H_r past I_r read as zero, so a k-block that reaches into the next expert's
// slice of W2_r adds nothing.
// Option TL_RS_BF16_PARTIALS: every partial is rounded to bf16 (RNE) before it
// is pushed and widened back to fp32 by the reducers (half the partial bytes).
// Launch 2, moe_combine_kernel: out[d][u] = bf16(sum over slots, in order, of
// gate * Y[sorted row of the pair]), t = d*T_r + u.
#include <algorithm>
#include <cstring>
#include <new>

#include "tl_internal.h"
#include "tl_moe_ws.cuh"
#include "tl_pair.cuh"

namespace tl {
namespace {

constexpr int MD_MAX_RANKS = 32;
constexpr int MD_MAX_E = 64;
constexpr int kWarpRed0 = kWarpEpi0 + kNumEpiWarps;  // first reducer warp
constexpr int kNumRedWarps = 8;
constexpr int kNumRedThreads = kNumRedWarps * 32;
constexpr int RB = 8;  // ranks loaded per batch in the reduce
constexpr int QU = 2;  // float4 elements per thread per round in the reduce
constexpr int MD_THREADS = (kWarpRed0 + kNumRedWarps) * 32;
constexpr uint32_t MD_SMEM_BARS = pair::SMEM_END;
constexpr uint32_t MD_SMEM_BYTES = MD_SMEM_BARS + sizeof(pair::Bars) + 1024;

struct MdParams {
  CUtensorMap map_h[MD_MAX_RANKS];  // H_r [P, I_r], box 128 rows x 64
  CUtensorMap map_w[MD_MAX_RANKS];  // W2_r [E*I_r, Hd], box 64 x 64
  float* Y;                         // [P, Hd] fp32
  float* slots;                     // [ring_items][2][half_floats] fp32 receive half-slots
  uint32_t* flags;                  // [2][max_items][2]: arrival, then reduced
  uint32_t* status;
  const int32_t* ws;                // routing workspace: tile count, tile table
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int32_t R, P, I_r, Hd, Nt, G, KB, max_tiles, max_items, slice_rows, ring_items, half_floats;
  uint32_t epoch;
};

struct MdItem {
  int tau, t, n, r, j, e, row0, rows;
};

// Output tile tau -> (expert tile t, column tile n): column tiles in groups of G,
// every tile (in expert order) inside a group, the group's column tiles innermost,
// so an expert's weight panels for a group are reused by all its tiles and a
// tile's rows by the group's column tiles.
__device__ __forceinline__ MdItem md_item(const MdParams& p, int i, int ntiles) {
  MdItem it;
  it.tau = i / p.R;
  it.j = i % p.R;
  const int per_group = ntiles * p.G;
  const int g = it.tau / per_group, rem = it.tau - g * per_group;
  it.t = rem / p.G;
  it.n = g * p.G + rem % p.G;
  it.r = (it.tau + it.j) % p.R;
  const int32_t* tr = p.ws + ws_tiles(p.max_tiles) + 6 * it.t;
  it.e = tr[0];
  it.row0 = tr[1];
  it.rows = tr[2];
  return it;
}

// kBf16: partials travel as bf16 (TL_RS_BF16_PARTIALS); one instantiation per partial type.
template <bool kBf16>
__global__ void __launch_bounds__(MD_THREADS, 1) moe_down_kernel(const __grid_constant__ MdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  pair::Bars* bars = reinterpret_cast<pair::Bars*>(smem + MD_SMEM_BARS);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const uint32_t rank = cluster_ctarank();
  const int h = int(rank);
  const int pair_id = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  const uint32_t tmem_base = pair::setup(bars, warp);
  volatile uint32_t* abort = &bars->abort;
  const int ntiles = min(p.ws[0], p.max_tiles);
  const int num_items = ntiles * p.Nt * p.R;
  const int my_items = pair_id < num_items ? (num_items - 1 - pair_id) / npairs + 1 : 0;
  uint32_t* arrived = p.flags;                         // 2*(tau*R + r) + h
  uint32_t* reduced = p.flags + 2 * size_t(p.max_items);  // 2*(tau*R + j) + h

  if (warp == kWarpTma) {
    // ---------------------------------------------------------------- TMA producer (this CTA's halves)
    if (lane == 0) {
      pair::Producer prod;
      // operands stay in L2 ahead of the streamed partials (as in the GEMM-RS kernel)
      const uint64_t keep = l2_policy_evict_last();
      for (int i = pair_id; i < num_items && !*abort; i += npairs) {
        const MdItem it = md_item(p, i, ntiles);
        for (int kb = 0; kb < p.KB; ++kb)
          if (!prod.load_hint(smem, bars, rank, &p.map_h[it.r], kb * pair::BK, it.row0 + h * pair::HM,
                              &p.map_w[it.r], it.n * pair::BN + h * pair::HN, it.e * p.I_r + kb * pair::BK, keep,
                              abort, p.status, p.pipe_timeout_ns))
            break;
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && rank == 0)
      pair::mma_loop(smem, bars, tmem_base, my_items, p.KB, abort, p.status, p.pipe_timeout_ns);
    __syncwarp();
  } else if (warp < kWarpRed0) {
    // ---------------------------------------------------------------- pushers
    const int wq = warp & 3;
    const int et = (warp - kWarpEpi0) * 32 + lane;
    const int row_in_half = wq * 32 + lane;
    // half-slot layout [slice][col/4][row in slice][4], one contiguous block per reducer slice
    const int my_slice = row_in_half / p.slice_rows, my_row = row_in_half % p.slice_rows;
    const size_t my_base = (size_t(my_slice) * 64 * p.slice_rows + my_row) * 4;
    int jj = 0;
    for (int i = pair_id; i < num_items; i += npairs, ++jj) {
      const MdItem it = md_item(p, i, ntiles);
      const int acc = jj & 1;
      const uint32_t acc_ph = uint32_t(jj >> 1) & 1u;
      // slot free: the R reducers of this half of the tile that last used the slot are done with it
      if (i >= p.ring_items && lane == 0) {
        const int prev_tau = (i - p.ring_items) / p.R;
        for (int j = 0; j < p.R; ++j) {
          const int f = 2 * (prev_tau * p.R + j) + h;
          wait_flag(reduced + f, p.epoch, p.status, p.timeout_ns, uint32_t(2 * p.max_items + f), TL_ERR_TIMEOUT);
        }
      }
      __syncwarp();
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      if (!named_bar_and(1, kNumEpiThreads, ok)) break;
      tc_fence_after();
      // element offset of this thread's first value in its half-slot (4-byte floats, or
      // 2-byte bf16 values in half the bytes)
      const size_t slot_el = (size_t(i % p.ring_items) * 2 + h) * p.half_floats + my_base;
      const uint64_t stream = l2_policy_evict_first();  // partial lines: written once, read once
      // a row past the tile's expert (the padding of its last tile) is neither pushed nor read
      const bool row_used = h * pair::HM + row_in_half < it.rows;
      for (int c = 0; c < pair::BN / 32; ++c) {
        if (it.n * pair::BN + c * 32 >= p.Hd) break;
        uint32_t v[32];
        tmem_ld_32cols(tmem_base + (uint32_t(wq * 32) << 16) + uint32_t(acc * pair::BN + c * 32), v);
        tmem_ld_wait();
        if (!row_used) continue;
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
      // produce_tile_notify: every pusher thread's writes are ordered before thread 0's release
      named_bar_sync(1, kNumEpiThreads);
      if (et == 0) st_release(arrived + 2 * (it.tau * p.R + it.r) + h, p.epoch);
    }
  } else {
    // ---------------------------------------------------------------- reducers (this CTA's half)
    const int et = (warp - kWarpRed0) * 32 + lane;
    for (int i = pair_id; i < num_items; i += npairs) {
      const MdItem it = md_item(p, i, ntiles);
      // consume_tile_wait / peer_tile_wait: all R partials of this half have arrived
      if (lane == 0) {
        for (int r = 0; r < p.R; ++r) {
          const int f = 2 * (it.tau * p.R + r) + h;
          wait_flag(arrived + f, p.epoch, p.status, p.timeout_ns, uint32_t(f), TL_ERR_TIMEOUT);
        }
      }
      __syncwarp();
      const int s0 = it.j * p.slice_rows;
      // rows of the slice that belong to the tile's expert (the pushers skip the others)
      const int s_rows = max(0, min(min(p.slice_rows, pair::HM - s0), it.rows - (h * pair::HM + s0)));
      const int n_cols = min(pair::BN, p.Hd - it.n * pair::BN);
      const int total = s_rows * (n_cols / 4);
      // rank r's partial was pushed by item tau*R + j(r), j(r) = (r - tau) mod R
      const uint64_t drop = l2_policy_evict_first();  // each partial line is read once, here
      const int jbase = ((-it.tau) % p.R + p.R) % p.R;
      const int ring_base = int((size_t(it.tau) * p.R) % size_t(p.ring_items));
      const int lrow_base = h * pair::HM + s0;  // row of the tile
      for (int e0 = et; e0 < total; e0 += kNumRedThreads * QU) {
        int off[QU];  // float offset inside a half-slot, -1 past the slice
        int lrow[QU];
        int ocol[QU];
#pragma unroll
        for (int u = 0; u < QU; ++u) {
          const int e = e0 + u * kNumRedThreads;
          const int c4 = e / s_rows, sr = e - c4 * s_rows;
          off[u] = e < total ? ((it.j * 64 + c4) * p.slice_rows + sr) * 4 : -1;
          lrow[u] = lrow_base + sr;
          ocol[u] = it.n * pair::BN + c4 * 4;
        }
        float4 acc4[QU];
        for (int rb = 0; rb < p.R; rb += RB) {
          // a batch of ranks loaded together, then added in rank order
          float4 v[RB][QU];
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) {
            if (rb + rr < p.R) {
              int j = jbase + rb + rr;
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
          // fixed rank order: ((P_0 + P_1) + P_2) + ...
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
        for (int u = 0; u < QU; ++u)
          if (off[u] >= 0)
            *reinterpret_cast<float4*>(p.Y + size_t(it.row0 + lrow[u]) * p.Hd + ocol[u]) = acc4[u];
      }
      // slice j of this half of tile tau is read: release its "reduced" flag (slot-free barrier)
      named_bar_sync(2, kNumRedThreads);
      if (et == 0) st_release(reduced + 2 * (it.tau * p.R + it.j) + h, p.epoch);
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
    }
  }
  pair::teardown(bars, warp, tmem_base);
}

struct CombineParams {
  const float* Y;         // [P, Hd] fp32
  const float* gates;     // [T, k]
  const int32_t* inv;     // [P] pair -> sorted row
  uint16_t* out[MD_MAX_RANKS];
  int32_t T, T_r, k, Hd;
};

// TopK-reduce and scatter: four columns of one token per thread.
__global__ void __launch_bounds__(256) moe_combine_kernel(const __grid_constant__ CombineParams p) {
  const int n4 = p.Hd / 4;
  const size_t total = size_t(p.T) * n4;
  for (size_t idx = size_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += size_t(gridDim.x) * blockDim.x) {
    const int t = int(idx / n4), c4 = int(idx % n4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.k; ++s) {
      // slot order: ((g_0 * Y_0) + g_1 * Y_1) + ..., products and sums rounded to fp32
      const int q = t * p.k + s;
      const float g = p.gates[q];
      const float4 y = __ldcg(reinterpret_cast<const float4*>(p.Y + size_t(p.inv[q]) * p.Hd) + c4);
      acc.x = __fadd_rn(acc.x, __fmul_rn(g, y.x));
      acc.y = __fadd_rn(acc.y, __fmul_rn(g, y.y));
      acc.z = __fadd_rn(acc.z, __fmul_rn(g, y.z));
      acc.w = __fadd_rn(acc.w, __fmul_rn(g, y.w));
    }
    const int d = t / p.T_r;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x, acc.y);
    pk.y = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(p.out[d] + size_t(t - d * p.T_r) * p.Hd + c4 * 4) = pk;
  }
}

int md_pairs(int max_items, int sm_count) { return std::max(1, std::min(sm_count / 2, max_items)); }
int md_ring_items(int max_items, int pairs) { return std::min(max_items, 3 * pairs); }
int md_half_floats(int R) { return R * cdiv(pair::HM, R) * pair::BN; }
int md_max_items(int R, int T_r, int topk, int E, int Hd) {
  const long long P = (long long)R * T_r * topk;
  return moe_max_tiles(int(P), E) * cdiv(Hd, pair::BN) * R;
}
size_t md_slots_bytes(int ring_items, int R) { return size_t(ring_items) * 2 * md_half_floats(R) * sizeof(float); }
size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace tl

extern "C" size_t tl_moe_down_workspace_size(int R, int T_r, int topk, int E, int Hd) {
  using namespace tl;
  if (R < 1 || T_r < 1 || topk < 1 || E < 1 || Hd < 1) return 0;
  const long long P = (long long)R * T_r * topk;
  if (P > (1ll << 30)) return 0;
  const int items = md_max_items(R, T_r, topk, E, Hd);
  DeviceInfo di{};
  const int sms = device_info(&di) == TL_OK ? di.sm_count : 0;
  const int ring = sms >= 2 ? md_ring_items(items, md_pairs(items, sms)) : items;
  return align256(md_slots_bytes(ring, R)) + size_t(P) * Hd * sizeof(float);
}

extern "C" int tl_moe_down_num_flags(int R, int T_r, int topk, int E, int Hd) {
  using namespace tl;
  if (R < 1 || T_r < 1 || topk < 1 || E < 1 || Hd < 1) return -1;
  const long long f = 4ll * md_max_items(R, T_r, topk, E, Hd);
  return f > (1ll << 30) ? -1 : int(f);
}

extern "C" tl_status tl_moe_down(const tl_moe_down_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_moe_down: NULL args");
  if (a->R < 1 || a->R > MD_MAX_RANKS) return fail(TL_ERR_UNSUPPORTED, "tl_moe_down: R=%d outside 1..%d", a->R, MD_MAX_RANKS);
  if (a->E < 1 || a->E > MD_MAX_E) return fail(TL_ERR_UNSUPPORTED, "tl_moe_down: E=%d outside 1..%d", a->E, MD_MAX_E);
  if (a->T_r < 1 || a->topk < 1 || a->topk > a->E || a->I_r < 1 || a->Hd < 1)
    return fail(TL_ERR_INVALID, "tl_moe_down: bad shape");
  if (a->I_r % 8 || a->Hd % 8)
    return fail(TL_ERR_UNSUPPORTED, "tl_moe_down: I_r (%d) and Hd (%d) must be multiples of 8", a->I_r, a->Hd);
  if (!a->H || !a->W2 || !a->gates || !a->routing || !a->out || !a->workspace || !a->signals)
    return fail(TL_ERR_INVALID, "tl_moe_down: NULL pointer argument");
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "tl_moe_down: epoch must be nonzero");
  if (a->options & ~TL_RS_BF16_PARTIALS) return fail(TL_ERR_INVALID, "tl_moe_down: unknown options 0x%x", a->options);
  for (int r = 0; r < a->R; ++r)
    if (!a->H[r] || !a->W2[r] || !a->out[r] || !aligned16(a->H[r]) || !aligned16(a->W2[r]) || !aligned16(a->out[r]))
      return fail(TL_ERR_INVALID, "tl_moe_down: rank %d pointer NULL or not 16-byte aligned", r);
  if (!aligned16(a->workspace) || !aligned16(a->gates) || !aligned16(a->routing))
    return fail(TL_ERR_INVALID, "tl_moe_down: workspace, gates and routing must be 16-byte aligned");
  const long long P = (long long)a->R * a->T_r * a->topk;
  if (P > (1ll << 30) || (long long)a->E * a->I_r > (1ll << 30))
    return fail(TL_ERR_UNSUPPORTED, "tl_moe_down: problem too large");
  const size_t need = tl_moe_down_workspace_size(a->R, a->T_r, a->topk, a->E, a->Hd);
  if (a->workspace_bytes < need)
    return fail(TL_ERR_INVALID, "tl_moe_down: workspace %zu bytes, need %zu", a->workspace_bytes, need);
  const int nflags = tl_moe_down_num_flags(a->R, a->T_r, a->topk, a->E, a->Hd);
  if (nflags < 0 || a->signals->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_moe_down: signals hold %d flags, need %d", a->signals->num_flags, nflags);
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  if (a->signals->device != di.device) return fail(TL_ERR_INVALID, "tl_moe_down: signals belong to another device");

  MdParams* p = new (std::nothrow) MdParams;
  if (!p) return fail(TL_ERR_INTERNAL, "out of host memory");
  std::memset(p, 0, sizeof(MdParams));
  const int max_tiles = moe_max_tiles(int(P), a->E);
  tl_status st = TL_OK;
  do {
    for (int r = 0; r < a->R && !st; ++r) {
      st = make_map_bf16(&p->map_h[r], a->H[r], uint64_t(P), a->I_r, size_t(a->I_r) * 2, pair::HM, pair::BK);
      if (!st)
        st = make_map_bf16(&p->map_w[r], a->W2[r], uint64_t(a->E) * a->I_r, a->Hd, size_t(a->Hd) * 2, pair::BK, 64);
    }
    if (st) break;
    const int max_items = md_max_items(a->R, a->T_r, a->topk, a->E, a->Hd);
    const int pairs = md_pairs(max_items, di.sm_count);
    p->ring_items = md_ring_items(max_items, pairs);
    p->slots = static_cast<float*>(a->workspace);
    p->Y = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) + align256(md_slots_bytes(p->ring_items, a->R)));
    p->flags = a->signals->flags;
    p->status = a->signals->status;
    p->ws = a->routing;
    p->timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
    p->pipe_timeout_ns = 2 * p->timeout_ns + 1000000000ull;
    p->R = a->R;
    p->P = int(P);
    p->I_r = a->I_r;
    p->Hd = a->Hd;
    p->Nt = cdiv(a->Hd, pair::BN);
    p->G = p->Nt % 4 == 0 ? 4 : (p->Nt % 2 == 0 ? 2 : 1);
    p->KB = cdiv(a->I_r, pair::BK);
    p->max_tiles = max_tiles;
    p->max_items = max_items;
    p->slice_rows = cdiv(pair::HM, a->R);
    p->half_floats = md_half_floats(a->R);
    p->epoch = a->epoch;
    void* args[] = {p};
    const void* kernel = (a->options & TL_RS_BF16_PARTIALS) ? reinterpret_cast<const void*>(&moe_down_kernel<true>)
                                                             : reinterpret_cast<const void*>(&moe_down_kernel<false>);
    st = launch_coop(kernel, 2 * pairs, MD_THREADS, MD_SMEM_BYTES, (cudaStream_t)stream, args, 2);
    if (st) break;
    CombineParams c{};
    c.Y = p->Y;
    c.gates = a->gates;
    c.inv = a->routing + ws_inv(max_tiles);
    for (int r = 0; r < a->R; ++r) c.out[r] = static_cast<uint16_t*>(a->out[r]);
    c.T = a->R * a->T_r;
    c.T_r = a->T_r;
    c.k = a->topk;
    c.Hd = a->Hd;
    const long long work = (long long)c.T * (a->Hd / 4);
    const int grid = int(std::min<long long>(std::max<long long>(1, (work + 255) / 256), 8ll * di.sm_count));
    moe_combine_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(c);
    st = cuda_ok(cudaGetLastError(), "combine launch");
  } while (false);
  delete p;
  return st;
}
