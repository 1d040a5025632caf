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
// tau = (expert tile t of the routing's tile table, 256-column tile n), tiles
// in expert order with the column tiles innermost.  The R partials of tau are added into its fp32 running sum rank after
// rank, the way a ring ReduceScatter passes a partial sum from rank to rank:
// pass j computes P_j = H_j[rows of t] . W2_j[expert slice, cols of n], waits
// for pass j-1 of the same tile, adds P_j to the sum and stores it back; pass
// R-1 writes the complete sum into Y.  Output tiles go in groups of
// kChainTiles, and inside a group pass by pass (item i -> group, pass j, tile),
// so a group's running sums stay in L2 from one pass to the next.  Items are
// taken round-robin by the CTA pairs.  Per CTA: warp 0 TMA producer, warp 1
// MMA issuer (leader), warps 2-9 epilogue (one row of the half-tile and half of
// its columns per thread; each warp frees the accumulator after its last read of
// it), warp 10 notifier (releases a pass's flag once every epilogue thread has
// stored its share).
// Only the rows of the tile's expert are summed and written: the padding rows
// of an expert's last tile are computed by the MMAs but belong to the next
// expert's rows of Y.  The K loop runs over I_r; columns of H_r past I_r read
// as zero, so a k-block that reaches into the next expert's slice of W2_r adds
// nothing.
// Option TL_RS_BF16_PARTIALS: every partial is rounded to bf16 (RNE) before it
// joins the fp32 sum.
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
// The epilogue has kEpiParts groups of four warps (one warp per TMEM lane quarter in each);
// group q drains and sums columns [q, q+1) * 256 / kEpiParts of the accumulator.
constexpr int kEpiParts = 2;
constexpr int kChunksPerPart = pair::BN / 32 / kEpiParts;
constexpr int kNumMdEpiThreads = kNumEpiThreads * kEpiParts;
constexpr int kWarpNotify = kWarpEpi0 + kNumMdEpiThreads / 32;  // releases each pass's flag
constexpr int MD_THREADS = (kWarpNotify + 1) * 32;
constexpr uint32_t MD_SMEM_BARS = pair::SMEM_END;
// per accumulator: the epilogue threads' sums and Y rows are stored (stored[a], one arrival
// per epilogue thread), and the notifier has released the item's flag (notified[a])
struct MdBars {
  uint64_t stored[2];
  uint64_t notified[2];
};
constexpr uint32_t MD_SMEM_MDBARS = MD_SMEM_BARS + (uint32_t(sizeof(pair::Bars)) + 7u) / 8u * 8u;
constexpr uint32_t MD_SMEM_BYTES = MD_SMEM_MDBARS + sizeof(MdBars) + 1024;
constexpr int kChainTiles = 96;                     // output tiles whose sums are in flight together
constexpr int kHalfFloats = pair::HM * pair::BN;     // one CTA's half of a tile's running sum

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

struct MdParams {
  CUtensorMap map_h[MD_MAX_RANKS];  // H_r [P, I_r], box 128 rows x 64
  CUtensorMap map_w[MD_MAX_RANKS];  // W2_r [E*I_r, Hd], box 64 x 64
  float* Y;                         // [P, Hd] fp32
  float* sums;                      // [max_tiles*Nt][2][col/4][row][4] fp32 running sums
  uint32_t* flags;                  // [max_items][2] pass arrival flags
  uint32_t* status;
  const int32_t* ws;                // routing workspace: tile count, tile table
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int32_t R, P, I_r, Hd, Nt, KB, max_tiles, max_items;
  uint32_t epoch;
};

struct MdItem {
  int tau, t, n, j, e, row0, rows;
};

// Item i -> (group of kChainTiles output tiles, pass j = rank, tile tau); tau ->
// (expert tile t, column tile n), column tiles innermost, so a tile's rows of
// H_j are reused by all its column tiles and an expert's W2_j panels by the
// expert's row tiles in the group.
__device__ __forceinline__ MdItem md_item(const MdParams& p, int i, int ntiles) {
  MdItem it;
  const int num_tiles = ntiles * p.Nt;
  const int tpg = min(num_tiles, kChainTiles);
  const int g = i / (p.R * tpg), rem = i - g * p.R * tpg;
  const int gt = min(tpg, num_tiles - g * tpg);  // tiles of this group (the last may be short)
  it.j = rem / gt;
  it.tau = g * tpg + (rem - it.j * gt);
  it.t = it.tau / p.Nt;
  it.n = it.tau - it.t * p.Nt;
  const int32_t* tr = p.ws + ws_tiles(p.max_tiles) + 6 * it.t;
  it.e = tr[0];
  it.row0 = tr[1];
  it.rows = tr[2];
  return it;
}

// kBf16: partials rounded to bf16 before they join the sum (TL_RS_BF16_PARTIALS).
template <bool kBf16>
__global__ void __launch_bounds__(MD_THREADS, 1) moe_down_kernel(const __grid_constant__ MdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  pair::Bars* bars = reinterpret_cast<pair::Bars*>(smem + MD_SMEM_BARS);
  MdBars* mdb = reinterpret_cast<MdBars*>(smem + MD_SMEM_MDBARS);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const uint32_t rank = cluster_ctarank();
  const int h = int(rank);
  const int pair_id = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  if (threadIdx.x == 0) {
    for (int a = 0; a < 2; ++a) {
      mbar_init(&mdb->stored[a], kNumMdEpiThreads);
      mbar_init(&mdb->notified[a], 1);
    }
  }
  // every epilogue warp of both CTAs frees the accumulator once it has read its columns
  const uint32_t tmem_base = pair::setup(bars, warp, 2 * (kNumMdEpiThreads / 32));
  volatile uint32_t* abort = &bars->abort;
  const int ntiles = min(p.ws[0], p.max_tiles);
  const int num_items = ntiles * p.Nt * p.R;
  const int my_items = pair_id < num_items ? (num_items - 1 - pair_id) / npairs + 1 : 0;
  uint32_t* arrived = p.flags;  // 2*(tau*R + j) + h

  if (warp == kWarpTma) {
    // ---------------------------------------------------------------- TMA producer (this CTA's halves)
    if (lane == 0) {
      pair::Producer prod;
      // the rows of H stay in L2 for the tile's column tiles (evict-last, like the running
      // sums); the weight panels, which small experts read once, do not push them out
      // (evict-normal)
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t norm = l2_policy_evict_normal();
      for (int i = pair_id; i < num_items && !*abort; i += npairs) {
        const MdItem it = md_item(p, i, ntiles);
        for (int kb = 0; kb < p.KB; ++kb)
          if (!prod.load_hint(smem, bars, rank, &p.map_h[it.j], kb * pair::BK, it.row0 + h * pair::HM,
                              &p.map_w[it.j], it.n * pair::BN + h * pair::HN, it.e * p.I_r + kb * pair::BK, keep, norm,
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
  } else if (warp == kWarpNotify) {
    // ---------------------------------------------------------------- notifier
    // produce_tile_notify for each pass, off the epilogue's path: once every epilogue
    // thread has stored its share of the item (their arrivals order their writes before
    // this thread's release), release the pass's arrival flag
    if (lane == 0) {
      int jj = 0;
      for (int i = pair_id; i < num_items; i += npairs, ++jj) {
        const MdItem it = md_item(p, i, ntiles);
        const int acc = jj & 1;
        if (!mbar_wait(&mdb->stored[acc], uint32_t(jj >> 1) & 1u, abort, p.status, p.pipe_timeout_ns, 6)) break;
        st_release(arrived + 2 * (it.tau * p.R + it.j) + h, p.epoch);
        mbar_arrive(&mdb->notified[acc]);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue: chain accumulation
    const int wq = warp & 3;                               // TMEM lane quarter of this warp
    const int part = (warp - kWarpEpi0) / kNumEpiWarps;    // its share of the columns
    const int row_in_half = wq * 32 + lane;
    int jj = 0;
    for (int i = pair_id; i < num_items; i += npairs, ++jj) {
      const MdItem it = md_item(p, i, ntiles);
      const int acc = jj & 1;
      const uint32_t acc_ph = uint32_t(jj >> 1) & 1u;
      // peer_tile_wait: the previous rank's partial is in the running sum (that pass ran a
      // whole pass of the group's tiles earlier)
      if (it.j > 0 && lane == 0) {
        const int f = 2 * (it.tau * p.R + it.j - 1) + h;
        wait_flag(arrived + f, p.epoch, p.status, p.timeout_ns, uint32_t(f), TL_ERR_TIMEOUT);
      }
      __syncwarp();
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      if (!named_bar_and(1, kNumMdEpiThreads, ok)) break;
      tc_fence_after();
      // half-tile layout [col/4][row][4]: a warp's 16-byte accesses cover 512 contiguous bytes
      float* S = p.sums + (size_t(it.tau) * 2 + h) * kHalfFloats + size_t(row_in_half) * 4;
      const bool first = it.j == 0, last = it.j == p.R - 1;
      // a row past the tile's expert (the padding of its last tile) is neither summed nor written
      const bool row_used = h * pair::HM + row_in_half < it.rows;
      float* yrow = p.Y + size_t(it.row0 + h * pair::HM + row_in_half) * p.Hd;
      const uint64_t keep = l2_policy_evict_last();  // the sum is read again by the next pass
      const int nch = min(pair::BN / 32, (p.Hd - it.n * pair::BN + 31) / 32);
      // this warp's share of the columns, and the running sums of its row one chunk of 32
      // columns ahead of the one being added: s0 = chunk c, s1 = chunk c+1
      const int c_lo = part * kChunksPerPart, c_hi = min(nch, c_lo + kChunksPerPart);
      const bool load = !first && row_used;
      float4 s0[8], s1[8];
      if (load && c_lo < c_hi) {
#pragma unroll
        for (int g = 0; g < 8; ++g) s1[g] = ld_global_cg_v4f_hint(S + size_t(c_lo * 8 + g) * pair::HM * 4, keep);
      }
      for (int c = c_lo; c < c_hi; ++c) {
        const int col0 = it.n * pair::BN + c * 32;
#pragma unroll
        for (int g = 0; g < 8; ++g) s0[g] = s1[g];
        if (load && c + 1 < c_hi) {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            s1[g] = ld_global_cg_v4f_hint(S + size_t((c + 1) * 8 + g) * pair::HM * 4, keep);
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
        if (!row_used) continue;
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
        if (!first) {
          // ((P_0 + P_1) + ...) + P_j in fp32, one rounding per pass
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            f[g * 4 + 0] = __fadd_rn(s0[g].x, f[g * 4 + 0]);
            f[g * 4 + 1] = __fadd_rn(s0[g].y, f[g * 4 + 1]);
            f[g * 4 + 2] = __fadd_rn(s0[g].z, f[g * 4 + 2]);
            f[g * 4 + 3] = __fadd_rn(s0[g].w, f[g * 4 + 3]);
          }
        }
        if (!last) {
          float* sc = S + size_t(c * 8) * pair::HM * 4;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            st_global_cg_v4f_hint(sc + size_t(g) * pair::HM * 4, f[g * 4], f[g * 4 + 1], f[g * 4 + 2],
                                  f[g * 4 + 3], keep);
        } else {
          // Y row of the complete sum (Hd is a multiple of 8, so a 4-column group is whole)
#pragma unroll
          for (int g = 0; g < 8; ++g)
            if (col0 + g * 4 < p.Hd)
              *reinterpret_cast<float4*>(yrow + col0 + g * 4) =
                  make_float4(f[g * 4], f[g * 4 + 1], f[g * 4 + 2], f[g * 4 + 3]);
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
      if (jj >= 2 && !mbar_wait(&mdb->notified[acc], (uint32_t(jj >> 1) & 1u) ^ 1u, abort, p.status,
                                p.pipe_timeout_ns, 7))
        break;
      mbar_arrive(&mdb->stored[acc]);
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
int md_max_items(int R, int T_r, int topk, int E, int Hd) {
  const long long P = (long long)R * T_r * topk;
  return moe_max_tiles(int(P), E) * cdiv(Hd, pair::BN) * R;
}
size_t md_sums_bytes(int max_tiles, int Hd) { return size_t(max_tiles) * cdiv(Hd, pair::BN) * 2 * kHalfFloats * sizeof(float); }
size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace tl

extern "C" size_t tl_moe_down_workspace_size(int R, int T_r, int topk, int E, int Hd) {
  using namespace tl;
  if (R < 1 || T_r < 1 || topk < 1 || E < 1 || Hd < 1) return 0;
  const long long P = (long long)R * T_r * topk;
  if (P > (1ll << 30)) return 0;
  return align256(md_sums_bytes(moe_max_tiles(int(P), E), Hd)) + size_t(P) * Hd * sizeof(float);
}

extern "C" int tl_moe_down_num_flags(int R, int T_r, int topk, int E, int Hd) {
  using namespace tl;
  if (R < 1 || T_r < 1 || topk < 1 || E < 1 || Hd < 1) return -1;
  const long long f = 2ll * md_max_items(R, T_r, topk, E, Hd);
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
    p->sums = static_cast<float*>(a->workspace);
    p->Y = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) + align256(md_sums_bytes(max_tiles, a->Hd)));
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
    p->KB = cdiv(a->I_r, pair::BK);
    p->max_tiles = max_tiles;
    p->max_items = max_items;
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
