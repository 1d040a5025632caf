// tl_ag_gemm.cu -- AllGather -> GEMM fused at tile granularity in one launch.
//
// TileLink talk summary ("TileLink: Generating Efficient Compute-Communication
// Overlapping Kernels using Tile-Centric Primitives"):
//  * Key Findings / Experimental Setup & Results -- AllGather-GEMM.
//  * Technical Deep Dive -- produce_tile_notify / consume_tile_wait signals;
//    pull mode (readiness barrier + completion barrier) and push mode (one
//    barrier); a wait's tile id maps affinely to (rank, barrier); consumer
//    tiles are swizzled into data-arrival order.
//
// A persistent grid of CTA pairs (clusters of two, one CTA per SM, sized so
// that every CTA is resident at once) computes 256 x 256 tiles with
// tcgen05.mma.cta_group::2.  Every CTA has:
//   warp 0      TMA producer: acquires the arrival flags of its 128 rows of a
//               tile, then streams its rows of A (gathered, or the self shard in
//               place) and its 128 columns of B into a 6-stage ring.
//   warp 1      MMA issuer (leader CTA of the pair only).
//   warps 2-5   epilogue: TMEM -> registers -> bf16 (and fp32) rows of C.
//   warp 6      copy (AllGather producer): bulk-TMA copies of shard row chunks
//               into `gathered`, then a release store of the chunk's flag.
// When the tiles would leave pairs idle and the caller gives a workspace, each
// tile's k-blocks are split over S units on S pairs (split-K, tl_splitk.cuh);
// the tile's rows are waited for by every unit of the tile.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "tl_copy.cuh"
#include "tl_epilogue.cuh"
#include "tl_internal.h"
#include "tl_pair.cuh"
#include "tl_splitk.cuh"

namespace tl {
namespace {

constexpr int AG_MAX_MTILES = 1024;  // 256-row pair tiles
constexpr int kWarpCopy = 6;
constexpr int AG_THREADS = 7 * 32;
// shared memory: the pipeline stages, the copy warp's staging (three buffers),
// then one 32 x 32 C box per epilogue warp for the TMA-store epilogue
constexpr int AG_COPY_NBUF = 3;
constexpr uint32_t AG_SMEM_COPY = pair::SMEM_END;
constexpr uint32_t AG_SMEM_CSTAGE = AG_SMEM_COPY + AG_COPY_NBUF * COPY_CHUNK;
constexpr uint32_t AG_SMEM_BARS = AG_SMEM_CSTAGE + kNumEpiWarps * C_BOX_BYTES;
constexpr uint32_t AG_SMEM_BYTES = AG_SMEM_BARS + sizeof(pair::Bars) + 1024;

struct AgParams {
  CUtensorMap map_g;     // gathered [M, K], box 128 rows
  CUtensorMap map_self;  // A_self [M_shard, K], box 128 rows
  CUtensorMap map_b;     // B [K, N], box 64 x 64
  CUtensorMap map_c;     // C [M, N], box 32 x 32, 64-byte swizzle (TMA stores)
  const uint8_t* shard[TL_MAX_RANKS];
  uint8_t* gathered;
  uint16_t* C;
  float* C_f32;
  uint32_t* flags;
  const uint32_t* ready;  // pull mode readiness flags, or nullptr
  uint32_t* status;
  int32_t* trace;
  uint64_t timeout_ns;       // bound of each flag wait
  uint64_t pipe_timeout_ns;  // bound of each pipeline (mbarrier) wait: 2 x flag bound + 1 s
  int32_t R, self, M_shard, K, N, M;
  int32_t rpb, bpr, Mt, Nt, KB, num_items;
  int32_t S, KBs, num_work;  // splits per tile, k-blocks per split, work units (tiles * S)
  splitk::Work sk;
  uint32_t epoch;
  uint64_t host_mask;  // shards in host memory (copied with plain loads)
  int32_t hold_first, hold_count;  // chunks the copy warps move last (tl_test_hold_chunks)
  uint64_t hold_ns;
  uint16_t m_order[AG_MAX_MTILES];
};

// Flag id guarding global row `row` of the gathered matrix (affine tile map).
__device__ __forceinline__ int row_flag(const AgParams& p, int row) {
  return (row / p.M_shard) * p.bpr + (row % p.M_shard) / p.rpb;
}

__global__ void __launch_bounds__(AG_THREADS, 1) ag_gemm_kernel(const __grid_constant__ AgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  pair::Bars* bars = reinterpret_cast<pair::Bars*>(smem + AG_SMEM_BARS);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const uint32_t rank = cluster_ctarank();
  const int pair_id = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&p.map_g);
    tma_prefetch_desc(&p.map_self);
    tma_prefetch_desc(&p.map_b);
  }
  const uint32_t tmem_base = pair::setup(bars, warp);
  volatile uint32_t* abort = &bars->abort;
  const int my_work = pair_id < p.num_work ? (p.num_work - 1 - pair_id) / npairs + 1 : 0;

  if (warp == kWarpTma) {
    // ---------------------------------------------------------------- TMA producer (this CTA's 128 rows)
    pair::Producer prod;
    int last_m = -1;
    for (int w = pair_id; w < p.num_work; w += npairs) {
      const int t = w / p.S, split = w % p.S;  // schedule slot of the tile, k range
      const int n = t % p.Nt;
      const int m = p.m_order[t / p.Nt];
      const int row0 = m * pair::BM + int(rank) * pair::HM;
      const bool any = row0 < p.M;
      const int row1 = min(p.M, row0 + pair::HM) - 1;
      const bool local = any && (row0 / p.M_shard == p.self) && (row1 / p.M_shard == p.self);
      if (any && !local && m != last_m) {
        // consume_tile_wait: every flag guarding this CTA's rows; lanes poll in parallel
        const int id0 = row_flag(p, row0), id1 = row_flag(p, row1);
        for (int id = id0 + lane; id <= id1; id += 32)
          wait_flag(p.flags + id, p.epoch, p.status, p.timeout_ns, uint32_t(id), TL_ERR_TIMEOUT);
      }
      last_m = m;
      __syncwarp();
      if (lane == 0) {
        if (p.trace && rank == 0 && split == 0) p.trace[t] = m * p.Nt + n;
        if (!local) fence_proxy_async_global();
        const CUtensorMap* ma = local ? &p.map_self : &p.map_g;
        const int a_y = local ? row0 - p.self * p.M_shard : row0;
        for (int kb = split * p.KBs; kb < (split + 1) * p.KBs; ++kb)
          if (!prod.load(smem, bars, rank, ma, kb * pair::BK, a_y, &p.map_b, n * pair::BN + int(rank) * pair::HN,
                         kb * pair::BK, abort, p.status, p.pipe_timeout_ns))
            break;
      }
      // warp-uniform exit decision
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer (leader CTA)
    if (lane == 0 && rank == 0)
      pair::mma_loop(smem, bars, tmem_base, my_work, p.KBs, abort, p.status, p.pipe_timeout_ns);
    __syncwarp();
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kNumEpiWarps) {
    // ---------------------------------------------------------------- epilogue (this CTA's 128 rows)
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* cbox = smem + AG_SMEM_CSTAGE + uint32_t(wq) * C_BOX_BYTES;
    int j = 0;
    for (int w = pair_id; w < p.num_work; w += npairs, ++j) {
      const int acc = j & 1;
      const uint32_t acc_ph = uint32_t(j >> 1) & 1u;
      const int t = w / p.S, split = w % p.S;
      const int n = t % p.Nt;
      const int m = p.m_order[t / p.Nt];
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      // split-K epilogues meet at named barriers, so all four warps leave together
      if (!(p.S > 1 ? named_bar_and(splitk::kBarrier, kNumEpiThreads, ok) : __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      const int row = m * pair::BM + int(rank) * pair::HM + wq * 32 + lane;
      const bool row_ok = row < p.M;
      const int row_base = m * pair::BM + int(rank) * pair::HM + wq * 32;
      const int nchunks = min(pair::BN / 32, (p.N - n * pair::BN + 31) / 32);
      const uint32_t tacc = tmem_base + (uint32_t(wq * 32) << 16) + uint32_t(acc * pair::BN);
      // chunk c of the finished tile (fp32 bits) to C and C_f32
      auto write_c = [&](int c, const uint32_t* v) {
        const int col0 = n * pair::BN + c * 32;
        // bf16 C: this warp's 32 x 32 box with one TMA store (rows past M are not written)
        if (row_base < p.M) store_box_bf16(&p.map_c, cbox, 1, lane, v, col0, row_base);
        if (row_ok && p.C_f32) {
          float* frow = p.C_f32 + size_t(row) * p.N + col0;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            if (col0 + g * 4 < p.N) {
              const float* f = reinterpret_cast<const float*>(v + g * 4);
              st_global_cg_v4f(frow + g * 4, f[0], f[1], f[2], f[3]);
            }
          }
        }
      };
      if (p.S > 1) {
        splitk::epilogue(p.sk, t, split, rank, wq, lane, tacc, nchunks, &bars->splitk_ok, p.status, write_c);
      } else {
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tmem_ld_32cols(tacc + uint32_t(c * 32), v);
          tmem_ld_wait();
          write_c(c, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) pair::release_accumulator(bars, acc, rank);
    }
    if (lane == 0) bulk_wait<0>();  // every store of this warp is complete
    __syncwarp();
  } else if (warp == kWarpCopy) {
    // ---------------------------------------------------------------- AllGather producer
    AgCopyJob job{p.shard, p.gathered, p.flags, p.ready, p.status, p.timeout_ns, p.pipe_timeout_ns,
                  p.R, p.self, p.M_shard, p.K, p.rpb, p.bpr, p.num_items, p.epoch, p.host_mask,
                  p.hold_first, p.hold_count, p.hold_ns};
    ag_copy_items<AG_COPY_NBUF>(job, smem + AG_SMEM_COPY, bars->copy, abort, int(blockIdx.x), int(gridDim.x));
  }
  pair::teardown(bars, warp, tmem_base);
}

int default_rpb(int K, int M_shard) {
  int rpb = std::max(1, int(131072 / (size_t(K) * 2)));  // about 128 KB of A per chunk
  return std::min(rpb, M_shard);
}

}  // namespace
}  // namespace tl

extern "C" int tl_ag_gemm_num_flags(int R, int M_shard, int K, int rows_per_barrier, int* effective_rpb) {
  if (R < 1 || M_shard < 1 || K < 1) return -1;
  int rpb = rows_per_barrier > 0 ? std::min(rows_per_barrier, M_shard) : tl::default_rpb(K, M_shard);
  if (effective_rpb) *effective_rpb = rpb;
  return R * tl::cdiv(M_shard, rpb);
}

extern "C" size_t tl_ag_gemm_workspace_size(int R, int M_shard, int K, int N, int sm_count) {
  if (R < 1 || M_shard < 1 || K < 1 || N < 1) return 0;
  if (sm_count <= 0) {
    tl::DeviceInfo di{};
    if (tl::device_info(&di)) return 0;
    sm_count = di.sm_count;
  }
  const long long tiles = ((long long)R * M_shard + tl::pair::BM - 1) / tl::pair::BM * tl::cdiv(N, tl::pair::BN);
  const int S = tl::splitk::choose(tiles, tl::cdiv(K, tl::pair::BK), sm_count / 2);
  return tl::splitk::workspace_bytes(tiles, S);
}

extern "C" tl_status tl_ag_gemm_tile_order(int R, int self_rank, int M_shard, int32_t* m_order, int capacity) {
  if (R < 1 || R > TL_MAX_RANKS || self_rank < 0 || self_rank >= R || M_shard < 1 || !m_order)
    return tl::fail(TL_ERR_INVALID, "tl_ag_gemm_tile_order: bad arguments");
  const long long M = (long long)R * M_shard;
  const int Mt = int((M + tl::pair::BM - 1) / tl::pair::BM);
  if (capacity < Mt) return tl::fail(TL_ERR_INVALID, "tl_ag_gemm_tile_order: capacity %d < %d tiles", capacity, Mt);
  // arrival position of shard r is (r - self) mod R; a row tile takes the latest
  // position among the shards its rows come from; stable by tile index
  std::vector<std::pair<int, int>> key(Mt);
  for (int m = 0; m < Mt; ++m) {
    const long long r0 = (long long)m * tl::pair::BM, r1 = std::min(M, r0 + tl::pair::BM) - 1;
    int best = 0;
    for (long long r = r0 / M_shard; r <= r1 / M_shard; ++r) best = std::max(best, int((r - self_rank + R) % R));
    key[m] = {best, m};
  }
  std::sort(key.begin(), key.end());
  for (int i = 0; i < Mt; ++i) m_order[i] = key[i].second;
  return TL_OK;
}

extern "C" tl_status tl_ag_gemm(const tl_ag_gemm_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_ag_gemm: NULL args");
  if (a->R < 1 || a->R > TL_MAX_RANKS) return fail(TL_ERR_INVALID, "tl_ag_gemm: R=%d outside 1..%d", a->R, TL_MAX_RANKS);
  if (a->self_rank < 0 || a->self_rank >= a->R) return fail(TL_ERR_INVALID, "tl_ag_gemm: self_rank %d", a->self_rank);
  if (a->M_shard < 1 || a->K < 1 || a->N < 1) return fail(TL_ERR_INVALID, "tl_ag_gemm: empty shape");
  if (a->K % 8 || a->N % 8)
    return fail(TL_ERR_UNSUPPORTED, "tl_ag_gemm: K (%d) and N (%d) must be multiples of 8", a->K, a->N);
  if (a->mode != TL_MODE_PULL && a->mode != TL_MODE_PUSH) return fail(TL_ERR_INVALID, "tl_ag_gemm: mode %d", a->mode);
  if (a->mode == TL_MODE_PULL && !a->src_ready)
    return fail(TL_ERR_INVALID, "tl_ag_gemm: pull mode needs src_ready flags");
  if (a->swizzle != TL_SWIZZLE_ARRIVAL && a->swizzle != TL_SWIZZLE_ROWS)
    return fail(TL_ERR_INVALID, "tl_ag_gemm: swizzle %d", a->swizzle);
  if (!a->A_shards || !a->B || !a->gathered || !a->C || !a->signals)
    return fail(TL_ERR_INVALID, "tl_ag_gemm: NULL pointer argument");
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "tl_ag_gemm: epoch must be nonzero");
  for (int r = 0; r < a->R; ++r)
    if (!a->A_shards[r] || !aligned16(a->A_shards[r])) return fail(TL_ERR_INVALID, "tl_ag_gemm: shard %d pointer", r);
  if (!aligned16(a->B) || !aligned16(a->gathered) || !aligned16(a->C) || (a->C_f32 && !aligned16(a->C_f32)) ||
      (a->workspace && !aligned16(a->workspace)))
    return fail(TL_ERR_INVALID, "tl_ag_gemm: pointers must be 16-byte aligned");
  const long long M = (long long)a->R * a->M_shard;
  const int Mt = int((M + pair::BM - 1) / pair::BM);
  if (M > (1ll << 30) || Mt > AG_MAX_MTILES)
    return fail(TL_ERR_UNSUPPORTED, "tl_ag_gemm: %lld rows exceeds %d row tiles", M, AG_MAX_MTILES);
  int rpb = 0;
  const int nflags = tl_ag_gemm_num_flags(a->R, a->M_shard, a->K, a->rows_per_barrier, &rpb);
  if (rpb < 1 || size_t(rpb) * a->K * 2 > (size_t(1) << 31))
    return fail(TL_ERR_INVALID, "tl_ag_gemm: rows_per_barrier %d", rpb);
  if (a->signals->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_ag_gemm: signals hold %d flags, need %d", a->signals->num_flags, nflags);
  if (a->mode == TL_MODE_PULL && a->src_ready->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_ag_gemm: src_ready holds %d flags, need %d", a->src_ready->num_flags, nflags);
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  if (a->signals->device != di.device) return fail(TL_ERR_INVALID, "tl_ag_gemm: signals belong to another device");
  const uint8_t* shard_dev[TL_MAX_RANKS];
  uint64_t host_mask = 0;
  if (tl_status s = classify_shards("tl_ag_gemm", a->A_shards, a->R, di.device, shard_dev, &host_mask)) return s;
  if ((host_mask >> a->self_rank) & 1ull)
    return fail(TL_ERR_UNSUPPORTED, "tl_ag_gemm: the self shard is read in place by TMA and must be device memory");

  AgParams* p = new (std::nothrow) AgParams;
  if (!p) return fail(TL_ERR_INTERNAL, "out of host memory");
  std::memset(p, 0, sizeof(AgParams));
  tl_status st = TL_OK;
  do {
    if ((st = make_map_bf16(&p->map_g, a->gathered, M, a->K, size_t(a->K) * 2, pair::HM, pair::BK))) break;
    if ((st = make_map_bf16(&p->map_self, a->A_shards[a->self_rank], a->M_shard, a->K, size_t(a->K) * 2, pair::HM,
                            pair::BK)))
      break;
    if ((st = make_map_bf16(&p->map_b, a->B, a->K, a->N, size_t(a->N) * 2, pair::BK, 64))) break;
    if ((st = make_map_bf16(&p->map_c, a->C, M, a->N, size_t(a->N) * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))) break;
    for (int r = 0; r < a->R; ++r) p->shard[r] = shard_dev[r];
    p->host_mask = host_mask;
    p->gathered = static_cast<uint8_t*>(a->gathered);
    p->C = static_cast<uint16_t*>(a->C);
    p->C_f32 = a->C_f32;
    p->flags = a->signals->flags;
    p->ready = a->mode == TL_MODE_PULL ? a->src_ready->flags : nullptr;
    p->status = a->signals->status;
    p->trace = a->trace;
    p->timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
    p->pipe_timeout_ns = 2 * p->timeout_ns + 1000000000ull;
    p->R = a->R;
    p->self = a->self_rank;
    p->M_shard = a->M_shard;
    p->K = a->K;
    p->N = a->N;
    p->M = int(M);
    p->rpb = rpb;
    p->bpr = cdiv(a->M_shard, rpb);
    p->Mt = Mt;
    p->Nt = cdiv(a->N, pair::BN);
    p->KB = cdiv(a->K, pair::BK);
    p->num_items = a->R * p->bpr;
    p->epoch = a->epoch;
    if ((st = test_hold("tl_ag_gemm", p->timeout_ns, &p->hold_first, &p->hold_count, &p->hold_ns))) break;
    // split-K when the tiles leave pairs idle and the caller gave a workspace
    const long long tiles = (long long)Mt * p->Nt;
    p->S = a->workspace ? splitk::choose(tiles, p->KB, di.sm_count / 2) : 1;
    if (p->S > 1) {
      const size_t need = splitk::workspace_bytes(tiles, p->S);
      if (a->workspace_bytes < need) {
        st = fail(TL_ERR_INVALID, "tl_ag_gemm: workspace of %zu bytes, split-K needs %zu", a->workspace_bytes, need);
        break;
      }
      uint8_t* ws = static_cast<uint8_t*>(a->workspace);
      p->sk.counters = reinterpret_cast<uint32_t*>(ws);
      p->sk.partials = reinterpret_cast<float*>(ws + splitk::counter_bytes(tiles));
      p->sk.tag = (a->epoch % 0xFFFFFFu + 1u) << 8;  // nonzero; repeats every 2^24 - 1 epochs
      p->sk.timeout_ns = p->timeout_ns;
      p->sk.S = p->S;
    }
    p->KBs = p->KB / p->S;
    p->num_work = int(tiles) * p->S;
    int32_t order[AG_MAX_MTILES];
    if ((st = tl_ag_gemm_tile_order(a->R, a->self_rank, a->M_shard, order, AG_MAX_MTILES))) break;
    for (int i = 0; i < Mt; ++i) p->m_order[i] = uint16_t(a->swizzle == TL_SWIZZLE_ROWS ? i : order[i]);
    const int pairs = std::max(1, std::min(di.sm_count / 2, std::max(p->num_work, (p->num_items + 1) / 2)));
    void* args[] = {p};
    st = launch_coop(reinterpret_cast<const void*>(&ag_gemm_kernel), 2 * pairs, AG_THREADS, AG_SMEM_BYTES,
                     (cudaStream_t)stream, args, 2);
  } while (false);
  delete p;
  return st;
}
