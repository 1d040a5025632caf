// tl_attn.cu -- AllGather-KV attention: the key/value AllGather fused with the
// attention that consumes it, at 128-token granularity, in one launch.
//
// TileLink talk summary ("TileLink: Generating Efficient Compute-Communication
// Overlapping Kernels using Tile-Centric Primitives"):
//  * Key Findings / Experimental Setup & Results -- attention layers: the
//    AllGather of the keys and values overlapped with the attention that
//    reads them (compared with Ring Attention).
//  * Technical Deep Dive -- produce_tile_notify / consume_tile_wait: the copy
//    of a chunk releases its flag; the consumer acquires it before loading.
//
// A persistent grid of single CTAs (one per SM) runs work units of (head h,
// 256 query rows): two 128-row query tiles A and B that share every key/value
// tile.
//   warp 0      TMA producer: the unit's Q tiles, then per key/value tile its
//               arrival flags (peers' shards only), K (128 keys x 128 dims)
//               and V (128 keys x 128 dims) into two- and three-stage rings.
//   warp 1      MMA issuer: S_X = Q_X K^T and O_X += P_X V with
//               tcgen05.mma.cta_group::1 (M = 128, N = 128), in the order
//               QK_A(0) QK_B(0) | PV_A(j) QK_A(j+1) PV_B(j) QK_B(j+1) | ...,
//               so that one tile's softmax runs while the tensor cores work on
//               the other tile.  P V takes its A operand (P) from TMEM.
//   warp 2      copy warp (AllGather producer): the AllGather-GEMM's item
//               order and flags, but plain 16-byte loads and stores instead of
//               bulk copies through shared memory, whose room holds the third
//               V stage (7.10 against 7.28 ms with two V stages and staging).
//   warp 3      idle.
//   warps 4-7   softmax of tile A, warps 8-11 of tile B, one query row per
//               thread: S from TMEM, running max m and sum l (base 2), P as
//               bf16 pairs written back over the first 64 columns of the
//               row's S (tcgen05.st), O in TMEM rescaled only when m grows by
//               more than 8 (P <= 2^8 between rescales), and the final O / l
//               and LSE.
//
// TMEM (lane = query row of the tile): S_A cols 0-127 (P_A in 0-63), S_B
// 128-255 (P_B in 128-191), O_A 256-383, O_B 384-511.  The tensor pipe runs
// one thread's MMAs in issue order, so the QK that overwrites S_X with the
// next tile's scores follows the P V that reads P_X from the same columns.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "tl_copy.cuh"
#include "tl_internal.h"

namespace tl {
namespace {

constexpr int HD = 128;          // head dim
constexpr int KV_TILE = 128;     // keys per tile (the flag granularity too)
constexpr int Q_ROWS = 128;      // query rows per tile
constexpr int UNIT_ROWS = 256;   // two 128-row tiles per unit
constexpr int KST = 2;           // K ring stages
constexpr int VST = 3;           // V ring stages
constexpr int ATT_THREADS = 12 * 32;
constexpr int kWarpCopyA = 2;
constexpr int kWarpSoftmax0 = 4;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the running max grows by more than this

constexpr uint32_t BOX = 128 * 64 * 2;         // 16 KB: 128 rows x 64 dims, one 128-byte swizzle span wide
constexpr uint32_t Q_TILE = 2 * BOX;           // 32 KB: 128 query rows x 128 dims (K-major)
constexpr uint32_t K_STAGE = 2 * BOX;          // 32 KB: 128 keys x 128 dims (K-major)
constexpr uint32_t V_STAGE = 2 * BOX;          // 32 KB: 128 keys x 128 dims (dims contiguous)
constexpr uint32_t SMEM_Q = 0;
constexpr uint32_t SMEM_K = SMEM_Q + 2 * Q_TILE;
constexpr uint32_t SMEM_V = SMEM_K + KST * K_STAGE;
constexpr uint32_t SMEM_BARS = SMEM_V + VST * V_STAGE;

constexpr uint32_t IDESC_QK = idesc_bf16_f32(Q_ROWS, KV_TILE, false);  // B = K rows, K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(Q_ROWS, HD, true);        // B = V [keys, dims], dims contiguous

struct __align__(8) AttnBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[2], p_full[2];
  uint64_t o_full[2], o_empty[2];
  uint32_t tmem_base;
  uint32_t abort;
};
constexpr uint32_t ATT_SMEM_BYTES = SMEM_BARS + sizeof(AttnBars) + 1024;
static_assert(ATT_SMEM_BYTES <= 232448, "attention shared memory above the per-CTA limit");

struct AttnParams {
  CUtensorMap map_q;   // Q [S, H*D], box 128 rows x 64 dims
  CUtensorMap map_kg;  // gathered K [R][S][Hkv*D], box 128 keys x 64 dims
  CUtensorMap map_vg;  // gathered V, box 128 keys x 64 dims
  CUtensorMap map_ks;  // self K shard [1][S][Hkv*D]
  CUtensorMap map_vs;  // self V shard
  const uint8_t* k_shard[TL_MAX_RANKS];
  const uint8_t* v_shard[TL_MAX_RANKS];
  uint8_t* kg;
  uint8_t* vg;
  uint16_t* O;
  float* lse;
  uint32_t* flags;  // K chunk flags [R*T], then V chunk flags [R*T]
  uint32_t* status;
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int32_t R, self, S, H, Hkv, group, causal;
  int32_t T;   // key tiles per shard
  int32_t QB;  // 256-row query blocks
  int32_t num_units, num_items;
  float scale_log2;
  uint32_t epoch;
};

__device__ __forceinline__ void unit_of(const AttnParams& p, int u, int& h, int& qb) {
  h = u / p.QB;
  qb = p.QB - 1 - u % p.QB;  // the longest causal block of a head first
}

// Key tiles of the unit's own shard that its rows can see.
__device__ __forceinline__ int self_tiles(const AttnParams& p, int qb) {
  if (!p.causal) return p.T;
  const int last_row = min(p.S - 1, qb * UNIT_ROWS + UNIT_ROWS - 1);
  return last_row / KV_TILE + 1;
}
__device__ __forceinline__ int unit_tiles(const AttnParams& p, int qb) {
  return p.causal ? self_tiles(p, qb) + p.self * p.T : p.R * p.T;
}
// Key tile j of a unit: the own shard first (in place), then the peers in copy
// order self+1, ... (causal: only the shards before self, in rank order).
__device__ __forceinline__ void tile_of(const AttnParams& p, int qb, int j, int& r, int& t) {
  if (!p.causal) {
    r = (p.self + j / p.T) % p.R;
    t = j % p.T;
    return;
  }
  const int ts = self_tiles(p, qb);
  if (j < ts) {
    r = p.self;
    t = j;
  } else {
    r = (j - ts) / p.T;
    t = (j - ts) % p.T;
  }
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]: A's rows in TMEM lanes, its K elements packed
// two bf16 per 32-bit column (16 elements = 8 columns per instruction).
__device__ __forceinline__ void tc_mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void issue_qk(uint8_t* smem, int X, int ks, uint32_t d_tmem) {
  const uint32_t q0 = smem_u32(smem + SMEM_Q + X * Q_TILE);
  const uint32_t k0 = smem_u32(smem + SMEM_K + ks * K_STAGE);
#pragma unroll
  for (int kk = 0; kk < HD / UMMA_K; ++kk) {
    const uint64_t ad = sdesc_sw128(q0 + (kk >> 2) * BOX + (kk & 3) * 32, 16, 1024);
    const uint64_t bd = sdesc_sw128(k0 + (kk >> 2) * BOX + (kk & 3) * 32, 16, 1024);
    tc_mma_bf16(d_tmem, ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
  }
}

// O += P V, P in the first 64 TMEM columns of the tile's S (keys 2c, 2c+1 in column c);
// V's two 64-dim halves are 128-byte swizzle spans BOX bytes apart.
__device__ __forceinline__ void issue_pv(uint8_t* smem, uint32_t p_tmem, int vs, uint32_t d_tmem, bool accumulate) {
  const uint32_t v0 = smem_u32(smem + SMEM_V + vs * V_STAGE);
#pragma unroll
  for (int kk = 0; kk < KV_TILE / UMMA_K; ++kk) {
    const uint64_t bd = sdesc_sw128(v0 + kk * 2048, BOX, 1024);
    tc_mma_bf16_tmem_a(d_tmem, p_tmem + uint32_t(kk * 8), bd, IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__global__ void __launch_bounds__(ATT_THREADS, 1) ag_attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  AttnBars* bars = reinterpret_cast<AttnBars*>(smem + SMEM_BARS);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const int cta = int(blockIdx.x), nctas = int(gridDim.x);
  volatile uint32_t* abort = &bars->abort;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_q);
    tma_prefetch_desc(&p.map_kg);
    tma_prefetch_desc(&p.map_vg);
    tma_prefetch_desc(&p.map_ks);
    tma_prefetch_desc(&p.map_vs);
  }
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->q_full[x], 1);
      mbar_init(&bars->q_empty[x], 1);
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->p_full[x], 4);
      mbar_init(&bars->o_full[x], 1);
      mbar_init(&bars->o_empty[x], 4);
    }
    for (int s = 0; s < KST; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    int ks = 0, vs = 0;
    uint32_t kph = 0, vph = 0;
    int iu = 0;
    for (int u = cta; u < p.num_units; u += nctas, ++iu) {
      int h, qb;
      unit_of(p, u, h, qb);
      const int hk = h / p.group;
      const int nkv = unit_tiles(p, qb);
      if (lane == 0) {
        for (int X = 0; X < 2; ++X) {
          if (!mbar_wait(&bars->q_empty[X], uint32_t(iu & 1) ^ 1u, abort, p.status, p.pipe_timeout_ns, 11)) break;
          mbar_arrive_expect_tx(&bars->q_full[X], Q_TILE);
          const int y = qb * UNIT_ROWS + X * Q_ROWS;
          uint8_t* dst = smem + SMEM_Q + X * Q_TILE;
          tma_load_2d(dst, &p.map_q, &bars->q_full[X], h * HD, y);
          tma_load_2d(dst + BOX, &p.map_q, &bars->q_full[X], h * HD + 64, y);
        }
      }
      for (int j = 0; j < nkv; ++j) {
        int r, t;
        tile_of(p, qb, j, r, t);
        const bool peer = r != p.self;
        if (peer && lane < 2) {
          // consume_tile_wait: the K (lane 0) and V (lane 1) flags of the chunk
          const int id = r * p.T + t + lane * p.R * p.T;
          wait_flag(p.flags + id, p.epoch, p.status, p.timeout_ns, uint32_t(id), TL_ERR_TIMEOUT);
        }
        __syncwarp();
        if (lane == 0) {
          if (peer) fence_proxy_async_global();
          const CUtensorMap* mk = peer ? &p.map_kg : &p.map_ks;
          const CUtensorMap* mv = peer ? &p.map_vg : &p.map_vs;
          const int z = peer ? r : 0;
          if (mbar_wait(&bars->k_empty[ks], kph ^ 1u, abort, p.status, p.pipe_timeout_ns, 12)) {
            mbar_arrive_expect_tx(&bars->k_full[ks], K_STAGE);
            uint8_t* dst = smem + SMEM_K + ks * K_STAGE;
            tma_load_3d(dst, mk, &bars->k_full[ks], hk * HD, t * KV_TILE, z);
            tma_load_3d(dst + BOX, mk, &bars->k_full[ks], hk * HD + 64, t * KV_TILE, z);
            if (++ks == KST) {
              ks = 0;
              kph ^= 1u;
            }
          }
          if (mbar_wait(&bars->v_empty[vs], vph ^ 1u, abort, p.status, p.pipe_timeout_ns, 13)) {
            mbar_arrive_expect_tx(&bars->v_full[vs], V_STAGE);
            uint8_t* dst = smem + SMEM_V + vs * V_STAGE;
            tma_load_3d(dst, mv, &bars->v_full[vs], hk * HD, t * KV_TILE, z);
            tma_load_3d(dst + BOX, mv, &bars->v_full[vs], hk * HD + 64, t * KV_TILE, z);
            if (++vs == VST) {
              vs = 0;
              vph ^= 1u;
            }
          }
        }
        if (__shfl_sync(0xffffffffu, *abort, 0)) break;
      }
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      uint32_t pcount[2] = {0, 0};
      int iu = 0;
      const uint32_t s_tmem[2] = {tmem_base, tmem_base + 128};
      const uint32_t o_tmem[2] = {tmem_base + 256, tmem_base + 384};
      for (int u = cta; u < p.num_units && !*abort; u += nctas, ++iu) {
        int h, qb;
        unit_of(p, u, h, qb);
        const int nkv = unit_tiles(p, qb);
        const uint32_t uph = uint32_t(iu & 1);
        bool ok = mbar_wait(&bars->q_full[0], uph, abort, p.status, p.pipe_timeout_ns, 21) &&
                  mbar_wait(&bars->q_full[1], uph, abort, p.status, p.pipe_timeout_ns, 21) &&
                  mbar_wait(&bars->k_full[ks], kph, abort, p.status, p.pipe_timeout_ns, 22);
        if (!ok) break;
        tc_fence_after();
        for (int X = 0; X < 2; ++X) {
          issue_qk(smem, X, ks, s_tmem[X]);
          tc_commit(&bars->s_full[X]);
          if (nkv == 1) tc_commit(&bars->q_empty[X]);
        }
        tc_commit(&bars->k_empty[ks]);
        if (++ks == KST) {
          ks = 0;
          kph ^= 1u;
        }
        for (int j = 0; j < nkv && ok; ++j) {
          if (!(ok = mbar_wait(&bars->v_full[vs], vph, abort, p.status, p.pipe_timeout_ns, 23))) break;
          for (int X = 0; X < 2; ++X) {
            ok = mbar_wait(&bars->p_full[X], pcount[X] & 1u, abort, p.status, p.pipe_timeout_ns, 24);
            ++pcount[X];
            if (ok && j == 0) ok = mbar_wait(&bars->o_empty[X], uph ^ 1u, abort, p.status, p.pipe_timeout_ns, 25);
            if (!ok) break;
            tc_fence_after();
            issue_pv(smem, s_tmem[X], vs, o_tmem[X], j > 0);
            if (X == 1) {
              tc_commit(&bars->v_empty[vs]);
              if (++vs == VST) {
                vs = 0;
                vph ^= 1u;
              }
            }
            if (j + 1 < nkv) {
              if (X == 0) {
                if (!(ok = mbar_wait(&bars->k_full[ks], kph, abort, p.status, p.pipe_timeout_ns, 26))) break;
                tc_fence_after();
              }
              issue_qk(smem, X, ks, s_tmem[X]);
              tc_commit(&bars->s_full[X]);
              if (j + 2 == nkv) tc_commit(&bars->q_empty[X]);
              if (X == 1) {
                tc_commit(&bars->k_empty[ks]);
                if (++ks == KST) {
                  ks = 0;
                  kph ^= 1u;
                }
              }
            } else {
              tc_commit(&bars->o_full[X]);
            }
          }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == kWarpCopyA) {
    // ---------------------------------------------------------------- AllGather producer (K and V chunks)
    // every shard, in device or pinned host memory, is copied with plain loads
    AgCopyJob jk{p.k_shard, p.kg, p.flags, nullptr, p.status, p.timeout_ns, p.pipe_timeout_ns,
                 p.R, p.self, p.S, p.Hkv * HD, KV_TILE, p.T, p.num_items, p.epoch, 0};
    AgCopyJob jv{p.v_shard, p.vg, p.flags + p.R * p.T, nullptr, p.status, p.timeout_ns, p.pipe_timeout_ns,
                 p.R, p.self, p.S, p.Hkv * HD, KV_TILE, p.T, p.num_items, p.epoch, 0};
    for (int it = cta; it < p.num_items; it += nctas) {
      ag_copy_one_plain(jk, it);
      ag_copy_one_plain(jv, it);
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
    }
  } else if (warp >= kWarpSoftmax0) {
    // ---------------------------------------------------------------- softmax warps (one row per thread)
    const int X = (warp - kWarpSoftmax0) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // row of the tile = TMEM lane
    const uint32_t lane_base = uint32_t(wq * 32) << 16;
    const uint32_t s_addr = tmem_base + lane_base + uint32_t(X * 128);
    const uint32_t o_addr = tmem_base + lane_base + uint32_t(256 + X * 128);
    uint32_t sc = 0;
    int iu = 0;
    bool ok = true;
    for (int u = cta; u < p.num_units && ok; u += nctas, ++iu) {
      int h, qb;
      unit_of(p, u, h, qb);
      const int nkv = unit_tiles(p, qb);
      const int qrow = qb * UNIT_ROWS + X * Q_ROWS + row;  // row in the shard
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < nkv; ++j) {
        int r, t;
        tile_of(p, qb, j, r, t);
        ok = mbar_wait(&bars->s_full[X], sc & 1u, abort, p.status, p.pipe_timeout_ns, 31);
        ++sc;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32cols(s_addr + uint32_t(c * 32), v[c]);
        tmem_ld_wait();
        // keys this row may not see: past the shard's end, or after the query (causal, own shard)
        int lim = min(KV_TILE, p.S - t * KV_TILE);
        if (p.causal && r == p.self) lim = min(lim, qrow - t * KV_TILE + 1);
        if (lim < KV_TILE) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i >= lim) v[c][i] = __float_as_uint(-INFINITY);
        }
        // row max in eight independent chains (a single chain would serialise 128 dependent maxima)
        float mq[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t* x = &v[q >> 1][(q & 1) * 16];
          float a = fmax3(__uint_as_float(x[0]), __uint_as_float(x[1]), __uint_as_float(x[2]));
#pragma unroll
          for (int i = 3; i < 15; i += 2) a = fmax3(a, __uint_as_float(x[i]), __uint_as_float(x[i + 1]));
          mq[q] = fmaxf(a, __uint_as_float(x[15]));
        }
        const float mx = fmaxf(fmax3(mq[0], mq[1], mq[2]), fmax3(fmax3(mq[3], mq[4], mq[5]), mq[6], mq[7]));
        const float mnew = fmaxf(m, mx * p.scale_log2);
        const bool resc = mnew > m + kRescaleLog2;
        float alpha = 1.0f;
        if (resc) {
          alpha = ex2_approx(m - mnew);
          m = mnew;
          l *= alpha;
        }
        const float neg_m = (m == -INFINITY) ? 0.0f : -m;
        float sq[8];  // eight partial row sums
#pragma unroll
        for (int q = 0; q < 8; ++q) sq[q] = 0.0f;
        // P as bf16 pairs over the first 64 columns of S (all of S is in registers by now)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = c * 64 + 2 * i;
            const float p0 = ex2_approx(fmaf(__uint_as_float(v[key >> 5][key & 31]), p.scale_log2, neg_m));
            const float p1 = ex2_approx(fmaf(__uint_as_float(v[(key + 1) >> 5][(key + 1) & 31]), p.scale_log2, neg_m));
            sq[i & 7] += p0 + p1;
            w[i] = pack_bf16x2(p0, p1);
          }
          tmem_st_32cols(s_addr + uint32_t(c * 32), w);
          if (c == 0 && j > 0 && __any_sync(0xffffffffu, resc)) {
            // O rescale, here where half of S is dead (fewer live registers)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t o[32];
              tmem_ld_32cols(o_addr + uint32_t(q * 32), o);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st_32cols(o_addr + uint32_t(q * 32), o);
            }
          }
        }
        l += ((sq[0] + sq[1]) + (sq[2] + sq[3])) + ((sq[4] + sq[5]) + (sq[6] + sq[7]));
        // P and the rescaled O are in TMEM before the next MMAs read them
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[X]);
      }
      if (!ok) break;
      ok = mbar_wait(&bars->o_full[X], uint32_t(iu & 1), abort, p.status, p.pipe_timeout_ns, 32);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const bool row_ok = qrow < p.S;
      uint16_t* orow = p.O + (size_t(qrow) * p.H + h) * HD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld_32cols(o_addr + uint32_t(c * 32), o);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[g * 8 + 2 * e]) * inv_l, __uint_as_float(o[g * 8 + 2 * e + 1]) * inv_l);
            st_global_v4(orow + c * 32 + g * 8, w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (row_ok && p.lse) p.lse[size_t(h) * p.S + qrow] = (m + log2f(l)) * 0.69314718055994531f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty[X]);
    }
  }

  // teardown: every thread is done with TMEM; after an abort, TMA loads that
  // nobody waits for land before the CTA's shared memory is released
  tc_fence_before();
  __syncthreads();
  if (bars->abort) {
    const uint64_t t0 = now_ns();
    while (now_ns() - t0 < 50000) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace
}  // namespace tl

extern "C" int tl_ag_attn_num_flags(int R, int S_shard) {
  if (R < 1 || S_shard < 1) return -1;
  return 2 * R * tl::cdiv(S_shard, tl::KV_TILE);
}

extern "C" tl_status tl_ag_attn(const tl_ag_attn_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_ag_attn: NULL args");
  if (a->R < 1 || a->R > TL_MAX_RANKS) return fail(TL_ERR_INVALID, "tl_ag_attn: R=%d outside 1..%d", a->R, TL_MAX_RANKS);
  if (a->self_rank < 0 || a->self_rank >= a->R) return fail(TL_ERR_INVALID, "tl_ag_attn: self_rank %d", a->self_rank);
  if (a->S_shard < 1 || a->H < 1 || a->H_kv < 1) return fail(TL_ERR_INVALID, "tl_ag_attn: empty shape");
  if (a->H % a->H_kv) return fail(TL_ERR_INVALID, "tl_ag_attn: H=%d is not a multiple of H_kv=%d", a->H, a->H_kv);
  if (a->head_dim != HD) return fail(TL_ERR_UNSUPPORTED, "tl_ag_attn: head_dim %d (only %d)", a->head_dim, HD);
  if (a->causal != 0 && a->causal != 1) return fail(TL_ERR_INVALID, "tl_ag_attn: causal %d", a->causal);
  if (!(a->scale >= 0.0f) || std::isinf(a->scale))
    return fail(TL_ERR_INVALID, "tl_ag_attn: scale must be positive and finite (0 = 1/sqrt(head_dim))");
  if (!a->Q || !a->K_shards || !a->V_shards || !a->K_gathered || !a->V_gathered || !a->O || !a->signals)
    return fail(TL_ERR_INVALID, "tl_ag_attn: NULL pointer argument");
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "tl_ag_attn: epoch must be nonzero");
  for (int r = 0; r < a->R; ++r)
    if (!a->K_shards[r] || !a->V_shards[r] || !aligned16(a->K_shards[r]) || !aligned16(a->V_shards[r]))
      return fail(TL_ERR_INVALID, "tl_ag_attn: shard %d pointer", r);
  if (!aligned16(a->Q) || !aligned16(a->K_gathered) || !aligned16(a->V_gathered) || !aligned16(a->O) ||
      (reinterpret_cast<uintptr_t>(a->lse) & 3u))
    return fail(TL_ERR_INVALID, "tl_ag_attn: pointers must be 16-byte aligned (lse 4-byte)");
  const long long S = a->S_shard;
  if ((long long)a->R * S > (1ll << 30) || (long long)a->H * HD > (1ll << 24) || (long long)a->H_kv * HD > (1ll << 24))
    return fail(TL_ERR_UNSUPPORTED, "tl_ag_attn: shape too large");
  const int T = cdiv(a->S_shard, KV_TILE);
  const int QB = cdiv(a->S_shard, UNIT_ROWS);
  if ((long long)a->H * QB > (1ll << 30)) return fail(TL_ERR_UNSUPPORTED, "tl_ag_attn: too many work units");
  const int nflags = tl_ag_attn_num_flags(a->R, a->S_shard);
  if (a->signals->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_ag_attn: signals hold %d flags, need %d", a->signals->num_flags, nflags);
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  if (a->signals->device != di.device) return fail(TL_ERR_INVALID, "tl_ag_attn: signals belong to another device");
  const uint8_t* kdev[TL_MAX_RANKS];
  const uint8_t* vdev[TL_MAX_RANKS];
  uint64_t kmask = 0, vmask = 0;
  if (tl_status s = classify_shards("tl_ag_attn (K)", a->K_shards, a->R, di.device, kdev, &kmask)) return s;
  if (tl_status s = classify_shards("tl_ag_attn (V)", a->V_shards, a->R, di.device, vdev, &vmask)) return s;
  if (((kmask | vmask) >> a->self_rank) & 1ull)
    return fail(TL_ERR_UNSUPPORTED, "tl_ag_attn: the self shards are read in place by TMA and must be device memory");

  AttnParams* p = new (std::nothrow) AttnParams;
  if (!p) return fail(TL_ERR_INTERNAL, "out of host memory");
  std::memset(p, 0, sizeof(AttnParams));
  tl_status st = TL_OK;
  const uint64_t kv_cols = uint64_t(a->H_kv) * HD;
  const uint64_t kv_pitch = kv_cols * 2;
  do {
    if ((st = make_map_bf16(&p->map_q, a->Q, S, uint64_t(a->H) * HD, uint64_t(a->H) * HD * 2, Q_ROWS, 64))) break;
    if ((st = make_map_bf16_3d(&p->map_kg, a->K_gathered, a->R, S, kv_cols, kv_pitch, S * kv_pitch, KV_TILE, 64)))
      break;
    if ((st = make_map_bf16_3d(&p->map_vg, a->V_gathered, a->R, S, kv_cols, kv_pitch, S * kv_pitch, KV_TILE, 64)))
      break;
    if ((st = make_map_bf16_3d(&p->map_ks, a->K_shards[a->self_rank], 1, S, kv_cols, kv_pitch, S * kv_pitch, KV_TILE,
                               64)))
      break;
    if ((st = make_map_bf16_3d(&p->map_vs, a->V_shards[a->self_rank], 1, S, kv_cols, kv_pitch, S * kv_pitch, KV_TILE,
                               64)))
      break;
    for (int r = 0; r < a->R; ++r) {
      p->k_shard[r] = kdev[r];
      p->v_shard[r] = vdev[r];
    }
    p->kg = static_cast<uint8_t*>(a->K_gathered);
    p->vg = static_cast<uint8_t*>(a->V_gathered);
    p->O = static_cast<uint16_t*>(a->O);
    p->lse = a->lse;
    p->flags = a->signals->flags;
    p->status = a->signals->status;
    p->timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
    p->pipe_timeout_ns = 2 * p->timeout_ns + 1000000000ull;
    p->R = a->R;
    p->self = a->self_rank;
    p->S = a->S_shard;
    p->H = a->H;
    p->Hkv = a->H_kv;
    p->group = a->H / a->H_kv;
    p->causal = a->causal;
    p->T = T;
    p->QB = QB;
    p->num_units = a->H * QB;
    p->num_items = a->R * T;
    const float scale = a->scale > 0.0f ? a->scale : 1.0f / std::sqrt(float(HD));
    p->scale_log2 = scale * 1.4426950408889634f;
    p->epoch = a->epoch;
    const int ctas = std::max(1, std::min(di.sm_count, std::max(p->num_units, p->num_items)));
    void* args[] = {p};
    st = launch_coop(reinterpret_cast<const void*>(&ag_attn_kernel), ctas, ATT_THREADS, ATT_SMEM_BYTES,
                     (cudaStream_t)stream, args, 1);
  } while (false);
  delete p;
  return st;
}
