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
// Work items: output tile tau = (dest d, m tile, n tile) in destination order,
// within a destination n tile by n tile with the m tiles innermost (a wave's
// tiles share B columns and the destination's A rows, which stay in L2); its R
// partial tiles P_r = A_r[rows of tau] . B_r[:, cols of tau] are items
// tau*R + j, rank r = (d + 1 + tau + j) mod R (the rotation spreads the
// destination rank's own item over the CTAs).  The grid is a multiple of R and
// items go round-robin, so the R items of a tile always run in the same wave.
//
// Receive slots form a ring of 2 * grid slots: item i pushes into slot
// i mod (2 * grid), after the R reducers of the tile that used the slot before
// have released their "reduced" flags.  The ring (about 38 MB for 152 SMs)
// stays in L2.  Deadlock freedom: every wait of a wave-w pusher is on waves
// <= w - 2 or on its own CTA's MMA; every wait of a wave-w reducer is on
// wave-w pushers; by induction on w every wave completes.
//
// Per CTA: warp 0 TMA producer (A_r, B_r k-blocks), warp 1 tcgen05 MMA issuer,
// warps 2-5 pushers, warps 6-9 reducers.  For item (tau, j):
//   push:   TMEM -> registers -> fp32 receive slot of the item; release the
//           arrival flag tau*R + r (produce_tile_notify).  Before reusing a ring
//           slot the pushers acquire the "reduced" flags of the tile that last
//           used it (the slot-free barrier of the pull protocol).
//   reduce: acquire the R arrival flags of tau (consume_tile_wait on its own
//           partial, peer_tile_wait on the others), sum row slice j of the tile
//           over the R slots in rank order 0..R-1 in fp32, store bf16 rows of
//           out[d], then release the "reduced" flag of (tau, j).
// Pushers never wait on peers' partials and reducers never hold TMEM, so the
// tensor pipe is not stalled by the reduction.  Flags: [0, items) arrival
// flags indexed tau*R + r; [items, 2*items) reduced flags indexed tau*R + j.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "tl_common.cuh"
#include "tl_internal.h"

namespace tl {
namespace {

constexpr int RS_MAX_RANKS = 32;
constexpr int kWarpRed0 = kWarpEpi0 + kNumEpiWarps;  // first reducer warp
constexpr int kNumRedWarps = 4;
constexpr int kNumRedThreads = kNumRedWarps * 32;
constexpr int RS_THREADS = (kWarpRed0 + kNumRedWarps) * 32;
constexpr uint32_t RS_SMEM_BARS = SMEM_GEMM_END;
constexpr uint32_t RS_SMEM_BYTES = RS_SMEM_BARS + sizeof(Barriers) + 1024;
constexpr int SLOT_FLOATS = BM * BN;  // one fp32 partial tile
constexpr int RB = 8;                 // ranks loaded per batch in the reduce
constexpr int QU = 2;                 // float4 elements per thread per round in the reduce

struct RsParams {
  CUtensorMap map_a[RS_MAX_RANKS];  // A_r [M, K_r]
  CUtensorMap map_b[RS_MAX_RANKS];  // B_r [K_r, N]
  uint16_t* out[RS_MAX_RANKS];      // out[d] [Md, N] bf16
  float* slots;                     // [ring_slots][BM*BN] fp32 receive slots
  uint32_t* flags;                  // [2][num_tiles][R]: arrival, then reduced
  uint32_t* status;
  int32_t* trace;                   // optional: tile and rank of each item
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int32_t R, M, Md, K, N;
  int32_t Mt_d, Nt, KB, num_tiles, num_items, slice_rows, ring_slots;
  uint32_t epoch;
};

struct Item {
  int tau, d, mt, nt, r, j;
};

__device__ __forceinline__ Item item_of(const RsParams& p, int i) {
  Item it;
  it.tau = i / p.R;
  it.j = i % p.R;
  const int per_d = p.Mt_d * p.Nt;
  it.d = it.tau / per_d;
  const int rem = it.tau % per_d;
  it.mt = rem % p.Mt_d;
  it.nt = rem / p.Mt_d;
  it.r = (it.d + 1 + it.tau + it.j) % p.R;
  return it;
}

__global__ void __launch_bounds__(RS_THREADS, 1) gemm_rs_kernel(const __grid_constant__ RsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + RS_SMEM_BARS);
  const int warp = int(warp_id());
  const int lane = int(lane_id());

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tmem_full[a], 1);
      mbar_init(&bars->tmem_empty[a], kNumEpiWarps);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  volatile uint32_t* abort = &bars->abort;

  if (warp == kWarpTma) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      for (int i = blockIdx.x; i < p.num_items && !*abort; i += gridDim.x) {
        const Item it = item_of(p, i);
        if (p.trace) p.trace[i] = ((it.d * p.Mt_d + it.mt) * p.Nt + it.nt) * p.R + it.r;
        const int row0 = it.d * p.Md + it.mt * BM;
        const CUtensorMap* ma = &p.map_a[it.r];
        const CUtensorMap* mb = &p.map_b[it.r];
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(&bars->empty[s], ph ^ 1u, abort, p.status, p.pipe_timeout_ns, 1)) break;
          mbar_arrive_expect_tx(&bars->full[s], STAGE_TX);
          tma_load_2d(smem + SMEM_A + s * A_STAGE_BYTES, ma, &bars->full[s], kb * BK, row0);
          uint8_t* b_dst = smem + SMEM_B + s * B_STAGE_BYTES;
#pragma unroll
          for (int q = 0; q < BN / 64; ++q)
            tma_load_2d(b_dst + q * B_BOX_BYTES, mb, &bars->full[s], it.nt * BN + q * 64, kb * BK);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int jj = 0;
      for (int i = blockIdx.x; i < p.num_items && !*abort; i += gridDim.x, ++jj) {
        const int acc = jj & 1;
        const uint32_t acc_ph = uint32_t(jj >> 1) & 1u;
        if (!mbar_wait(&bars->tmem_empty[acc], acc_ph ^ 1u, abort, p.status, p.pipe_timeout_ns, 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(&bars->full[s], ph, abort, p.status, p.pipe_timeout_ns, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_kblock(smem, s, d_tmem, kb == 0);
          tc_commit(&bars->empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&bars->tmem_full[acc]);
      }
    }
    __syncwarp();
  } else if (warp < kWarpRed0) {
    // ---------------------------------------------------------------- pushers
    const int wq = warp & 3;                         // TMEM lane quarter of this warp
    const int et = (warp - kWarpEpi0) * 32 + lane;  // 0..127 among pusher threads
    const int row_in_tile = wq * 32 + lane;
    uint32_t* reduced = p.flags + p.num_items;
    int jj = 0;
    for (int i = blockIdx.x; i < p.num_items; i += gridDim.x, ++jj) {
      const Item it = item_of(p, i);
      const int acc = jj & 1;
      const uint32_t acc_ph = uint32_t(jj >> 1) & 1u;
      // slot free: the R reducers of the tile that last used this ring slot are done with it
      if (i >= p.ring_slots && lane == 0) {
        const int prev_tau = (i - p.ring_slots) / p.R;
        for (int j = 0; j < p.R; ++j)
          wait_flag(reduced + size_t(prev_tau) * p.R + j, p.epoch, p.status, p.timeout_ns,
                    uint32_t(p.num_items + prev_tau * p.R + j), TL_ERR_TIMEOUT);
      }
      __syncwarp();
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      // all four pusher warps leave together (they meet at a named barrier below)
      if (!named_bar_and(1, kNumEpiThreads, ok)) break;
      tc_fence_after();
      // slot layout [col/4][row][4]: a warp writes 512 contiguous bytes per store
      float* slot = p.slots + size_t(i % p.ring_slots) * SLOT_FLOATS;
      for (int c = 0; c < BN / 32; ++c) {
        if (it.nt * BN + c * 32 >= p.N) break;
        uint32_t v[32];
        tmem_ld_32cols(tmem_base + (uint32_t(wq * 32) << 16) + uint32_t(acc * BN + c * 32), v);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float* f = reinterpret_cast<const float*>(v + g * 4);
          st_global_cg_v4f(slot + (size_t(c * 8 + g) * BM + row_in_tile) * 4, f[0], f[1], f[2], f[3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tmem_empty[acc]);
      // produce_tile_notify: the barrier orders every pusher thread's writes before
      // thread 0's gpu-scope release, which makes them visible to its acquirers
      named_bar_sync(1, kNumEpiThreads);
      if (et == 0) st_release(p.flags + size_t(it.tau) * p.R + it.r, p.epoch);
    }
  } else {
    // ---------------------------------------------------------------- reducers
    const int et = (warp - kWarpRed0) * 32 + lane;  // 0..127 among reducer threads
    uint32_t* reduced = p.flags + p.num_items;
    for (int i = blockIdx.x; i < p.num_items; i += gridDim.x) {
      const Item it = item_of(p, i);
      // consume_tile_wait / peer_tile_wait: all R partials of the tile have arrived
      if (lane == 0) {
        for (int r = 0; r < p.R; ++r)
          wait_flag(p.flags + size_t(it.tau) * p.R + r, p.epoch, p.status, p.timeout_ns,
                    uint32_t(it.tau * p.R + r), TL_ERR_TIMEOUT);
      }
      __syncwarp();
      const int s0 = it.j * p.slice_rows;
      const int s_rows = max(0, min(p.slice_rows, BM - s0));
      const int n_cols = min(BN, p.N - it.nt * BN);  // valid columns in this tile (multiple of 8)
      const int total = s_rows * (n_cols / 4);       // float4 elements of the slice
      // rank r's partial of this tile was pushed by item tau*R + j(r), j(r) = (r - d - 1 - tau) mod R,
      // into ring slot (tau*R + j(r)) mod ring_slots
      const int jbase = ((-(it.d + 1 + it.tau)) % p.R + p.R) % p.R;
      const int ring_base = int((size_t(it.tau) * p.R) % size_t(p.ring_slots));
      uint16_t* out = p.out[it.d];
      for (int e0 = et; e0 < total; e0 += kNumRedThreads * QU) {
        int off[QU];  // float offset of each element inside a slot, -1 when past the slice
        int orow[QU];
        int ocol[QU];
#pragma unroll
        for (int u = 0; u < QU; ++u) {
          const int e = e0 + u * kNumRedThreads;
          const int c4 = e / s_rows, sr = e - c4 * s_rows;
          off[u] = e < total ? (c4 * BM + s0 + sr) * 4 : -1;
          orow[u] = it.mt * BM + s0 + sr;
          ocol[u] = it.nt * BN + c4 * 4;
        }
        float4 acc4[QU];
        for (int rb = 0; rb < p.R; rb += RB) {
          float4 v[RB][QU];
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) {
            if (rb + rr < p.R) {
              int j = jbase + rb + rr;
              j -= j >= p.R ? p.R : 0;
              int slot = ring_base + j;
              slot -= slot >= p.ring_slots ? p.ring_slots : 0;
              const float* src = p.slots + size_t(slot) * SLOT_FLOATS;
#pragma unroll
              for (int u = 0; u < QU; ++u)
                if (off[u] >= 0) v[rr][u] = __ldcg(reinterpret_cast<const float4*>(src + off[u]));
            }
          }
          // fixed rank order: acc = ((P_0 + P_1) + P_2) + ...
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
      // slice j of tile tau is read: release its "reduced" flag (slot-free barrier)
      named_bar_sync(2, kNumRedThreads);
      if (et == 0) st_release(reduced + size_t(it.tau) * p.R + it.j, p.epoch);
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort) {
    const uint64_t t0 = now_ns();
    while (now_ns() - t0 < 50000) {
    }
  }
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

int rs_num_tiles(int R, int M, int N) {
  const int Md = M / R;
  return cdiv(Md, BM) * cdiv(N, BN) * R;
}

// CTAs of a launch: a multiple of R (so a tile's R items share a wave), at most the SMs.
int rs_grid(int R, int num_items, int sm_count) {
  int grid = (sm_count / R) * R;
  return std::min(grid, ((num_items + R - 1) / R) * R);
}

// Receive slots in the ring: two waves of items, or every item when fewer.
int rs_ring_slots(int num_items, int grid) { return std::min(num_items, 2 * grid); }

int current_sm_count() {
  DeviceInfo di{};
  return device_info(&di) == TL_OK ? di.sm_count : 0;
}

}  // namespace
}  // namespace tl

extern "C" size_t tl_gemm_rs_workspace_size(int R, int M, int N) {
  if (R < 1 || M < R || N < 1 || M % R) return 0;
  const int items = tl::rs_num_tiles(R, M, N) * R;
  const int sms = tl::current_sm_count();
  // without a usable device, size for every item (always enough)
  const int slots = sms >= R ? tl::rs_ring_slots(items, tl::rs_grid(R, items, sms)) : items;
  return size_t(slots) * tl::SLOT_FLOATS * sizeof(float);
}

extern "C" int tl_gemm_rs_num_flags(int R, int M, int N) {
  if (R < 1 || M < R || N < 1 || M % R) return -1;
  return 2 * tl::rs_num_tiles(R, M, N) * R;  // arrival flags, then reduced flags
}

extern "C" tl_status tl_gemm_rs(const tl_gemm_rs_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_gemm_rs: NULL args");
  if (a->R < 1 || a->R > RS_MAX_RANKS)
    return fail(a->R > RS_MAX_RANKS ? TL_ERR_UNSUPPORTED : TL_ERR_INVALID, "tl_gemm_rs: R=%d outside 1..%d", a->R,
                RS_MAX_RANKS);
  if (a->M < a->R || a->M % a->R) return fail(TL_ERR_INVALID, "tl_gemm_rs: M=%d must be a positive multiple of R", a->M);
  if (a->K_r < 1 || a->N < 1) return fail(TL_ERR_INVALID, "tl_gemm_rs: empty shape");
  if (a->K_r % 8 || a->N % 8)
    return fail(TL_ERR_UNSUPPORTED, "tl_gemm_rs: K_r (%d) and N (%d) must be multiples of 8", a->K_r, a->N);
  if (!a->A || !a->B || !a->out || !a->workspace || !a->signals)
    return fail(TL_ERR_INVALID, "tl_gemm_rs: NULL pointer argument");
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "tl_gemm_rs: epoch must be nonzero");
  for (int r = 0; r < a->R; ++r) {
    if (!a->A[r] || !a->B[r] || !a->out[r] || !aligned16(a->A[r]) || !aligned16(a->B[r]) || !aligned16(a->out[r]))
      return fail(TL_ERR_INVALID, "tl_gemm_rs: rank %d pointer NULL or not 16-byte aligned", r);
  }
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
  const int num_tiles = rs_num_tiles(a->R, a->M, a->N);
  if ((long long)num_tiles * a->R > (1ll << 30)) return fail(TL_ERR_UNSUPPORTED, "tl_gemm_rs: too many tiles");

  RsParams* p = new (std::nothrow) RsParams;
  if (!p) return fail(TL_ERR_INTERNAL, "out of host memory");
  std::memset(p, 0, sizeof(RsParams));
  tl_status st = TL_OK;
  do {
    for (int r = 0; r < a->R && !st; ++r) {
      st = make_map_bf16(&p->map_a[r], a->A[r], a->M, a->K_r, size_t(a->K_r) * 2, BM, BK);
      if (!st) st = make_map_bf16(&p->map_b[r], a->B[r], a->K_r, a->N, size_t(a->N) * 2, BK, 64);
      p->out[r] = static_cast<uint16_t*>(a->out[r]);
    }
    if (st) break;
    p->slots = static_cast<float*>(a->workspace);
    p->flags = a->signals->flags;
    p->status = a->signals->status;
    p->trace = a->trace;
    p->timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
    p->pipe_timeout_ns = 2 * p->timeout_ns + 1000000000ull;
    p->R = a->R;
    p->M = a->M;
    p->Md = a->M / a->R;
    p->K = a->K_r;
    p->N = a->N;
    p->Mt_d = cdiv(p->Md, BM);
    p->Nt = cdiv(a->N, BN);
    p->KB = cdiv(a->K_r, BK);
    p->num_tiles = num_tiles;
    p->num_items = num_tiles * a->R;
    p->slice_rows = cdiv(BM, a->R);
    p->epoch = a->epoch;
    // a multiple of R CTAs, so the R items of a tile share a wave (their waits never form a cycle)
    const int grid = rs_grid(a->R, p->num_items, di.sm_count);
    p->ring_slots = rs_ring_slots(p->num_items, grid);
    if (grid < a->R) {
      st = fail(TL_ERR_UNSUPPORTED, "tl_gemm_rs: R=%d exceeds the %d SMs", a->R, di.sm_count);
      break;
    }
    void* args[] = {p};
    st = launch_coop(reinterpret_cast<const void*>(&gemm_rs_kernel), grid, RS_THREADS, RS_SMEM_BYTES,
                     (cudaStream_t)stream, args);
  } while (false);
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
  if (!a) return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: NULL args");
  if (a->workspace || a->workspace_bytes || a->signals)
    return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: workspace and signals must be NULL (the scratch is static)");
  if (a->R < 1 || a->R > RS_MAX_RANKS)
    return fail(a->R > RS_MAX_RANKS ? TL_ERR_UNSUPPORTED : TL_ERR_INVALID, "tl_gemm_rs_noalloc: R=%d outside 1..%d",
                a->R, RS_MAX_RANKS);
  if (a->M < a->R || a->M % a->R)
    return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: M=%d must be a positive multiple of R", a->M);
  if (a->K_r < 1 || a->N < 1) return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: empty shape");
  if (a->K_r % 8 || a->N % 8)
    return fail(TL_ERR_UNSUPPORTED, "tl_gemm_rs_noalloc: K_r (%d) and N (%d) must be multiples of 8", a->K_r, a->N);
  if (!a->A || !a->B || !a->out) return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: NULL pointer argument");
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: epoch must be nonzero");
  if (dev_status && !aligned16(dev_status)) return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: dev_status alignment");
  for (int r = 0; r < a->R; ++r) {
    if (!a->A[r] || !a->B[r] || !a->out[r] || !aligned16(a->A[r]) || !aligned16(a->B[r]) || !aligned16(a->out[r]))
      return fail(TL_ERR_INVALID, "tl_gemm_rs_noalloc: rank %d pointer NULL or not 16-byte aligned", r);
  }
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

  const int num_tiles = rs_num_tiles(a->R, a->M, a->N);
  const int nitems = num_tiles * a->R;
  const int nflags = 2 * nitems;
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
  for (int r = 0; r < a->R; ++r) {
    if (tl_status s = make_map_bf16(&p.map_a[r], a->A[r], a->M, a->K_r, size_t(a->K_r) * 2, BM, BK)) return s;
    if (tl_status s = make_map_bf16(&p.map_b[r], a->B[r], a->K_r, a->N, size_t(a->N) * 2, BK, 64)) return s;
    p.out[r] = static_cast<uint16_t*>(a->out[r]);
  }
  p.slots = slots;
  p.flags = flags;
  p.status = dev_status ? dev_status : status;
  p.trace = a->trace;
  p.timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
  p.pipe_timeout_ns = 2 * p.timeout_ns + 1000000000ull;
  p.R = a->R;
  p.M = a->M;
  p.Md = a->M / a->R;
  p.K = a->K_r;
  p.N = a->N;
  p.Mt_d = cdiv(p.Md, BM);
  p.Nt = cdiv(a->N, BN);
  p.KB = cdiv(a->K_r, BK);
  p.num_tiles = num_tiles;
  p.num_items = nitems;
  p.slice_rows = cdiv(BM, a->R);
  p.epoch = a->epoch;
  const int grid = rs_grid(a->R, p.num_items, di.sm_count);
  p.ring_slots = rs_ring_slots(p.num_items, grid);
  if (grid < a->R) return fail(TL_ERR_UNSUPPORTED, "tl_gemm_rs_noalloc: R=%d exceeds the %d SMs", a->R, di.sm_count);
  void* args[] = {&p};
  return launch_coop(reinterpret_cast<const void*>(&gemm_rs_kernel), grid, RS_THREADS, RS_SMEM_BYTES, st, args);
}

namespace {
size_t noalloc_scratch_needed(int R, int M, int N, int sm_count) {
  if (R < 1 || M < R || N < 1 || M % R || sm_count < R) return 0;
  const int nitems = tl::rs_num_tiles(R, M, N) * R;
  const size_t nflags = 2 * size_t(nitems);
  const int slots = tl::rs_ring_slots(nitems, tl::rs_grid(R, nitems, sm_count));
  return align_up(kNoAllocHeader + nflags * 4, 256) + size_t(slots) * tl::SLOT_FLOATS * sizeof(float);
}
}  // namespace
