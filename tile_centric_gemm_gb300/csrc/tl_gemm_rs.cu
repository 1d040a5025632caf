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
// Work items: output tile tau = (dest d, m tile, n tile) in destination order;
// its R partial tiles P_r = A_r[rows of tau] . B_r[:, cols of tau] are items
// tau*R + j, rank r = (d + 1 + tau + j) mod R (the rotation spreads the
// destination rank's own item over the CTAs).  The grid is a multiple of R and
// items go round-robin, so the R items of a tile always run in the same wave.
//
// Per CTA: warp 0 TMA producer (A_r, B_r k-blocks), warp 1 tcgen05 MMA issuer,
// warps 2-5 epilogue.  The epilogue of item (tau, j):
//   1. push: TMEM -> registers -> fp32 receive slot (tau, r) in the workspace;
//      release flag tau*R + r (produce_tile_notify);
//   2. reduce: acquire all R flags of tau, then sum row slice j of the tile over
//      the R slots in rank order 0..R-1 in fp32 and store it as bf16 rows of
//      out[d].
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "tl_common.cuh"
#include "tl_internal.h"

namespace tl {
namespace {

constexpr int RS_MAX_RANKS = 32;
constexpr int RS_THREADS = 6 * 32;
constexpr uint32_t RS_SMEM_BARS = SMEM_GEMM_END;
constexpr uint32_t RS_SMEM_BYTES = RS_SMEM_BARS + sizeof(Barriers) + 1024;
constexpr int SLOT_FLOATS = BM * BN;  // one fp32 partial tile
constexpr int RB = 8;                 // ranks loaded per batch in the reduce
constexpr int QU = 4;                 // float4 elements per thread per round in the reduce

struct RsParams {
  CUtensorMap map_a[RS_MAX_RANKS];  // A_r [M, K_r]
  CUtensorMap map_b[RS_MAX_RANKS];  // B_r [K_r, N]
  uint16_t* out[RS_MAX_RANKS];      // out[d] [Md, N] bf16
  float* slots;                     // [num_tiles][R][BM*BN] fp32 receive slots
  uint32_t* flags;                  // [num_tiles][R]
  uint32_t* status;
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int32_t R, M, Md, K, N;
  int32_t Mt_d, Nt, KB, num_tiles, num_items, slice_rows;
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
  it.mt = rem / p.Nt;
  it.nt = rem % p.Nt;
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
  } else {
    // ---------------------------------------------------------------- epilogue: push + slice reduce
    const int wq = warp & 3;             // TMEM lane quarter of this warp
    const int et = (warp - kWarpEpi0) * 32 + lane;  // 0..127 among epilogue threads
    const int row_in_tile = wq * 32 + lane;
    int jj = 0;
    for (int i = blockIdx.x; i < p.num_items; i += gridDim.x, ++jj) {
      const Item it = item_of(p, i);
      const int acc = jj & 1;
      const uint32_t acc_ph = uint32_t(jj >> 1) & 1u;
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      // all four epilogue warps leave together (they meet at a named barrier below)
      if (!named_bar_and(1, kNumEpiThreads, ok)) break;
      tc_fence_after();
      // 1. push the fp32 partial: slot layout [col/4][row][4] so a warp writes 512 contiguous bytes
      float* slot = p.slots + (size_t(it.tau) * p.R + it.r) * SLOT_FLOATS;
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
      // produce_tile_notify: every epilogue thread's writes, then one release
      __threadfence();
      named_bar_sync(1, kNumEpiThreads);
      if (et == 0) st_release(p.flags + size_t(it.tau) * p.R + it.r, p.epoch);

      // 2. reduce row slice j of the tile: wait on all R partials (own and peers')
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
      const float* tile_slots = p.slots + size_t(it.tau) * p.R * SLOT_FLOATS;
      uint16_t* out = p.out[it.d];
      for (int e0 = et; e0 < total; e0 += kNumEpiThreads * QU) {
        float4 acc4[QU];
        for (int rb = 0; rb < p.R; rb += RB) {
          float4 v[RB][QU];
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) {
#pragma unroll
            for (int u = 0; u < QU; ++u) {
              const int e = e0 + u * kNumEpiThreads;
              if (rb + rr < p.R && e < total) {
                const int c4 = e / s_rows, sr = e - c4 * s_rows;
                v[rr][u] = ld_global_cg_v4f(tile_slots + size_t(rb + rr) * SLOT_FLOATS +
                                            (size_t(c4) * BM + s0 + sr) * 4);
              }
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
          const int e = e0 + u * kNumEpiThreads;
          if (e < total) {
            const int c4 = e / s_rows, sr = e - c4 * s_rows;
            const int orow = it.mt * BM + s0 + sr;
            if (orow < p.Md) {
              uint2 pk;
              pk.x = pack_bf16x2(acc4[u].x, acc4[u].y);
              pk.y = pack_bf16x2(acc4[u].z, acc4[u].w);
              *reinterpret_cast<uint2*>(out + size_t(orow) * p.N + it.nt * BN + c4 * 4) = pk;
            }
          }
        }
      }
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

}  // namespace
}  // namespace tl

extern "C" size_t tl_gemm_rs_workspace_size(int R, int M, int N) {
  if (R < 1 || M < R || N < 1 || M % R) return 0;
  return size_t(tl::rs_num_tiles(R, M, N)) * size_t(R) * tl::SLOT_FLOATS * sizeof(float);
}

extern "C" int tl_gemm_rs_num_flags(int R, int M, int N) {
  if (R < 1 || M < R || N < 1 || M % R) return -1;
  return tl::rs_num_tiles(R, M, N) * R;
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
  const size_t need = tl_gemm_rs_workspace_size(a->R, a->M, a->N);
  if (a->workspace_bytes < need)
    return fail(TL_ERR_INVALID, "tl_gemm_rs: workspace %zu bytes, need %zu", a->workspace_bytes, need);
  const int nflags = tl_gemm_rs_num_flags(a->R, a->M, a->N);
  if (a->signals->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_gemm_rs: signals hold %d flags, need %d", a->signals->num_flags, nflags);
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
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
    int grid = (di.sm_count / a->R) * a->R;
    grid = std::min(grid, ((p->num_items + a->R - 1) / a->R) * a->R);
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
size_t noalloc_scratch_needed(int R, int M, int N);
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
  const size_t need = noalloc_scratch_needed(a->R, a->M, a->N);
  if (need == 0 || need > kNoAllocScratchBytes)
    return fail(TL_ERR_UNSUPPORTED,
                "tl_gemm_rs_noalloc: R=%d M=%d N=%d needs %zu bytes of scratch; the static scratch holds %zu "
                "(use tl_gemm_rs with a caller-allocated workspace)",
                a->R, a->M, a->N, need, kNoAllocScratchBytes);
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  uint8_t* scratch = nullptr;
  if (tl_status s = noalloc_scratch(di.device, &scratch)) return s;

  const int num_tiles = rs_num_tiles(a->R, a->M, a->N);
  const int nflags = num_tiles * a->R;
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
  p.num_items = nflags;
  p.slice_rows = cdiv(BM, a->R);
  p.epoch = a->epoch;
  int grid = (di.sm_count / a->R) * a->R;
  grid = std::min(grid, ((p.num_items + a->R - 1) / a->R) * a->R);
  if (grid < a->R) return fail(TL_ERR_UNSUPPORTED, "tl_gemm_rs_noalloc: R=%d exceeds the %d SMs", a->R, di.sm_count);
  void* args[] = {&p};
  return launch_coop(reinterpret_cast<const void*>(&gemm_rs_kernel), grid, RS_THREADS, RS_SMEM_BYTES, st, args);
}

namespace {
size_t noalloc_scratch_needed(int R, int M, int N) {
  if (R < 1 || M < R || N < 1 || M % R) return 0;
  const size_t nflags = size_t(tl::rs_num_tiles(R, M, N)) * R;
  return align_up(kNoAllocHeader + nflags * 4, 256) + nflags * size_t(tl::SLOT_FLOATS) * sizeof(float);
}
}  // namespace
