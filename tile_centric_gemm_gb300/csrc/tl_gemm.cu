// tl_gemm.cu -- plain GEMM C = A . B on the CTA-pair tcgen05 core.
//
// The compute half of AllGather-GEMM without any communication or waits: the
// "GEMM alone" arm against which the fused kernels' overlap is measured, and a
// building block of the decomposed (per-shard, multi-stream) baseline the
// TileLink talk summary describes as prior art (Background: decomposition-
// based overlap).  With a workspace, grids with fewer tiles than CTA pairs are
// split over K (tl_splitk.cuh), as in the AllGather-GEMM.
#include <algorithm>
#include <cstring>
#include <new>

#include "tl_epilogue.cuh"
#include "tl_internal.h"
#include "tl_pair.cuh"
#include "tl_splitk.cuh"

namespace tl {
namespace {

constexpr int GEMM_THREADS = 6 * 32;
// C staging for TMA stores: per epilogue warp two buffers of one 32 x 32 box
constexpr uint32_t GEMM_SMEM_CSTAGE = pair::SMEM_END;
constexpr uint32_t GEMM_SMEM_BARS = GEMM_SMEM_CSTAGE + kNumEpiWarps * 2 * C_BOX_BYTES;
constexpr uint32_t GEMM_SMEM_BYTES = GEMM_SMEM_BARS + sizeof(pair::Bars) + 1024;

struct GemmParams {
  CUtensorMap map_a;  // A [M, K]
  CUtensorMap map_b;  // B [K, N]
  CUtensorMap map_c;  // C [M, N], box 32 x 32, 64-byte swizzle (TMA stores)
  uint16_t* C;
  float* C_f32;
  uint32_t* status;
  uint64_t pipe_timeout_ns;
  int32_t M, N, K, Mt, Nt, KB;
  int32_t S, KBs, num_work;  // splits per tile, k-blocks per split, work units (tiles * S)
  splitk::Work sk;
};

__global__ void __launch_bounds__(GEMM_THREADS, 1) gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  pair::Bars* bars = reinterpret_cast<pair::Bars*>(smem + GEMM_SMEM_BARS);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  const uint32_t rank = cluster_ctarank();
  const int pair_id = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  const uint32_t tmem_base = pair::setup(bars, warp);
  volatile uint32_t* abort = &bars->abort;
  const int my_work = pair_id < p.num_work ? (p.num_work - 1 - pair_id) / npairs + 1 : 0;

  if (warp == kWarpTma) {
    if (lane == 0) {
      pair::Producer prod;
      for (int w = pair_id; w < p.num_work && !*abort; w += npairs) {
        const int t = w / p.S, split = w % p.S;
        const int m = t / p.Nt, n = t % p.Nt;
        for (int kb = split * p.KBs; kb < (split + 1) * p.KBs; ++kb)
          if (!prod.load(smem, bars, rank, &p.map_a, kb * pair::BK, m * pair::BM + int(rank) * pair::HM, &p.map_b,
                         n * pair::BN + int(rank) * pair::HN, kb * pair::BK, abort, p.status, p.pipe_timeout_ns))
            break;
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0 && rank == 0)
      pair::mma_loop(smem, bars, tmem_base, my_work, p.KBs, abort, p.status, p.pipe_timeout_ns);
    __syncwarp();
  } else {
    const int wq = warp & 3;
    uint8_t* cstage = smem + GEMM_SMEM_CSTAGE + uint32_t(wq) * 2 * C_BOX_BYTES;
    int nbox = 0;  // boxes this warp has stored (buffer nbox & 1)
    int j = 0;
    for (int w = pair_id; w < p.num_work; w += npairs, ++j) {
      const int acc = j & 1;
      const uint32_t acc_ph = uint32_t(j >> 1) & 1u;
      const int t = w / p.S, split = w % p.S;
      const int m = t / p.Nt, n = t % p.Nt;
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
        if (p.C && row_base < p.M) {
          // this warp's 32 x 32 box through shared memory, one TMA store (rows and
          // columns past the matrix are not written)
          store_box_bf16(&p.map_c, cstage + (nbox & 1) * C_BOX_BYTES, 2, lane, v, col0, row_base);
          ++nbox;
        }
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
  }
  pair::teardown(bars, warp, tmem_base);
}

}  // namespace
}  // namespace tl

extern "C" size_t tl_gemm_workspace_size(int M, int N, int K, int sm_count) {
  if (M < 1 || N < 1 || K < 1) return 0;
  if (sm_count <= 0) {
    tl::DeviceInfo di{};
    if (tl::device_info(&di)) return 0;
    sm_count = di.sm_count;
  }
  const long long tiles = (long long)tl::cdiv(M, tl::pair::BM) * tl::cdiv(N, tl::pair::BN);
  return tl::splitk::workspace_bytes(tiles, tl::splitk::choose(tiles, tl::cdiv(K, tl::pair::BK), sm_count / 2));
}

extern "C" tl_status tl_gemm(const tl_gemm_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_gemm: NULL args");
  if (a->M < 1 || a->N < 1 || a->K < 1) return fail(TL_ERR_INVALID, "tl_gemm: empty shape");
  if (a->K % 8 || a->N % 8)
    return fail(TL_ERR_UNSUPPORTED, "tl_gemm: K (%d) and N (%d) must be multiples of 8", a->K, a->N);
  if (!a->A || !a->B || (!a->C && !a->C_f32) || !a->signals)
    return fail(TL_ERR_INVALID, "tl_gemm: NULL pointer argument");
  if (!aligned16(a->A) || !aligned16(a->B) || (a->C && !aligned16(a->C)) || (a->C_f32 && !aligned16(a->C_f32)) ||
      (a->workspace && !aligned16(a->workspace)))
    return fail(TL_ERR_INVALID, "tl_gemm: pointers must be 16-byte aligned");
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  GemmParams* p = new (std::nothrow) GemmParams;
  if (!p) return fail(TL_ERR_INTERNAL, "out of host memory");
  std::memset(p, 0, sizeof(GemmParams));
  tl_status st = TL_OK;
  do {
    if ((st = make_map_bf16(&p->map_a, a->A, a->M, a->K, size_t(a->K) * 2, pair::HM, pair::BK))) break;
    if ((st = make_map_bf16(&p->map_b, a->B, a->K, a->N, size_t(a->N) * 2, pair::BK, 64))) break;
    if (a->C && (st = make_map_bf16(&p->map_c, a->C, a->M, a->N, size_t(a->N) * 2, 32, 32,
                                    CU_TENSOR_MAP_SWIZZLE_64B)))
      break;
    p->C = static_cast<uint16_t*>(a->C);
    p->C_f32 = a->C_f32;
    p->status = a->signals->status;
    p->pipe_timeout_ns = 2 * (a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs) + 1000000000ull;
    p->M = a->M;
    p->N = a->N;
    p->K = a->K;
    p->Mt = cdiv(a->M, pair::BM);
    p->Nt = cdiv(a->N, pair::BN);
    p->KB = cdiv(a->K, pair::BK);
    const long long tiles = (long long)p->Mt * p->Nt;
    p->S = a->workspace ? splitk::choose(tiles, p->KB, di.sm_count / 2) : 1;
    if (p->S > 1) {
      const size_t need = splitk::workspace_bytes(tiles, p->S);
      if (a->workspace_bytes < need) {
        st = fail(TL_ERR_INVALID, "tl_gemm: workspace of %zu bytes, split-K needs %zu", a->workspace_bytes, need);
        break;
      }
      uint8_t* ws = static_cast<uint8_t*>(a->workspace);
      p->sk.counters = reinterpret_cast<uint32_t*>(ws);
      p->sk.partials = reinterpret_cast<float*>(ws + splitk::counter_bytes(tiles));
      p->sk.tag = 1u << 8;
      p->sk.timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
      p->sk.S = p->S;
    }
    p->KBs = p->KB / p->S;
    if (tiles * p->S > (1ll << 30)) {
      st = fail(TL_ERR_UNSUPPORTED, "tl_gemm: %lld tiles", tiles);
      break;
    }
    p->num_work = int(tiles) * p->S;
    const int pairs = std::max(1, std::min(di.sm_count / 2, p->num_work));
    void* args[] = {p};
    st = launch_coop(reinterpret_cast<const void*>(&gemm_pair_kernel), 2 * pairs, GEMM_THREADS, GEMM_SMEM_BYTES,
                     (cudaStream_t)stream, args, 2);
  } while (false);
  delete p;
  return st;
}
