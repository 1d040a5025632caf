// tl_gemm.cu -- plain GEMM C = A . B on the CTA-pair tcgen05 core.
//
// The compute half of AllGather-GEMM without any communication or waits: the
// "GEMM alone" arm against which the fused kernels' overlap is measured, and a
// building block of the decomposed (per-shard, multi-stream) baseline the
// TileLink talk summary describes as prior art (Background: decomposition-
// based overlap).
#include <algorithm>
#include <cstring>
#include <new>

#include "tl_epilogue.cuh"
#include "tl_internal.h"
#include "tl_pair.cuh"

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
  int32_t M, N, K, Mt, Nt, KB, num_tiles;
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
  const int my_tiles = pair_id < p.num_tiles ? (p.num_tiles - 1 - pair_id) / npairs + 1 : 0;

  if (warp == kWarpTma) {
    if (lane == 0) {
      pair::Producer prod;
      for (int t = pair_id; t < p.num_tiles && !*abort; t += npairs) {
        const int m = t / p.Nt, n = t % p.Nt;
        for (int kb = 0; kb < p.KB; ++kb)
          if (!prod.load(smem, bars, rank, &p.map_a, kb * pair::BK, m * pair::BM + int(rank) * pair::HM, &p.map_b,
                         n * pair::BN + int(rank) * pair::HN, kb * pair::BK, abort, p.status, p.pipe_timeout_ns))
            break;
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0 && rank == 0)
      pair::mma_loop(smem, bars, tmem_base, my_tiles, p.KB, abort, p.status, p.pipe_timeout_ns);
    __syncwarp();
  } else {
    const int wq = warp & 3;
    uint8_t* cstage = smem + GEMM_SMEM_CSTAGE + uint32_t(wq) * 2 * C_BOX_BYTES;
    int nbox = 0;  // boxes this warp has stored (buffer nbox & 1)
    int j = 0;
    for (int t = pair_id; t < p.num_tiles; t += npairs, ++j) {
      const int acc = j & 1;
      const uint32_t acc_ph = uint32_t(j >> 1) & 1u;
      const int m = t / p.Nt, n = t % p.Nt;
      const bool ok = mbar_wait(&bars->tmem_full[acc], acc_ph, abort, p.status, p.pipe_timeout_ns, 4);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int row = m * pair::BM + int(rank) * pair::HM + wq * 32 + lane;
      const bool row_ok = row < p.M;
      for (int c = 0; c < pair::BN / 32; ++c) {
        const int col0 = n * pair::BN + c * 32;
        if (col0 >= p.N) break;
        uint32_t v[32];
        tmem_ld_32cols(tmem_base + (uint32_t(wq * 32) << 16) + uint32_t(acc * pair::BN + c * 32), v);
        tmem_ld_wait();
        const int row_base = m * pair::BM + int(rank) * pair::HM + wq * 32;
        if (p.C && row_base < p.M) {
          // this warp's 32 x 32 box through shared memory, one TMA store (rows and
          // columns past the matrix are not written)
          store_box_bf16(&p.map_c, cstage + (nbox & 1) * C_BOX_BYTES, 2, lane, v, col0, row_base);
          ++nbox;
        }
        if (row_ok && p.C_f32) {
          {
            float* frow = p.C_f32 + size_t(row) * p.N + col0;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              if (col0 + g * 4 < p.N) {
                const float* f = reinterpret_cast<const float*>(v + g * 4);
                st_global_cg_v4f(frow + g * 4, f[0], f[1], f[2], f[3]);
              }
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
  }
  pair::teardown(bars, warp, tmem_base);
}

}  // namespace
}  // namespace tl

extern "C" tl_status tl_gemm(const tl_gemm_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_gemm: NULL args");
  if (a->M < 1 || a->N < 1 || a->K < 1) return fail(TL_ERR_INVALID, "tl_gemm: empty shape");
  if (a->K % 8 || a->N % 8)
    return fail(TL_ERR_UNSUPPORTED, "tl_gemm: K (%d) and N (%d) must be multiples of 8", a->K, a->N);
  if (!a->A || !a->B || (!a->C && !a->C_f32) || !a->signals)
    return fail(TL_ERR_INVALID, "tl_gemm: NULL pointer argument");
  if (!aligned16(a->A) || !aligned16(a->B) || (a->C && !aligned16(a->C)) || (a->C_f32 && !aligned16(a->C_f32)))
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
    p->num_tiles = p->Mt * p->Nt;
    const int pairs = std::max(1, std::min(di.sm_count / 2, p->num_tiles));
    void* args[] = {p};
    st = launch_coop(reinterpret_cast<const void*>(&gemm_pair_kernel), 2 * pairs, GEMM_THREADS, GEMM_SMEM_BYTES,
                     (cudaStream_t)stream, args, 2);
  } while (false);
  delete p;
  return st;
}
