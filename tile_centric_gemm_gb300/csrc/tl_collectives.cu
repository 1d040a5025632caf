// tl_collectives.cu -- the communication halves of the fused operations on
// their own: AllGather with per-chunk signals (the producer of AllGather-GEMM)
// and a rank-ordered ReduceScatter of fp32 partials (the reduce stage of
// GEMM-ReduceScatter).  TileLink talk summary ("TileLink: Generating Efficient
// Compute-Communication Overlapping Kernels using Tile-Centric Primitives"):
// Technical Deep Dive -- produce_tile_notify after each moved tile, pull and
// push modes; Background -- the decomposed (separate communication and
// compute) schedule that fused kernels are measured against.
#include <algorithm>

#include "tl_copy.cuh"
#include "tl_internal.h"

namespace tl {
namespace {

constexpr uint32_t AGC_SMEM_BYTES = COPY_NBUF * COPY_CHUNK + COPY_NBUF * 8 + 1024;

struct AllgatherParams {
  const uint8_t* shard[TL_MAX_RANKS];
  AgCopyJob job;
};

// One warp per CTA, one CTA per SM: the same copy routine and staging as the
// copy warp of the fused kernel.
__global__ void __launch_bounds__(32, 1) allgather_kernel(const __grid_constant__ AllgatherParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + COPY_NBUF * COPY_CHUNK);
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    for (int b = 0; b < COPY_NBUF; ++b) mbar_init(&bars[b], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  AgCopyJob job = p.job;
  job.shard = p.shard;
  ag_copy_items(job, stage, bars, &abort_flag, int(blockIdx.x), int(gridDim.x));
}

struct ReduceParams {
  const float* part[TL_MAX_RANKS];  // R partials [M, N] fp32
  uint16_t* out[TL_MAX_RANKS];      // R row shards [M/R, N] bf16
  int R, M, Md, N;
};

// out[row / Md][row % Md] = bf16(((P_0 + P_1) + P_2) + ...), four columns per thread.
__global__ void __launch_bounds__(256) reduce_scatter_kernel(const __grid_constant__ ReduceParams p) {
  const size_t n4 = size_t(p.N) / 4;
  const size_t total = size_t(p.M) * n4;
  for (size_t e = size_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += size_t(gridDim.x) * blockDim.x) {
    const size_t row = e / n4, c4 = e % n4;
    float4 acc = __ldcs(reinterpret_cast<const float4*>(p.part[0]) + e);
    for (int r = 1; r < p.R; ++r) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(p.part[r]) + e);
      acc.x = __fadd_rn(acc.x, v.x);
      acc.y = __fadd_rn(acc.y, v.y);
      acc.z = __fadd_rn(acc.z, v.z);
      acc.w = __fadd_rn(acc.w, v.w);
    }
    uint2 pk;
    pk.x = pack_bf16x2(acc.x, acc.y);
    pk.y = pack_bf16x2(acc.z, acc.w);
    const int d = int(row / p.Md);
    *reinterpret_cast<uint2*>(p.out[d] + (row - size_t(d) * p.Md) * p.N + c4 * 4) = pk;
  }
}

}  // namespace
}  // namespace tl

extern "C" tl_status tl_allgather(const tl_allgather_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_allgather: NULL args");
  if (a->R < 1 || a->R > TL_MAX_RANKS) return fail(TL_ERR_INVALID, "tl_allgather: R=%d", a->R);
  if (a->self_rank < 0 || a->self_rank >= a->R) return fail(TL_ERR_INVALID, "tl_allgather: self_rank");
  if (a->M_shard < 1 || a->K < 1) return fail(TL_ERR_INVALID, "tl_allgather: empty shape");
  if (a->K % 8) return fail(TL_ERR_UNSUPPORTED, "tl_allgather: K (%d) must be a multiple of 8", a->K);
  if (a->mode != TL_MODE_PULL && a->mode != TL_MODE_PUSH) return fail(TL_ERR_INVALID, "tl_allgather: mode");
  if (a->mode == TL_MODE_PULL && !a->src_ready) return fail(TL_ERR_INVALID, "tl_allgather: pull mode needs src_ready");
  if (!a->A_shards || !a->gathered || !a->signals) return fail(TL_ERR_INVALID, "tl_allgather: NULL pointer argument");
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "tl_allgather: epoch must be nonzero");
  for (int r = 0; r < a->R; ++r)
    if (!a->A_shards[r] || !aligned16(a->A_shards[r])) return fail(TL_ERR_INVALID, "tl_allgather: shard %d", r);
  if (!aligned16(a->gathered)) return fail(TL_ERR_INVALID, "tl_allgather: gathered alignment");
  int rpb = 0;
  const int nflags = tl_ag_gemm_num_flags(a->R, a->M_shard, a->K, a->rows_per_barrier, &rpb);
  if (a->signals->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_allgather: signals hold %d flags, need %d", a->signals->num_flags, nflags);
  if (a->mode == TL_MODE_PULL && a->src_ready->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_allgather: src_ready holds %d flags, need %d", a->src_ready->num_flags, nflags);
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  AllgatherParams p{};
  if (tl_status s = classify_shards("tl_allgather", a->A_shards, a->R, di.device, p.shard, &p.job.host_mask))
    return s;
  p.job.gathered = static_cast<uint8_t*>(a->gathered);
  p.job.flags = a->signals->flags;
  p.job.ready = a->mode == TL_MODE_PULL ? a->src_ready->flags : nullptr;
  p.job.status = a->signals->status;
  p.job.timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
  p.job.pipe_timeout_ns = 2 * p.job.timeout_ns + 1000000000ull;
  p.job.R = a->R;
  p.job.self = a->self_rank;
  p.job.M_shard = a->M_shard;
  p.job.K = a->K;
  p.job.rpb = rpb;
  p.job.bpr = cdiv(a->M_shard, rpb);
  p.job.num_items = a->R * p.job.bpr;
  p.job.epoch = a->epoch;
  if (tl_status s = test_hold("tl_allgather", p.job.timeout_ns, &p.job.hold_first, &p.job.hold_count, &p.job.hold_ns))
    return s;
  const int grid = std::max(1, std::min(di.sm_count, p.job.num_items));
  void* args[] = {&p};
  return launch_coop(reinterpret_cast<const void*>(&allgather_kernel), grid, 32, AGC_SMEM_BYTES,
                     (cudaStream_t)stream, args);
}

extern "C" tl_status tl_reduce_scatter(const tl_reduce_scatter_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_reduce_scatter: NULL args");
  if (a->R < 1 || a->R > TL_MAX_RANKS) return fail(TL_ERR_INVALID, "tl_reduce_scatter: R=%d", a->R);
  if (a->M < a->R || a->M % a->R) return fail(TL_ERR_INVALID, "tl_reduce_scatter: M must be a multiple of R");
  if (a->N < 1) return fail(TL_ERR_INVALID, "tl_reduce_scatter: empty shape");
  if (a->N % 8) return fail(TL_ERR_UNSUPPORTED, "tl_reduce_scatter: N (%d) must be a multiple of 8", a->N);
  if (!a->partials || !a->out) return fail(TL_ERR_INVALID, "tl_reduce_scatter: NULL pointer argument");
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  ReduceParams p{};
  for (int r = 0; r < a->R; ++r) {
    if (!a->partials[r] || !a->out[r] || !aligned16(a->partials[r]) || !aligned16(a->out[r]))
      return fail(TL_ERR_INVALID, "tl_reduce_scatter: rank %d pointer", r);
    p.part[r] = a->partials[r];
    p.out[r] = static_cast<uint16_t*>(a->out[r]);
  }
  p.R = a->R;
  p.M = a->M;
  p.Md = a->M / a->R;
  p.N = a->N;
  reduce_scatter_kernel<<<di.sm_count * 8, 256, 0, (cudaStream_t)stream>>>(p);
  return cuda_ok(cudaGetLastError(), "reduce_scatter launch");
}
