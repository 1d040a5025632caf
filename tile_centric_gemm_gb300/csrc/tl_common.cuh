// tl_common.cuh -- constants and device pieces shared by the GEMM-shaped kernels:
// tile shape, shared-memory layout, and the TMA-producer / tcgen05-MMA /
// TMEM-epilogue warp roles of a persistent warp-specialised CTA.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "tl_ptx.cuh"

namespace tl {

// GEMM tile: 128 x 256 fp32 accumulator in TMEM, K step 64 (one 128-byte swizzle atom of bf16).
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr uint32_t A_STAGE_BYTES = BM * BK * 2;  // 16 KB
constexpr uint32_t B_BOX_BYTES = BK * 64 * 2;    // 8 KB: 64 K-rows x 64 N-cols
constexpr uint32_t B_STAGE_BYTES = BK * BN * 2;  // 32 KB = 4 boxes
constexpr uint32_t STAGE_TX = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr uint32_t TMEM_COLS = 512;  // two 256-column fp32 accumulators
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, true);

// Warp roles.
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpEpi0 = 2;
constexpr int kNumEpiWarps = 4;
constexpr int kNumEpiThreads = kNumEpiWarps * 32;

// Copy-warp staging (producer of the AllGather): NBUF buffers of CHUNK bytes.
constexpr int COPY_NBUF = 4;
constexpr uint32_t COPY_CHUNK = 8192;

// Shared-memory carve-up, offsets from a 1024-aligned base.
constexpr uint32_t SMEM_A = 0;
constexpr uint32_t SMEM_B = SMEM_A + STAGES * A_STAGE_BYTES;
constexpr uint32_t SMEM_GEMM_END = SMEM_B + STAGES * B_STAGE_BYTES;  // 192 KB

struct __align__(8) Barriers {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t copy[COPY_NBUF];
  uint32_t tmem_base;
  uint32_t abort;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// Issue the four UMMA_K steps of one 64-deep k-block from stage `s`.
__device__ __forceinline__ void mma_kblock(uint8_t* smem, int s, uint32_t d_tmem, bool first) {
  const uint32_t a0 = smem_u32(smem + SMEM_A + s * A_STAGE_BYTES);
  const uint32_t b0 = smem_u32(smem + SMEM_B + s * B_STAGE_BYTES);
#pragma unroll
  for (int kk = 0; kk < BK / UMMA_K; ++kk) {
    // A (K-major): advance 16 bf16 = 32 B inside the swizzle atom; SBO = 8 rows x 128 B.
    const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
    // B (MN-major): advance 16 K-rows = 2 atoms; LBO = next 64-column box; SBO = 8 K-rows x 128 B.
    const uint64_t bd = sdesc_sw128(b0 + kk * 2048, B_BOX_BYTES, 1024);
    tc_mma_bf16(d_tmem, ad, bd, IDESC, (first && kk == 0) ? 0u : 1u);
  }
}

}  // namespace tl
