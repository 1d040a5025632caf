// tl_common.cuh -- constants shared by the GEMM-shaped kernels: the tcgen05 K
// step, the B staging box, the TMEM accumulators, the TMA-producer /
// tcgen05-MMA / TMEM-epilogue warp roles of a persistent warp-specialised CTA,
// and the copy-warp staging.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "tl_ptx.cuh"

namespace tl {

// tcgen05 K step of bf16 and the B staging box (64 K-rows x 64 N-columns, one
// 128-byte swizzle atom wide); TMEM holds two 256-column fp32 accumulators.
constexpr int UMMA_K = 16;
constexpr uint32_t B_BOX_BYTES = 64 * 64 * 2;  // 8 KB
constexpr uint32_t TMEM_COLS = 512;

// Warp roles.
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpEpi0 = 2;
constexpr int kNumEpiWarps = 4;
constexpr int kNumEpiThreads = kNumEpiWarps * 32;

// Copy-warp staging (producer of the AllGather): NBUF buffers of CHUNK bytes.
constexpr int COPY_NBUF = 4;
constexpr uint32_t COPY_CHUNK = 8192;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

}  // namespace tl
