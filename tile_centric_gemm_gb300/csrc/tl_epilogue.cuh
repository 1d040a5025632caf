// tl_epilogue.cuh -- TMA-store epilogue pieces for the bf16 outputs of the
// GEMM-shaped kernels: an epilogue warp converts its 32 rows x 32 columns of the
// fp32 accumulator to bf16, writes them into a shared-memory box laid out as the
// 64-byte swizzle of the output's tensor map, and one lane stores the box with a
// bulk tensor copy (rows and columns outside the matrix are not written).
#pragma once

#include "tl_ptx.cuh"

namespace tl {

constexpr uint32_t C_BOX_BYTES = 32 * 64;  // 32 rows x 32 bf16 columns

// This lane's row r of the box from 32 fp32 values: 16-byte chunk q of row r
// sits at chunk q ^ ((r >> 1) & 3) (64-byte swizzle; the buffer is 512-byte aligned).
__device__ __forceinline__ void stage_row_bf16(uint8_t* buf, int r, const uint32_t* v) {
  const uint32_t base = smem_u32(buf) + uint32_t(r) * 64u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float* f = reinterpret_cast<const float*>(v + q * 8);
    st_shared_v4(base + uint32_t((q ^ ((r >> 1) & 3)) * 16), pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                 pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
  }
}

// The warp's box at (col0, row0) of `map` from `buf`.  `nbuf` staging buffers per
// warp: before overwriting one, the store that last used it must have read it.
__device__ __forceinline__ void store_box_bf16(const CUtensorMap* map, uint8_t* buf, int nbuf, int lane,
                                               const uint32_t* v, int col0, int row0) {
  if (lane == 0) {
    if (nbuf >= 2) bulk_wait_read<1>();
    else bulk_wait_read<0>();
  }
  __syncwarp();
  stage_row_bf16(buf, lane, v);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, col0, row0, buf);
    bulk_commit();
  }
}

}  // namespace tl
