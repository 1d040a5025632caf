// tl_moe_ws.cuh -- layout of the MoE routing workspace (int32 words, documented
// in tilelink.h) shared by the AllGather + grouped GEMM call that writes it and
// the down-projection call that reads it.
#pragma once

namespace tl {

constexpr int MOE_TILE_ROWS = 256;  // sorted rows of an expert tile (one CTA pair)
constexpr int WS_HEADER = 16;       // [0] = number of tiles
__host__ __device__ inline int ws_tiles(int) { return WS_HEADER; }
__host__ __device__ inline int ws_order(int max_tiles) { return WS_HEADER + 6 * max_tiles; }
__host__ __device__ inline int ws_inv(int max_tiles) { return WS_HEADER + 7 * max_tiles; }
// Tiles of at most MOE_TILE_ROWS sorted rows, one expert each: at most ceil(P / rows) + E.
inline int moe_max_tiles(int P, int E) { return (P + MOE_TILE_ROWS - 1) / MOE_TILE_ROWS + E; }

}  // namespace tl
