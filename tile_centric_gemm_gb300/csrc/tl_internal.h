// tl_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tilelink.h"

struct tl_signals {
  int device;
  int num_flags;
  uint32_t* flags;   // device, num_flags words
  uint32_t* status;  // device, 4 words: code, where, seen, expected
};

namespace tl {

constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s

// Record a message for tl_last_error() and return `code`.
tl_status fail(tl_status code, const char* fmt, ...);
// Map a CUDA runtime error to TL_ERR_CUDA with a message; TL_OK on success.
tl_status cuda_ok(cudaError_t e, const char* what);

struct DeviceInfo {
  int device;
  int sm_count;
  int max_smem_optin;
  int cc_major;
  int cc_minor;
  int coop_launch;
};
tl_status device_info(DeviceInfo* out);

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with the given row
// pitch; box = box_rows x box_cols elements; 128-byte swizzle unless given;
// out-of-range elements read as zero (and are not written by stores).
tl_status make_map_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        uint64_t row_pitch_bytes, uint32_t box_rows, uint32_t box_cols,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// 3-D bf16 tensor map over `planes` stacked row-major [rows, cols] matrices
// (plane pitch in bytes); box = box_rows x box_cols elements of one plane,
// 128-byte swizzle.  Rows past `rows` read as zero, so a box never reaches
// into the next plane.
tl_status make_map_bf16_3d(CUtensorMap* map, const void* base, uint64_t planes, uint64_t rows, uint64_t cols,
                           uint64_t row_pitch_bytes, uint64_t plane_pitch_bytes, uint32_t box_rows,
                           uint32_t box_cols);

// Launch a grid whose CTAs must all be resident at once: a cooperative launch
// for single CTAs, a cluster launch sized within the device's resident-cluster
// capacity for clusters of `cluster` CTAs.  Fails instead of launching when the
// grid cannot be resident at once.
// early_start (clusters only): programmatic dependent launch -- the grid may start
// before the previous kernel on the stream has finished, and must wait for it
// (griddepcontrol.wait) before it reads what that kernel wrote.
tl_status launch_coop(const void* kernel, int grid, int block, size_t smem, cudaStream_t st, void** args,
                      int cluster = 1, bool early_start = false);

// Where each of R shard pointers lives: device memory of `device` (bulk TMA
// copies), or pinned host / managed memory (plain loads; bit r of *host_mask).
// dev[r] receives the address the device uses.  Pageable host memory and other
// devices' memory are rejected (TL_ERR_UNSUPPORTED) before any launch.
tl_status classify_shards(const char* who, const void* const* shards, int R, int device, const uint8_t** dev,
                          uint64_t* host_mask);

// The calling thread's held-chunk setting (tl_test_hold_chunks) for a copy-warp launch
// whose flag waits are bounded by timeout_ns: count 0 when none.  Rejects a hold that
// would not end well inside the waits' bound.
tl_status test_hold(const char* who, uint64_t timeout_ns, int32_t* first, int32_t* count, uint64_t* hold_ns);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

}  // namespace tl
