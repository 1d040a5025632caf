// tl_host.cu -- error reporting, device queries, tensor maps, co-resident launches,
// and the signal primitives of the C ABI (tl_signals_*, tl_tile_notify,
// tl_tile_wait, tl_query_status).
//
// Signal semantics follow the TileLink talk summary ("TileLink: Generating
// Efficient Compute-Communication Overlapping Kernels using Tile-Centric
// Primitives", Technical Deep Dive): produce_tile_notify lowers to a
// synchronisation followed by an atomic flag update, consume_tile_wait polls
// the flag a tile id maps to.  Here a notify is a gpu-scope release store and a
// wait a gpu-scope acquire load in a bounded loop.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "tl_internal.h"
#include "tl_ptx.cuh"

namespace {
thread_local char g_last_error[512] = "";
// tl_test_hold_chunks: chunks [first, first + count) are copied last, after hold_ns
struct Hold {
  int first, count;
  uint64_t ns;
};
thread_local Hold g_hold = {0, 0, 0};
}

namespace tl {

tl_status fail(tl_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

tl_status test_hold(const char* who, uint64_t timeout_ns, int32_t* first, int32_t* count, uint64_t* hold_ns) {
  *first = g_hold.first;
  *count = g_hold.count;
  *hold_ns = g_hold.ns;
  if (g_hold.count > 0 && 2 * g_hold.ns >= timeout_ns)
    return fail(TL_ERR_INVALID, "%s: held chunks wait %llu ns, which is not below half the timeout (%llu ns)", who,
                (unsigned long long)g_hold.ns, (unsigned long long)timeout_ns);
  return TL_OK;
}

tl_status cuda_ok(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return TL_OK;
  return fail(TL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

tl_status device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  if (tl_status s = cuda_ok(cudaGetDevice(&dev), "cudaGetDevice")) return s;
  if (dev < 0 || dev >= 64) return fail(TL_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    DeviceInfo d{};
    d.device = dev;
    if (tl_status s = cuda_ok(cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev), "sm count"))
      return s;
    if (tl_status s = cuda_ok(
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev), "smem optin"))
      return s;
    if (tl_status s = cuda_ok(cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev), "cc"))
      return s;
    if (tl_status s = cuda_ok(cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev), "cc"))
      return s;
    if (tl_status s = cuda_ok(cudaDeviceGetAttribute(&d.coop_launch, cudaDevAttrCooperativeLaunch, dev), "coop"))
      return s;
    cache[dev] = d;
    have[dev] = true;
  }
  *out = cache[dev];
  if (out->cc_major != 10 || out->cc_minor != 3)
    return fail(TL_ERR_UNSUPPORTED, "kernels are built for sm_103a; device is sm_%d%d", out->cc_major, out->cc_minor);
  return TL_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

tl_status make_map_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t row_pitch_bytes,
                        uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return fail(TL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  // TMA operands must be memory of the current device
  cudaPointerAttributes at{};
  int dev = -1;
  if (cudaPointerGetAttributes(&at, base) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(TL_ERR_UNSUPPORTED, "tensor operand %p is not memory the device can address", base);
  }
  if (at.type != cudaMemoryTypeDevice || at.device != dev)
    return fail(TL_ERR_UNSUPPORTED, "tensor operand %p must be device memory of device %d (TMA-loaded)", base, dev);
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TL_ERR_INVALID, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] pitch %llu", int(r),
                (unsigned long long)rows, (unsigned long long)cols, (unsigned long long)row_pitch_bytes);
  return TL_OK;
}

tl_status make_map_bf16_3d(CUtensorMap* map, const void* base, uint64_t planes, uint64_t rows, uint64_t cols,
                           uint64_t row_pitch_bytes, uint64_t plane_pitch_bytes, uint32_t box_rows,
                           uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn) return fail(TL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cudaPointerAttributes at{};
  int dev = -1;
  if (cudaPointerGetAttributes(&at, base) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(TL_ERR_UNSUPPORTED, "tensor operand %p is not memory the device can address", base);
  }
  if (at.type != cudaMemoryTypeDevice || at.device != dev)
    return fail(TL_ERR_UNSUPPORTED, "tensor operand %p must be device memory of device %d (TMA-loaded)", base, dev);
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {row_pitch_bytes, plane_pitch_bytes};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TL_ERR_INVALID, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu x %llu]", int(r),
                (unsigned long long)planes, (unsigned long long)rows, (unsigned long long)cols);
  return TL_OK;
}

tl_status classify_shards(const char* who, const void* const* shards, int R, int device, const uint8_t** dev,
                          uint64_t* host_mask) {
  *host_mask = 0;
  for (int r = 0; r < R; ++r) {
    cudaPointerAttributes at{};
    const cudaError_t e = cudaPointerGetAttributes(&at, shards[r]);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return fail(TL_ERR_UNSUPPORTED, "%s: shard %d is not memory the device can address (%s)", who, r,
                  cudaGetErrorName(e));
    }
    if (at.type == cudaMemoryTypeDevice) {
      if (at.device != device)
        return fail(TL_ERR_UNSUPPORTED, "%s: shard %d lives on device %d, the call runs on device %d", who, r,
                    at.device, device);
      dev[r] = static_cast<const uint8_t*>(shards[r]);
    } else if (at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged) {
      if (!at.devicePointer)
        return fail(TL_ERR_UNSUPPORTED, "%s: host shard %d is not mapped into the device's address space", who, r);
      dev[r] = static_cast<const uint8_t*>(at.devicePointer);
      *host_mask |= 1ull << r;
    } else {
      return fail(TL_ERR_UNSUPPORTED, "%s: shard %d is pageable host memory; pin it (cudaHostAlloc / "
                                      "cudaHostRegister) or place it on the device", who, r);
    }
    if (!aligned16(dev[r])) return fail(TL_ERR_INVALID, "%s: shard %d device address is not 16-byte aligned", who, r);
  }
  return TL_OK;
}

namespace {
// The dynamic shared-memory limit of a kernel is raised per device to the most
// any launch has asked for (never lowered: a kernel whose launches ask for
// different sizes keeps a limit that fits them all); the resident capacity
// (CTAs per SM, or clusters) is queried once per (device, kernel, block, smem,
// cluster) and reused.
struct LaunchKey {
  int device;
  const void* kernel;
  int block;
  size_t smem;
  int cluster;
  bool operator==(const LaunchKey& o) const {
    return device == o.device && kernel == o.kernel && block == o.block && smem == o.smem && cluster == o.cluster;
  }
};
struct LaunchEntry {
  LaunchKey key;
  int capacity;
};
struct SmemLimit {
  int device;
  const void* kernel;
  size_t smem;
};
std::mutex g_launch_mu;
LaunchEntry g_launch_cache[64];
int g_launch_n = 0;
SmemLimit g_smem_limit[64];
int g_smem_n = 0;

// Raise `kernel`'s dynamic shared-memory limit on `device` to at least `smem`.
tl_status ensure_smem_limit(int device, const void* kernel, size_t smem) {
  std::lock_guard<std::mutex> lock(g_launch_mu);
  int slot = -1;
  for (int i = 0; i < g_smem_n; ++i)
    if (g_smem_limit[i].device == device && g_smem_limit[i].kernel == kernel) slot = i;
  if (slot >= 0 && g_smem_limit[slot].smem >= smem) return TL_OK;
  if (tl_status s = cuda_ok(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                            "cudaFuncSetAttribute(max dynamic smem)"))
    return s;
  if (slot >= 0) g_smem_limit[slot].smem = smem;
  else if (g_smem_n < 64) g_smem_limit[g_smem_n++] = SmemLimit{device, kernel, smem};
  return TL_OK;
}
}  // namespace

tl_status launch_coop(const void* kernel, int grid, int block, size_t smem, cudaStream_t st, void** args,
                      int cluster, bool early_start) {
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  if (cluster < 1 || grid % cluster) return fail(TL_ERR_INTERNAL, "grid %d is not a multiple of cluster %d", grid, cluster);
  if (tl_status s = ensure_smem_limit(di.device, kernel, smem)) return s;
  const LaunchKey key{di.device, kernel, block, smem, cluster};
  int capacity = -1;
  {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    for (int i = 0; i < g_launch_n; ++i)
      if (g_launch_cache[i].key == key) capacity = g_launch_cache[i].capacity;
  }
  if (capacity < 0) {
    if (cluster > 1) {
      cudaLaunchConfig_t q{};
      q.gridDim = dim3(grid);
      q.blockDim = dim3(block);
      q.dynamicSmemBytes = smem;
      cudaLaunchAttribute ca[1];
      ca[0].id = cudaLaunchAttributeClusterDimension;
      ca[0].val.clusterDim.x = unsigned(cluster);
      ca[0].val.clusterDim.y = 1;
      ca[0].val.clusterDim.z = 1;
      q.attrs = ca;
      q.numAttrs = 1;
      if (tl_status s = cuda_ok(cudaOccupancyMaxActiveClusters(&capacity, kernel, &q), "cluster occupancy")) return s;
      capacity *= cluster;
    } else {
      int per_sm = 0;
      if (tl_status s = cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, smem),
                                "occupancy"))
        return s;
      capacity = per_sm * di.sm_count;
    }
    std::lock_guard<std::mutex> lock(g_launch_mu);
    if (g_launch_n < 64) g_launch_cache[g_launch_n++] = LaunchEntry{key, capacity};
  }
  if (grid > capacity)
    return fail(TL_ERR_UNSUPPORTED, "grid of %d CTAs (clusters of %d) cannot be co-resident (at most %d)", grid,
                cluster, capacity);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  if (cluster > 1) {
    // Clusters: the grid is sized to the number of clusters the device holds at
    // once, so every CTA is resident together (the cooperative attribute is not
    // combined with clusters: profilers cannot launch that combination).  Every
    // cross-CTA wait in the kernels is bounded in any case.
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (early_start) {
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.numAttrs = 2;
    }
    return cuda_ok(cudaLaunchKernelExC(&cfg, kernel, args), "cluster launch");
  }
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelExC(&cfg, kernel, args), "cooperative launch");
}

}  // namespace tl

// ---------------------------------------------------------------- kernels of the signal API
namespace {

__global__ void notify_kernel(uint32_t* flags, int first, int count, uint32_t value) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) tl::st_release(flags + first + i, value);
}

// One warp; lane l polls flags first+l, first+l+32, ...
__global__ void wait_kernel(const uint32_t* flags, uint32_t* status, int first, int count, uint32_t value,
                            uint64_t timeout_ns) {
  for (int i = threadIdx.x; i < count; i += 32) {
    if (!tl::wait_flag(flags + first + i, value, status, timeout_ns, uint32_t(first + i), TL_ERR_TIMEOUT)) break;
  }
}

}  // namespace

extern "C" {

int tl_version(void) { return TL_VERSION; }
const char* tl_last_error(void) { return g_last_error; }

tl_status tl_signals_create(int num_flags, tl_signals** out) {
  if (!out) return tl::fail(TL_ERR_INVALID, "tl_signals_create: out is NULL");
  *out = nullptr;
  if (num_flags < 1) return tl::fail(TL_ERR_INVALID, "tl_signals_create: num_flags %d < 1", num_flags);
  int dev = 0;
  if (tl_status s = tl::cuda_ok(cudaGetDevice(&dev), "cudaGetDevice")) return s;
  uint32_t* mem = nullptr;
  size_t bytes = (size_t(num_flags) + 4) * sizeof(uint32_t);
  if (tl_status s = tl::cuda_ok(cudaMalloc(&mem, bytes), "cudaMalloc(signals)")) return s;
  if (tl_status s = tl::cuda_ok(cudaMemset(mem, 0, bytes), "cudaMemset(signals)")) {
    cudaFree(mem);
    return s;
  }
  auto* sig = new (std::nothrow) tl_signals;
  if (!sig) {
    cudaFree(mem);
    return tl::fail(TL_ERR_INTERNAL, "out of host memory");
  }
  sig->device = dev;
  sig->num_flags = num_flags;
  sig->status = mem;
  sig->flags = mem + 4;
  *out = sig;
  return TL_OK;
}

tl_status tl_signals_destroy(tl_signals* s) {
  if (!s) return TL_OK;
  tl_status st = tl::cuda_ok(cudaFree(s->status), "cudaFree(signals)");
  delete s;
  return st;
}

tl_status tl_signals_flags(const tl_signals* s, uint32_t** dev_flags, int* num_flags) {
  if (!s) return tl::fail(TL_ERR_INVALID, "tl_signals_flags: NULL signals");
  if (dev_flags) *dev_flags = s->flags;
  if (num_flags) *num_flags = s->num_flags;
  return TL_OK;
}

tl_status tl_signals_reset(tl_signals* s, void* stream) {
  if (!s) return tl::fail(TL_ERR_INVALID, "tl_signals_reset: NULL signals");
  return tl::cuda_ok(cudaMemsetAsync(s->status, 0, (size_t(s->num_flags) + 4) * 4, (cudaStream_t)stream),
                     "cudaMemsetAsync(signals)");
}

tl_status tl_tile_notify(tl_signals* s, int first, int count, uint32_t value, void* stream) {
  if (!s) return tl::fail(TL_ERR_INVALID, "tl_tile_notify: NULL signals");
  if (first < 0 || count < 0 || first + count > s->num_flags)
    return tl::fail(TL_ERR_INVALID, "tl_tile_notify: range [%d, %d) outside %d flags", first, first + count,
                    s->num_flags);
  if (count == 0) return TL_OK;
  notify_kernel<<<(count + 255) / 256, 256, 0, (cudaStream_t)stream>>>(s->flags, first, count, value);
  return tl::cuda_ok(cudaGetLastError(), "notify launch");
}

tl_status tl_tile_wait(tl_signals* s, int first, int count, uint32_t value, uint64_t timeout_ns, void* stream) {
  if (!s) return tl::fail(TL_ERR_INVALID, "tl_tile_wait: NULL signals");
  if (first < 0 || count < 0 || first + count > s->num_flags)
    return tl::fail(TL_ERR_INVALID, "tl_tile_wait: range [%d, %d) outside %d flags", first, first + count,
                    s->num_flags);
  if (count == 0) return TL_OK;
  if (timeout_ns == 0) timeout_ns = tl::kDefaultTimeoutNs;
  wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(s->flags, s->status, first, count, value, timeout_ns);
  return tl::cuda_ok(cudaGetLastError(), "wait launch");
}

tl_status tl_query_status(tl_signals* s, void* stream, int* code, int* where) {
  if (!s) return tl::fail(TL_ERR_INVALID, "tl_query_status: NULL signals");
  cudaStream_t st = (cudaStream_t)stream;
  if (tl_status e = tl::cuda_ok(cudaStreamSynchronize(st), "cudaStreamSynchronize")) return e;
  uint32_t h[4] = {0, 0, 0, 0};
  if (tl_status e = tl::cuda_ok(cudaMemcpy(h, s->status, sizeof(h), cudaMemcpyDeviceToHost), "read status"))
    return e;
  if (h[0] != 0) {
    if (tl_status e = tl::cuda_ok(cudaMemset(s->status, 0, sizeof(h)), "clear status")) return e;
  }
  if (code) *code = int(h[0]);
  if (where) *where = h[0] ? int(h[1]) : -1;
  if (h[0] == 0) return TL_OK;
  if (h[0] == TL_ERR_TIMEOUT)
    return tl::fail(TL_ERR_TIMEOUT, "device wait timed out at %d (flag value %u, expected epoch %u)", int(h[1]), h[2],
                    h[3]);
  return tl::fail(tl_status(h[0]), "device error %u at 0x%x", h[0], h[1]);
}

}  // extern "C"

extern "C" tl_status tl_test_hold_chunks(int first_flag, int count, uint64_t hold_ns) {
  if (count < 0 || first_flag < 0) return tl::fail(TL_ERR_INVALID, "tl_test_hold_chunks: negative range");
  if (hold_ns > 100000000ull) return tl::fail(TL_ERR_INVALID, "tl_test_hold_chunks: hold above 100 ms");
  g_hold = Hold{first_flag, count, hold_ns};
  return TL_OK;
}
