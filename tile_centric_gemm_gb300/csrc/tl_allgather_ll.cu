// tl_allgather_ll.cu -- AllGather through a slow link with a low-latency
// protocol that carries the flag inside the data.
//
// TileLink talk summary ("TileLink: Generating Efficient Compute-Communication
// Overlapping Kernels using Tile-Centric Primitives"), Experimental Setup &
// Results, further results: an AllGather over PCIe with a low-latency protocol
// runs about three times faster than NCCL's.  The summary gives no format; the
// reading here is the classic flag-in-data one: every 8-byte link word holds 4
// bytes of data and 4 bytes of the call's epoch, written and read as one
// single-copy-atomic 64-bit access, so a receiver that sees the epoch in a word
// also sees that word's data -- no fence on the sender's side between data and
// flag, and no separate flag to poll on the receiver's side.  The price is
// twice the bytes on the link, so the protocol is for small messages, where the
// round trips of the flag protocol dominate.
//
// One launch emulates both sides of a push AllGather of R ranks on one GPU (all
// CTAs co-resident: receivers wait for senders of the same launch):
//   send    -- for every rank r != self in send_mask: the rank's shard A_r is
//              written into its region of the link buffer (pinned host memory:
//              the stand-in for the slow link; or device memory);
//   receive -- rank self's receiver takes every peer's region from the link
//              into `gathered` (rows r*M_shard ...), chunk by chunk, and
//              releases one flag per chunk for local consumers
//              (produce_tile_notify, the flag ids of tl_allgather);
//   the self shard is copied into `gathered` directly (it crosses no link).
// Two protocols on the same link buffer, so they can be timed against each
// other:
//   TL_LL_FLAG_IN_DATA  -- link word = {data[4 bytes], epoch}; the receiver
//                          polls each word until it carries the epoch (bounded);
//   TL_LL_SEPARATE_FLAG -- the sender writes the raw data, fences at system
//                          scope and release-stores the chunk's flag in the
//                          link buffer; the receiver acquires the flag, then
//                          reads the data (two round trips over the link).
// Ranks outside send_mask are not sent by this launch: their link regions are
// filled by another agent (the host, or an earlier launch) with the same
// epoch, and the receiver waits for them like for any other.
#include <algorithm>

#include "tl_internal.h"
#include "tl_ptx.cuh"

namespace tl {
namespace {

constexpr int LL_WARPS = 4;
constexpr int LL_THREADS = LL_WARPS * 32;
constexpr uint32_t LL_FLAG_STRIDE = 128;  // bytes between two chunk flags of the separate-flag protocol
constexpr int LL_VEC = 8;                 // 16-byte vectors in flight per lane (link reads are round trips)

struct LlParams {
  const uint8_t* shard[TL_MAX_RANKS];  // sources [M_shard, K] bf16 (device or host memory)
  uint8_t* link;                       // link buffer
  uint8_t* gathered;                   // [R*M_shard, K] bf16
  uint32_t* flags;                     // one per chunk, for local consumers
  uint32_t* status;
  uint64_t timeout_ns;
  uint64_t send_mask;
  size_t raw_bytes;                    // R * M_shard * K * 2: start of the separate-flag area
  int32_t R, self, M_shard, K, rpb, bpr, protocol;
  uint32_t epoch;
};

__device__ __forceinline__ void st_volatile_v2u64(void* p, uint64_t a, uint64_t b) {
  asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_volatile_v2u64(const void* p) {
  ulonglong2 v;
  asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_volatile_v4u32(const void* p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_release_sys(uint32_t* p, uint32_t v) {
  asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Chunk c of rank r: rows [lo, lo + rows) of the shard, `bytes` of data starting
// at data offset `off` of the gathered layout (also the raw link layout).
struct Chunk {
  int r, lo, rows, flag_id;
  size_t off;
  uint32_t bytes;
};
__device__ __forceinline__ Chunk chunk_of(const LlParams& p, int r, int c) {
  Chunk x;
  x.r = r;
  x.lo = c * p.rpb;
  x.rows = min(p.rpb, p.M_shard - x.lo);
  x.flag_id = r * p.bpr + c;
  x.off = (size_t(r) * p.M_shard + x.lo) * size_t(p.K) * 2;
  x.bytes = uint32_t(x.rows) * uint32_t(p.K) * 2u;
  return x;
}

// Sender of one chunk (all 32 lanes).
__device__ void send_chunk(const LlParams& p, const Chunk& x, int lane) {
  const uint4* src = reinterpret_cast<const uint4*>(p.shard[x.r] + size_t(x.lo) * p.K * 2);
  const uint32_t n16 = x.bytes / 16u;
  if (p.protocol == TL_LL_FLAG_IN_DATA) {
    // 16 data bytes -> two 16-byte link stores of {data, epoch} word pairs
    uint8_t* dst = p.link + x.off * 2;
    const uint64_t e = uint64_t(p.epoch) << 32;
    for (uint32_t base = 0; base < n16; base += 32u * LL_VEC) {
      uint4 v[LL_VEC];  // every source read of the batch in flight before the first store
#pragma unroll
      for (int u = 0; u < LL_VEC; ++u) {
        const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
        if (i < n16) v[u] = __ldcg(src + i);
      }
#pragma unroll
      for (int u = 0; u < LL_VEC; ++u) {
        const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
        if (i < n16) {
          st_volatile_v2u64(dst + size_t(i) * 32, e | v[u].x, e | v[u].y);
          st_volatile_v2u64(dst + size_t(i) * 32 + 16, e | v[u].z, e | v[u].w);
        }
      }
    }
  } else {
    uint4* dst = reinterpret_cast<uint4*>(p.link + x.off);
    for (uint32_t base = 0; base < n16; base += 32u * LL_VEC) {
      uint4 v[LL_VEC];
#pragma unroll
      for (int u = 0; u < LL_VEC; ++u) {
        const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
        if (i < n16) v[u] = __ldcg(src + i);
      }
#pragma unroll
      for (int u = 0; u < LL_VEC; ++u) {
        const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
        if (i < n16) __stcg(dst + i, v[u]);
      }
    }
    // the data reaches the link before the flag: system-scope fence, then release
    __threadfence_system();
    __syncwarp();
    if (lane == 0)
      st_release_sys(reinterpret_cast<uint32_t*>(p.link + p.raw_bytes + size_t(x.flag_id) * LL_FLAG_STRIDE), p.epoch);
  }
}

// Receiver of one chunk (all 32 lanes).  Returns false if a bounded wait ran out.
// Every lane keeps LL_VEC link reads in flight at once (a read of host memory is
// a round trip over the link), then re-polls only the words not yet valid.
__device__ bool recv_chunk(const LlParams& p, const Chunk& x, int lane) {
  uint4* dst = reinterpret_cast<uint4*>(p.gathered + x.off);
  const uint32_t n16 = x.bytes / 16u;
  bool ok = true;
  if (p.protocol == TL_LL_FLAG_IN_DATA) {
    const uint8_t* src = p.link + x.off * 2;
    const uint64_t t0 = now_ns();
    for (uint32_t base = 0; base < n16 && ok; base += 32u * LL_VEC) {
      ulonglong2 a[LL_VEC], b[LL_VEC];
#pragma unroll
      for (int u = 0; u < LL_VEC; ++u) {
        const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
        if (i < n16) {
          a[u] = ld_volatile_v2u64(src + size_t(i) * 32);
          b[u] = ld_volatile_v2u64(src + size_t(i) * 32 + 16);
        }
      }
      uint32_t spins = 0;
      while (true) {
        // words of this batch still without the epoch: read them again
        bool all = true;
#pragma unroll
        for (int u = 0; u < LL_VEC; ++u) {
          const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
          if (i >= n16) continue;
          if (!epoch_reached(uint32_t(a[u].x >> 32), p.epoch) || !epoch_reached(uint32_t(a[u].y >> 32), p.epoch)) {
            a[u] = ld_volatile_v2u64(src + size_t(i) * 32);
            all = false;
          }
          if (!epoch_reached(uint32_t(b[u].x >> 32), p.epoch) || !epoch_reached(uint32_t(b[u].y >> 32), p.epoch)) {
            b[u] = ld_volatile_v2u64(src + size_t(i) * 32 + 16);
            all = false;
          }
        }
        if (all) break;
        if ((++spins & 15u) == 0u) {
          if (ld_volatile(p.status) != 0u) {
            ok = false;
            break;
          }
          if (now_ns() - t0 > p.timeout_ns) {
            // the flag half of the first link word of this lane that is not set yet
            uint32_t seen = p.epoch;
#pragma unroll
            for (int u = LL_VEC - 1; u >= 0; --u) {
              const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
              if (i >= n16) continue;
              const uint32_t f[4] = {uint32_t(a[u].x >> 32), uint32_t(a[u].y >> 32), uint32_t(b[u].x >> 32),
                                     uint32_t(b[u].y >> 32)};
              for (int q = 3; q >= 0; --q)
                if (!epoch_reached(f[q], p.epoch)) seen = f[q];
            }
            record_error(p.status, TL_ERR_TIMEOUT, uint32_t(x.flag_id), seen, p.epoch);
            ok = false;
            break;
          }
        }
      }
      if (!ok) break;
#pragma unroll
      for (int u = 0; u < LL_VEC; ++u) {
        const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
        if (i < n16) __stcg(dst + i, make_uint4(uint32_t(a[u].x), uint32_t(a[u].y), uint32_t(b[u].x), uint32_t(b[u].y)));
      }
    }
  } else {
    if (lane == 0) {
      const uint32_t* f = reinterpret_cast<const uint32_t*>(p.link + p.raw_bytes + size_t(x.flag_id) * LL_FLAG_STRIDE);
      const uint64_t t0 = now_ns();
      uint32_t spins = 0, v = ld_acquire_sys(f);
      while (!epoch_reached(v, p.epoch)) {
        if ((++spins & 31u) == 0u) {
          if (ld_volatile(p.status) != 0u) {
            ok = false;
            break;
          }
          if (now_ns() - t0 > p.timeout_ns) {
            record_error(p.status, TL_ERR_TIMEOUT, uint32_t(x.flag_id), v, p.epoch);
            ok = false;
            break;
          }
        }
        v = ld_acquire_sys(f);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();  // every lane's data loads come after lane 0's acquire
    if (ok) {
      const uint8_t* src = p.link + x.off;
      for (uint32_t base = 0; base < n16; base += 32u * LL_VEC) {
        uint4 v[LL_VEC];
#pragma unroll
        for (int u = 0; u < LL_VEC; ++u) {
          const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
          if (i < n16) v[u] = ld_volatile_v4u32(src + size_t(i) * 16);
        }
#pragma unroll
        for (int u = 0; u < LL_VEC; ++u) {
          const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
          if (i < n16) __stcg(dst + i, v[u]);
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// Warps take send items (peer chunks of the ranks in send_mask), then the self
// shard's chunks, then receive items, each in rank order self+1, ..., self-1.
__global__ void __launch_bounds__(LL_THREADS) allgather_ll_kernel(const __grid_constant__ LlParams p) {
  const int lane = int(lane_id());
  const int gw = int(blockIdx.x) * LL_WARPS + int(warp_id());
  const int nw = int(gridDim.x) * LL_WARPS;
  const int peer_items = (p.R - 1) * p.bpr;
  // 1. send
  for (int it = gw; it < peer_items; it += nw) {
    const int r = (p.self + 1 + it / p.bpr) % p.R;
    if ((p.send_mask >> r) & 1ull) send_chunk(p, chunk_of(p, r, it % p.bpr), lane);
  }
  // 2. the self shard, straight into gathered
  for (int c = gw; c < p.bpr; c += nw) {
    const Chunk x = chunk_of(p, p.self, c);
    const uint4* src = reinterpret_cast<const uint4*>(p.shard[p.self] + size_t(x.lo) * p.K * 2);
    uint4* dst = reinterpret_cast<uint4*>(p.gathered + x.off);
    const uint32_t n16 = x.bytes / 16u;
    for (uint32_t base = 0; base < n16; base += 32u * LL_VEC) {
      uint4 v[LL_VEC];
#pragma unroll
      for (int u = 0; u < LL_VEC; ++u) {
        const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
        if (i < n16) v[u] = __ldcg(src + i);
      }
#pragma unroll
      for (int u = 0; u < LL_VEC; ++u) {
        const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
        if (i < n16) __stcg(dst + i, v[u]);
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release(p.flags + x.flag_id, p.epoch);
  }
  // 3. receive
  for (int it = gw; it < peer_items; it += nw) {
    const Chunk x = chunk_of(p, (p.self + 1 + it / p.bpr) % p.R, it % p.bpr);
    if (!recv_chunk(p, x, lane)) break;
    // produce_tile_notify for local consumers of `gathered`
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release(p.flags + x.flag_id, p.epoch);
  }
}

int ll_default_rpb(int M_shard, int K) { return std::max(1, std::min(M_shard, int(8192 / (size_t(K) * 2)))); }

}  // namespace
}  // namespace tl

extern "C" size_t tl_allgather_ll_link_bytes(int R, int M_shard, int K, int rows_per_barrier) {
  if (R < 1 || M_shard < 1 || K < 1) return 0;
  const int rpb = rows_per_barrier > 0 ? std::min(rows_per_barrier, M_shard) : tl::ll_default_rpb(M_shard, K);
  const size_t raw = size_t(R) * M_shard * size_t(K) * 2;
  const size_t flags = size_t(R) * tl::cdiv(M_shard, rpb) * tl::LL_FLAG_STRIDE;
  return std::max(2 * raw, raw + flags);
}

extern "C" tl_status tl_allgather_ll(const tl_allgather_ll_args* a, void* stream) {
  using namespace tl;
  if (!a) return fail(TL_ERR_INVALID, "tl_allgather_ll: NULL args");
  if (a->R < 1 || a->R > TL_MAX_RANKS) return fail(TL_ERR_INVALID, "tl_allgather_ll: R=%d", a->R);
  if (a->self_rank < 0 || a->self_rank >= a->R) return fail(TL_ERR_INVALID, "tl_allgather_ll: self_rank");
  if (a->M_shard < 1 || a->K < 1) return fail(TL_ERR_INVALID, "tl_allgather_ll: empty shape");
  if (a->K % 8) return fail(TL_ERR_UNSUPPORTED, "tl_allgather_ll: K (%d) must be a multiple of 8", a->K);
  if (a->protocol != TL_LL_FLAG_IN_DATA && a->protocol != TL_LL_SEPARATE_FLAG)
    return fail(TL_ERR_INVALID, "tl_allgather_ll: protocol %d", a->protocol);
  if (!a->A_shards || !a->link || !a->gathered || !a->signals)
    return fail(TL_ERR_INVALID, "tl_allgather_ll: NULL pointer argument");
  if (a->epoch == 0) return fail(TL_ERR_INVALID, "tl_allgather_ll: epoch must be nonzero");
  if (!aligned16(a->link) || !aligned16(a->gathered)) return fail(TL_ERR_INVALID, "tl_allgather_ll: alignment");
  const size_t need = tl_allgather_ll_link_bytes(a->R, a->M_shard, a->K, a->rows_per_barrier);
  if (a->link_bytes < need)
    return fail(TL_ERR_INVALID, "tl_allgather_ll: link buffer %zu bytes, need %zu", a->link_bytes, need);
  for (int r = 0; r < a->R; ++r)
    if (!a->A_shards[r] || !aligned16(a->A_shards[r])) return fail(TL_ERR_INVALID, "tl_allgather_ll: shard %d", r);
  const int rpb = a->rows_per_barrier > 0 ? std::min(a->rows_per_barrier, a->M_shard) : ll_default_rpb(a->M_shard, a->K);
  const int bpr = cdiv(a->M_shard, rpb);
  const int nflags = a->R * bpr;
  if (a->signals->num_flags < nflags)
    return fail(TL_ERR_INVALID, "tl_allgather_ll: signals hold %d flags, need %d", a->signals->num_flags, nflags);
  DeviceInfo di{};
  if (tl_status s = device_info(&di)) return s;
  if (a->signals->device != di.device) return fail(TL_ERR_INVALID, "tl_allgather_ll: signals belong to another device");
  LlParams p{};
  uint64_t host_mask = 0;
  if (tl_status s = classify_shards("tl_allgather_ll", a->A_shards, a->R, di.device, p.shard, &host_mask)) return s;
  {
    // the link buffer: device memory of this device, or pinned host / managed memory
    const void* lp[1] = {a->link};
    const uint8_t* ld[1];
    uint64_t lm = 0;
    if (tl_status s = classify_shards("tl_allgather_ll (link)", lp, 1, di.device, ld, &lm)) return s;
    p.link = const_cast<uint8_t*>(ld[0]);
  }
  p.gathered = static_cast<uint8_t*>(a->gathered);
  p.flags = a->signals->flags;
  p.status = a->signals->status;
  p.timeout_ns = a->timeout_ns ? a->timeout_ns : kDefaultTimeoutNs;
  p.send_mask = a->send_mask;
  p.raw_bytes = size_t(a->R) * a->M_shard * size_t(a->K) * 2;
  p.R = a->R;
  p.self = a->self_rank;
  p.M_shard = a->M_shard;
  p.K = a->K;
  p.rpb = rpb;
  p.bpr = bpr;
  p.protocol = a->protocol;
  p.epoch = a->epoch;
  const int items = std::max(1, std::max((a->R - 1) * bpr, bpr));
  const int grid = std::max(1, std::min(di.sm_count, cdiv(items, LL_WARPS)));
  void* args[] = {&p};
  return launch_coop(reinterpret_cast<const void*>(&allgather_ll_kernel), grid, LL_THREADS, 0, (cudaStream_t)stream,
                     args);
}
