// tl_copy.cuh -- the AllGather producer shared by the fused AllGather-GEMM
// kernel and the stand-alone AllGather: one warp moves row chunks of the shards
// into the gathered buffer and releases one flag per chunk once its writes are
// complete (produce_tile_notify).  Pull mode first acquires the source's
// readiness flag of the same chunk.
//  * Shards in device memory: one lane streams the chunk through a ring of
//    shared-memory buffers with bulk TMA copies (global -> shared -> global),
//    the source lines marked evict-first in L2 (they are read once).
//  * Shards in pinned host (or managed) memory -- the stand-in for a slower
//    link: all 32 lanes copy 16-byte vectors with plain loads and stores, many
//    loads in flight per lane, then fence before the release.
#pragma once

#include "tilelink.h"
#include "tl_common.cuh"

namespace tl {

struct AgCopyJob {
  const uint8_t* const* shard;  // R source shards [M_shard, K]
  uint8_t* gathered;            // [R*M_shard, K]
  uint32_t* flags;              // R * bpr arrival flags
  const uint32_t* ready;        // pull mode readiness flags, or nullptr
  uint32_t* status;
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int R, self, M_shard, K, rpb, bpr, num_items;
  uint32_t epoch;
  uint64_t host_mask;  // bit r: shard r is host (or managed) memory, copied with plain loads
  // held chunks (a test facility that forces an arrival order): chunks whose flag id lies in
  // [hold_first, hold_first + hold_count) are copied after every other chunk of the copy
  // warp, and not before hold_ns have passed since the warp started
  int hold_first, hold_count;
  uint64_t hold_ns;
};

__device__ __forceinline__ bool ag_item_held(const AgCopyJob& j, int it) {
  if (j.hold_count <= 0) return false;
  const int r = (j.self + 1 + it / j.bpr) % j.R;
  const int f = r * j.bpr + it % j.bpr;
  return f >= j.hold_first && f < j.hold_first + j.hold_count;
}

// Lane 0 spins until hold_ns have passed since t0 (a bounded wait: hold_ns is
// checked on the host against the call's timeout), or the launch has aborted.
__device__ __forceinline__ void hold_until(uint64_t t0, uint64_t hold_ns, volatile uint32_t* abort,
                                           const uint32_t* status) {
  while (now_ns() - t0 < hold_ns) {
    if (*abort || ld_volatile(status) != 0u) break;
    __nanosleep(1000);
  }
}

// Copy `bytes` (a multiple of 16) from src (host or device memory) to dst with
// every lane of the warp: kVec 16-byte loads in flight per lane.
__device__ __forceinline__ void copy_rows_plain(const uint8_t* src, uint8_t* dst, uint32_t bytes, int lane) {
  constexpr int kVec = 8;
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  const uint32_t n = bytes / 16u;
  for (uint32_t base = 0; base < n; base += 32u * kVec) {
    uint4 v[kVec];
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
      if (i < n) v[u] = __ldcg(s + i);
    }
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const uint32_t i = base + uint32_t(u) * 32u + uint32_t(lane);
      if (i < n) __stcg(d + i, v[u]);
    }
  }
}

// Item `it` of the job: shard (self + 1 + it / bpr) mod R, row chunk it % bpr.
struct AgItem {
  const uint8_t* src;
  uint8_t* dst;
  uint32_t bytes;
  int flag_id;
  int r;
};
__device__ __forceinline__ AgItem ag_item(const AgCopyJob& j, int it) {
  const int jj = it / j.bpr, b = it % j.bpr;
  const int r = (j.self + 1 + jj) % j.R;
  const int lo = b * j.rpb;
  const int rows = min(j.rpb, j.M_shard - lo);
  return AgItem{j.shard[r] + size_t(lo) * j.K * 2, j.gathered + (size_t(r) * j.M_shard + lo) * size_t(j.K) * 2,
                uint32_t(rows) * uint32_t(j.K) * 2u, r * j.bpr + b, r};
}
// Pull mode: the source publishes readiness first (first barrier of the pull
// protocol); a chunk whose source never became ready is neither copied nor
// announced.  Returns whether to copy (on every lane).
__device__ __forceinline__ bool ag_item_ready(const AgCopyJob& j, const AgItem& x, int lane) {
  bool ready = true;
  if (j.ready && lane == 0)
    ready = wait_flag(j.ready + x.flag_id, j.epoch, j.status, j.timeout_ns, uint32_t(x.flag_id), TL_ERR_TIMEOUT);
  return __shfl_sync(0xffffffffu, ready, 0);
}
// Plain 16-byte loads and stores by every lane, then the release of the chunk's flag.
__device__ __forceinline__ void ag_item_copy_plain(const AgCopyJob& j, const AgItem& x, int lane) {
  copy_rows_plain(x.src, x.dst, x.bytes, lane);
  // produce_tile_notify: every lane's stores are ordered before lane 0's release
  __threadfence();
  __syncwarp();
  if (lane == 0) st_release(j.flags + x.flag_id, j.epoch);
}

// Copy item `it` with plain loads and stores only (no shared-memory staging):
// for a kernel whose shared memory holds other stages.  Called by all 32 lanes
// of one warp; consumers fence the async proxy before their TMA loads of it.
__device__ __forceinline__ void ag_copy_one_plain(const AgCopyJob& j, int it) {
  const int lane = int(lane_id());
  const AgItem x = ag_item(j, it);
  if (ag_item_ready(j, x, lane)) ag_item_copy_plain(j, x, lane);
}

// Copy item `it` into the gathered buffer and release its flag: bulk copies
// through shared memory, or plain loads for a shard in host memory.  Called by
// all 32 lanes of one warp.  `stage` holds NBUF buffers of COPY_CHUNK bytes; `bars`
// NBUF mbarriers initialised with count 1; `seq` (lane 0's count of chunks
// staged so far: buffer seq % NBUF, parity (seq / NBUF) & 1) carries the
// staging ring's state from one call to the next.  Returns true (on every
// lane) if a pipeline wait gave up.
template <int NBUF = COPY_NBUF>
__device__ __forceinline__ bool ag_copy_one(const AgCopyJob& j, int it, uint8_t* stage, uint64_t* bars,
                                            volatile uint32_t* abort, uint32_t& seq) {
  static_assert(NBUF >= 1 && NBUF <= COPY_NBUF, "staging buffers");
  const int lane = int(lane_id());
  const AgItem x = ag_item(j, it);
  const uint8_t* src = x.src;
  uint8_t* dst = x.dst;
  const uint32_t bytes = x.bytes;
  const int flag_id = x.flag_id;
  if (!ag_item_ready(j, x, lane)) return false;
  if ((j.host_mask >> x.r) & 1ull) {
    ag_item_copy_plain(j, x, lane);
    return false;
  }
  bool dead = false;
  if (lane == 0) {
    // each source line is read once: let it leave L2 before the gathered rows and B
    const uint64_t once = l2_policy_evict_first();
    const int nch = int((bytes + COPY_CHUNK - 1) / COPY_CHUNK);
    int issued = 0, stored = 0;
    while (stored < nch) {
      while (issued < nch && issued - stored < NBUF) {
        const uint32_t q = seq + uint32_t(issued);
        const int buf = int(q % NBUF);
        // the store that last read `buf` (chunk q - NBUF) must have finished reading it
        bulk_wait_read_dyn(stored - issued + NBUF - 1);
        const uint32_t off = uint32_t(issued) * COPY_CHUNK;
        const uint32_t sz = min(COPY_CHUNK, bytes - off);
        mbar_arrive_expect_tx(&bars[buf], sz);
        bulk_g2s_hint(stage + buf * COPY_CHUNK, src + off, sz, &bars[buf], once);
        ++issued;
      }
      const uint32_t q = seq + uint32_t(stored);
      const int buf = int(q % NBUF);
      if (!mbar_wait(&bars[buf], (q / NBUF) & 1u, abort, j.status, j.pipe_timeout_ns, 5)) {
        dead = true;
        break;
      }
      const uint32_t off = uint32_t(stored) * COPY_CHUNK;
      bulk_s2g(dst + off, stage + buf * COPY_CHUNK, min(COPY_CHUNK, bytes - off));
      bulk_commit();
      ++stored;
    }
    seq += uint32_t(nch);
    // produce_tile_notify: writes complete -> order with the generic proxy -> release
    bulk_wait<0>();
    if (!dead) {
      fence_proxy_async_global();
      st_release(j.flags + flag_id, j.epoch);
    }
  }
  return __shfl_sync(0xffffffffu, dead, 0);
}

// Items first, first + stride, ... in copy order: shards self+1, ..., self+R-1,
// then self; chunks ascending.  Called by all 32 lanes of one warp.
// Held chunks (see AgCopyJob) come after all the others.
template <int NBUF = COPY_NBUF>
__device__ __forceinline__ void ag_copy_items(const AgCopyJob& j, uint8_t* stage, uint64_t* bars,
                                              volatile uint32_t* abort, int first, int stride) {
  const uint64_t t0 = now_ns();
  uint32_t seq = 0;
  bool dead = false, any_held = false;
  for (int it = first; it < j.num_items && !dead; it += stride) {
    if (ag_item_held(j, it)) {
      any_held = true;
      continue;
    }
    dead = ag_copy_one<NBUF>(j, it, stage, bars, abort, seq);
  }
  if (any_held && !dead) {
    if (lane_id() == 0) hold_until(t0, j.hold_ns, abort, j.status);
    __syncwarp();
    for (int it = first; it < j.num_items && !dead; it += stride)
      if (ag_item_held(j, it)) dead = ag_copy_one<NBUF>(j, it, stage, bars, abort, seq);
  }
  if (lane_id() == 0) bulk_wait<0>();
  __syncwarp();
}

}  // namespace tl
