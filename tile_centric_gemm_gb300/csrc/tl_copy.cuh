// tl_copy.cuh -- the AllGather producer shared by the fused AllGather-GEMM
// kernel and the stand-alone AllGather: one warp lane moves row chunks of the
// shards into the gathered buffer through a ring of shared-memory buffers with
// bulk TMA copies, and releases one flag per chunk once its writes are
// complete (produce_tile_notify).  Pull mode first acquires the source's
// readiness flag of the same chunk.
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
};

// Items first, first + stride, ... in copy order: shards self+1, ..., self+R-1,
// then self; chunks ascending.  `stage` holds COPY_NBUF buffers of COPY_CHUNK
// bytes; `bars` COPY_NBUF mbarriers initialised with count 1.
__device__ __forceinline__ void ag_copy_items(const AgCopyJob& j, uint8_t* stage, uint64_t* bars,
                                              volatile uint32_t* abort, int first, int stride) {
  uint32_t seq = 0;  // chunks loaded so far: buffer seq % NBUF, parity (seq / NBUF) & 1
  bool dead = false;
  for (int it = first; it < j.num_items && !dead; it += stride) {
    const int jj = it / j.bpr, b = it % j.bpr;
    const int r = (j.self + 1 + jj) % j.R;
    const int lo = b * j.rpb;
    const int rows = min(j.rpb, j.M_shard - lo);
    const uint8_t* src = j.shard[r] + size_t(lo) * j.K * 2;
    uint8_t* dst = j.gathered + (size_t(r) * j.M_shard + lo) * size_t(j.K) * 2;
    const uint32_t bytes = uint32_t(rows) * uint32_t(j.K) * 2u;
    const int flag_id = r * j.bpr + b;
    // pull mode: the source publishes readiness first (first barrier of the pull protocol);
    // a chunk whose source never became ready is neither copied nor announced
    if (j.ready && !wait_flag(j.ready + flag_id, j.epoch, j.status, j.timeout_ns, uint32_t(flag_id), TL_ERR_TIMEOUT))
      continue;
    const int nch = int((bytes + COPY_CHUNK - 1) / COPY_CHUNK);
    int issued = 0, stored = 0;
    while (stored < nch) {
      while (issued < nch && issued - stored < COPY_NBUF) {
        const uint32_t q = seq + uint32_t(issued);
        const int buf = int(q % COPY_NBUF);
        // the store that last read `buf` (chunk q - NBUF) must have finished reading it
        bulk_wait_read_dyn(stored - issued + COPY_NBUF - 1);
        const uint32_t off = uint32_t(issued) * COPY_CHUNK;
        const uint32_t sz = min(COPY_CHUNK, bytes - off);
        mbar_arrive_expect_tx(&bars[buf], sz);
        bulk_g2s(stage + buf * COPY_CHUNK, src + off, sz, &bars[buf]);
        ++issued;
      }
      const uint32_t q = seq + uint32_t(stored);
      const int buf = int(q % COPY_NBUF);
      if (!mbar_wait(&bars[buf], (q / COPY_NBUF) & 1u, abort, j.status, j.pipe_timeout_ns, 5)) {
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
    if (dead) break;
    fence_proxy_async_global();
    st_release(j.flags + flag_id, j.epoch);
  }
  bulk_wait<0>();
}

}  // namespace tl
