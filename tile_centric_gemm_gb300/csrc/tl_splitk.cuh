// tl_splitk.cuh -- split-K for CTA-pair GEMMs whose 256 x 256 tiles leave pairs
// idle.
//
// A tile's k-blocks are cut into S equal ranges that run as separate work units
// (unit = tile * S + split) on separate pairs, all in one wave of a launch
// whose grid the device holds at once (tiles * S <= pairs, one unit per pair).
// Each CTA of a unit writes its fp32 128 x 256 half of the partial tile into
// its own workspace slot and counts itself in on that half-tile's counter; once
// all S have counted in (a bounded wait), split s sums the S partials of its
// share of the columns, in split order 0, 1, ..., S-1 (its own from TMEM, the
// others through L2), and writes that share of C.  The fixed order makes the
// result independent of the schedule; spreading the sums over the S CTAs keeps
// each one's reads at (S-1)/S of a half-tile.
//
// Each half-tile has an arrival and a departure counter holding
// (tag << 8) | count; the split that departs last zeroes both, so a completed
// call (or a replayed graph of calls) leaves them ready for the next.  A count
// with another tag starts over at 1: an AllGather-GEMM tags with its epoch,
// which also makes counters left behind by an aborted call harmless; a plain
// GEMM uses one fixed tag, so after a call that reported a device error its
// counters must be zeroed before the workspace is reused.
//
// Workspace: counters [tiles][2 halves][arrive, depart] uint32 (padded to a
// multiple of 1 KB), then partial halves [tiles][S][2] of 128 x 256 fp32 each,
// stored per epilogue warp (32 rows) as [32-column chunk][group of 4 columns]
// [row][4]: one warp-wide 16-byte access covers 512 contiguous bytes.
#pragma once

#include "tl_epilogue.cuh"
#include "tl_pair.cuh"

namespace tl {
namespace splitk {

constexpr int MAX_SPLITS = 16;
constexpr int MIN_KB_PER_SPLIT = 8;   // 512 of K per split keeps the six-stage ring full
constexpr uint32_t kBarrier = 3;      // named barrier of the four epilogue warps
constexpr size_t HALF_FLOATS = size_t(pair::HM) * pair::BN;
constexpr int kMaxCasTries = 4096;    // each failed CAS means another split got in; at most S-1 do
constexpr int kBatch = 2;             // partial slots loaded together before they are added in order

// Splits for `tiles` tiles of KB k-blocks on `pairs` CTA pairs: the largest S
// that divides KB, leaves every split at least MIN_KB_PER_SPLIT k-blocks and
// keeps all tiles * S units in one wave; 1 (no split) when the tiles already
// fill the pairs or no S >= 2 qualifies.
inline int choose(long long tiles, int KB, int pairs) {
  if (tiles < 1 || tiles >= pairs) return 1;
  for (int S = MAX_SPLITS; S >= 2; --S)
    if (KB % S == 0 && KB / S >= MIN_KB_PER_SPLIT && tiles * S <= pairs) return S;
  return 1;
}
inline size_t counter_bytes(long long tiles) { return (size_t(tiles) * 4 * 4 + 1023) / 1024 * 1024; }
inline size_t workspace_bytes(long long tiles, int S) {
  return S <= 1 ? 0 : counter_bytes(tiles) + size_t(tiles) * S * 2 * HALF_FLOATS * 4;
}

struct Work {
  uint32_t* counters;  // [tiles][2 halves][arrive, depart]
  float* partials;     // [tiles][S][2][HALF_FLOATS]
  uint64_t timeout_ns; // bound of the wait for the other splits
  uint32_t tag;        // nonzero multiple of 256
  int32_t S;
};

// Count one on `ctr` under `tag`; returns the count reached, or 0 if the CAS
// never got in (recorded as an internal error).
__device__ __forceinline__ uint32_t count_in(uint32_t* ctr, uint32_t tag, uint32_t* status, uint32_t where) {
  uint32_t cur = *reinterpret_cast<volatile uint32_t*>(ctr);
  for (int i = 0; i < kMaxCasTries; ++i) {
    const uint32_t next = ((cur & 0xFFFFFF00u) == tag) ? cur + 1u : (tag | 1u);
    const uint32_t prev = atomicCAS(ctr, cur, next);
    if (prev == cur) return next & 0xFFu;
    cur = prev;
  }
  record_error(status, TL_ERR_INTERNAL, where, cur, tag);
  return 0;
}

// Bounded wait until `ctr` holds tag | S (every split of the half-tile arrived).
__device__ __forceinline__ bool wait_all(const uint32_t* ctr, uint32_t want, uint32_t* status, uint64_t timeout_ns,
                                         uint32_t where) {
  uint32_t v = ld_acquire(ctr);
  if (v == want) return true;
  const uint64_t t0 = now_ns();
  uint32_t spins = 0;
  while (true) {
    v = ld_acquire(ctr);
    if (v == want) return true;
    if ((++spins & 63u) == 0u) {
      if (ld_volatile(status) != 0u) return false;
      if (now_ns() - t0 > timeout_ns) {
        record_error(status, TL_ERR_TIMEOUT, where, v, want);
        return false;
      }
    }
    __nanosleep(32);
  }
}

// The epilogue of one split unit for one epilogue warp (all four warps of the
// CTA call it): rows wq*32 .. wq*32+31 of this CTA's half, `nchunks` 32-column
// chunks of the accumulator at TMEM address `tacc` (this warp's lanes).
// `ok_flag` is a shared word; write_c(c, v) writes chunk c of the final sum
// (32 fp32 values as bits) to C.  Split s sums chunks [s*nchunks/S, (s+1)*nchunks/S).
template <class WriteC>
__device__ __forceinline__ void epilogue(const Work& w, int tile, int split, uint32_t rank, int wq, int lane,
                                         uint32_t tacc, int nchunks, volatile uint32_t* ok_flag, uint32_t* status,
                                         WriteC&& write_c) {
  const size_t stride = 2 * HALF_FLOATS / 4;  // float4s from one split's slot to the next
  // split 0's slot of this half-tile, this warp's 32 rows, this lane
  const float4* base = reinterpret_cast<const float4*>(w.partials + (size_t(tile) * w.S * 2 + rank) * HALF_FLOATS +
                                                       size_t(wq) * 32 * pair::BN) + lane;
  float4* mine = const_cast<float4*>(base) + size_t(split) * stride;
  for (int c = 0; c < nchunks; ++c) {
    uint32_t v[32];
    tmem_ld_32cols(tacc + uint32_t(c * 32), v);
    tmem_ld_wait();
#pragma unroll
    for (int g = 0; g < 8; ++g)
      __stcg(mine + (c * 8 + g) * 32, make_float4(__uint_as_float(v[g * 4]), __uint_as_float(v[g * 4 + 1]),
                                                  __uint_as_float(v[g * 4 + 2]), __uint_as_float(v[g * 4 + 3])));
  }
  __threadfence();  // this thread's partial is visible before the arrival below
  named_bar_sync(kBarrier, kNumEpiThreads);
  if (threadIdx.x == kWarpEpi0 * 32) {
    uint32_t* ctr = w.counters + (size_t(tile) * 2 + rank) * 2;  // arrive, depart
    const uint32_t where = uint32_t(tile) * 2 + rank;
    bool ok = count_in(ctr, w.tag, status, where) != 0 &&
              wait_all(ctr, w.tag | uint32_t(w.S), status, w.timeout_ns, where);
    if (ok) {
      __threadfence();  // the other splits' partials are read after their arrivals
      const uint32_t gone = count_in(ctr + 1, w.tag, status, where);
      ok = gone != 0;
      if (gone == uint32_t(w.S)) {  // every split has seen all arrivals: ready for the next call
        atomicExch(ctr, 0u);
        atomicExch(ctr + 1, 0u);
      }
    }
    *ok_flag = ok ? 1u : 0u;
  }
  named_bar_sync(kBarrier, kNumEpiThreads);
  if (!*ok_flag) return;
  const int c0 = split * nchunks / w.S, c1 = (split + 1) * nchunks / w.S;
  for (int c = c0; c < c1; ++c) {
    uint32_t own[32];
    tmem_ld_32cols(tacc + uint32_t(c * 32), own);
    tmem_ld_wait();
    float acc[32];
    for (int s0 = 0; s0 < w.S; s0 += kBatch) {
      // the batch's slots in flight together, then added in split order
      float4 x[kBatch][8];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int s = s0 + b;
        if (s < w.S && s != split) {
#pragma unroll
          for (int g = 0; g < 8; ++g) x[b][g] = __ldcg(base + size_t(s) * stride + (c * 8 + g) * 32);
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int s = s0 + b;
        if (s >= w.S) break;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          float4 f;
          if (s == split)
            f = make_float4(__uint_as_float(own[g * 4]), __uint_as_float(own[g * 4 + 1]),
                            __uint_as_float(own[g * 4 + 2]), __uint_as_float(own[g * 4 + 3]));
          else
            f = x[b][g];
          if (s == 0) {
            acc[g * 4] = f.x;
            acc[g * 4 + 1] = f.y;
            acc[g * 4 + 2] = f.z;
            acc[g * 4 + 3] = f.w;
          } else {
            acc[g * 4] += f.x;
            acc[g * 4 + 1] += f.y;
            acc[g * 4 + 2] += f.z;
            acc[g * 4 + 3] += f.w;
          }
        }
      }
    }
    uint32_t out[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) out[i] = __float_as_uint(acc[i]);
    write_c(c, out);
  }
}

}  // namespace splitk
}  // namespace tl
