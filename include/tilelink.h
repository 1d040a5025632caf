/*
 * tilelink.h -- C ABI of libtilelink: tile-centric compute/communication
 * overlap on one NVIDIA GB300 (sm_103a).
 *
 * The method follows the TileLink talk summary ("TileLink: Generating Efficient
 * Compute-Communication Overlapping Kernels using Tile-Centric Primitives",
 * MLSys 2025): producers and consumers of tiles synchronise through per-tile
 * signals (Technical Deep Dive: signal primitives consume_tile_wait,
 * produce_tile_notify, peer_tile_wait; data primitives push and pull; tile-id
 * to rank/barrier maps; swizzled tile orders), applied to AllGather-GEMM,
 * GEMM-ReduceScatter and the AllGather + GroupGEMM part of an MoE layer (Key
 * Findings; Experimental Setup & Results).
 *
 * The R communicating ranks are emulated on one GPU: every rank's data is a
 * separate allocation that the caller passes as an array of pointers, and
 * "communication" is a copy between those allocations performed by the
 * library's own copy warps.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Matrices are row-major.  bf16 = IEEE bfloat16 (uint16 storage).
 *  - Pointers named "device" must be device memory of the current device,
 *    16-byte aligned; operands the kernels load with TMA are checked and any
 *    other memory is rejected with TL_ERR_UNSUPPORTED before a launch.  Arrays
 *    of pointers (A_shards, A, B, out, X, W) are HOST arrays read during the
 *    call; the pointers in them are device pointers.
 *  - AllGather shards (tl_ag_gemm other than the self shard, tl_allgather) may
 *    also be pinned host or managed memory, the stand-in for a slower link:
 *    those are copied with plain loads by the copy warps.  Pageable host
 *    memory and other devices' memory are rejected (TL_ERR_UNSUPPORTED).
 *  - Ownership: the caller owns every buffer passed in.  The library allocates
 *    only the flag/status memory of a tl_signals object.
 *  - Ordering: every call that takes a stream is asynchronous and ordered on
 *    that stream (a cudaStream_t passed as void*, NULL = legacy default
 *    stream).  Argument errors are returned synchronously and launch nothing.
 *    Device-side errors (a bounded wait that ran out) are recorded in the
 *    signals object's status word and read with tl_query_status.
 *  - Epochs: a flag is "set for epoch E" when its value v satisfies
 *    (int32_t)(v - E) >= 0.  Each call that uses a signals object releases its
 *    flags with the caller's epoch, so flags are never reset between calls; a
 *    later call on the same object must use a larger epoch (mod 2^32).
 *  - Every wait inside a kernel is bounded by timeout_ns (0 = 1 s).  When a
 *    bound runs out the kernel records TL_ERR_TIMEOUT, stops waiting for the
 *    rest of the launch, and finishes; its outputs are then undefined.
 *  - Failure: no call aborts the process; no exception crosses the ABI.
 *    tl_last_error() returns a message for the calling thread's last error.
 *  - Calls that take an epoch are not capturable into CUDA graphs for replay:
 *    the epoch is a launch parameter.  tl_gemm and tl_reduce_scatter take none;
 *    they may be captured once a first call outside any capture has set up
 *    their kernel on the device (launch attributes are set on first use).
 */
#ifndef TILELINK_H
#define TILELINK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TL_VERSION 1
#define TL_MAX_RANKS 64
#define TL_MAX_EXPERTS 256

typedef enum {
  TL_OK = 0,
  TL_ERR_INVALID = 1,      /* bad argument (null, negative, misaligned, too small) */
  TL_ERR_CUDA = 2,         /* a CUDA runtime/driver call failed */
  TL_ERR_TIMEOUT = 3,      /* a bounded device wait ran out (see tl_query_status) */
  TL_ERR_UNSUPPORTED = 4,  /* valid but outside what the kernels handle */
  TL_ERR_INTERNAL = 5      /* a device-side consistency check failed */
} tl_status;

typedef enum { TL_MODE_PULL = 0, TL_MODE_PUSH = 1 } tl_mode;

/* Consumer row-tile order of AllGather-GEMM (talk summary, Technical Deep Dive:
 * swizzling lines the consumption order up with the arrival order). */
typedef enum {
  TL_SWIZZLE_ARRIVAL = 0, /* row tiles in the order their shards arrive: self, self+1, ... (default) */
  TL_SWIZZLE_ROWS = 1     /* row tiles in index order 0, 1, ..., whatever the arrival order
                             (the unswizzled schedule, kept for comparison) */
} tl_swizzle;

/* Opaque per-tile signal buffer: device uint32 flags plus a device status word. */
typedef struct tl_signals tl_signals;

/* Library version (TL_VERSION) and the last error message of this thread. */
int tl_version(void);
const char* tl_last_error(void);

/* ---------------------------------------------------------------- signals
 * Signal primitives (talk summary, Technical Deep Dive: produce_tile_notify,
 * consume_tile_wait).  A signals object owns num_flags device uint32 flags,
 * zero at creation, and a status word.  The object belongs to the device that
 * is current at creation.
 */
tl_status tl_signals_create(int num_flags, tl_signals** out);
tl_status tl_signals_destroy(tl_signals* s);
/* Device pointer to the flags (for tests and for the caller's own kernels). */
tl_status tl_signals_flags(const tl_signals* s, uint32_t** dev_flags, int* num_flags);
/* Zero every flag and the status word (stream-ordered). */
tl_status tl_signals_reset(tl_signals* s, void* stream);

/* produce_tile_notify: release-store `value` into flags [first, first+count)
 * after all earlier work on `stream` (one thread per flag, st.release.gpu). */
tl_status tl_tile_notify(tl_signals* s, int first, int count, uint32_t value, void* stream);

/* consume_tile_wait: block `stream` until every flag in [first, first+count)
 * is set for epoch `value` (acquire loads), or until timeout_ns elapses; on
 * timeout the status word records TL_ERR_TIMEOUT with the flag index.  The
 * wait must be satisfiable by work already ordered before it: a flag that only
 * a later or concurrent launch would set is a timeout, never a hang. */
tl_status tl_tile_wait(tl_signals* s, int first, int count, uint32_t value,
                       uint64_t timeout_ns, void* stream);

/* Synchronise `stream`, return the first device error recorded since the last
 * query (TL_OK if none) and clear it.  *where receives the flag index or tile
 * that failed (-1 if none).  Either out pointer may be NULL. */
tl_status tl_query_status(tl_signals* s, void* stream, int* code, int* where);

/* ---------------------------------------------------------------- test facility: forced arrival order
 * Not part of the method: a way for tests to make chunks arrive in an order
 * other than the one the consumers take them in, so that a missing or wrong
 * wait shows up as a wrong result instead of passing by luck.  On the calling
 * thread, every later tl_ag_gemm, tl_allgather and tl_moe_ag_gemm call has its
 * copy warps move the chunks whose flag ids lie in [first_flag, first_flag +
 * count) after all their other chunks, and not before hold_ns have passed since
 * the copy warp started (a bounded spin on the global timer).  count 0 turns it
 * off.  A call whose timeout_ns is not above twice hold_ns is rejected
 * (TL_ERR_INVALID), so that the consumers' bounded waits outlast the hold.
 * hold_ns at most 100 ms.  The results of the calls do not change.
 */
tl_status tl_test_hold_chunks(int first_flag, int count, uint64_t hold_ns);

/* ---------------------------------------------------------------- GEMM
 * C = A . B, bf16 in, fp32 accumulate, bf16 (and optionally fp32) out, with no
 * communication and no waits: the compute half of AllGather-GEMM alone, used to
 * measure the fused kernels' overlap and as the compute step of a decomposed
 * (per-shard, multi-stream) baseline (talk summary, Background: decomposition-
 * based overlap splits operators into sub-operators on several streams).
 * tcgen05 MMAs of pairs of CTAs (cta_group::2), 256 x 256 tiles.
 */
typedef struct tl_gemm_args {
  int32_t M;                   /* rows of A and C, >= 1 */
  int32_t N;                   /* columns of B and C, multiple of 8 */
  int32_t K;                   /* contraction, multiple of 8 */
  int32_t reserved0;
  const void* A;               /* device bf16 [M, K] */
  const void* B;               /* device bf16 [K, N] */
  void* C;                     /* device bf16 [M, N], written; may be NULL when C_f32 is given */
  float* C_f32;                /* optional device float [M, N], written; NULL = none */
  tl_signals* signals;         /* receives device-side errors in its status word (any size >= 1) */
  uint64_t timeout_ns;         /* bound of the pipeline waits is 2 * timeout + 1 s; 0 = 1 s */
  void* workspace;             /* optional device scratch for split-K (see tl_ag_gemm_workspace_size),
                                  16-byte aligned, zeroed before its first use; NULL = no split */
  size_t workspace_bytes;      /* >= tl_gemm_workspace_size(M, N, K, 0) when workspace is given */
} tl_gemm_args;

size_t tl_gemm_workspace_size(int M, int N, int K, int sm_count);
tl_status tl_gemm(const tl_gemm_args* args, void* stream);

/* ---------------------------------------------------------------- AllGather-GEMM
 * C = G . B with G = [A_0; A_1; ...; A_{R-1}] (talk summary, Key Findings and
 * Experimental Setup & Results: AllGather-GEMM).  One launch holds both sides:
 *  - producer: copy warps move each shard, rows_per_barrier rows at a time, into
 *    `gathered` with bulk TMA copies and release one flag per row chunk
 *    (produce_tile_notify).  Pull mode first waits on the source's readiness
 *    flag of the same id (two barriers per tile); push mode has one barrier.
 *  - consumer: tcgen05 GEMM tiles of 256 x 256 on pairs of CTAs
 *    (cta_group::2); each CTA acquires every flag guarding its 128 rows
 *    (consume_tile_wait; flag id = rank * barriers_per_rank +
 *    row_in_shard / rows_per_barrier, an affine map of the row) before loading
 *    them, and tiles run in arrival order: shards self, self+1, ..., self+R-1
 *    (consume_tile_swizzle; TL_SWIZZLE_ROWS runs them in index order instead).  Row halves wholly inside the self shard read
 *    A_self in place and never wait, so the self shard must be device memory.
 *    Copies run in the order self+1, ..., self+R-1, self.
 * Output is independent of self_rank, mode and rows_per_barrier.
 */
typedef struct tl_ag_gemm_args {
  int32_t R;                   /* ranks, 1..TL_MAX_RANKS */
  int32_t self_rank;           /* 0..R-1 */
  int32_t M_shard;             /* rows per shard, >= 1 */
  int32_t K;                   /* contraction, >= 8, multiple of 8 */
  int32_t N;                   /* output columns, >= 8, multiple of 8 */
  int32_t mode;                /* tl_mode */
  int32_t rows_per_barrier;    /* rows per producer tile / flag; 0 = about 128 KB of A */
  int32_t swizzle;             /* tl_swizzle: consumer row-tile order; 0 = arrival order */
  const void* const* A_shards; /* host array of R device pointers, bf16 [M_shard, K] */
  const void* B;               /* device bf16 [K, N] */
  void* gathered;              /* device bf16 [R*M_shard, K], written (the gathered A) */
  void* C;                     /* device bf16 [R*M_shard, N], written */
  float* C_f32;                /* optional device float [R*M_shard, N], written; NULL = none */
  tl_signals* signals;         /* arrival flags, >= tl_ag_gemm_num_flags(...) */
  const tl_signals* src_ready; /* pull mode: source readiness flags (same ids); else NULL */
  uint32_t epoch;              /* nonzero */
  uint32_t reserved1;
  uint64_t timeout_ns;         /* 0 = 1 s */
  int32_t* trace;              /* optional device int32 [ceil(M/256) * ceil(N/256)]:
                                  trace[slot] = m_tile * n_tiles + n_tile of the 256 x 256
                                  tile the consumer ran at schedule slot `slot` */
  void* workspace;             /* optional device scratch for split-K, 16-byte aligned; NULL = no split */
  size_t workspace_bytes;      /* >= tl_ag_gemm_workspace_size(...) when workspace is given */
} tl_ag_gemm_args;

/* Split-K (both AG-GEMM and GEMM): when the 256 x 256 tiles are fewer than the
 * CTA pairs (SMs / 2) and a workspace is given, every tile's k-blocks are cut
 * into S equal ranges (the largest S <= 16 that divides ceil(K/64), keeps at
 * least 8 k-blocks per range and keeps tiles * S <= pairs), run on S pairs at
 * once; each writes an fp32 partial tile to the workspace, and once all S have
 * (a bounded wait, TL_ERR_TIMEOUT) each adds the S partials of 1/S of the
 * tile's columns in range order 0..S-1 and writes them to C.  Results are
 * deterministic (fixed order) and differ from the unsplit product only by fp32
 * rounding.  The workspace's counters are left zeroed by every call that
 * completes; an AG-GEMM tags them with its epoch, a GEMM with a fixed tag, so
 * after a tl_gemm call that reported a device error the first 2 KB of its
 * workspace must be zeroed before it is used again.  Calls sharing a workspace
 * must not run concurrently.  The S units of a tile wait for one another, so a
 * split call needs its whole grid resident at once: with other kernels holding
 * SMs at the same time it can fail with TL_ERR_TIMEOUT (the AG-GEMM's flag
 * waits already need the same).
 * Workspace bytes for a shape: 0 when no split would be used.  sm_count 0 =
 * the current device's SM count (the launch uses the device's own count). */
size_t tl_ag_gemm_workspace_size(int R, int M_shard, int K, int N, int sm_count);
/* Flags an AG-GEMM call needs: R * ceil(M_shard / rows_per_barrier) (after
 * replacing 0 by the default); also returns the effective rows_per_barrier. */
int tl_ag_gemm_num_flags(int R, int M_shard, int K, int rows_per_barrier, int* effective_rpb);
/* Host copy of the consumer's row-tile order (the swizzle): writes the
 * ceil(R*M_shard/256) m-tile indices (256-row tiles) in the order the consumer
 * runs them. */
tl_status tl_ag_gemm_tile_order(int R, int self_rank, int M_shard, int32_t* m_order, int capacity);
tl_status tl_ag_gemm(const tl_ag_gemm_args* args, void* stream);

/* ---------------------------------------------------------------- GEMM-ReduceScatter
 * out[d] = rows [d*M/R, (d+1)*M/R) of S = (((P_0 + P_1) + P_2) + ...), P_r =
 * A_r . B_r (talk summary, Key Findings and Technical Deep Dive: a persistent
 * GEMM that notifies each finished partial tile, and a reduce stage that waits
 * on its own and its peers' tiles).  One launch on pairs of CTAs
 * (cta_group::2, 256 x 256 tiles; CTA h of a pair owns rows h*128..h*128+127
 * of every tile); output tiles tau run in destination order, n tile by n tile
 * with the m tiles innermost.  Two schedules, with the same result bits:
 *  - chain (tl_gemm_rs): the partials are summed on the way, like the partial
 *    sums of a ring reduce passing from rank to rank.  Destinations are taken
 *    in groups of two; within a group, pass j produces every tile's partial of
 *    the j-th rank of the summation order (rank j, or rank d+1+j mod R with
 *    TL_RS_RING_ORDER); the pushers of pass j wait for pass j-1's arrival flag
 *    of the tile, add their fp32 partial (rounded to bf16 first with
 *    TL_RS_BF16_PARTIALS) to the tile's running sum in `workspace` (one fp32
 *    tile per output tile), and release the arrival and reduced flags of
 *    (tile, j); pass R-1 writes bf16 of the sum into out[d].  A group's sums
 *    stay in L2 from pass to pass and each rank's operands are read from
 *    memory about once per group.
 *  - push and reduce (tl_gemm_rs_noalloc): every partial half-tile is pushed
 *    into a receive slot of `workspace` (a ring of three waves of slots,
 *    reused as the launch proceeds) and its arrival flag released; the R
 *    partials of one output tile are produced back to back, rank
 *    (d + 1 + tau + j) mod R at position j of output tile tau.  Reducer warps
 *    of the CTAs that computed them each reduce one row slice of their half
 *    after acquiring its R arrival flags, adding the partials in rank order
 *    (or ring order) in fp32, write bf16 rows into out[d], and release a
 *    "reduced" flag; a pusher reuses a ring slot only after the reduced flags
 *    of the tile that used it before.
 */
/* GEMM-RS options (bits of tl_gemm_rs_args.options), closer to a real
 * ReduceScatter's traffic; the default (0) is fp32 partials summed in rank order. */
#define TL_RS_BF16_PARTIALS 1u /* round each partial to bf16 (RNE) before it is pushed */
#define TL_RS_RING_ORDER 2u    /* destination d sums ranks d+1, d+2, ..., d (mod R) */

typedef struct tl_gemm_rs_args {
  int32_t R;                   /* ranks, 1..32 (TL_ERR_UNSUPPORTED above) */
  int32_t M;                   /* rows of every A_r; multiple of R */
  int32_t K_r;                 /* per-rank contraction, >= 8, multiple of 8 */
  int32_t N;                   /* >= 8, multiple of 8 */
  const void* const* A;        /* host array of R device pointers, bf16 [M, K_r] */
  const void* const* B;        /* host array of R device pointers, bf16 [K_r, N] */
  void* const* out;            /* host array of R device pointers, bf16 [M/R, N] */
  void* workspace;             /* device, >= tl_gemm_rs_workspace_size(R, M, N) bytes */
  size_t workspace_bytes;
  tl_signals* signals;         /* >= tl_gemm_rs_num_flags(R, M, N) flags */
  uint32_t epoch;              /* nonzero */
  uint32_t options;            /* TL_RS_* bits; 0 = fp32 partials, rank order */
  uint64_t timeout_ns;         /* 0 = 1 s */
  int32_t* trace;              /* optional device int32 [tl_gemm_rs_num_flags(R, M, N) / 4]:
                                  trace[item] = ((d * m_tiles + m) * n_tiles + n) * R + r,
                                  the output tile and rank of each produced partial in
                                  production order (the schedule's), m_tiles =
                                  ceil(M/R/256), n_tiles = ceil(N/256) */
} tl_gemm_rs_args;

/* Workspace bytes for the current device: the larger of the chain schedule's
 * running sums (tiles fp32 tiles, tiles = R * ceil(M/R/256) * ceil(N/256)) and
 * the push schedule's ring, min(items, 3 * pairs) items of two half-slots of
 * R * ceil(128/R) * 256 floats, pairs = half the SM count.  Both are laid out
 * in half-tiles [slice][column/4][row in slice][4], one contiguous block per
 * row slice. */
size_t tl_gemm_rs_workspace_size(int R, int M, int N);
/* Flags a GEMM-RS call needs: 4 * R * tiles (arrival and reduced flags for
 * both halves), tiles = R * ceil(M/R/256) * ceil(N/256). */
int tl_gemm_rs_num_flags(int R, int M, int N);
tl_status tl_gemm_rs(const tl_gemm_rs_args* args, void* stream);

/* ---------------------------------------------------------------- GEMM-RS without allocation
 * The talk summary has no counterpart of this entry point.  It exists for
 * callers that cannot allocate device memory -- a runtime whose allocator owns
 * the device and forbids cudaMalloc on its hot path, code that runs before any
 * allocator exists, or an embedding that may only pass the buffers it already
 * holds.  Same operation and arguments as tl_gemm_rs, always with the push and
 * reduce schedule (the same result bits as the chain schedule), except:
 *  - args->workspace, args->workspace_bytes and args->signals must be NULL/0.
 *    The flags, a status word and the fp32 receive slots live in one static
 *    device array of TL_GEMM_RS_NOALLOC_MAX_BYTES (64 MiB), which every GPU
 *    that loads the library holds until the process exits.
 *  - A problem that needs more scratch than that fails with
 *    TL_ERR_UNSUPPORTED and launches nothing.  It needs roundup256(256 + 4*F)
 *    bytes of flags plus the ring of receive slots described under
 *    tl_gemm_rs_workspace_size, F = tl_gemm_rs_num_flags(R, M, N).
 *  - dev_status: optional caller-owned device pointer to 4 uint32 words
 *    (16-byte aligned) where the kernel records its first device-side error
 *    (code, where, value seen, value expected); the caller zeroes it.  With
 *    NULL, device-side timeouts go unreported.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process: after a cudaDeviceReset of that device the module is loaded
 *    anew and the kept address is stale, so the entry point must not be
 *    called on a device that was reset after its first call.
 *  - Every call shares the array and it keeps the last call's contents: each
 *    call clears the flags (a stream-ordered memset) before its launch.  Calls
 *    that overlap on the GPU (different streams without ordering) race.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define TL_GEMM_RS_NOALLOC_MAX_BYTES (64ull << 20)
tl_status tl_gemm_rs_noalloc(const tl_gemm_rs_args* args, uint32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- communication halves alone
 * tl_allgather: the AllGather-GEMM producer without the GEMM -- the same copy
 * routine moves every shard into `gathered`, rows_per_barrier rows at a time,
 * and releases one flag per chunk (flag ids and modes as for tl_ag_gemm, so a
 * caller's own consumer can tl_tile_wait on them).  One warp on every SM.
 * tl_reduce_scatter: the GEMM-ReduceScatter reduce stage without the GEMM --
 * out[d] = rows [d*M/R, (d+1)*M/R) of (((P_0 + P_1) + P_2) + ...) with the fp32
 * partials P_r [M, N] given, summed in rank order in fp32, one bf16 rounding.
 * Both serve as the separate communication step of a decomposed schedule
 * (talk summary, Background) and to measure the fused kernels' overlap.
 */
typedef struct tl_allgather_args {
  int32_t R, self_rank, M_shard, K;  /* as tl_ag_gemm_args */
  int32_t mode, rows_per_barrier;
  const void* const* A_shards;       /* host array of R device pointers, bf16 [M_shard, K] */
  void* gathered;                    /* device bf16 [R*M_shard, K], written */
  tl_signals* signals;               /* >= tl_ag_gemm_num_flags(...) flags, released per chunk */
  const tl_signals* src_ready;       /* pull mode readiness flags, else NULL */
  uint32_t epoch;                    /* nonzero */
  uint32_t reserved0;
  uint64_t timeout_ns;               /* 0 = 1 s */
} tl_allgather_args;

typedef struct tl_reduce_scatter_args {
  int32_t R, M, N, reserved0;        /* M multiple of R, N multiple of 8 */
  const float* const* partials;      /* host array of R device pointers, float [M, N] */
  void* const* out;                  /* host array of R device pointers, bf16 [M/R, N], written */
} tl_reduce_scatter_args;

tl_status tl_allgather(const tl_allgather_args* args, void* stream);
tl_status tl_reduce_scatter(const tl_reduce_scatter_args* args, void* stream);

/* ---------------------------------------------------------------- AllGather through a slow link, low latency
 * The talk summary (Experimental Setup & Results, further results) reports an
 * AllGather over PCIe with a low-latency protocol about three times faster
 * than NCCL's; it gives no format.  This call reads it as the flag-in-data
 * protocol: every 8-byte link word holds 4 bytes of data and 4 bytes of the
 * call's epoch and is written and read as one 64-bit access, so a receiver that
 * sees the epoch also sees the data -- the sender needs no fence between data
 * and flag and the receiver polls no separate flag -- at twice the bytes on
 * the link.  One launch emulates both sides of a push AllGather on one GPU:
 *  - send: the shard of every rank r != self_rank with bit r of send_mask is
 *    written into rank r's region of `link` (TL_LL_FLAG_IN_DATA: packed words;
 *    TL_LL_SEPARATE_FLAG: the raw data, a system-scope fence, then a release
 *    of the chunk's flag in the link buffer -- the protocol it is compared with);
 *  - receive: rank self_rank's receiver polls each peer chunk in the link
 *    (bounded by timeout_ns; TL_ERR_TIMEOUT in the status word with the flag
 *    id) and writes it into rows r*M_shard ... of `gathered`, then releases the
 *    chunk's flag in `signals` (the flag ids of tl_allgather: r * chunks + c);
 *  - the self shard is copied into `gathered` directly.
 * Ranks without their send_mask bit are not sent by this launch: their link
 * regions must be filled, with the same epoch and layout, by another agent
 * (the host, or an earlier launch).  Link layout: TL_LL_FLAG_IN_DATA -- data
 * word w of the gathered matrix (4 bytes, row-major [R*M_shard, K] bf16) at
 * link byte 8*w as {data (low 32 bits), epoch (high 32 bits)};
 * TL_LL_SEPARATE_FLAG -- the gathered matrix's bytes at the same offsets, then
 * chunk flag f (uint32) at byte R*M_shard*K*2 + 128*f.  Words of an earlier
 * epoch are never mistaken for this call's; the caller zero-fills the link
 * buffer before its first use (its last epoch is then 0), since leftover bytes
 * could read as a later epoch.  All CTAs of the launch must be
 * co-resident (receivers wait for senders of the same launch).
 */
typedef enum { TL_LL_FLAG_IN_DATA = 0, TL_LL_SEPARATE_FLAG = 1 } tl_ll_protocol;

typedef struct tl_allgather_ll_args {
  int32_t R, self_rank, M_shard, K;  /* as tl_allgather_args; K multiple of 8 */
  int32_t protocol;                  /* tl_ll_protocol */
  int32_t rows_per_barrier;          /* rows per chunk / flag; 0 = about 8 KB of a shard */
  const void* const* A_shards;       /* host array of R pointers (device or pinned host), bf16 [M_shard, K] */
  void* link;                        /* pinned host (the slow link) or device memory, 16-byte aligned */
  size_t link_bytes;                 /* >= tl_allgather_ll_link_bytes(R, M_shard, K, rows_per_barrier) */
  void* gathered;                    /* device bf16 [R*M_shard, K], written */
  tl_signals* signals;               /* >= R * chunks flags, released per chunk */
  uint64_t send_mask;                /* bit r: this launch sends rank r's shard (self_rank's bit is ignored) */
  uint32_t epoch;                    /* nonzero, larger than the link buffer's last epoch */
  uint32_t reserved0;
  uint64_t timeout_ns;               /* 0 = 1 s */
} tl_allgather_ll_args;

/* Link bytes for a shape (the larger of the two protocols' layouts). */
size_t tl_allgather_ll_link_bytes(int R, int M_shard, int K, int rows_per_barrier);
tl_status tl_allgather_ll(const tl_allgather_ll_args* args, void* stream);

/* ---------------------------------------------------------------- AllGather + grouped MoE GEMM
 * The AllGather + GroupGEMM part of an MoE layer (talk summary, Key Findings
 * and Experimental Setup & Results: MoE layers; Technical Deep Dive: lookup
 * tables built from the routing carry the tile -> rank/barrier map of a
 * dynamic workload).  T = R*T_r tokens, P = T*topk routed rows.
 *   perm[i]            sorted row i -> token*topk + slot, rows sorted by
 *                      (expert, global token id, slot); global id = r*T_r + local
 *   expert_offsets[e]  first sorted row of expert e; expert_offsets[E] = P
 *   sorted_tokens[i]   = token perm[i]/topk  (the gathered tokens, expert order)
 *   Y[i, :]            = sorted_tokens[i] . W_{expert of row i}   (fp32 accumulate, bf16)
 * Two stream-ordered launches: a routing kernel on a cluster of 8 CTAs
 * (histogram, scan, stable counting sort, tile table, tile order) and one
 * persistent kernel launched with programmatic dependent launch (its launch is
 * set up while the routing runs; it waits for the routing's tables), in
 * which copy warps move token rows into `sorted_tokens` while tcgen05 GEMM
 * tiles of 256 rows of one expert wait on the flags their lookup-table entry
 * names and multiply their sorted rows by their expert's weight.  The two data
 * modes of the talk summary (Technical Deep Dive: push sends, pull fetches
 * with finer control of arrival order) move the same rows:
 *  - push: source shards, in the order self, self+1, ..., scatter each token
 *    to its topk sorted rows; one flag per chunk of rows_per_barrier tokens of
 *    a shard (barrier id of token t: (t / T_r) * chunks + (t % T_r) /
 *    rows_per_barrier, chunks = ceil(T_r / rows_per_barrier)); a tile waits on
 *    every barrier from its tokens' lowest to highest and tiles run by the
 *    latest arrival position among those, barrier (r, c) arriving at
 *    ((r - self) mod R) * chunks + c;
 *  - pull: the consumer side gathers the sorted rows in order, one flag per
 *    chunk of rows_per_barrier sorted rows; a tile waits on its own chunks and
 *    tiles run in sorted order.
 * No gate weighting, no combine.
 * Workspace layout (int32 words; read-only for the caller, documented for
 * tests), max_tiles = ceil(P/256) + E, tiles of 256 sorted rows computed by
 * pairs of CTAs (cta_group::2):
 *   [0]                         number of tiles
 *   [16 + 6*t .. 16 + 6*t + 5]  tile t: expert, first sorted row, rows,
 *                               lowest barrier, highest barrier, source-rank mask
 *   [16 + 6*max_tiles + i]      i-th tile in consumer order (the swizzle above)
 *   [16 + 7*max_tiles + q]      sorted row of pair q (the inverse of perm)
 * Limits: R <= 32, E <= 64, H and N
 * multiples of 8.  A topk id outside [0, E) records TL_ERR_INVALID in the
 * status word (the pair is clamped into range).
 */
typedef struct tl_moe_args {
  int32_t R;                    /* ranks, 1..32 */
  int32_t self_rank;            /* 0..R-1 */
  int32_t T_r;                  /* tokens per shard */
  int32_t H;                    /* hidden size (contraction), multiple of 8 */
  int32_t N;                    /* expert output columns, multiple of 8 */
  int32_t E;                    /* experts, 1..64 */
  int32_t topk;                 /* routed experts per token, 1..E */
  int32_t rows_per_barrier;     /* rows per producer chunk / flag: push = tokens of a shard
                                   (0 = about 128 KB), pull = sorted rows (0 = about 64 KB) */
  const void* const* X;         /* host array of R device pointers, bf16 [T_r, H] */
  const int32_t* topk_ids;      /* device int32 [R*T_r, topk] */
  const void* const* W;         /* host array of E device pointers, bf16 [H, N] */
  void* sorted_tokens;          /* device bf16 [P, H], written */
  void* Y;                      /* device bf16 [P, N], written */
  int32_t* perm;                /* device int32 [P], written */
  int32_t* expert_offsets;      /* device int32 [E+1], written */
  void* workspace;              /* device, >= tl_moe_workspace_size(...) bytes, 16-byte aligned */
  size_t workspace_bytes;
  tl_signals* signals;          /* >= tl_moe_num_flags(...) flags */
  uint32_t epoch;               /* nonzero */
  int32_t mode;                 /* tl_mode: TL_MODE_PULL (default, 0) or TL_MODE_PUSH */
  uint64_t timeout_ns;          /* 0 = 1 s */
  int32_t* trace;               /* optional device int32 [max_tiles * ceil(N/256)]:
                                   tile * n_tiles + n of the work run at each schedule slot */
} tl_moe_args;

size_t tl_moe_workspace_size(int R, int T_r, int E, int topk);
/* Flags an MoE call needs in `mode`: push R * ceil(T_r / rpb), pull ceil(P / rpb). */
int tl_moe_num_flags(int mode, int R, int T_r, int H, int topk, int rows_per_barrier, int* effective_rpb);
tl_status tl_moe_ag_gemm(const tl_moe_args* args, void* stream);

/* ---------------------------------------------------------------- MoE down-projection side
 * The rest of the MoE layer after the up-projection (talk summary, Key Findings
 * and Experimental Setup & Results: GroupGEMM, ReduceScatter, TopK-reduce and a
 * scatter back to the token order).  Every expert's weights are split over the R
 * ranks along the intermediate dimension: rank r holds H_r [P, I_r], the
 * intermediate activations of the P = R*T_r*topk routed rows in expert-sorted
 * order, and W2_r [E*I_r, Hd] with expert e's slice at rows e*I_r.  With i a
 * sorted row of expert e and pos(t, s) the sorted row of pair t*topk + s:
 *   Y[i]      = sum over ranks r = 0..R-1, in order, of H_r[i] . W2_r[e slice]   (fp32)
 *   out[d][u] = bf16( sum over slots s = 0..topk-1, in order, of
 *                     gates[t, s] * Y[pos(t, s)] ),   t = d*T_r + u          (fp32)
 * Two stream-ordered launches: a grouped GEMM-ReduceScatter on pairs of CTAs
 * (items = (expert tile, 256-column tile, rank); each tile's partials are added
 * into its fp32 running sum rank after rank, rank r's pass waiting on rank
 * r-1's arrival flag, and rank R-1's pass writes the sum into Y: the chain
 * schedule of tl_gemm_rs, output tiles in groups of 96), then the TopK-reduce
 * that combines and scatters.  The routing
 * (sorted rows, tile table, inverse permutation) is the workspace a
 * tl_moe_ag_gemm call on the same topk_ids, R, T_r, E and topk left behind.
 * Limits: R <= 32, E <= 64, I_r and Hd multiples of 8.
 */
typedef struct tl_moe_down_args {
  int32_t R;                   /* ranks, 1..32 */
  int32_t T_r;                 /* tokens per rank */
  int32_t topk;                /* routed experts per token */
  int32_t E;                   /* experts, 1..64 */
  int32_t I_r;                 /* intermediate columns per rank (contraction), multiple of 8 */
  int32_t Hd;                  /* output hidden size, multiple of 8 */
  const void* const* H;        /* host array of R device pointers, bf16 [P, I_r], expert-sorted rows */
  const void* const* W2;       /* host array of R device pointers, bf16 [E*I_r, Hd] */
  const float* gates;          /* device fp32 [R*T_r, topk] */
  const int32_t* routing;      /* device: the workspace of the matching tl_moe_ag_gemm call */
  void* const* out;            /* host array of R device pointers, bf16 [T_r, Hd], written */
  void* workspace;             /* device, >= tl_moe_down_workspace_size(...) bytes, 16-byte aligned */
  size_t workspace_bytes;
  tl_signals* signals;         /* >= tl_moe_down_num_flags(...) flags */
  uint32_t epoch;              /* nonzero */
  uint32_t options;            /* 0, or TL_RS_BF16_PARTIALS: each rank's partial is rounded to bf16 (RNE)
                                  before it joins the fp32 running sum */
  uint64_t timeout_ns;         /* 0 = 1 s */
} tl_moe_down_args;

/* Workspace bytes: the fp32 running sums of every output tile (max_tiles * ceil(Hd/256)
 * tiles of 256 x 256) and Y [P, Hd] fp32.  0 for invalid sizes. */
size_t tl_moe_down_workspace_size(int R, int T_r, int topk, int E, int Hd);
/* Flags: 2 * R * max_tiles * ceil(Hd/256) (one per pass and CTA half of every output
 * tile), max_tiles = ceil(P/256) + E; -1 for invalid sizes. */
int tl_moe_down_num_flags(int R, int T_r, int topk, int E, int Hd);
tl_status tl_moe_down(const tl_moe_down_args* args, void* stream);

/* ---------------------------------------------------------------- AllGather-KV attention
 * Sequence-parallel attention with the key/value AllGather overlapped with the
 * attention that consumes it (talk summary, Key Findings and Experimental Setup
 * & Results: attention layers, AllGather-KV against Ring Attention).  Rank
 * `self_rank` holds the queries Q of its S_shard tokens; every rank r holds the
 * keys K_r and values V_r of its own tokens.  With Kg, Vg the shards gathered in
 * rank order (token self_rank*S_shard + t is query t's global position), for
 * every query t and head h, with kv head hk = h / (H / H_kv):
 *   s_j   = scale * <Q[t, h], Kg[j, hk]>        over the visible keys j
 *           (all keys; causal: j <= self_rank*S_shard + t)
 *   O[t, h] = bf16( sum_j exp(s_j - lse) Vg[j, hk] ),  lse[h, t] = log sum_j exp(s_j)
 * One launch of single CTAs, one per SM (tcgen05.mma.cta_group::1):
 *  - producer: a copy warp per CTA moves the peers' key and value shards, 128
 *    tokens at a time, into K_gathered / V_gathered (plain 16-byte loads and
 *    stores, from device or pinned host memory) and releases one flag per
 *    chunk of each (produce_tile_notify), shards self+1, ..., self+R-1, then
 *    self;
 *  - consumer: work units of one head and 256 query rows (two 128-row tiles
 *    that share every key/value tile); each unit streams its own shard's keys
 *    and values first (in place, no wait), then the peers' in copy order,
 *    acquiring each chunk's flags before loading it (consume_tile_wait).
 *    S = Q K^T and O += P V run on the tensor cores with S and O in tensor
 *    memory and P written back into tensor memory over S; the online softmax
 *    (running max, rescaling of O only when the max grows by more than 2^8)
 *    runs in between on the CTA's softmax warps.
 * The result does not depend on the copy order or the schedule; it is one
 * evaluation of the formula above with P rounded to bf16 for the P V product.
 * Flags: K chunk (r, c) uses flag r * ceil(S_shard/128) + c, V chunk the same
 * id plus R * ceil(S_shard/128).
 * Limits: head_dim = 128; R <= TL_MAX_RANKS; H % H_kv == 0; the self shards and
 * Q, O, K_gathered, V_gathered must be device memory; peer shards device or
 * pinned host memory.
 */
typedef struct tl_ag_attn_args {
  int32_t R;                   /* ranks, 1..TL_MAX_RANKS */
  int32_t self_rank;           /* 0..R-1 */
  int32_t S_shard;             /* tokens per rank, >= 1 */
  int32_t H;                   /* query heads, >= 1 */
  int32_t H_kv;                /* key/value heads, divides H */
  int32_t head_dim;            /* 128 */
  int32_t causal;              /* 0 = every key, 1 = keys at or before the query's position */
  float scale;                 /* softmax scale; 0 = 1/sqrt(head_dim) */
  const void* Q;               /* device bf16 [S_shard, H, head_dim] */
  const void* const* K_shards; /* host array of R pointers, bf16 [S_shard, H_kv, head_dim] */
  const void* const* V_shards; /* host array of R pointers, bf16 [S_shard, H_kv, head_dim] */
  void* K_gathered;            /* device bf16 [R*S_shard, H_kv, head_dim], written */
  void* V_gathered;            /* device bf16 [R*S_shard, H_kv, head_dim], written */
  void* O;                     /* device bf16 [S_shard, H, head_dim], written */
  float* lse;                  /* optional device float [H, S_shard] (natural log), written; NULL = none */
  tl_signals* signals;         /* >= tl_ag_attn_num_flags(R, S_shard) flags */
  uint32_t epoch;              /* nonzero */
  uint32_t reserved0;
  uint64_t timeout_ns;         /* 0 = 1 s */
} tl_ag_attn_args;

/* Flags an AllGather-KV attention call needs: 2 * R * ceil(S_shard / 128). */
int tl_ag_attn_num_flags(int R, int S_shard);
tl_status tl_ag_attn(const tl_ag_attn_args* args, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TILELINK_H */
