"""AllGather -> GEMM oracle (test infrastructure only).

Follows the TileLink talk summary ("TileLink: Generating Efficient
Compute-Communication Overlapping Kernels using Tile-Centric Primitives"):

* Key Findings / Experimental Setup & Results: AllGather-GEMM gathers the row
  shards that R ranks hold and multiplies the gathered matrix by B.  The result
  is defined by the gather and the product alone; the order in which tiles are
  moved or multiplied never changes it.
* Technical Deep Dive, tile-id mapping: a wait on a tile id is resolved to the
  (rank id, barrier id) pairs that guard its rows; for a static workload this
  is an affine function of the tile id, the tiles per rank and the barriers per
  rank.
* Technical Deep Dive, swizzle: producers and consumers walk tiles in an order
  that follows the data's arrival, so early shards are consumed first.

Arithmetic: bf16 inputs decoded exactly to float64, products and sums in
float64 (the exact result up to float64 rounding of the sums).
"""
from __future__ import annotations

import numpy as np

from . import bf16


def gathered(A_shards):
    """G = [A_0; A_1; ...; A_{R-1}] as bf16 bits (rank order; self rank does not matter)."""
    return np.concatenate([np.asarray(a, dtype=np.uint16) for a in A_shards], axis=0)


def ag_gemm(A_shards, B):
    """C = G . B in float64, G the row concatenation of the shards."""
    G = bf16.decode(gathered(A_shards))
    return G @ bf16.decode(B)


def ag_gemm_at(A_shards, B, rows, cols):
    """C[rows[i], cols[i]] one element at a time (for full-size sampled checks)."""
    M_shard = A_shards[0].shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    out = np.empty(rows.shape[0], dtype=np.float64)
    for i, (row, col) in enumerate(zip(rows, cols)):
        a = bf16.decode(A_shards[row // M_shard][row % M_shard, :])
        b = bf16.decode(B[:, col])
        out[i] = np.dot(a, b)
    return out


# ---------------------------------------------------------------- tile bookkeeping

def barriers_per_rank(M_shard, rows_per_barrier):
    return -(-M_shard // rows_per_barrier)


def barrier_of_row(row, M_shard, rows_per_barrier):
    """Global row of G -> (rank, barrier within rank, global barrier id)."""
    r = row // M_shard
    b = (row % M_shard) // rows_per_barrier
    return r, b, r * barriers_per_rank(M_shard, rows_per_barrier) + b


def tile_barriers(m_tile, BM, R, M_shard, rows_per_barrier):
    """Sorted global barrier ids guarding the rows of consumer row tile m_tile (brute force)."""
    M = R * M_shard
    ids = set()
    for row in range(m_tile * BM, min((m_tile + 1) * BM, M)):
        ids.add(barrier_of_row(row, M_shard, rows_per_barrier)[2])
    return sorted(ids)


def tile_is_local(m_tile, BM, R, M_shard, self_rank):
    """True when every row of the tile lies in the self rank's shard (read in place, no wait)."""
    M = R * M_shard
    lo, hi = m_tile * BM, min((m_tile + 1) * BM, M)
    return all(row // M_shard == self_rank for row in range(lo, hi))


def consumer_order(R, self_rank, M_shard, N, BM, BN):
    """Arrival-ordered list of (m_tile, n_tile).

    A shard's arrival position is (rank - self) mod R.  A row tile is ordered
    by the latest arrival position among its rows, then by its index; the N
    tiles of a row tile are consecutive (innermost)."""
    M = R * M_shard
    Mt, Nt = -(-M // BM), -(-N // BN)

    def key(m):
        pos = [((row // M_shard) - self_rank) % R for row in range(m * BM, min((m + 1) * BM, M))]
        return (max(pos), m)

    return [(m, n) for m in sorted(range(Mt), key=key) for n in range(Nt)]


def copy_order(R, self_rank, M_shard, rows_per_barrier):
    """Producer order: shards self+1, ..., self+R-1, then self; barriers ascending.

    Returns (rank, barrier, first_row_in_G, rows)."""
    bpr = barriers_per_rank(M_shard, rows_per_barrier)
    items = []
    for j in list(range(1, R)) + [0]:
        r = (self_rank + j) % R
        for b in range(bpr):
            lo = b * rows_per_barrier
            rows = min(rows_per_barrier, M_shard - lo)
            items.append((r, b, r * M_shard + lo, rows))
    return items
