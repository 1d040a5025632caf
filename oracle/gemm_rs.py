"""GEMM -> ReduceScatter oracle (test infrastructure only).

Follows the TileLink talk summary ("TileLink: Generating Efficient
Compute-Communication Overlapping Kernels using Tile-Centric Primitives"):

* Key Findings / Experimental Setup & Results: GEMM-ReduceScatter; every rank
  r holds A_r and B_r (the contraction dimension is split across ranks) and
  computes its partial product; the partials are summed and row shard d of the
  sum ends on rank d.
* Technical Deep Dive, persistent kernels: the GEMM part notifies each finished
  partial tile; a reduce stage waits on its own tile and on its peers' tiles
  before summing.

The sum runs in fixed rank order, S = (((P_0 + P_1) + P_2) + ... ), P_r in
float64 from exactly decoded bf16 inputs.

Two variants closer to a real ReduceScatter's traffic (the options of the
library's GEMM-RS):
* bf16 partials -- every partial is rounded to bf16 (round to nearest even)
  before it is summed, as a rank that sends its partial in the output type;
* ring order -- destination d sums the partials in the order a ring
  ReduceScatter accumulates them, ranks d+1, d+2, ..., d (mod R): the running
  sum starts next to d and travels around the ring back to d.
"""
from __future__ import annotations

import numpy as np

from . import bf16


def partial(A_r, B_r):
    """P_r = A_r . B_r in float64."""
    return bf16.decode(A_r) @ bf16.decode(B_r)


def reduced(A_list, B_list):
    """S = sum of the partials in rank order 0..R-1 (float64), full [M, N]."""
    S = None
    for A_r, B_r in zip(A_list, B_list):
        P = partial(A_r, B_r)
        S = P if S is None else S + P
    return S


def gemm_rs(A_list, B_list):
    """Row shards out[d] = S[d*M/R:(d+1)*M/R, :] for d = 0..R-1 (float64)."""
    R = len(A_list)
    M = A_list[0].shape[0]
    if M % R:
        raise ValueError("M must be a multiple of R")
    Md = M // R
    S = reduced(A_list, B_list)
    return [S[d * Md:(d + 1) * Md, :] for d in range(R)]


def summation_order(R, d, order="rank"):
    """Ranks in the order destination d adds their partials."""
    if order == "rank":
        return list(range(R))
    if order == "ring":
        return [(d + 1 + i) % R for i in range(R)]
    raise ValueError(order)


def gemm_rs_variant(A_list, B_list, partials="f32", order="rank"):
    """Row shards out[d] (float64) with the partials optionally rounded to bf16
    first and summed in rank or ring order; the float64 sum follows that order."""
    R = len(A_list)
    M = A_list[0].shape[0]
    if M % R:
        raise ValueError("M must be a multiple of R")
    Md = M // R
    P = []
    for A_r, B_r in zip(A_list, B_list):
        p = partial(A_r, B_r)
        if partials == "bf16":
            p = bf16.decode(bf16.encode_rne(p))
        elif partials != "f32":
            raise ValueError(partials)
        P.append(p)
    out = []
    for d in range(R):
        S = None
        for r in summation_order(R, d, order):
            blk = P[r][d * Md:(d + 1) * Md, :]
            S = blk if S is None else S + blk
        out.append(S)
    return out


def partial_abs_sum(A_list, B_list):
    """sum_r |P_r| (float64), full [M, N]: scales the rounding error of bf16 partials."""
    S = None
    for A_r, B_r in zip(A_list, B_list):
        P = np.abs(partial(A_r, B_r))
        S = P if S is None else S + P
    return S


def gemm_rs_at(A_list, B_list, rows, cols):
    """S[rows[i], cols[i]] one element at a time, rank-ordered sum of per-rank dots."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    out = np.empty(rows.shape[0], dtype=np.float64)
    for i, (row, col) in enumerate(zip(rows, cols)):
        s = 0.0
        for A_r, B_r in zip(A_list, B_list):
            s = s + float(np.dot(bf16.decode(A_r[row, :]), bf16.decode(B_r[:, col])))
        out[i] = s
    return out


# ---------------------------------------------------------------- tile bookkeeping

def output_tiles(R, M, N, BM, BN):
    """Output tiles (d, m_tile_in_d, n_tile) in destination order, and within a
    destination n-tile by n-tile with the m tiles innermost (the tiles that run
    side by side share B columns and the destination's A rows); tiles never
    straddle a destination's row shard."""
    Md = M // R
    Mt, Nt = -(-Md // BM), -(-N // BN)
    return [(d, m, n) for d in range(R) for n in range(Nt) for m in range(Mt)]


CHAIN_GROUP = 2  # destinations whose tiles form one group of the chain order


def chain_order(R, M, N, BM, BN, group=CHAIN_GROUP, order="rank"):
    """Production order of the chain accumulation: (tau, d, m, n, r).

    The ordered sum accumulated on the way, like the partial sums of a ring
    reduce passing from rank to rank.  The destinations are taken in groups of
    `group` (the last group may be smaller); within a group, pass j adds every
    tile's partial of the j-th rank of its summation order (rank j, or rank
    d+1+j mod R in ring order; see summation_order), the tiles in the order of
    output_tiles, so that a tile's pass-j partial joins the running sum left by
    pass j-1."""
    tiles = output_tiles(R, M, N, BM, BN)
    items = []
    for g0 in range(0, R, group):
        members = [(tau, t) for tau, t in enumerate(tiles) if g0 <= t[0] < g0 + group]
        for j in range(R):
            items += [(tau, d, m, n, summation_order(R, d, order)[j]) for tau, (d, m, n) in members]
    return items


def item_order(R, M, N, BM, BN):
    """Production order of partial tiles: (tau, d, m, n, r).

    Tile tau's R partials are consecutive; the j-th has rank
    r = (d + 1 + tau + j) mod R, so the destination rank's own partial (the one
    that also reduces, r == d) sits at a position that rotates with tau."""
    items = []
    for tau, (d, m, n) in enumerate(output_tiles(R, M, N, BM, BN)):
        for j in range(R):
            items.append((tau, d, m, n, (d + 1 + tau + j) % R))
    return items
