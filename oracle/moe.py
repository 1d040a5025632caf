"""AllGather + grouped MoE GEMM oracle (test infrastructure only).

Follows the TileLink talk summary ("TileLink: Generating Efficient
Compute-Communication Overlapping Kernels using Tile-Centric Primitives"):

* Key Findings / Experimental Setup & Results: the MoE layer gathers the
  token shards of all ranks and runs a grouped GEMM (one GEMM per expert over
  the tokens routed to it); this module covers that AllGather + GroupGEMM
  part, with no gate weighting and no combine.
* Technical Deep Dive, dynamic workloads: routing makes the tile -> rank
  dependencies data dependent, so they are handed to the kernel as lookup
  tables built from the routing.
* Key Findings / Experimental Setup & Results, the rest of the MoE layer (the
  down-projection side): a GroupGEMM per rank over the expert-sorted rows, a
  ReduceScatter of the ranks' partial outputs, a TopK-reduce that combines
  each token's k expert outputs with its gate weights, and a scatter back to
  the token order on the token's own rank (moe_down).

Routing bookkeeping (integer, plain loops):
  counts[e]   number of (token, slot) pairs routed to expert e
  offsets     exclusive prefix sum of counts, offsets[E] = T*k
  perm[i]     sorted position i -> token*k + slot, sorted by
              (expert, global token id, slot); global token id = r*T_r + local
  tile table  for each expert, ceil(count/BM) row tiles (expert, first row, rows)
  per tile    the bitmask of source ranks of its tokens, and the lowest and
              highest producer barrier (token chunk) its tokens come from.
Products: bf16 inputs decoded exactly, float64 arithmetic.
"""
from __future__ import annotations

import numpy as np

from . import bf16


def route(topk_ids, E):
    """(counts[E], offsets[E+1], perm[T*k]) as int64 arrays, by plain loops and a sort."""
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    counts = [0] * E
    for t in range(T):
        for s in range(k):
            counts[int(ids[t, s])] += 1
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + counts[e])
    pairs = sorted((int(ids[t, s]), t, s) for t in range(T) for s in range(k))
    perm = [t * k + s for (_, t, s) in pairs]
    return (np.array(counts, dtype=np.int64), np.array(offsets, dtype=np.int64),
            np.array(perm, dtype=np.int64))


def tile_table(counts, offsets, BM):
    """[(expert, first_sorted_row, rows)] in expert order."""
    out = []
    for e in range(len(counts)):
        c = int(counts[e])
        for j in range(-(-c // BM)):
            out.append((e, int(offsets[e]) + j * BM, min(BM, c - j * BM)))
    return out


def tile_sources(perm, k, table, T_r, rows_per_barrier):
    """Per tile: (rank bitmask, lowest barrier id, highest barrier id) of its tokens."""
    bpr = -(-T_r // rows_per_barrier)
    out = []
    for (_, start, rows) in table:
        mask, lo, hi = 0, None, None
        for i in range(start, start + rows):
            tok = int(perm[i]) // k
            r = tok // T_r
            b = r * bpr + (tok % T_r) // rows_per_barrier
            mask |= 1 << r
            lo = b if lo is None else min(lo, b)
            hi = b if hi is None else max(hi, b)
        out.append((mask, lo, hi))
    return out


def tile_sources_pull(perm, k, table, T_r, rows_per_barrier):
    """Pull mode: the consumer side gathers sorted rows in order, one barrier per
    chunk of rows_per_barrier sorted rows.  Per tile: (rank bitmask of its
    tokens, first chunk, last chunk) -- the chunks holding its rows."""
    out = []
    for (mask, _, _), (_, start, rows) in zip(tile_sources(perm, k, table, T_r, 1), table):
        out.append((mask, start // rows_per_barrier, (start + rows - 1) // rows_per_barrier))
    return out


def tile_order_pull(sources):
    """Pull mode: chunks arrive in sorted-row order, so tiles run by their last chunk, then index."""
    return [t for (_, t) in sorted((hi, t) for t, (_, _, hi) in enumerate(sources))]


def tile_order(sources, R, self_rank, T_r, rows_per_barrier):
    """Consumer order of the tiles (the swizzle for a dynamic workload).

    Producer barriers arrive shard by shard starting at the self shard: barrier
    (rank r, chunk c) has arrival position ((r - self) mod R) * chunks + c.  A
    tile is keyed by the latest position among the barriers it waits on (every
    id from its lowest to its highest barrier) and tiles run by (key, index)."""
    bpr = -(-T_r // rows_per_barrier)
    keys = []
    for t, (_, lo, hi) in enumerate(sources):
        key = max(((b // bpr - self_rank) % R) * bpr + b % bpr for b in range(lo, hi + 1))
        keys.append((key, t))
    return [t for (_, t) in sorted(keys)]


def sorted_tokens(X_shards, perm, k):
    """Row i = gathered token perm[i] // k (bf16 bits): the gathered tokens in expert order."""
    G = np.concatenate([np.asarray(x, dtype=np.uint16) for x in X_shards], axis=0)
    return G[np.asarray(perm, dtype=np.int64) // k]


def moe_ag_gemm(X_shards, topk_ids, W):
    """Y [T*k, N] float64: Y[i] = token(perm[i]) . W_{expert of row i}."""
    E = len(W)
    k = np.asarray(topk_ids).shape[1]
    counts, offsets, perm = route(topk_ids, E)
    Gs = bf16.decode(sorted_tokens(X_shards, perm, k))
    N = W[0].shape[1]
    Y = np.zeros((Gs.shape[0], N), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            Y[lo:hi] = Gs[lo:hi] @ bf16.decode(W[e])
    return Y


def moe_at(X_shards, topk_ids, W, rows, cols, route_result=None):
    """Y[rows[i], cols[i]] one element at a time."""
    E = len(W)
    k = np.asarray(topk_ids).shape[1]
    counts, offsets, perm = route_result if route_result is not None else route(topk_ids, E)
    T_r = X_shards[0].shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    out = np.empty(rows.shape[0], dtype=np.float64)
    for i, (row, col) in enumerate(zip(rows, cols)):
        e = int(np.searchsorted(offsets, row, side="right") - 1)
        tok = int(perm[row]) // k
        x = bf16.decode(X_shards[tok // T_r][tok % T_r, :])
        out[i] = np.dot(x, bf16.decode(W[e][:, col]))
    return out


def _rank_partial(p, partials):
    """A rank's partial as it is summed: as is ("f32": exact here), or rounded to
    bf16 first ("bf16": a rank that sends its partial in the output type)."""
    if partials == "bf16":
        return bf16.decode(bf16.encode_rne(p))
    if partials != "f32":
        raise ValueError(partials)
    return p


def moe_down(H_list, W2_list, topk_ids, gates, E, T_r, partials="f32"):
    """The down-projection side of the MoE layer, float64.

    Every expert's weights are split over the R ranks along the intermediate
    dimension: rank r holds H_r [P, I_r] (the intermediate activations of the
    P = T*k routed rows, in expert-sorted order) and W2_r [E*I_r, Hd] (expert
    e's slice at rows e*I_r .. (e+1)*I_r - 1).  With i a sorted row of expert e,
      Y[i]   = sum over ranks r = 0..R-1, in order, of H_r[i] . W2_r[e slice]
      out[t] = sum over slots s = 0..k-1, in order, of gates[t, s] * Y[pos(t, s)]
    where pos(t, s) is the sorted row of pair t*k + s; row shard d of out
    (tokens d*T_r .. (d+1)*T_r - 1) is returned as out[d].  With partials="bf16"
    each rank's term H_r[i] . W2_r[e slice] is rounded to bf16 (nearest even)
    before it enters the rank-ordered sum."""
    R = len(H_list)
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    counts, offsets, perm = route(ids, E)
    I_r = H_list[0].shape[1]
    Hd = W2_list[0].shape[1]
    P = T * k
    Y = np.zeros((P, Hd), dtype=np.float64)
    for H_r, W2_r in zip(H_list, W2_list):
        Hr, Wr = bf16.decode(H_r), bf16.decode(W2_r)
        for e in range(E):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            if hi > lo:
                Y[lo:hi] = Y[lo:hi] + _rank_partial(Hr[lo:hi] @ Wr[e * I_r:(e + 1) * I_r], partials)
    pos = np.empty(P, dtype=np.int64)
    pos[np.asarray(perm, dtype=np.int64)] = np.arange(P)
    g = np.asarray(gates, dtype=np.float64)
    out = np.zeros((T, Hd), dtype=np.float64)
    for s in range(k):
        out = out + g[:, s:s + 1] * Y[pos[np.arange(T) * k + s]]
    return [out[d * T_r:(d + 1) * T_r] for d in range(T // T_r)]


def moe_down_at(H_list, W2_list, topk_ids, gates, E, toks, cols, route_result=None, partials="f32"):
    """out[toks[i], cols[i]] (global token index) one element at a time."""
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    counts, offsets, perm = route_result if route_result is not None else route(ids, E)
    P = T * k
    pos = np.empty(P, dtype=np.int64)
    pos[np.asarray(perm, dtype=np.int64)] = np.arange(P)
    I_r = H_list[0].shape[1]
    out = np.empty(len(toks), dtype=np.float64)
    for n, (t, c) in enumerate(zip(toks, cols)):
        acc = 0.0
        for s in range(k):
            i = int(pos[int(t) * k + s])
            e = int(ids[int(t), s])
            y = 0.0
            for H_r, W2_r in zip(H_list, W2_list):
                y += float(_rank_partial(np.dot(bf16.decode(H_r[i, :]), bf16.decode(W2_r[e * I_r:(e + 1) * I_r, int(c)])),
                                         partials))
            acc += float(gates[int(t), s]) * y
        out[n] = acc
    return out
