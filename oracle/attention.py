"""AllGather-KV attention oracle (test infrastructure only).

Follows the TileLink talk summary ("TileLink: Generating Efficient
Compute-Communication Overlapping Kernels using Tile-Centric Primitives"):

* Key Findings / Experimental Setup & Results, attention: a sequence-parallel
  attention layer in which every rank holds the queries, keys and values of
  its own block of tokens; the key and value shards of all ranks are gathered
  (AllGather-KV) and each rank attends with its own queries over the gathered
  keys and values.  The talk compares this with Ring Attention, which passes
  the shards around a ring and merges per-shard results instead.

The talk gives no formula, so the operation is the standard scaled
dot-product attention (softmax over the keys, no dropout, no bias), per query
head, with these readings where the talk is silent:

* gather order: the gathered keys are the shards in rank order, token order
  inside a shard (as for the AllGather of the GEMM workloads);
* grouped query heads: with H query heads and H_kv key/value heads, query head
  h reads key/value head h // (H / H_kv);
* causal masking (optional): query t of rank `self_rank` sits at global
  position self_rank * S_kv + t and sees the gathered keys at positions
  0 .. that position (every query sees at least one key);
* scale: 1/sqrt(D) unless given; LSE is the natural logarithm of the sum of
  exp(scaled scores) over the visible keys.

Arithmetic: bf16 inputs decoded exactly to float64; scores, exponentials and
sums in float64 (numpy's matmul serves as the dot-product step).

Layouts (bf16 bit arrays): Q [S_q, H, D]; K_r, V_r [S_kv, H_kv, D].
"""
from __future__ import annotations

import math

import numpy as np

from . import bf16


def gather(shards):
    """The AllGather: shards in rank order, rows (tokens) in order."""
    return np.concatenate([np.asarray(s) for s in shards], axis=0)


def _setup(Q, K_shards, V_shards, scale):
    q = bf16.decode(Q)
    k = bf16.decode(gather(K_shards))
    v = bf16.decode(gather(V_shards))
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    assert H % Hkv == 0 and k.shape[2] == D and v.shape == k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return q, k, v, H, Hkv, D, float(scale)


def _visible(t_rows, n_keys, self_rank, S_kv, causal):
    """[len(t_rows), n_keys] mask of the keys each query row sees."""
    keys = np.arange(n_keys)
    if not causal:
        return np.ones((len(t_rows), n_keys), dtype=bool)
    pos = self_rank * S_kv + np.asarray(t_rows)
    return keys[None, :] <= pos[:, None]


def _attend(q_rows, k, v, vis, scale):
    """Softmax attention of query rows [n, D] over keys k [S, D], values v [S, D]."""
    s = (q_rows @ k.T) * scale
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1)
    w = np.exp(s - m[:, None])
    l = w.sum(axis=1)
    o = (w @ v) / l[:, None]
    lse = m + np.log(l)
    # error scale of a bf16 evaluation: sum_j softmax_j * |v_j| (bounds every
    # rounding of an individual weight or value relative to its size)
    a = (w @ np.abs(v)) / l[:, None]
    return o, lse, a


def ag_kv_attention(Q, K_shards, V_shards, self_rank, scale=None, causal=False):
    """(O [S_q, H, D], lse [H, S_q], err_scale [S_q, H, D]) in float64."""
    q, k, v, H, Hkv, D, scale = _setup(Q, K_shards, V_shards, scale)
    S_q, S_kv = q.shape[0], np.asarray(K_shards[0]).shape[0]
    g = H // Hkv
    vis = _visible(range(S_q), k.shape[0], self_rank, S_kv, causal)
    O = np.zeros((S_q, H, D))
    A = np.zeros((S_q, H, D))
    L = np.zeros((H, S_q))
    for h in range(H):
        o, lse, a = _attend(q[:, h, :], k[:, h // g, :], v[:, h // g, :], vis, scale)
        O[:, h, :] = o
        A[:, h, :] = a
        L[h] = lse
    return O, L, A


def ag_kv_attention_at(Q, K_shards, V_shards, self_rank, rows, heads, scale=None, causal=False):
    """Only the sampled (row, head) pairs: (O [n, D], lse [n], err_scale [n, D])."""
    q, k, v, H, Hkv, D, scale = _setup(Q, K_shards, V_shards, scale)
    S_kv = np.asarray(K_shards[0]).shape[0]
    g = H // Hkv
    O, L, A = [], [], []
    for t, h in zip(rows, heads):
        vis = _visible([t], k.shape[0], self_rank, S_kv, causal)
        o, lse, a = _attend(q[t:t + 1, h, :], k[:, h // g, :], v[:, h // g, :], vis, scale)
        O.append(o[0])
        L.append(lse[0])
        A.append(a[0])
    return np.array(O), np.array(L), np.array(A)
