"""Pin checks for the oracle, written as functions of the implementation under
test so that the same checks run on the oracle itself (must pass) and on
copies of it with a planted mistake (must fail).

Each check compares against something other than the oracle: brute-force
loops, closed forms, invariants that a plausible mistake breaks, or the
hand-worked fixtures in tests/golden/.
"""
import itertools
import math
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_json(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(x):
    """Exact small values -> bf16 bits, by the binary32 upper-half definition (no rounding needed)."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def _rand_bits(rng, shape, lo=-4, hi=4):
    """Random small integers / 8 -> exact bf16 values (brute force stays exact)."""
    return _bits(rng.integers(lo * 8, hi * 8 + 1, size=shape).astype(np.float32) / 8.0)


# ------------------------------------------------------------------ AG-GEMM

def brute_ag(A_shards, B):
    """Triple loop over plain Python floats; the gather is explicit row copying."""
    rows = []
    for a in A_shards:
        for i in range(a.shape[0]):
            rows.append([float(np.float32(np.uint32(int(v) << 16).view(np.float32))) for v in a[i]])
    Bv = [[float(np.uint32(int(v) << 16).view(np.float32)) for v in row] for row in B]
    M, K, N = len(rows), len(Bv), len(Bv[0])
    C = [[0.0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s += rows[i][k] * Bv[k][j]
            C[i][j] = s
    return np.array(C)


def check_ag_gemm(ag_gemm, ag_gemm_at, gathered, decode):
    rng = np.random.default_rng(7)
    # brute force, uneven shapes so that a transposed operand cannot pass
    A = [_rand_bits(rng, (3, 5)) for _ in range(3)]
    B = _rand_bits(rng, (5, 4))
    C = ag_gemm(A, B)
    assert C.shape == (9, 4)
    np.testing.assert_array_equal(C, brute_ag(A, B))
    # shard order: shard r constant (r+1) -> its rows are (r+1) * column sums of B
    A = [_bits(np.full((2, 6), r + 1.0)) for r in range(4)]
    B = _rand_bits(rng, (6, 3))
    C = ag_gemm(A, B)
    colsum = decode(B).sum(axis=0)
    for r in range(4):
        np.testing.assert_array_equal(C[2 * r:2 * r + 2], np.tile((r + 1) * colsum, (2, 1)))
    # closed forms: identity B returns the gathered rows exactly; all-ones gives K
    A = [_rand_bits(rng, (4, 8)) for _ in range(2)]
    np.testing.assert_array_equal(ag_gemm(A, _bits(np.eye(8))), decode(gathered(A)))
    ones = [_bits(np.ones((3, 7))) for _ in range(2)]
    np.testing.assert_array_equal(ag_gemm(ones, _bits(np.ones((7, 5)))), np.full((6, 5), 7.0))
    # R = 1 is a plain GEMM (brute force)
    A1 = [_rand_bits(rng, (4, 3))]
    B1 = _rand_bits(rng, (3, 2))
    np.testing.assert_array_equal(ag_gemm(A1, B1), brute_ag(A1, B1))
    # element sampler agrees with the full product at every element
    A = [_rand_bits(rng, (3, 6)) for _ in range(2)]
    B = _rand_bits(rng, (6, 5))
    C = ag_gemm(A, B)
    ii, jj = np.meshgrid(np.arange(6), np.arange(5), indexing="ij")
    np.testing.assert_array_equal(ag_gemm_at(A, B, ii.ravel(), jj.ravel()), C.ravel())
    # gathered buffer: rank order, exact bits
    A = [_rand_bits(rng, (2, 3)) for _ in range(3)]
    G = gathered(A)
    for r in range(3):
        np.testing.assert_array_equal(G[2 * r:2 * r + 2], A[r])


def check_ag_tile_maps(consumer_order, tile_barriers, copy_order, tile_is_local):
    fx = golden_json("ag_tile_maps_small.json")
    for c in fx["cases"]:
        got = consumer_order(c["R"], c["self"], c["M_shard"], c["N"], c["BM"], c["BN"])
        assert [list(t) for t in got] == c["consumer_order"]
    b = fx["barriers"]
    got = [tile_barriers(m, b["BM"], b["R"], b["M_shard"], b["rows_per_barrier"]) for m in range(3)]
    assert got == b["tile_barriers"]
    got = copy_order(b["R"], 0, b["M_shard"], b["rows_per_barrier"])
    assert [list(t) for t in got] == b["copy_order_self0"]
    # properties on a mid case: a permutation of all tiles; self tiles first; each
    # shard's tiles are contiguous and shards come in arrival order
    R, s, Ms, N, BM, BN = 4, 2, 256, 512, 128, 256
    order = consumer_order(R, s, Ms, N, BM, BN)
    assert sorted(order) == list(itertools.product(range(R * Ms // BM), range(N // BN)))
    shard_seq = [(m * BM) // Ms for (m, _) in order]
    assert shard_seq == sorted(shard_seq, key=lambda r: (r - s) % R)
    assert shard_seq[0] == s
    assert all(tile_is_local(m, BM, R, Ms, s) == ((m * BM) // Ms == s) for m in range(R * Ms // BM))
    # every copied row appears exactly once, self shard last
    items = copy_order(R, s, Ms, 96)
    rows = sorted(row for (_, _, g, n) in items for row in range(g, g + n))
    assert rows == list(range(R * Ms))
    assert all(it[0] == s for it in items[-3:]) and items[0][0] == (s + 1) % R


# ------------------------------------------------------------------ GEMM-RS

def check_gemm_rs(gemm_rs, gemm_rs_at, reduced):
    rng = np.random.default_rng(11)
    # brute force against per-rank triple loops summed in rank order
    R, M, Kr, N = 3, 6, 4, 5
    A = [_rand_bits(rng, (M, Kr)) for _ in range(R)]
    B = [_rand_bits(rng, (Kr, N)) for _ in range(R)]
    S = None
    for r in range(R):
        P = brute_ag([A[r]], B[r])
        S = P if S is None else S + P
    out = gemm_rs(A, B)
    assert len(out) == R
    for d in range(R):
        np.testing.assert_array_equal(out[d], S[2 * d:2 * d + 2])
    # scatter mapping: A_r[:,0] = global row index, B_r[0,:] = 1 -> out[d][i,j] = R*(d*Md+i)
    R, M, Kr, N = 4, 8, 3, 3
    A = []
    for r in range(R):
        a = np.zeros((M, Kr), dtype=np.float32)
        a[:, 0] = np.arange(M)
        A.append(_bits(a))
    Bm = np.zeros((Kr, N), dtype=np.float32)
    Bm[0, :] = 1.0
    B = [_bits(Bm)] * R
    out = gemm_rs(A, B)
    for d in range(R):
        expect = R * (d * 2 + np.arange(2))[:, None] * np.ones((1, N))
        np.testing.assert_array_equal(out[d], expect)
    # rank weights: A_r = (r+1) ones, B_r = ones -> every element K_r * sum(r+1)
    A = [_bits(np.full((4, 5), r + 1.0)) for r in range(4)]
    B = [_bits(np.ones((5, 2)))] * 4
    for d, o in enumerate(gemm_rs(A, B)):
        np.testing.assert_array_equal(o, np.full((1, 2), 5.0 * 10))
    # fixed rank order of the float64 sum: P_0 = 2^53, P_1 = 1, P_2 = -2^53.
    # ((2^53 + 1) - 2^53) = 0 in float64 (2^53+1 rounds to 2^53); any order that
    # adds P_2 before P_1 gives 1.
    A = [_bits(np.array([[2.0 ** 53]])), _bits(np.array([[1.0]])), _bits(np.array([[-(2.0 ** 53)]]))]
    B = [_bits(np.array([[1.0]]))] * 3
    assert reduced(A, B)[0, 0] == 0.0
    assert gemm_rs_at(A, B, [0], [0])[0] == 0.0
    # element sampler agrees with the full reduction
    R, M, Kr, N = 2, 4, 3, 3
    A = [_rand_bits(rng, (M, Kr)) for _ in range(R)]
    B = [_rand_bits(rng, (Kr, N)) for _ in range(R)]
    S = reduced(A, B)
    ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    np.testing.assert_array_equal(gemm_rs_at(A, B, ii.ravel(), jj.ravel()), S.ravel())


def check_rs_item_order(item_order):
    fx = golden_json("rs_item_order_small.json")
    for c in fx["cases"]:
        got = item_order(c["R"], c["M"], c["N"], c["BM"], c["BN"])
        assert [list(t) for t in got] == c["items"]
    # properties: every (tile, rank) once; the reducer (r == d) position rotates
    R, M, N, BM, BN = 8, 2048, 512, 128, 256
    items = item_order(R, M, N, BM, BN)
    assert sorted((t, r) for (t, _, _, _, r) in items) == [(t, r) for t in range(len(items) // R) for r in range(R)]
    pos = [j for j, it in enumerate(items) if it[4] == it[1]]
    assert len({p % R for p in pos}) == R


def check_rs_chain_order(chain_order):
    fx = golden_json("rs_chain_order_small.json")
    for c in fx["cases"]:
        got = chain_order(c["R"], c["M"], c["N"], c["BM"], c["BN"])
        assert [list(t) for t in got] == c["items"]
    for c in fx["ring_cases"]:
        got = chain_order(c["R"], c["M"], c["N"], c["BM"], c["BN"], order="ring")
        assert [list(t) for t in got] == c["items"]
    # properties: every (tile, rank) once; destination groups of two in order, within a
    # group ranks never decrease and the group's tiles run in index order at every
    # rank; tile indices follow destination, then n, then m
    R, M, N, BM, BN = 5, 2560, 512, 256, 256
    items = chain_order(R, M, N, BM, BN)
    ntiles = len(items) // R
    assert sorted((t, r) for (t, _, _, _, r) in items) == [(t, r) for t in range(ntiles) for r in range(R)]
    groups = [d // 2 for (_, d, _, _, _) in items]
    assert groups == sorted(groups)
    for g in set(groups):
        sub = [(t, r) for (t, d, _, _, r) in items if d // 2 == g]
        tiles = sorted({t for t, _ in sub})
        assert sub == [(t, r) for r in range(R) for t in tiles]
    Mt, Nt = -(-(M // R) // BM), -(-N // BN)
    assert all(t == (d * Nt + n) * Mt + m for (t, d, m, n, _) in items)


# ------------------------------------------------------------------ MoE

def check_moe_tile_order(tile_order, tile_sources):
    fx = golden_json("moe_routing_small.json")
    src = [tuple(t) for t in fx["tile_sources"]]
    assert tile_order(src, fx["R"], 0, fx["T_r"], fx["rows_per_barrier"]) == fx["tile_order_self0"]
    assert tile_order(src, fx["R"], 1, fx["T_r"], fx["rows_per_barrier"]) == fx["tile_order_self1"]
    # a permutation whose keys never decrease, on a random case
    rng = np.random.default_rng(9)
    R, T_r, rpb = 4, 64, 8
    src = []
    for _ in range(40):
        lo = int(rng.integers(0, R * T_r // rpb))
        hi = int(rng.integers(lo, R * T_r // rpb))
        src.append((0, lo, hi))
    order = tile_order(src, R, 2, T_r, rpb)
    assert sorted(order) == list(range(40))
    bpr = T_r // rpb
    key = lambda t: max(((b // bpr - 2) % R) * bpr + b % bpr for b in range(src[t][1], src[t][2] + 1))
    ks = [key(t) for t in order]
    assert ks == sorted(ks)


def check_moe_pull(tile_sources_pull, tile_order_pull, route, tile_table):
    fx = golden_json("moe_routing_small.json")
    ids = np.array(fx["topk_ids"])
    counts, offsets, perm = route(ids, fx["E"])
    table = tile_table(counts, offsets, fx["BM"])
    for rpb, key in ((1, "pull_sources_rpb1"), (2, "pull_sources_rpb2")):
        src = tile_sources_pull(perm, fx["k"], table, fx["T_r"], rpb)
        assert [list(t) for t in src] == fx[key]
    assert tile_order_pull([tuple(t) for t in fx["pull_sources_rpb2"]]) == fx["pull_order"]
    # every sorted row's chunk lies in its tile's range and ranges never go backwards
    rng = np.random.default_rng(4)
    T, k, E = 300, 2, 9
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = route(ids, E)
    table = tile_table(counts, offsets, 16)
    src = tile_sources_pull(perm, k, table, 100, 8)
    for (_, start, rows), (_, lo, hi) in zip(table, src):
        assert lo == start // 8 and hi == (start + rows - 1) // 8
    assert [h for (_, _, h) in src] == sorted(h for (_, _, h) in src)


def check_moe_routing(route, tile_table, tile_sources):
    fx = golden_json("moe_routing_small.json")
    ids = np.array(fx["topk_ids"])
    counts, offsets, perm = route(ids, fx["E"])
    assert list(counts) == fx["counts"]
    assert list(offsets) == fx["offsets"]
    assert list(perm) == fx["perm"]
    table = tile_table(counts, offsets, fx["BM"])
    assert [list(t) for t in table] == fx["tile_table"]
    src = tile_sources(perm, fx["k"], table, fx["T_r"], fx["rows_per_barrier"])
    assert [list(t) for t in src] == fx["tile_sources"]
    # invariants on a random routing
    rng = np.random.default_rng(3)
    T, k, E = 200, 2, 7
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = route(ids, E)
    np.testing.assert_array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert sorted(perm) == list(range(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert all(ids[p // k, p % k] == e for p in seg)
        toks = [p // k for p in seg]
        assert toks == sorted(toks)                      # stable by global token id
    table = tile_table(counts, offsets, 16)
    assert sum(t[2] for t in table) == T * k
    assert all(0 < t[2] <= 16 for t in table)


def check_moe_gemm(moe_ag_gemm, moe_at, sorted_tokens, route, ag_gemm, decode):
    rng = np.random.default_rng(5)
    # E = 1, k = 1 routing is a plain AllGather-GEMM
    X = [_rand_bits(rng, (3, 4)) for _ in range(2)]
    W = [_rand_bits(rng, (4, 5))]
    ids = np.zeros((6, 1), dtype=np.int32)
    np.testing.assert_array_equal(moe_ag_gemm(X, ids, W), ag_gemm(X, W[0]))
    # identity routing token t -> expert t mod E, k = 1: sorted rows are the
    # tokens of each residue class, each times its own expert's weight
    E = 3
    X = [_rand_bits(rng, (4, 3)) for _ in range(2)]
    W = [_rand_bits(rng, (3, 2)) for _ in range(E)]
    ids = (np.arange(8) % E).astype(np.int32)[:, None]
    Y = moe_ag_gemm(X, ids, W)
    G = np.concatenate(X)
    row = 0
    for e in range(E):
        for t in range(e, 8, E):
            np.testing.assert_array_equal(Y[row], brute_ag([G[t:t + 1]], W[e])[0])
            row += 1
    # top-2 brute force: every sorted row is token . W_expert, and rows are
    # grouped by expert with tokens ascending
    X = [_rand_bits(rng, (3, 4)) for _ in range(2)]
    W = [_rand_bits(rng, (4, 3)) for _ in range(3)]
    ids = np.array([[0, 2], [1, 0], [2, 1], [0, 1], [2, 0], [1, 2]], dtype=np.int32)
    Y = moe_ag_gemm(X, ids, W)
    G = np.concatenate(X)
    expect = []
    for e in range(3):
        for t in range(6):
            if e in ids[t]:
                expect.append(brute_ag([G[t:t + 1]], W[e])[0])
    np.testing.assert_array_equal(Y, np.array(expect))
    counts, offsets, perm = route(ids, 3)
    Gs = sorted_tokens(X, perm, 2)
    for i in range(12):
        np.testing.assert_array_equal(Gs[i], G[perm[i] // 2])
    ii, jj = np.meshgrid(np.arange(12), np.arange(3), indexing="ij")
    np.testing.assert_array_equal(moe_at(X, ids, W, ii.ravel(), jj.ravel()), Y.ravel())


def check_gemm_rs_variant(variant, gemm_rs):
    """Pins of the bf16-partial / ring-order GEMM-RS variant."""
    rng = np.random.default_rng(19)
    # f32 partials in rank order are the plain definition
    R, M, Kr, N = 3, 6, 4, 5
    A = [_rand_bits(rng, (M, Kr)) for _ in range(R)]
    B = [_rand_bits(rng, (Kr, N)) for _ in range(R)]
    for a, b in zip(variant(A, B, "f32", "rank"), gemm_rs(A, B)):
        np.testing.assert_array_equal(a, b)
    # bf16 rounding of each partial: P_0 = 1 + 2^-8 is a tie between 1 and 1 + 2^-7
    # and rounds to the even 1.0; P_1 = 1 is exact.  bf16 partials sum to 2, fp32 ones
    # to 2 + 2^-8.  Partials that bf16 holds exactly are not changed.
    A = [_bits(np.array([[1.0, 2.0 ** -8]] * 2)), _bits(np.array([[1.0, 0.0]] * 2))]
    B = [_bits(np.array([[1.0], [1.0]]))] * 2
    for o in variant(A, B, "bf16", "rank"):
        np.testing.assert_array_equal(o, [[2.0]])
    for o in variant(A, B, "f32", "rank"):
        np.testing.assert_array_equal(o, [[2.0 + 2.0 ** -8]])
    A = [_bits(np.array([[1.5, 0.25]] * 2)), _bits(np.array([[3.0, -1.0]] * 2))]
    for x, y in zip(variant(A, B, "bf16", "rank"), variant(A, B, "f32", "rank")):
        np.testing.assert_array_equal(x, y)
    # ring order, by hand: R = 4 partials 1, 2^53, -2^53, 0 on every row; destination d
    # adds ranks d+1, d+2, d+3, d.  In float64 (1 + 2^53) rounds to 2^53, so a row sums
    # to 0 exactly when 1 and 2^53 are both added before -2^53:
    #   d=0: 2^53, -2^53, 0, 1 -> 1     d=1: -2^53, 0, 1, 2^53 -> 1
    #   d=2: 0, 1, 2^53, -2^53 -> 0     d=3: 1, 2^53, -2^53, 0 -> 0
    # (rank order gives 0 everywhere; the reversed ring gives 1, 1, 0, 1)
    vals = [1.0, 2.0 ** 53, -(2.0 ** 53), 0.0]
    A = [_bits(np.full((4, 1), v)) for v in vals]
    B = [_bits(np.array([[1.0]]))] * 4
    np.testing.assert_array_equal([o[0, 0] for o in variant(A, B, "f32", "ring")], [1.0, 1.0, 0.0, 0.0])
    np.testing.assert_array_equal([o[0, 0] for o in variant(A, B, "f32", "rank")], [0.0, 0.0, 0.0, 0.0])


def check_partial_abs_sum(partial_abs_sum):
    """sum_r |P_r| by hand.  One element, three ranks with one-term partials 1, -2,
    3: the magnitudes add to 6 (the signed sum is 2).  Then a partial that cancels
    inside its own dot product: P_0 = 1*2 + (-1)*3 = -1 and P_1 = 2*1 + 0*5 = 2
    give 3 -- not 7, the sum of |a_k| |b_k| over the terms, nor 1, the magnitude
    of the summed partials.  Finally a 2 x 2 case by hand, rows and columns
    distinct so a transposed operand shows."""
    one = _bits(np.array([[1.0]]))
    T = partial_abs_sum([_bits(np.array([[v]])) for v in (1.0, -2.0, 3.0)], [one] * 3)
    np.testing.assert_array_equal(T, [[6.0]])
    A = [_bits(np.array([[1.0, -1.0]])), _bits(np.array([[2.0, 0.0]]))]
    B = [_bits(np.array([[2.0], [3.0]])), _bits(np.array([[1.0], [5.0]]))]
    np.testing.assert_array_equal(partial_abs_sum(A, B), [[3.0]])
    # P_0 = [[1, 2], [3, 4]] @ [[1, 0], [-1, 1]] = [[-1, 2], [-1, 4]]; P_1 = -I
    A = [_bits(np.array([[1.0, 2.0], [3.0, 4.0]])), _bits(np.array([[-1.0, 0.0], [0.0, -1.0]]))]
    B = [_bits(np.array([[1.0, 0.0], [-1.0, 1.0]])), _bits(np.eye(2))]
    np.testing.assert_array_equal(partial_abs_sum(A, B), [[2.0, 2.0], [1.0, 5.0]])


def check_moe_down(moe_down, route, moe_down_at):
    """Pins of the MoE down-projection side: brute force on a tiny case, the
    plain-GEMM special case, and linearity in the ranks and in the gates.  The
    element-at-a-time sampler moe_down_at is held to the same brute force at
    every (token, column) of the tiny case, with both gates and with slot 1's
    gate zeroed."""
    rng = np.random.default_rng(23)
    # brute force: R = 2 ranks, T = 6 tokens of T_r = 3, top-2 of E = 3, I_r = 2, Hd = 3
    R, T_r, E, k, I_r, Hd = 2, 3, 3, 2, 2, 3
    T, P = R * T_r, R * T_r * k
    ids = np.array([[0, 2], [1, 0], [2, 1], [0, 1], [2, 0], [1, 2]], dtype=np.int32)
    H = [_rand_bits(rng, (P, I_r)) for _ in range(R)]
    W2 = [_rand_bits(rng, (E * I_r, Hd)) for _ in range(R)]
    gates = rng.uniform(0.0, 1.0, (T, k)).astype(np.float32)
    out = moe_down(H, W2, ids, gates, E, T_r)
    # sorted rows by (expert, token, slot), written out by hand from ids
    sorted_pairs = [(e, t, s) for e in range(E) for t in range(T) for s in range(k) if ids[t, s] == e]
    pos = {(t, s): i for i, (_, t, s) in enumerate(sorted_pairs)}
    dec = lambda b: np.asarray(b, dtype=np.uint32).astype(np.uint32) << 16
    Hf = [dec(h).view(np.float32).astype(np.float64) for h in H]
    Wf = [dec(w).view(np.float32).astype(np.float64) for w in W2]
    brute = np.zeros((T, Hd))
    for t in range(T):
        for c in range(Hd):
            want = 0.0
            for s in range(k):
                i = pos[(t, s)]
                e = ids[t, s]
                y = 0.0
                for r in range(R):
                    for j in range(I_r):
                        y += Hf[r][i, j] * Wf[r][e * I_r + j, c]
                want += float(gates[t, s]) * y
            assert abs(out[t // T_r][t % T_r, c] - want) <= 1e-12 * max(1.0, abs(want)), (t, c)
            brute[t, c] = want
    # E = 1, k = 1, R = 1, gate 1: sorted rows are the tokens in order, out = H . W2
    H1 = [_rand_bits(rng, (4, 3))]
    W1 = [_rand_bits(rng, (3, 5))]
    o = moe_down(H1, W1, np.zeros((4, 1), np.int32), np.ones((4, 1), np.float32), 1, 4)
    Hf1, Wf1 = dec(H1[0]).view(np.float32).astype(np.float64), dec(W1[0]).view(np.float32).astype(np.float64)
    np.testing.assert_allclose(o[0], Hf1 @ Wf1, rtol=1e-12, atol=0)
    # linearity in the ranks: the R-rank result is the sum of the one-rank results
    parts = [moe_down([H[r]], [W2[r]], ids, gates, E, T) for r in range(R)]
    whole = np.concatenate(out)
    np.testing.assert_allclose(whole, parts[0][0] + parts[1][0], rtol=1e-12, atol=1e-12)
    # gates: zeroing slot 1 leaves only slot 0's expert output
    g0 = gates.copy()
    g0[:, 1] = 0.0
    o0 = np.concatenate(moe_down(H, W2, ids, g0, E, T_r))
    for t in range(T):
        i = pos[(t, 0)]
        e = ids[t, 0]
        y = sum(Hf[r][i] @ Wf[r][e * I_r:(e + 1) * I_r] for r in range(R))
        np.testing.assert_allclose(o0[t], float(gates[t, 0]) * y, rtol=1e-12, atol=1e-12)
    # the sampler, every element, in a scrambled visiting order (so a mix-up of the
    # token and column lists cannot pass), against the brute force and the zeroed gate
    tt, cc = np.meshgrid(np.arange(T), np.arange(Hd), indexing="ij")
    order = np.random.default_rng(29).permutation(T * Hd)
    toks, cols = tt.ravel()[order], cc.ravel()[order]
    np.testing.assert_allclose(moe_down_at(H, W2, ids, gates, E, toks, cols), brute[toks, cols],
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(moe_down_at(H, W2, ids, g0, E, toks, cols), o0[toks, cols], rtol=1e-12, atol=1e-12)


def check_moe_down_bf16(moe_down, moe_down_at):
    """Pins of the bf16-partials variant of the MoE down side, by hand.  Two
    tokens of two ranks route to the one expert (k = 1, I_r = 2, Hd = 1); rank 1
    adds 3*2^-8 to both.  Rank 0's term is 1 + 2^-8 for token 0 (a tie between 1
    and 1 + 2^-7, to even: 1) and 1 + 3*2^-9 for token 1 (three quarters of a
    step: 1 + 2^-7).  So with bf16 partials token 0 gives 1 + 3*2^-8 and token 1,
    gated by 1/2, (1 + 2^-7 + 3*2^-8) / 2; with fp32 partials 1 + 2^-6 and
    (1 + 9*2^-9) / 2.  Rounding the sum instead of each partial gives 1 + 2^-6
    for token 0; truncating instead of rounding gives (1 + 3*2^-8) / 2 for token 1."""
    H = [_bits(np.array([[1.0, 2.0 ** -8], [1.0, 3 * 2.0 ** -9]])), _bits(np.array([[0.0, 3 * 2.0 ** -8]] * 2))]
    W2 = [_bits(np.array([[1.0], [1.0]]))] * 2
    ids = np.zeros((2, 1), dtype=np.int32)
    gates = np.array([[1.0], [0.5]], dtype=np.float32)
    want_bf16 = [1 + 3 * 2.0 ** -8, (1 + 2.0 ** -7 + 3 * 2.0 ** -8) / 2]
    want_f32 = [1 + 2.0 ** -6, (1 + 9 * 2.0 ** -9) / 2]
    for partials, want in (("bf16", want_bf16), ("f32", want_f32)):
        out = moe_down(H, W2, ids, gates, 1, 1, partials=partials)
        np.testing.assert_array_equal([out[0][0, 0], out[1][0, 0]], want)
        np.testing.assert_array_equal(moe_down_at(H, W2, ids, gates, 1, [0, 1], [0, 0], partials=partials), want)


# ------------------------------------------------------------------ AllGather-KV attention

def check_ag_attention(attn, gather):
    """Pins of the AllGather-KV attention oracle.

    * the gather: explicit row copying, shards in rank order;
    * non-causal, grouped heads: torch's scaled_dot_product_attention in
      float64 on the CPU (an independent library routine; default scale and an
      explicit one);
    * closed forms: values constant per key/value head give that constant;
      zero queries give the mean of the visible values and LSE = log(count);
      the first query of rank 0 under the causal mask sees one key;
    * the causal result of a query equals the non-causal result over the
      gathered prefix up to its position;
    * the Ring-Attention merge: the attention over all shards equals the
      exp(lse_r - lse)-weighted sum of the per-shard results;
    * the error scale sum_j softmax_j |v_j| is 1 when every |v| is 1.
    """
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(29)
    R, S, H, Hkv, D = 3, 5, 4, 2, 8
    g = H // Hkv
    dec = lambda b: (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    Q = _rand_bits(rng, (S, H, D), -2, 2)
    K = [_rand_bits(rng, (S, Hkv, D), -2, 2) for _ in range(R)]
    V = [_rand_bits(rng, (S, Hkv, D), -4, 4) for _ in range(R)]
    # gather by explicit copying
    Kg = gather(K)
    assert Kg.shape == (R * S, Hkv, D)
    for r in range(R):
        for u in range(S):
            np.testing.assert_array_equal(Kg[r * S + u], K[r][u])
    Kf, Vf = dec(gather(K)), dec(gather(V))
    q_t = torch.from_numpy(dec(Q)).permute(1, 0, 2).contiguous()
    k_t = torch.from_numpy(Kf).permute(1, 0, 2).contiguous()
    v_t = torch.from_numpy(Vf).permute(1, 0, 2).contiguous()
    for scale in (None, 0.3):
        want = F.scaled_dot_product_attention(q_t, k_t, v_t, scale=scale, enable_gqa=True).permute(1, 0, 2).numpy()
        for self_rank in (0, 2):
            O, L, A = attn(Q, K, V, self_rank, scale=scale, causal=False)
            np.testing.assert_allclose(O, want, rtol=1e-10, atol=1e-12)
    # constant values per key/value head
    c = np.array([[1.5] * D, [-0.25] * D])
    Vc = [_bits(np.broadcast_to(c, (S, Hkv, D)).copy()) for _ in range(R)]
    for causal in (False, True):
        O, _, _ = attn(Q, K, Vc, 1, causal=causal)
        for h in range(H):
            np.testing.assert_allclose(O[:, h, :], np.broadcast_to(c[h // g], (S, D)), rtol=1e-13, atol=0)
    # zero queries: uniform weights over the visible keys
    Z = _bits(np.zeros((S, H, D), dtype=np.float32))
    for causal in (False, True):
        for self_rank in (0, 1, 2):
            O, L, _ = attn(Z, K, V, self_rank, causal=causal)
            for t in range(S):
                n = (self_rank * S + t + 1) if causal else R * S
                for h in range(H):
                    want = sum(Vf[j, h // g] for j in range(n)) / n
                    np.testing.assert_allclose(O[t, h], want, rtol=1e-12, atol=1e-13)
                    assert abs(L[h, t] - math.log(n)) <= 1e-12, (causal, self_rank, t, h)
    # first query of rank 0, causal: one visible key (K_0 row 0)
    O, L, _ = attn(Q, K, V, 0, causal=True)
    qf = dec(Q)
    for h in range(H):
        np.testing.assert_allclose(O[0, h], dec(V[0])[0, h // g], rtol=0, atol=0)
        dot = 0.0
        for e in range(D):
            dot += qf[0, h, e] * dec(K[0])[0, h // g, e]
        assert abs(L[h, 0] - dot / math.sqrt(D)) <= 1e-12
    # causal = non-causal over the prefix up to the query's position
    for self_rank in (1, 2):
        O, L, _ = attn(Q, K, V, self_rank, causal=True)
        for t in range(S):
            n = self_rank * S + t + 1
            Kp, Vp = [Kg[:n]], [gather(V)[:n]]
            o1, l1, _ = attn(Q[t:t + 1], Kp, Vp, 0, causal=False)
            np.testing.assert_allclose(O[t], o1[0], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(L[:, t], l1[:, 0], rtol=1e-12, atol=1e-13)
    # Ring-Attention merge of per-shard results (pins LSE, including its scale)
    for scale in (None, 0.7):
        O, L, _ = attn(Q, K, V, 1, scale=scale, causal=False)
        parts = [attn(Q, [K[r]], [V[r]], 0, scale=scale, causal=False) for r in range(R)]
        lse = np.logaddexp.reduce(np.stack([p[1] for p in parts]), axis=0)
        np.testing.assert_allclose(L, lse, rtol=1e-12, atol=1e-12)
        merged = sum(np.exp(p[1] - lse).T[:, :, None] * p[0] for p in parts)
        np.testing.assert_allclose(O, merged, rtol=1e-10, atol=1e-12)
    # error scale with |v| = 1 everywhere
    Vs = [_bits(np.where(rng.integers(0, 2, (S, Hkv, D)) == 1, 1.0, -1.0).astype(np.float32)) for _ in range(R)]
    _, _, A = attn(Q, K, Vs, 2, causal=True)
    np.testing.assert_allclose(A, 1.0, rtol=1e-13, atol=0)
