"""The oracle pins must catch plausible mistakes.  Each test plants one mistake
in a copy of an oracle function (on the CPU, never in the oracle itself) and
checks that the corresponding pin check fails."""
import numpy as np
import pytest

import oracle
from oracle import bf16
from tests import oracle_checks as C

A = oracle.ag_gemm
G = oracle.gemm_rs
M = oracle.moe


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_pins_catch_dropped_k_term():
    def bad(A_shards, B):
        Gm = bf16.decode(A.gathered(A_shards))[:, :-1]
        return Gm @ bf16.decode(B)[:-1]
    _fails(C.check_ag_gemm, bad, A.ag_gemm_at, A.gathered, bf16.decode)


def test_pins_catch_reversed_shard_order():
    def bad_gathered(A_shards):
        return np.concatenate([np.asarray(a) for a in A_shards[::-1]])
    def bad(A_shards, B):
        return bf16.decode(bad_gathered(A_shards)) @ bf16.decode(B)
    _fails(C.check_ag_gemm, bad, A.ag_gemm_at, bad_gathered, bf16.decode)


def test_pins_catch_wrong_sign():
    def bad(A_shards, B):
        return -A.ag_gemm(A_shards, B)
    _fails(C.check_ag_gemm, bad, A.ag_gemm_at, A.gathered, bf16.decode)


def test_pins_catch_sampler_index_swap():
    def bad_at(A_shards, B, rows, cols):
        return A.ag_gemm_at(A_shards, B, cols, rows) if max(rows) < B.shape[1] else A.ag_gemm_at(A_shards, B, rows, cols[::-1])
    _fails(C.check_ag_gemm, A.ag_gemm, bad_at, A.gathered, bf16.decode)


def test_pins_catch_n_outer_consumer_order():
    def bad(R, s, Ms, N, BM, BN):
        order = A.consumer_order(R, s, Ms, N, BM, BN)
        return sorted(order, key=lambda t: (t[1], order.index(t)))
    _fails(C.check_ag_tile_maps, bad, A.tile_barriers, A.copy_order, A.tile_is_local)


def test_pins_catch_off_by_one_barrier():
    def bad(m, BM, R, Ms, rpb):
        return A.tile_barriers(m, BM, R, Ms, rpb + 1)
    _fails(C.check_ag_tile_maps, A.consumer_order, bad, A.copy_order, A.tile_is_local)


def test_pins_catch_reverse_rank_order_sum():
    def bad_reduced(A_list, B_list):
        return G.reduced(A_list[::-1], B_list[::-1])
    def bad_rs(A_list, B_list):
        R = len(A_list)
        S = bad_reduced(A_list, B_list)
        Md = S.shape[0] // R
        return [S[d * Md:(d + 1) * Md] for d in range(R)]
    _fails(C.check_gemm_rs, bad_rs, G.gemm_rs_at, bad_reduced)


def test_pins_catch_scatter_to_wrong_destination():
    def bad_rs(A_list, B_list):
        out = G.gemm_rs(A_list, B_list)
        return out[1:] + out[:1]
    _fails(C.check_gemm_rs, bad_rs, G.gemm_rs_at, G.reduced)


def test_pins_catch_transposed_partial():
    def bad_reduced(A_list, B_list):
        S = None
        for a, b in zip(A_list, B_list):
            P = bf16.decode(a) @ bf16.decode(b)
            P = P[::-1]
            S = P if S is None else S + P
        return S
    def bad_rs(A_list, B_list):
        R = len(A_list)
        S = bad_reduced(A_list, B_list)
        Md = S.shape[0] // R
        return [S[d * Md:(d + 1) * Md] for d in range(R)]
    _fails(C.check_gemm_rs, bad_rs, G.gemm_rs_at, bad_reduced)


def test_pins_catch_unrotated_rs_order():
    def bad(R, Mm, N, BM, BN):
        return [(t, d, m, n, j) for (t, d, m, n, _), j in
                zip(G.item_order(R, Mm, N, BM, BN), [j for _ in range(10 ** 6) for j in range(R)])]
    _fails(C.check_rs_item_order, bad)


def test_pins_catch_unstable_sort():
    def bad_route(ids, E):
        counts, offsets, perm = M.route(ids, E)
        k = ids.shape[1]
        out = perm.copy()
        for e in range(E):
            seg = out[offsets[e]:offsets[e + 1]]
            out[offsets[e]:offsets[e + 1]] = seg[::-1]
        return counts, offsets, out
    _fails(C.check_moe_routing, bad_route, M.tile_table, M.tile_sources)


def test_pins_catch_inclusive_scan():
    def bad_route(ids, E):
        counts, offsets, perm = M.route(ids, E)
        return counts, np.concatenate([offsets[1:], offsets[-1:]]), perm
    _fails(C.check_moe_routing, bad_route, M.tile_table, M.tile_sources)


def test_pins_catch_wrong_expert_weight():
    def bad(X, ids, W):
        return M.moe_ag_gemm(X, ids, W[1:] + W[:1])
    _fails(C.check_moe_gemm, bad, M.moe_at, M.sorted_tokens, M.route, A.ag_gemm, bf16.decode)


def test_pins_catch_slot_for_token_confusion():
    def bad_sorted(X, perm, k):
        Gm = np.concatenate([np.asarray(x) for x in X])
        return Gm[np.asarray(perm) % Gm.shape[0]]
    _fails(C.check_moe_gemm, M.moe_ag_gemm, M.moe_at, bad_sorted, M.route, A.ag_gemm, bf16.decode)


def test_pins_catch_n_innermost_rs_tiles():
    def bad(R, Mm, N, BM, BN):
        Md = Mm // R
        Mt, Nt = -(-Md // BM), -(-N // BN)
        tiles = [(d, m, n) for d in range(R) for m in range(Mt) for n in range(Nt)]
        return [(t, d, m, n, (d + 1 + t + j) % R) for t, (d, m, n) in enumerate(tiles) for j in range(R)]
    _fails(C.check_rs_item_order, bad)


def test_pins_catch_moe_order_by_lowest_barrier():
    def bad(sources, R, s, T_r, rpb):
        bpr = -(-T_r // rpb)
        keys = [(((lo // bpr - s) % R) * bpr + lo % bpr, t) for t, (_, lo, hi) in enumerate(sources)]
        return [t for (_, t) in sorted(keys)]
    _fails(C.check_moe_tile_order, bad, M.tile_sources)


def test_pins_catch_pull_range_off_by_one():
    def bad(perm, k, table, T_r, rpb):
        return [(m, lo, hi + 1) for (m, lo, hi) in M.tile_sources_pull(perm, k, table, T_r, rpb)]
    _fails(C.check_moe_pull, bad, M.tile_order_pull, M.route, M.tile_table)


def test_pins_catch_reversed_ring():
    def bad(A, B, partials="f32", order="rank"):
        if order != "ring":
            return G.gemm_rs_variant(A, B, partials, order)
        R = len(A)
        Md = A[0].shape[0] // R
        P = [G.partial(a, b) for a, b in zip(A, B)]
        out = []
        for d in range(R):
            S = None
            for r in [(d - 1 - i) % R for i in range(R)]:
                blk = P[r][d * Md:(d + 1) * Md]
                S = blk if S is None else S + blk
            out.append(S)
        return out
    _fails(C.check_gemm_rs_variant, bad, G.gemm_rs)


def test_pins_catch_unrounded_bf16_partials():
    def bad(A, B, partials="f32", order="rank"):
        return G.gemm_rs_variant(A, B, "f32", order)
    _fails(C.check_gemm_rs_variant, bad, G.gemm_rs)


def test_pins_catch_swapped_gates():
    def bad(H, W2, ids, gates, E, T_r):
        return M.moe_down(H, W2, ids, np.ascontiguousarray(gates[:, ::-1]), E, T_r)
    _fails(C.check_moe_down, bad, M.route, M.moe_down_at)


def test_pins_catch_wrong_expert_slice():
    def bad(H, W2, ids, gates, E, T_r):
        I_r = H[0].shape[1]
        rolled = [np.roll(w, I_r, axis=0) for w in W2]
        return M.moe_down(H, rolled, ids, gates, E, T_r)
    _fails(C.check_moe_down, bad, M.route, M.moe_down_at)


def test_pins_catch_sorted_row_for_pair_index():
    def bad(H, W2, ids, gates, E, T_r):
        # reads row t*k + s of Y instead of the pair's sorted position
        T, k = np.asarray(ids).shape
        ident = np.arange(T * k)
        old_route = M.route
        try:
            M.route = lambda i, e: (lambda c, o, p: (c, o, ident))(*old_route(i, e))
            return M.moe_down(H, W2, ids, gates, E, T_r)
        finally:
            M.route = old_route
    _fails(C.check_moe_down, bad, M.route, M.moe_down_at)


def _mutated_attention(old, new):
    """A copy of the attention oracle with one source substitution, loaded as a
    fresh module (the oracle itself is untouched)."""
    import importlib.util
    import inspect
    import types
    src = inspect.getsource(oracle.attention)
    assert src.count(old) == 1, old
    mod = types.ModuleType("attention_mutant")
    mod.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(old, new), "attention_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("old,new", [
    ("o, lse, a = _attend(q[:, h, :], k[:, h // g, :], v[:, h // g, :], vis, scale)",
     "o, lse, a = _attend(q[:, h, :], k[:, h % Hkv, :], v[:, h % Hkv, :], vis, scale)"),  # head grouping
    ("s = (q_rows @ k.T) * scale", "s = (q_rows @ k.T)"),                                # dropped scale
    ("return keys[None, :] <= pos[:, None]", "return keys[None, :] < pos[:, None]"),     # causal off by one
    ("pos = self_rank * S_kv + np.asarray(t_rows)", "pos = np.asarray(t_rows)"),         # rank offset lost
    ("lse = m + np.log(l)", "lse = np.log(l)"),                                          # LSE without the max
    ("o = (w @ v) / l[:, None]", "o = (w @ v)"),                                         # no normalisation
    ("for s in shards], axis=0)", "for s in shards[::-1]], axis=0)"),                    # reversed gather
    ("o, lse, a = _attend(q[:, h, :], k[:, h // g, :], v[:, h // g, :], vis, scale)",
     "o, lse, a = _attend(q[:, h, :], k[:, h // g, :], k[:, h // g, :], vis, scale)"),  # keys as values
    ("a = (w @ np.abs(v)) / l[:, None]", "a = (w @ v) / l[:, None]"),                    # error scale signed
    ("scale = 1.0 / math.sqrt(D)", "scale = 1.0 / D"),                                    # default scale
])
def test_pins_catch_attention_mistakes(old, new):
    m = _mutated_attention(old, new)
    with np.errstate(all="ignore"):
        _fails(C.check_ag_attention, m.ag_kv_attention, m.gather)


def _mutated_module(module, name, old, new):
    """A copy of an oracle module with one source substitution, loaded as a fresh
    module (the oracle itself is untouched)."""
    import inspect
    import types
    src = inspect.getsource(module)
    assert src.count(old) == 1, old
    mod = types.ModuleType(name)
    mod.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(old, new), name, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("old,new", [
    # slot s's expert output weighted by the other slot's gate
    ("acc += float(gates[int(t), s]) * y", "acc += float(gates[int(t), k - 1 - s]) * y"),
    # the first slot's expert slice used for every slot
    ("e = int(ids[int(t), s])", "e = int(ids[int(t), 0])"),
    # the pair's index read as its sorted row
    ("i = int(pos[int(t) * k + s])", "i = int(t) * k + s"),
    # the expert slice one expert off
    ("W2_r[e * I_r:(e + 1) * I_r, int(c)]", "W2_r[(e + 1) % E * I_r:((e + 1) % E + 1) * I_r, int(c)]"),
    # only the first rank's partial
    ("for H_r, W2_r in zip(H_list, W2_list):\n                y +=", "for H_r, W2_r in zip(H_list[:1], W2_list[:1]):\n                y +="),
])
def test_pins_catch_moe_down_sampler_mistakes(old, new):
    m = _mutated_module(M, "moe_mutant", old, new)
    _fails(C.check_moe_down, M.moe_down, M.route, m.moe_down_at)


@pytest.mark.parametrize("old,new", [
    ("P = np.abs(partial(A_r, B_r))", "P = len(A_list) * np.abs(partial(A_r, B_r))"),        # scaled by R
    ("P = np.abs(partial(A_r, B_r))", "P = partial(A_r, B_r)"),                              # signed partials
    ("P = np.abs(partial(A_r, B_r))", "P = np.abs(bf16.decode(A_r)) @ np.abs(bf16.decode(B_r))"),  # |A||B|
])
def test_pins_catch_partial_abs_sum_mistakes(old, new):
    m = _mutated_module(G, "gemm_rs_mutant", old, new)
    _fails(C.check_partial_abs_sum, m.partial_abs_sum)


@pytest.mark.parametrize("old,new", [
    # the partials summed unrounded
    ('    if partials == "bf16":\n        return bf16.decode(bf16.encode_rne(p))',
     '    if partials == "bf16":\n        return p'),
    # rounded toward zero instead of to nearest even
    ('    if partials == "bf16":\n        return bf16.decode(bf16.encode_rne(p))',
     '    if partials == "bf16":\n        return np.trunc(np.asarray(p) * 128.0) / 128.0'),
])
def test_pins_catch_moe_down_bf16_partial_mistakes(old, new):
    m = _mutated_module(M, "moe_bf16_mutant", old, new)
    _fails(C.check_moe_down_bf16, m.moe_down, m.moe_down_at)


def test_pins_catch_moe_down_sum_rounded_instead_of_partials():
    def bad(H, W2, ids, gates, E, T_r, partials="f32"):
        if partials != "bf16":
            return M.moe_down(H, W2, ids, gates, E, T_r)
        R = len(H)
        T, k = np.asarray(ids).shape
        counts, offsets, perm = M.route(ids, E)
        I_r = H[0].shape[1]
        Y = np.zeros((T * k, W2[0].shape[1]))
        for h, w in zip(H, W2):
            hd, wd = bf16.decode(h), bf16.decode(w)
            for e in range(E):
                lo, hi = int(offsets[e]), int(offsets[e + 1])
                Y[lo:hi] += hd[lo:hi] @ wd[e * I_r:(e + 1) * I_r]
        Y = bf16.decode(bf16.encode_rne(Y))
        pos = np.empty(T * k, dtype=np.int64)
        pos[np.asarray(perm)] = np.arange(T * k)
        out = np.zeros((T, Y.shape[1]))
        for s in range(k):
            out = out + np.asarray(gates, np.float64)[:, s:s + 1] * Y[pos[np.arange(T) * k + s]]
        return [out[d * T_r:(d + 1) * T_r] for d in range(T // T_r)]
    _fails(C.check_moe_down_bf16, bad, M.moe_down_at)


def test_pins_catch_tile_major_chain_order():
    # the push schedule's order (a tile's ranks together) in place of rank by rank
    def bad(R, Mm, N, BM, BN):
        return [(t, d, m, n, r) for t, (d, m, n) in enumerate(G.output_tiles(R, Mm, N, BM, BN)) for r in range(R)]
    _fails(C.check_rs_chain_order, bad)


def test_pins_catch_chain_order_with_n_innermost_tiles():
    def bad(R, Mm, N, BM, BN):
        Md = Mm // R
        Mt, Nt = -(-Md // BM), -(-N // BN)
        tiles = [(d, m, n) for d in range(R) for m in range(Mt) for n in range(Nt)]
        return [(t, d, m, n, r) for r in range(R) for t, (d, m, n) in enumerate(tiles)]
    _fails(C.check_rs_chain_order, bad)


def test_pins_catch_chain_order_without_destination_groups():
    def bad(R, Mm, N, BM, BN):
        return G.chain_order(R, Mm, N, BM, BN, group=R)
    _fails(C.check_rs_chain_order, bad)


def test_pins_catch_chain_ring_order_from_rank_zero():
    # ring order started at rank d instead of d + 1
    def bad(R, Mm, N, BM, BN, group=G.CHAIN_GROUP, order="rank"):
        items = G.chain_order(R, Mm, N, BM, BN, group=group)
        if order == "ring":
            items = [(t, d, m, n, (d + r) % R) for (t, d, m, n, r) in items]
        return items
    _fails(C.check_rs_chain_order, bad)
