"""Oracle pins (CPU only): the oracle against definitions, closed forms,
brute force, invariants, hand-worked fixtures and an independent library."""
import os
import re

import numpy as np
import pytest
import torch

import oracle
from oracle import bf16
from tests import oracle_checks as C

GOLDEN = C.GOLDEN


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(re.split(r"\s{2,}", line))
    return rows


def test_bf16_decode_matches_format_definition():
    for bits, value in _read_table("bf16_patterns.txt"):
        got = bf16.decode(np.array([int(bits, 16)], dtype=np.uint16))[0]
        want = float(value)
        assert got == want and np.signbit(got) == np.signbit(want), (bits, got, want)


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = bf16.decode(bits)
    fin = np.isfinite(t)
    np.testing.assert_array_equal(got[fin], t[fin])
    assert np.all(np.isnan(got[np.isnan(t)]))


def test_bf16_encode_ties_fixture():
    for row in _read_table("bf16_rne_ties.txt"):
        expr, bits = row[0], row[1]
        x = eval(expr, {"__builtins__": {}})
        got = int(bf16.encode_rne(np.array([x]))[0])
        assert got == int(bits, 16), (expr, hex(got), bits)


def test_bf16_encode_matches_torch_on_float32_values():
    # torch's float32 -> bfloat16 conversion rounds to nearest even; for float32
    # inputs a direct float64 rounding must agree with it bit for bit.
    rng = np.random.default_rng(0)
    u = rng.integers(0, 1 << 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    # add exact ties and near-ties around random bf16 values
    base = (rng.integers(0, 1 << 16, size=50_000).astype(np.uint32) << 16).view(np.float32)
    base = base[np.isfinite(base)]
    ties = (base.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, base, ties, np.array([0.0, -0.0, 1e-45, -1e-45], dtype=np.float32)])
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = bf16.encode_rne(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_roundtrip_all_finite_patterns():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bf16.decode(bits)
    fin = np.isfinite(v)
    np.testing.assert_array_equal(bf16.encode_rne(v[fin]), bits[fin])


def test_ag_gemm_pins():
    C.check_ag_gemm(oracle.ag_gemm.ag_gemm, oracle.ag_gemm.ag_gemm_at, oracle.ag_gemm.gathered, bf16.decode)


def test_ag_tile_map_pins():
    A = oracle.ag_gemm
    C.check_ag_tile_maps(A.consumer_order, A.tile_barriers, A.copy_order, A.tile_is_local)


def test_ag_tile_barriers_affine_closed_form():
    # barrier ids of a row tile form the contiguous range between its first and
    # last row's barrier (rows are contiguous and barriers ascend with rows)
    A = oracle.ag_gemm
    for (R, Ms, BM, rpb) in [(3, 100, 64, 16), (8, 1024, 128, 32), (2, 37, 16, 5)]:
        for m in range(-(-R * Ms // BM)):
            ids = A.tile_barriers(m, BM, R, Ms, rpb)
            lo = A.barrier_of_row(m * BM, Ms, rpb)[2]
            hi = A.barrier_of_row(min((m + 1) * BM, R * Ms) - 1, Ms, rpb)[2]
            assert ids == list(range(lo, hi + 1))


def test_gemm_rs_pins():
    G = oracle.gemm_rs
    C.check_gemm_rs(G.gemm_rs, G.gemm_rs_at, G.reduced)


def test_rs_item_order_pins():
    C.check_rs_item_order(oracle.gemm_rs.item_order)


def test_rs_chain_order_pins():
    C.check_rs_chain_order(oracle.gemm_rs.chain_order)


def test_moe_routing_pins():
    M = oracle.moe
    C.check_moe_routing(M.route, M.tile_table, M.tile_sources)


def test_moe_tile_order_pins():
    C.check_moe_tile_order(oracle.moe.tile_order, oracle.moe.tile_sources)


def test_moe_pull_pins():
    M = oracle.moe
    C.check_moe_pull(M.tile_sources_pull, M.tile_order_pull, M.route, M.tile_table)


def test_moe_gemm_pins():
    M = oracle.moe
    C.check_moe_gemm(M.moe_ag_gemm, M.moe_at, M.sorted_tokens, M.route, oracle.ag_gemm.ag_gemm, bf16.decode)


def test_gemm_matches_float32_library_matmul_mid_size():
    # library special case: at a mid size the float64 oracle agrees with torch's
    # float32 CPU matmul of the same bf16 values to float32 accuracy
    from tile_centric_gemm_gb300 import inputs
    A, B = inputs.ag_gemm_inputs(2, 64, 256, 96, "normal", seed=1)
    want = oracle.ag_gemm.ag_gemm(A, B)
    tA = torch.cat([inputs.to_torch_bf16(a).float() for a in A])
    tB = inputs.to_torch_bf16(B).float()
    got = (tA @ tB).double().numpy()
    assert np.max(np.abs(got - want)) <= 1e-5 * np.max(np.abs(want))


def test_gemm_rs_variant_pins():
    C.check_gemm_rs_variant(oracle.gemm_rs.gemm_rs_variant, oracle.gemm_rs.gemm_rs)


def test_gemm_rs_partial_abs_sum_pins():
    C.check_partial_abs_sum(oracle.gemm_rs.partial_abs_sum)


def test_gemm_rs_partial_abs_sum_bounds_the_sum():
    from tile_centric_gemm_gb300 import inputs
    A = [inputs.normal_bf16((8, 16), 300 + r) for r in range(3)]
    B = [inputs.normal_bf16((16, 4), 400 + r) for r in range(3)]
    S = oracle.gemm_rs.reduced(A, B)
    T = oracle.gemm_rs.partial_abs_sum(A, B)
    assert np.all(np.abs(S) <= T * (1 + 1e-12)) and np.all(T >= 0)


def test_moe_down_pins():
    C.check_moe_down(oracle.moe.moe_down, oracle.moe.route, oracle.moe.moe_down_at)


def test_moe_down_bf16_partials_pins():
    C.check_moe_down_bf16(oracle.moe.moe_down, oracle.moe.moe_down_at)


def test_ag_attention_pins():
    C.check_ag_attention(oracle.attention.ag_kv_attention, oracle.attention.gather)


def test_ag_attention_sampled_matches_full():
    from tile_centric_gemm_gb300 import inputs
    Q, K, V = inputs.ag_attention_inputs(R=3, S_shard=37, H=4, H_kv=2, D=16, seed=3)
    for causal in (False, True):
        O, L, A = oracle.attention.ag_kv_attention(Q, K, V, 1, causal=causal)
        rows, heads = [0, 5, 36, 17], [0, 3, 1, 2]
        o, l, a = oracle.attention.ag_kv_attention_at(Q, K, V, 1, rows, heads, causal=causal)
        for i, (t, h) in enumerate(zip(rows, heads)):
            np.testing.assert_allclose(o[i], O[t, h], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(a[i], A[t, h], rtol=1e-12, atol=1e-14)
            assert abs(l[i] - L[h, t]) <= 1e-12
