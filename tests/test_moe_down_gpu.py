"""The MoE down-projection side (grouped GEMM -> ReduceScatter over ranks ->
gate-weighted TopK-reduce -> scatter to the token's rank) through the C ABI
against the oracle.  The routing comes from an AllGather + grouped GEMM call on
the same topk_ids, as in a layer; every output is poisoned with NaN first."""
import numpy as np
import pytest

import oracle
from tests.helpers import check_bf16, dev_bf16, to_f64
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


_epoch = [0]


def routing_workspace(B, R, T_r, E, k, ids, seed):
    """Run the up-projection call on small random tokens and weights: its
    workspace holds the routing of ids (sorted rows, tile table, inverse)."""
    import torch
    H_up, N_up = 64, 64
    X = [inputs.normal_bf16((T_r, H_up), seed + r) for r in range(R)]
    W = [inputs.normal_bf16((H_up, N_up), seed + 100 + e, 0.02) for e in range(E)]
    P = R * T_r * k
    S = torch.empty(P, H_up, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(P, N_up, dtype=torch.bfloat16, device="cuda")
    perm = torch.empty(P, dtype=torch.int32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.tl_moe_workspace_size(R, T_r, E, k) // 4, dtype=torch.int32, device="cuda")
    sig = B.Signals(B.tl_moe_num_flags(R, T_r, H_up, k)[0])
    dids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    _epoch[0] += 1
    B.tl_moe_ag_gemm([dev_bf16(x) for x in X], dids, [dev_bf16(w) for w in W], S, Y, perm, offs, ws, sig, _epoch[0])
    assert B.tl_query_status(sig) == (0, -1)
    return ws


def run_down(B, R, T_r, E, k, I_r, Hd, seed, options=0):
    import torch
    ids = inputs.zipf_topk(R * T_r, E, k, 1.2, seed + 3000)
    H, W2, gates = inputs.moe_down_inputs(R, T_r, k, E, I_r, Hd, seed)
    ws_route = routing_workspace(B, R, T_r, E, k, ids, seed)
    out = [torch.full((T_r, Hd), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    work = torch.full((B.tl_moe_down_workspace_size(R, T_r, k, E, Hd) // 4,), float("nan"), dtype=torch.float32,
                      device="cuda")
    sig = B.Signals(B.tl_moe_down_num_flags(R, T_r, k, E, Hd))
    _epoch[0] += 1
    B.tl_moe_down([dev_bf16(h) for h in H], [dev_bf16(w) for w in W2], torch.from_numpy(gates).cuda(), ws_route,
                  out, work, sig, _epoch[0], topk=k, E=E, options=options)
    return dict(out=out, status=B.tl_query_status(sig), ids=ids, H=H, W2=W2, gates=gates)


@pytest.mark.parametrize("R,T_r,E,k,I_r,Hd", [(2, 64, 5, 2, 72, 264), (4, 256, 8, 2, 256, 512),
                                              (32, 4, 64, 2, 8, 8),  # the most ranks and experts, smallest sizes
                                              (3, 100, 6, 3, 136, 136), (1, 300, 4, 1, 64, 256),
                                              (2, 16, 12, 9, 64, 136)])  # topk above 8: the generic combine
def test_moe_down_parity(B, R, T_r, E, k, I_r, Hd):
    r = run_down(B, R, T_r, E, k, I_r, Hd, seed=80 + R + E)
    assert r["status"] == (0, -1), r["status"]
    want = oracle.moe.moe_down(r["H"], r["W2"], r["ids"], r["gates"], E, T_r)
    for d in range(R):
        check_bf16(to_f64(r["out"][d]), want[d], f"out[{d}]")


def test_moe_down_repeated_calls(B):
    # a second call on the same routing and signals (new epoch) gives the same result
    import torch
    R, T_r, E, k, I_r, Hd = 2, 128, 4, 2, 128, 256
    ids = inputs.zipf_topk(R * T_r, E, k, 1.2, 11)
    H, W2, gates = inputs.moe_down_inputs(R, T_r, k, E, I_r, Hd, 11)
    ws_route = routing_workspace(B, R, T_r, E, k, ids, 11)
    work = torch.empty(B.tl_moe_down_workspace_size(R, T_r, k, E, Hd) // 4, dtype=torch.float32, device="cuda")
    sig = B.Signals(B.tl_moe_down_num_flags(R, T_r, k, E, Hd))
    want = oracle.moe.moe_down(H, W2, ids, gates, E, T_r)
    dH, dW, dg = [dev_bf16(h) for h in H], [dev_bf16(w) for w in W2], torch.from_numpy(gates).cuda()
    for e in (1, 4):
        out = [torch.full((T_r, Hd), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        B.tl_moe_down(dH, dW, dg, ws_route, out, work, sig, e, topk=k, E=E)
        assert B.tl_query_status(sig) == (0, -1)
        for d in range(R):
            check_bf16(to_f64(out[d]), want[d], f"epoch {e} out[{d}]")


@pytest.mark.slow
def test_moe_down_full_size_sampled(B):
    R, T_r, E, k, I_r, Hd = 8, 1024, 32, 2, 1408, 4096
    r = run_down(B, R, T_r, E, k, I_r, Hd, seed=0)
    assert r["status"] == (0, -1)
    rng = np.random.default_rng(4)
    toks = np.concatenate([rng.integers(0, R * T_r, 400), [0, R * T_r - 1]])
    cols = np.concatenate([rng.integers(0, Hd, 400), [Hd - 1, 0]])
    want = oracle.moe.moe_down_at(r["H"], r["W2"], r["ids"], r["gates"], E, toks, cols)
    got = np.array([to_f64(r["out"][t // T_r][t % T_r:t % T_r + 1, c:c + 1])[0, 0] for t, c in zip(toks, cols)])
    check_bf16(got, want, "out sampled")
    for d in range(R):
        assert np.isfinite(to_f64(r["out"][d])).all()


@pytest.mark.parametrize("R,T_r,E,k,I_r,Hd", [(2, 64, 5, 2, 72, 264), (4, 256, 8, 2, 256, 512),
                                              (3, 100, 6, 3, 136, 136), (8, 128, 32, 2, 128, 512)])
def test_moe_down_bf16_partials_parity(B, R, T_r, E, k, I_r, Hd):
    # each rank's partial rounded to bf16 before it is pushed: against the oracle's bf16-partials
    # variant.  The GPU rounds its fp32 accumulation of a partial, which may land one bf16 step
    # from the exact partial rounded (a step is at most 2^-7 |P_r|); the final rounding adds
    # 2^-9 |o|.  The magnitudes sum_s g_s sum_r |P_r| are bounded by the same oracle on |H|,
    # |W2| and |g| (bf16 magnitudes: the sign bit cleared).
    r = run_down(B, R, T_r, E, k, I_r, Hd, seed=120 + R + E, options=B.TL_RS_BF16_PARTIALS)
    assert r["status"] == (0, -1), r["status"]
    want = oracle.moe.moe_down(r["H"], r["W2"], r["ids"], r["gates"], E, T_r, partials="bf16")
    mag = oracle.moe.moe_down([(h & 0x7FFF).astype(np.uint16) for h in r["H"]],
                              [(w & 0x7FFF).astype(np.uint16) for w in r["W2"]], r["ids"], np.abs(r["gates"]), E, T_r)
    for d in range(R):
        got, o = to_f64(r["out"][d]), want[d]
        assert np.isfinite(got).all()
        bound = 2.0 ** -7 * mag[d] + 2.0 ** -8 * np.abs(o) + 1e-3 * np.abs(o).max()
        assert np.all(np.abs(got - o) <= bound), f"out[{d}]: max excess {np.max(np.abs(got - o) - bound):.3e}"
        assert np.abs(got - o).max() / np.abs(o).max() <= 2e-2


@pytest.mark.parametrize("options", [0, 1])
def test_moe_down_sums_ranks_in_order(B, options):
    # every routed row's partials are 2^24, 1 and -2^24 from ranks 0, 1 and 2 (one-hot H_r rows,
    # W2_r rows of those values).  Their fp32 sum in rank order is exactly 0, since 2^24 + 1
    # rounds to 2^24; adding 1 last, or -2^24 before 2^24, gives 1.  All three values are bf16,
    # so the bf16-partials option gives the same.
    import torch
    R, T_r, E, k, I_r, Hd = 3, 64, 4, 2, 64, 264
    ids = inputs.zipf_topk(R * T_r, E, k, 1.2, 7)
    P = R * T_r * k
    ws_route = routing_workspace(B, R, T_r, E, k, ids, 7)
    H = np.zeros((P, I_r), dtype=np.uint16)
    H[:, 0] = 0x3F80  # 1.0
    W2 = []
    for v in (0x4B80, 0x3F80, 0xCB80):  # 2^24, 1, -2^24
        w = np.zeros((E * I_r, Hd), dtype=np.uint16)
        w[np.arange(E) * I_r, :] = v
        W2.append(w)
    gates = np.random.default_rng(7).uniform(0.5, 1.0, (R * T_r, k)).astype(np.float32)
    out = [torch.full((T_r, Hd), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    work = torch.full((B.tl_moe_down_workspace_size(R, T_r, k, E, Hd) // 4,), float("nan"), dtype=torch.float32,
                      device="cuda")
    sig = B.Signals(B.tl_moe_down_num_flags(R, T_r, k, E, Hd))
    _epoch[0] += 1
    B.tl_moe_down([dev_bf16(H)] * R, [dev_bf16(w) for w in W2], torch.from_numpy(gates).cuda(), ws_route,
                  out, work, sig, _epoch[0], topk=k, E=E, options=options)
    assert B.tl_query_status(sig) == (0, -1)
    for d in range(R):
        assert (to_f64(out[d]) == 0).all(), f"out[{d}] not exactly 0: ranks summed out of order"
