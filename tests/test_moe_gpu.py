"""AllGather + grouped MoE GEMM through the C ABI against the oracle.

Bookkeeping (expert offsets, perm, tile table, tile order, gathered sorted
tokens, flags, trace) must match bit for bit; Y within the bf16 tolerance.
sorted_tokens and Y are poisoned with NaN before every call."""
import numpy as np
import pytest

import oracle
from tests.helpers import check_bf16, dev_bf16, to_bits, to_f64
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


_epoch = [0]


def run_moe(B, X, ids, W, *, self_rank=0, rpb=0, timeout_ns=0, mode=None):
    import torch
    R, (T_r, H), E, N, k = len(X), X[0].shape, len(W), W[0].shape[1], ids.shape[1]
    P = R * T_r * k
    dX = [dev_bf16(x) for x in X]
    dW = [dev_bf16(w) for w in W]
    dids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    S = torch.full((P, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((P, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    perm = torch.full((P,), -1, dtype=torch.int32, device="cuda")
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.tl_moe_workspace_size(R, T_r, E, k) // 4, dtype=torch.int32, device="cuda")
    mode = B.TL_MODE_PULL if mode is None else mode
    nflags, eff = B.tl_moe_num_flags(R, T_r, H, k, rpb, mode)
    sig = B.Signals(nflags)
    max_tiles = -(-P // 256) + E
    Nt = -(-N // 256)
    trace = torch.full((max_tiles * Nt,), -1, dtype=torch.int32, device="cuda")
    _epoch[0] += 1
    B.tl_moe_ag_gemm(dX, dids, dW, S, Y, perm, offs, ws, sig, _epoch[0], self_rank=self_rank,
                     rows_per_barrier=rpb, mode=mode, timeout_ns=timeout_ns, trace=trace)
    status = B.tl_query_status(sig)
    return dict(S=S, Y=Y, perm=perm, offs=offs, ws=ws.cpu().numpy(), sig=sig, status=status, rpb=eff,
                nflags=nflags, epoch=_epoch[0], max_tiles=max_tiles, Nt=Nt, trace=trace, mode=mode)


def check_moe(B, X, ids, W, r, self_rank=0, full_y=True):
    assert r["status"] == (0, -1), r["status"]
    R, T_r, E, k = len(X), X[0].shape[0], len(W), ids.shape[1]
    counts, offsets, perm = oracle.moe.route(ids, E)
    np.testing.assert_array_equal(r["offs"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(r["perm"].cpu().numpy(), perm)
    table = oracle.moe.tile_table(counts, offsets, 256)
    pull = r["mode"] == B.TL_MODE_PULL
    sources = (oracle.moe.tile_sources_pull if pull else oracle.moe.tile_sources)(perm, k, table, T_r, r["rpb"])
    ws, mt = r["ws"], r["max_tiles"]
    n = int(ws[0])
    assert n == len(table)
    got = ws[16:16 + 6 * n].reshape(n, 6).astype(np.int64)
    got[:, 5] &= 0xFFFFFFFF  # the source-rank mask is a 32-bit word (bit 31 = rank 31)
    want = np.array([[e, s0, rows, lo, hi, mask] for (e, s0, rows), (mask, lo, hi) in zip(table, sources)])
    np.testing.assert_array_equal(got, want)
    order = (oracle.moe.tile_order_pull(sources) if pull else
             oracle.moe.tile_order(sources, R, self_rank, T_r, r["rpb"]))
    assert ws[16 + 6 * mt:16 + 6 * mt + n].tolist() == order
    inv = ws[16 + 7 * mt:16 + 7 * mt + len(perm)]
    np.testing.assert_array_equal(inv[perm], np.arange(len(perm)))
    np.testing.assert_array_equal(to_bits(r["S"]), oracle.moe.sorted_tokens(X, perm, k))
    assert np.all(r["sig"].read_flags()[:r["nflags"]] == r["epoch"])
    Nt = r["Nt"]
    assert r["trace"].cpu().tolist()[:n * Nt] == [t * Nt + j for t in order for j in range(Nt)]
    if full_y:
        check_bf16(to_f64(r["Y"]), oracle.moe.moe_ag_gemm(X, ids, W), "Y")


@pytest.mark.parametrize("R,T_r,H,N,E,k,self_rank,rpb", [
    (2, 64, 256, 256, 5, 2, 0, 0),
    (3, 50, 136, 264, 7, 3, 2, 8),     # ragged everything, three slots per token
    (4, 128, 512, 512, 16, 2, 1, 16),
    (1, 200, 64, 72, 3, 1, 0, 0),      # one rank, top-1
    (32, 8, 128, 256, 8, 2, 31, 0),    # the largest rank count, 8 tokens per rank
    (2, 1, 8, 8, 64, 2, 1, 0),         # 64 experts (the most) for 4 routed rows: nearly all empty
])
@pytest.mark.parametrize("mode", ["pull", "push"])
def test_moe_parity(B, R, T_r, H, N, E, k, self_rank, rpb, mode):
    X, ids, W = inputs.moe_inputs(R, T_r, H, N, E, k, 1.2, seed=R * 31 + E)
    m = B.TL_MODE_PULL if mode == "pull" else B.TL_MODE_PUSH
    r = run_moe(B, X, ids, W, self_rank=self_rank, rpb=rpb, mode=m)
    check_moe(B, X, ids, W, r, self_rank)


def test_moe_single_expert_is_allgather_gemm(B):
    X, _, W = inputs.moe_inputs(2, 96, 128, 256, 1, 1, 1.2, seed=4)
    ids = np.zeros((192, 1), dtype=np.int32)
    r = run_moe(B, X, ids, W)
    check_moe(B, X, ids, W, r)
    check_bf16(to_f64(r["Y"]), oracle.ag_gemm.ag_gemm(X, W[0]), "Y vs AG-GEMM")


def test_moe_empty_experts_and_identity_routing(B):
    # token t -> expert (t mod 3) of E = 6: experts 3..5 get no rows
    X, _, W = inputs.moe_inputs(2, 80, 128, 256, 6, 1, 1.2, seed=5)
    ids = (np.arange(160) % 3).astype(np.int32)[:, None]
    r = run_moe(B, X, ids, W, self_rank=1)
    check_moe(B, X, ids, W, r, self_rank=1)
    offs = r["offs"].cpu().numpy()
    assert offs[3] == offs[4] == offs[5] == offs[6] == 160


def test_moe_invalid_expert_id_is_reported(B):
    X, ids, W = inputs.moe_inputs(2, 32, 64, 64, 4, 2, 1.2, seed=6)
    ids = ids.copy()
    ids[5, 1] = 9
    r = run_moe(B, X, ids, W)
    assert r["status"][0] == B.TL_ERR_INVALID


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["pull", "push"])
def test_moe_llm_full_size(B, mode):
    c = inputs.CONFIGS["moe_llm"]
    X, ids, W = inputs.moe_inputs(c["R"], c["T_r"], c["H"], c["N"], c["E"], c["topk"], c["zipf_s"], seed=0)
    r = run_moe(B, X, ids, W, mode=B.TL_MODE_PULL if mode == "pull" else B.TL_MODE_PUSH)
    check_moe(B, X, ids, W, r, full_y=False)
    rng = np.random.default_rng(8)
    P = c["R"] * c["T_r"] * c["topk"]
    rows = np.concatenate([rng.integers(0, P, 2500), [0, P - 1]])
    cols = np.concatenate([rng.integers(0, c["N"], 2500), [0, c["N"] - 1]])
    want = oracle.moe.moe_at(X, ids, W, rows, cols)
    check_bf16(to_f64(r["Y"])[rows, cols], want, "Y sampled")
    assert np.isfinite(to_f64(r["Y"])).all()
