"""AllGather-KV attention through the C ABI against the oracle.

Tolerance (derived from the arithmetic): the kernel rounds every softmax
weight P to bf16 for the P V product (relative error <= 2^-9 of each term,
so at most 2^-9 * sum_j w_j |v_j| = 2^-9 * err_scale on an output) and rounds
O to bf16 (<= 2^-9 |o|); the fp32 score, exponential and accumulation errors
are orders of magnitude below.  Every element must satisfy
|got - want| <= 2^-8 (|want| + err_scale), plus the stated normwise gate
||got - want||_inf / ||want||_inf <= 2e-2.  LSE (fp32, natural log) within
1e-3 absolute.  The gathered keys and values must equal the shards exactly.
Every output is poisoned with NaN first."""
import numpy as np
import pytest

import oracle
from tests.helpers import BF16_NORM_TOL, dev_bf16, pinned_bf16, to_bits, to_f64
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


_epoch = [0]


def run_attn(B, R, S, H, Hkv, *, self_rank=0, causal=False, scale=0.0, seed=0, host_ranks=(), sig=None, bufs=None):
    import torch
    Q, K, V = inputs.ag_attention_inputs(R, S, H, Hkv, D, seed)
    dQ = dev_bf16(Q)
    dK = [pinned_bf16(k) if r in host_ranks else dev_bf16(k) for r, k in enumerate(K)]
    dV = [pinned_bf16(v) if r in host_ranks else dev_bf16(v) for r, v in enumerate(V)]
    if bufs is None:
        Kg = torch.full((R * S, Hkv, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        Vg = torch.full((R * S, Hkv, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        O = torch.full((S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        L = torch.full((H, S), float("nan"), dtype=torch.float32, device="cuda")
    else:
        Kg, Vg, O, L = bufs
    if sig is None:
        sig = B.Signals(B.tl_ag_attn_num_flags(R, S))
    _epoch[0] += 1
    B.tl_ag_attn(dQ, dK, dV, Kg, Vg, O, sig, _epoch[0], self_rank=self_rank, causal=causal, scale=scale, lse=L)
    torch.cuda.synchronize()
    return dict(Q=Q, K=K, V=V, Kg=Kg, Vg=Vg, O=O, L=L, status=B.tl_query_status(sig), sig=sig)


def check_attn(got_o, got_l, want_o, want_l, err_scale, name=""):
    got_o = np.asarray(got_o, dtype=np.float64)
    assert got_o.shape == want_o.shape, (name, got_o.shape, want_o.shape)
    assert np.all(np.isfinite(got_o)), f"{name}: non-finite output"
    err = np.abs(got_o - want_o)
    norm_rel = float(err.max() / max(float(np.abs(want_o).max()), 1e-300))
    assert norm_rel <= BF16_NORM_TOL, f"{name}: normwise rel err {norm_rel:.3e}"
    bound = 2.0 ** -8 * (np.abs(want_o) + err_scale)
    bad = err > bound
    assert not bad.any(), f"{name}: {int(bad.sum())} elements beyond bound, worst {float((err - bound).max()):.3e}"
    dl = np.abs(np.asarray(got_l, dtype=np.float64) - want_l)
    assert np.all(np.isfinite(dl)) and float(dl.max()) <= 1e-3, f"{name}: LSE error {float(np.nanmax(dl)):.3e}"
    return norm_rel


def check_gathered(res):
    np.testing.assert_array_equal(to_bits(res["Kg"]), oracle.attention.gather(res["K"]))
    np.testing.assert_array_equal(to_bits(res["Vg"]), oracle.attention.gather(res["V"]))


def check_full(res, self_rank, causal, scale=None):
    assert res["status"] == (0, -1), res["status"]
    check_gathered(res)
    O, L, A = oracle.attention.ag_kv_attention(res["Q"], res["K"], res["V"], self_rank, scale=scale, causal=causal)
    return check_attn(to_f64(res["O"]), to_f64(res["L"]), O, L, A)


@pytest.mark.parametrize("R,S,H,Hkv,self_rank,causal", [
    (1, 128, 2, 1, 0, False),   # one key tile, one query tile
    (2, 300, 4, 2, 1, False),   # ragged shard (three key tiles, the last 44 keys), grouped heads
    (3, 300, 4, 2, 1, True),    # causal, ragged, diagonal tiles
    (3, 300, 4, 2, 0, True),    # causal on rank 0: only the own shard
    (2, 520, 2, 2, 1, True),    # two 512-row query blocks, no head grouping
    (4, 64, 8, 1, 3, False),    # shard shorter than a tile, 8 query heads on one kv head
    (8, 1, 4, 4, 5, True),      # one token per rank
    (5, 200, 2, 1, 2, False),   # odd rank count
    (64, 8, 2, 1, 63, True),    # the largest rank count, causal on the last rank
    (2, 1100, 40, 8, 1, True),  # 200 work units on 152 SMs: CTAs run two units (barrier phases across units)
    (64, 3, 2, 2, 10, False),   # 64 ranks of three tokens
    (1, 1, 1, 1, 0, False),     # one token, one head
    (1, 1, 1, 1, 0, True),
])
def test_attn_parity(B, R, S, H, Hkv, self_rank, causal):
    res = run_attn(B, R, S, H, Hkv, self_rank=self_rank, causal=causal, seed=R * 100 + S)
    check_full(res, self_rank, causal)


@pytest.mark.parametrize("scale", [0.35, 0.02])
def test_attn_explicit_scale(B, scale):
    # 0.35 ~ 4/sqrt(128): peaked weights, the running max grows often (rescaling path)
    res = run_attn(B, 2, 384, 2, 1, self_rank=1, scale=scale, seed=7)
    check_full(res, 1, False, scale=scale)


def test_attn_pinned_host_peer_shards(B):
    res = run_attn(B, 3, 256, 4, 2, self_rank=1, host_ranks=(0, 2), seed=11)
    check_full(res, 1, False)


def test_attn_repeated_calls_same_signals(B):
    r1 = run_attn(B, 2, 256, 2, 1, self_rank=0, causal=True, seed=13)
    o1 = to_bits(r1["O"]).copy()
    r2 = run_attn(B, 2, 256, 2, 1, self_rank=0, causal=True, seed=13, sig=r1["sig"])
    assert r2["status"] == (0, -1)
    np.testing.assert_array_equal(to_bits(r2["O"]), o1)


def test_attn_without_lse(B):
    # the LSE output is optional; O must not depend on whether it is written
    import torch
    R, S, H, Hkv = 2, 300, 4, 2
    res = run_attn(B, R, S, H, Hkv, self_rank=1, causal=True, seed=17)
    check_full(res, 1, True)
    O2 = torch.full_like(res["O"], float("nan"))
    sig = B.Signals(B.tl_ag_attn_num_flags(R, S))
    B.tl_ag_attn(dev_bf16(res["Q"]), [dev_bf16(k) for k in res["K"]], [dev_bf16(v) for v in res["V"]],
                 res["Kg"], res["Vg"], O2, sig, 1, self_rank=1, causal=True)
    torch.cuda.synchronize()
    assert B.tl_query_status(sig) == (0, -1)
    np.testing.assert_array_equal(to_bits(O2), to_bits(res["O"]))


def test_attn_full_size_sampled(B):
    # the sequence-parallel layer size: 8 ranks x 8192 tokens (64K context),
    # 32 query heads over 8 key/value heads, head dim 128, non-causal and causal
    import torch
    R, S, H, Hkv = 8, 8192, 32, 8
    rng = np.random.default_rng(5)
    rows = np.concatenate([[0, 1, 127, 128, 255, 256, 511, 512, S - 1], rng.integers(0, S, 23)])
    heads = np.concatenate([[0, 31, 3, 4, 7, 8, 30, 1, 17], rng.integers(0, H, 23)])
    for self_rank, causal in ((3, False), (7, True)):
        res = run_attn(B, R, S, H, Hkv, self_rank=self_rank, causal=causal, seed=21)
        assert res["status"] == (0, -1), res["status"]
        assert bool(torch.isfinite(res["O"]).all()) and bool(torch.isfinite(res["L"]).all())
        assert torch.equal(res["Kg"], torch.cat([dev_bf16(k) for k in res["K"]]))
        assert torch.equal(res["Vg"], torch.cat([dev_bf16(v) for v in res["V"]]))
        o, l, a = oracle.attention.ag_kv_attention_at(res["Q"], res["K"], res["V"], self_rank, rows, heads,
                                                      causal=causal)
        got_o = to_f64(res["O"])[rows, heads]
        got_l = to_f64(res["L"])[heads, rows]
        check_attn(got_o, got_l, o, l, a, name=f"self={self_rank} causal={causal}")


def test_attn_rejects_bad_arguments(B):
    import torch
    R, S, H, Hkv = 2, 128, 4, 2
    Q, K, V = inputs.ag_attention_inputs(R, S, H, Hkv, D, 1)
    dQ, dK, dV = dev_bf16(Q), [dev_bf16(k) for k in K], [dev_bf16(v) for v in V]
    Kg = torch.empty(R * S, Hkv, D, dtype=torch.bfloat16, device="cuda")
    Vg = torch.empty_like(Kg)
    O = torch.empty(S, H, D, dtype=torch.bfloat16, device="cuda")
    sig = B.Signals(B.tl_ag_attn_num_flags(R, S))
    with pytest.raises(B.TLError):  # head_dim 64
        B.tl_ag_attn(dQ[:, :, :64].contiguous(), [k[:, :, :64].contiguous() for k in dK],
                     [v[:, :, :64].contiguous() for v in dV], Kg, Vg, O, sig, 1)
    with pytest.raises(B.TLError):  # H not a multiple of H_kv
        B.tl_ag_attn(dQ[:, :3].contiguous(), dK, dV, Kg, Vg, O, sig, 1)
    with pytest.raises(B.TLError):  # negative scale
        B.tl_ag_attn(dQ, dK, dV, Kg, Vg, O, sig, 1, scale=-1.0)
    with pytest.raises(B.TLError):  # self shard in host memory
        B.tl_ag_attn(dQ, [pinned_bf16(K[0]), dK[1]], dV, Kg, Vg, O, sig, 1, self_rank=0)
    with pytest.raises(B.TLError):  # too few flags
        B.tl_ag_attn(dQ, dK, dV, Kg, Vg, O, B.Signals(3), 1)
    with pytest.raises(B.TLError):  # epoch 0
        B.tl_ag_attn(dQ, dK, dV, Kg, Vg, O, sig, 0)
