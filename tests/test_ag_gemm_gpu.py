"""AllGather-GEMM through the C ABI against the oracle.

Every call poisons `gathered` and C with NaN first, so a consumer tile that
reads rows before their arrival flag is set shows up as a mismatch."""
import numpy as np
import pytest

import oracle
from tests.helpers import check_bf16, check_f32, dev_bf16, pinned_bf16, to_bits, to_f64
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


class Epoch:
    v = 0

    @classmethod
    def next(cls):
        cls.v += 1
        return cls.v


def run_ag(B, A, Bm, *, self_rank=0, mode=None, rpb=0, f32=False, notify_ready=True, timeout_ns=0,
           withhold=None, trace=False, host_ranks=(), swizzle=0, ws=None):
    import torch
    R, (Ms, K), N = len(A), A[0].shape, Bm.shape[1]
    mode = B.TL_MODE_PUSH if mode is None else mode
    dA = [pinned_bf16(a) if r in host_ranks else dev_bf16(a) for r, a in enumerate(A)]
    dB = dev_bf16(Bm)
    G = torch.full((R * Ms, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = torch.full((R * Ms, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    C32 = torch.full((R * Ms, N), float("nan"), dtype=torch.float32, device="cuda") if f32 else None
    nflags, eff_rpb = B.tl_ag_gemm_num_flags(R, Ms, K, rpb)
    sig = B.Signals(nflags)
    ready = None
    epoch = Epoch.next()
    if mode == B.TL_MODE_PULL:
        ready = B.Signals(nflags)
        if notify_ready:
            B.tl_tile_notify(ready, 0, nflags, epoch)
            if withhold is not None:
                B.tl_tile_notify(ready, withhold, 1, epoch - 1)
    Mt, Nt = -(-R * Ms // 256), -(-N // 256)
    tr = torch.full((Mt * Nt,), -1, dtype=torch.int32, device="cuda") if trace else None
    B.tl_ag_gemm(dA, dB, G, C, sig, epoch, self_rank=self_rank, C_f32=C32, mode=mode, src_ready=ready,
                 rows_per_barrier=rpb, timeout_ns=timeout_ns, trace=tr, swizzle=swizzle, workspace=ws)
    status = B.tl_query_status(sig)
    out = dict(G=G, C=C, C32=C32, sig=sig, ready=ready, epoch=epoch, status=status, nflags=nflags,
               rpb=eff_rpb, trace=tr, Mt=Mt, Nt=Nt)
    return out


def check_all(B, A, Bm, r, self_rank=0):
    assert r["status"] == (0, -1), r["status"]
    want = oracle.ag_gemm.ag_gemm(A, Bm)
    check_bf16(to_f64(r["C"]), want, "C")
    if r["C32"] is not None:
        check_f32(to_f64(r["C32"]), want, "C_f32")
    np.testing.assert_array_equal(to_bits(r["G"]), oracle.ag_gemm.gathered(A))
    flags = r["sig"].read_flags()
    assert np.all(flags[:r["nflags"]] == r["epoch"])
    if r["trace"] is not None:
        R, Ms, N = len(A), A[0].shape[0], Bm.shape[1]
        order = oracle.ag_gemm.consumer_order(R, self_rank, Ms, N, 256, 256)
        want_trace = [m * r["Nt"] + n for (m, n) in order]
        assert r["trace"].cpu().tolist() == want_trace


def test_ag_tiny_bf16_and_fp32(B):
    c = inputs.CONFIGS["ag_tiny"]
    A, Bm = inputs.ag_gemm_inputs(c["R"], c["M_shard"], c["K"], c["N"], c["dist"], seed=0)
    r = run_ag(B, A, Bm, f32=True, trace=True)
    check_all(B, A, Bm, r)


def test_ag_identity_b_returns_gathered_rows_exactly(B):
    rng = np.random.default_rng(0)
    A = [inputs.uniform_bf16((128, 256), 10 + r) for r in range(2)]
    eye = inputs.bf16_bits_from_f32(np.eye(256, dtype=np.float32))
    r = run_ag(B, A, eye, self_rank=1)
    assert r["status"] == (0, -1)
    np.testing.assert_array_equal(to_bits(r["C"]), oracle.ag_gemm.gathered(A))


@pytest.mark.parametrize("R,Ms,K,N,self_rank,rpb", [
    (3, 100, 136, 264, 1, 16),     # tiles straddle shards; K and N tails
    (5, 77, 64, 8, 4, 0),          # tiny N, ragged everything
    (1, 300, 520, 512, 0, 0),      # one rank: plain GEMM
    (4, 256, 1024, 768, 2, 32),    # several tiles per shard, rotation from rank 2
    (2, 1, 8, 8, 1, 0),            # smallest shapes: one row per shard, K = N = 8
])
def test_ag_ragged_shapes(B, R, Ms, K, N, self_rank, rpb):
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=R * 100 + Ms)
    r = run_ag(B, A, Bm, self_rank=self_rank, rpb=rpb, f32=True, trace=True)
    check_all(B, A, Bm, r, self_rank)


def test_ag_pull_mode_matches_push(B):
    A, Bm = inputs.ag_gemm_inputs(4, 256, 512, 512, "normal", seed=5)
    r1 = run_ag(B, A, Bm, self_rank=3, mode=B.TL_MODE_PULL, trace=True)
    check_all(B, A, Bm, r1, 3)
    r2 = run_ag(B, A, Bm, self_rank=3, mode=B.TL_MODE_PUSH)
    check_all(B, A, Bm, r2, 3)
    np.testing.assert_array_equal(to_bits(r1["C"]), to_bits(r2["C"]))


def test_ag_pull_missing_source_flag_times_out(B):
    import torch
    A, Bm = inputs.ag_gemm_inputs(2, 128, 256, 256, "normal", seed=6)
    nflags, _ = B.tl_ag_gemm_num_flags(2, 128, 256)
    r = run_ag(B, A, Bm, mode=B.TL_MODE_PULL, withhold=nflags - 1, timeout_ns=20_000_000)
    assert r["status"][0] == B.TL_ERR_TIMEOUT
    # the withheld flag, or a consumer flag that depends on it, is reported
    assert 0 <= r["status"][1] < nflags
    # the context stays usable: the same call with every flag set now succeeds
    r = run_ag(B, A, Bm, mode=B.TL_MODE_PULL)
    check_all(B, A, Bm, r)
    assert float(torch.ones(8, device="cuda").sum()) == 8.0


def test_ag_repeated_calls_same_signals_advance_epoch(B):
    import torch
    A, Bm = inputs.ag_gemm_inputs(2, 256, 256, 256, "normal", seed=8)
    dA = [dev_bf16(a) for a in A]
    dB = dev_bf16(Bm)
    nflags, _ = B.tl_ag_gemm_num_flags(2, 256, 256)
    sig = B.Signals(nflags)
    want = oracle.ag_gemm.ag_gemm(A, Bm)
    for e in range(1, 4):
        G = torch.full((512, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
        C = torch.full((512, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.tl_ag_gemm(dA, dB, G, C, sig, e, self_rank=e % 2)
        assert B.tl_query_status(sig) == (0, -1)
        check_bf16(to_f64(C), want, f"C epoch {e}")
        assert np.all(sig.read_flags() == e)


@pytest.mark.slow
def test_ag_llm_full_size_sampled(B):
    c = inputs.CONFIGS["ag_llm"]
    A, Bm = inputs.ag_gemm_inputs(c["R"], c["M_shard"], c["K"], c["N"], c["dist"], seed=0)
    r = run_ag(B, A, Bm, trace=True)
    assert r["status"] == (0, -1)
    np.testing.assert_array_equal(to_bits(r["G"]), oracle.ag_gemm.gathered(A))
    assert np.all(r["sig"].read_flags() == r["epoch"])
    rng = np.random.default_rng(1)
    M, N = c["R"] * c["M_shard"], c["N"]
    rows = np.concatenate([rng.integers(0, M, 3000), [0, M - 1, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 3000), [0, 0, N - 1]])
    want = oracle.ag_gemm.ag_gemm_at(A, Bm, rows, cols)
    got = to_f64(r["C"])[rows, cols]
    check_bf16(got, want, "C sampled")
    # every element: finite (no NaN left from the poison) and the trace is the swizzle
    assert np.isfinite(to_f64(r["C"])).all()
    order = oracle.ag_gemm.consumer_order(c["R"], 0, c["M_shard"], N, 256, 256)
    assert r["trace"].cpu().tolist() == [m * r["Nt"] + n for (m, n) in order]


@pytest.mark.slow
@pytest.mark.parametrize("R,M", [(4, 4096), (2, 1024), (8, 16384)])
def test_ag_sweep_points(B, R, M):
    # AG sweep workload: K=8192, N=1024, activations N(0,1), weights N(0,0.02),
    # with the split-K workspace the sweep gives (M=1024: 16 tiles split 4 ways)
    A, Bm = inputs.ag_gemm_inputs(R, M // R, 8192, 1024, "normal", seed=M + R)
    r = run_ag(B, A, Bm, self_rank=R - 1, trace=True, ws=splitk_ws(B, R, M // R, 8192, 1024))
    assert r["status"] == (0, -1)
    np.testing.assert_array_equal(to_bits(r["G"]), oracle.ag_gemm.gathered(A))
    rng = np.random.default_rng(R)
    rows, cols = rng.integers(0, M, 2000), rng.integers(0, 1024, 2000)
    check_bf16(to_f64(r["C"])[rows, cols], oracle.ag_gemm.ag_gemm_at(A, Bm, rows, cols), "C sampled")
    order = oracle.ag_gemm.consumer_order(R, R - 1, M // R, 1024, 256, 256)
    assert r["trace"].cpu().tolist() == [m * r["Nt"] + n for (m, n) in order]


@pytest.mark.parametrize("mode", ["push", "pull"])
def test_ag_pinned_host_peer_shards(B, mode):
    # the slower-link stand-in: every shard but the self shard in pinned host memory
    R, Ms, K, N, self_rank = 4, 300, 520, 264, 2
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=41)
    m = B.TL_MODE_PUSH if mode == "push" else B.TL_MODE_PULL
    r = run_ag(B, A, Bm, self_rank=self_rank, mode=m, rpb=13, trace=True,
               host_ranks=[x for x in range(R) if x != self_rank])
    check_all(B, A, Bm, r, self_rank)


def test_ag_rejects_host_self_shard_and_host_b(B):
    import torch
    R, Ms, K, N = 2, 128, 256, 256
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=43)
    G = torch.zeros(R * Ms, K, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(R * Ms, N, dtype=torch.bfloat16, device="cuda")
    sig = B.Signals(B.tl_ag_gemm_num_flags(R, Ms, K)[0])
    with pytest.raises(B.TLError) as e:
        B.tl_ag_gemm([pinned_bf16(A[0]), dev_bf16(A[1])], dev_bf16(Bm), G, C, sig, 1, self_rank=0)
    assert e.value.code == B.TL_ERR_UNSUPPORTED and "self shard" in str(e.value)
    with pytest.raises(B.TLError) as e:
        B.tl_ag_gemm([dev_bf16(a) for a in A], pinned_bf16(Bm), G, C, sig, 1)
    assert e.value.code == B.TL_ERR_UNSUPPORTED
    assert np.all(sig.read_flags() == 0)


def test_ag_rows_swizzle_runs_tiles_in_index_order(B):
    # the unswizzled schedule: same result, row tiles 0, 1, ... whatever the arrival order
    R, Ms, K, N, self_rank = 4, 300, 520, 264, 2
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=47)
    r = run_ag(B, A, Bm, self_rank=self_rank, rpb=11, trace=True, swizzle=B.TL_SWIZZLE_ROWS)
    assert r["status"] == (0, -1)
    check_bf16(to_f64(r["C"]), oracle.ag_gemm.ag_gemm(A, Bm), "C")
    np.testing.assert_array_equal(to_bits(r["G"]), oracle.ag_gemm.gathered(A))
    assert r["trace"].cpu().tolist() == [m * r["Nt"] + n for m in range(r["Mt"]) for n in range(r["Nt"])]


def splitk_ws(B, R, Ms, K, N):
    import torch
    n = B.tl_ag_gemm_workspace_size(R, Ms, K, N)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("R,Ms,K,N,self_rank,splits", [
    (2, 300, 2048, 520, 1, 4),     # 3 x 3 ragged tiles, 32 k-blocks in 4 ranges of 8
    (8, 128, 8192, 1024, 7, 4),    # the smallest sweep point: 16 tiles, 128 k-blocks
    (1, 256, 1024, 256, 0, 2),     # one tile, 16 k-blocks in two ranges
    (3, 100, 1000, 264, 2, 2),     # K tail inside the last range (16 k-blocks, the last partial)
    (3, 100, 136, 264, 1, 1),      # too few k-blocks to split: the workspace is left unused
    (64, 4, 8192, 256, 37, 16),    # the most ranks and the most splits: one tile over 64 shards, 16 ranges
])
def test_ag_splitk_parity(B, R, Ms, K, N, self_rank, splits):
    n = B.tl_ag_gemm_workspace_size(R, Ms, K, N)
    tiles = -(-R * Ms // 256) * -(-N // 256)
    assert n == (0 if splits == 1 else 1024 + tiles * splits * 256 * 256 * 4)
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=R * 31 + Ms + K)
    r = run_ag(B, A, Bm, self_rank=self_rank, f32=True, trace=True, ws=splitk_ws(B, R, Ms, K, N))
    check_all(B, A, Bm, r, self_rank)


def test_ag_splitk_deterministic_and_stale_counters(B):
    # the sum of the ranges runs in range order whichever finishes last, so two
    # calls give the same bits; counters left at another epoch's values (an
    # aborted call) start over instead of miscounting
    R, Ms, K, N = 2, 300, 2048, 520
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=5)
    ws = splitk_ws(B, R, Ms, K, N)
    r1 = run_ag(B, A, Bm, self_rank=0, ws=ws)
    check_all(B, A, Bm, r1)
    c1 = to_bits(r1["C"]).copy()
    ws[:1024] = 0x37  # every counter 0x37373737: a foreign tag with 0x37 arrivals
    r2 = run_ag(B, A, Bm, self_rank=0, ws=ws)
    check_all(B, A, Bm, r2)
    np.testing.assert_array_equal(to_bits(r2["C"]), c1)
    r3 = run_ag(B, A, Bm, self_rank=0)  # unsplit: the same product up to fp32 rounding
    check_all(B, A, Bm, r3)


@pytest.mark.parametrize("mode,host_ranks", [("pull", ()), ("push", (0, 2)), ("pull", (0, 2))])
def test_ag_splitk_pull_mode_and_host_shards(B, mode, host_ranks):
    # split units of one tile each wait for the tile's rows, whichever path brings them
    R, Ms, K, N = 3, 100, 2048, 264
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=71 + len(host_ranks))
    m = B.TL_MODE_PULL if mode == "pull" else B.TL_MODE_PUSH
    r = run_ag(B, A, Bm, self_rank=1, mode=m, f32=True, trace=True, host_ranks=host_ranks,
               ws=splitk_ws(B, R, Ms, K, N))
    check_all(B, A, Bm, r, self_rank=1)


def test_ag_splitk_rejects_small_workspace(B):
    import torch
    R, Ms, K, N = 2, 300, 2048, 520
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=6)
    small = torch.zeros(B.tl_ag_gemm_workspace_size(R, Ms, K, N) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.TLError) as e:
        run_ag(B, A, Bm, ws=small)
    assert e.value.code == B.TL_ERR_INVALID


def test_ag_max_ranks(B):
    # TL_MAX_RANKS = 64 shards of 16 rows: 64 flags, one 256-row tile per 16 shards
    R, Ms, K, N = 64, 16, 64, 64
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=64)
    r = run_ag(B, A, Bm, self_rank=37, trace=True)
    check_all(B, A, Bm, r, self_rank=37)
