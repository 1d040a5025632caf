"""GEMM-ReduceScatter through the C ABI against the oracle.

Outputs and the receive workspace are poisoned with NaN before every call, so a
reduce that read a partial before its flag was released shows up."""
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


def run_rs(B, A, Bl, *, timeout_ns=0, options=0):
    import torch
    R = len(A)
    M, K_r = A[0].shape
    N = Bl[0].shape[1]
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in Bl]
    out = [torch.full((M // R, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    ws_bytes = B.tl_gemm_rs_workspace_size(R, M, N)
    ws = torch.full((ws_bytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    nflags = B.tl_gemm_rs_num_flags(R, M, N)
    sig = B.Signals(nflags)
    trace = torch.full((nflags,), -1, dtype=torch.int32, device="cuda")
    _epoch[0] += 1
    B.tl_gemm_rs(dA, dB, out, ws, sig, _epoch[0], timeout_ns=timeout_ns, trace=trace, options=options)
    status = B.tl_query_status(sig)
    return dict(out=out, sig=sig, status=status, epoch=_epoch[0], nflags=nflags, items=nflags // 4, trace=trace)


def expected_trace(R, M, N, options=0):
    """Production order of tl_gemm_rs: the chain accumulation, in rank or ring order."""
    Mt, Nt = -(-(M // R) // 256), -(-N // 256)
    order = "ring" if options & 2 else "rank"
    items = oracle.gemm_rs.chain_order(R, M, N, 256, 256, order=order)
    return [((d * Mt + m) * Nt + n) * R + r for (_, d, m, n, r) in items]


def check_flags(r):
    """Every arrival and reduced flag holds the call's epoch."""
    assert np.all(r["sig"].read_flags()[:r["nflags"]] == r["epoch"])


def check(B, A, Bl, r):
    assert r["status"] == (0, -1), r["status"]
    want = oracle.gemm_rs.gemm_rs(A, Bl)
    for d, (o, w) in enumerate(zip(r["out"], want)):
        check_bf16(to_f64(o), w, f"out[{d}]")
    check_flags(r)
    R, M, N = len(A), A[0].shape[0], Bl[0].shape[1]
    assert r["trace"].cpu().tolist()[:r["items"]] == expected_trace(R, M, N)


@pytest.mark.parametrize("R,M,K_r,N", [
    (2, 256, 128, 256),
    (3, 300, 72, 264),      # ragged rows per destination, K and N tails
    (8, 2048, 256, 512),
    (1, 200, 64, 136),      # one rank: plain GEMM, bf16 out
    (5, 5 * 130, 520, 72),  # R that does not divide the tile height
    (4, 4, 8, 8),           # smallest shapes: one row per destination, K_r = N = 8
])
def test_rs_parity(B, R, M, K_r, N):
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=R * 7 + M)
    r = run_rs(B, A, Bl)
    check(B, A, Bl, r)


def test_rs_sums_partials_in_rank_order(B):
    # P_0 = 2^24, P_1 = 1, P_2 = -2^24 in every element (exact tensor-core products).
    # In fp32, ((2^24 + 1) + -2^24) = 0 because 2^24 + 1 rounds to 2^24; every
    # other order gives 1.  The output must be exactly 0.
    R, M, K_r, N = 3, 384, 8, 256
    vals = [(2.0 ** 12, 2.0 ** 12), (1.0, 1.0), (-(2.0 ** 12), 2.0 ** 12)]
    A, Bl = [], []
    for a, b in vals:
        Am = np.zeros((M, K_r), np.float32)
        Am[:, 0] = a
        Bm = np.zeros((K_r, N), np.float32)
        Bm[0, :] = b
        A.append(inputs.bf16_bits_from_f32(Am))
        Bl.append(inputs.bf16_bits_from_f32(Bm))
    r = run_rs(B, A, Bl)
    assert r["status"] == (0, -1)
    p = [np.float32(a * b) for a, b in vals]
    want = np.float32(np.float32(p[0] + p[1]) + p[2])
    assert want == 0.0
    for o in r["out"]:
        assert np.all(to_f64(o) == float(want))


def test_rs_repeated_calls_reuse_signals(B):
    import torch
    R, M, K_r, N = 4, 512, 128, 256
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=3)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in Bl]
    ws = torch.empty(B.tl_gemm_rs_workspace_size(R, M, N) // 4, dtype=torch.float32, device="cuda")
    sig = B.Signals(B.tl_gemm_rs_num_flags(R, M, N))
    want = oracle.gemm_rs.gemm_rs(A, Bl)
    # epochs need only increase between calls on the same signals
    for e in (1, 2, 5, 9):
        ws.fill_(float("nan"))
        out = [torch.full((M // R, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        B.tl_gemm_rs(dA, dB, out, ws, sig, e)
        assert B.tl_query_status(sig) == (0, -1)
        for d in range(R):
            check_bf16(to_f64(out[d]), want[d], f"epoch {e} out[{d}]")


def test_rs_workspace_aligned_to_16_bytes_only(B):
    # the workspace needs only 16-byte alignment
    import torch
    R, M, K_r, N = 4, 1024, 192, 512
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=21)
    n = B.tl_gemm_rs_workspace_size(R, M, N) // 4
    ws = torch.full((n + 64,), float("nan"), dtype=torch.float32, device="cuda")[4:4 + n]
    assert ws.data_ptr() % 128 == 16
    out = [torch.full((M // R, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    sig = B.Signals(B.tl_gemm_rs_num_flags(R, M, N))
    B.tl_gemm_rs([dev_bf16(a) for a in A], [dev_bf16(b) for b in Bl], out, ws, sig, 1)
    assert B.tl_query_status(sig) == (0, -1)
    want = oracle.gemm_rs.gemm_rs(A, Bl)
    for d in range(R):
        check_bf16(to_f64(out[d]), want[d], f"out[{d}]")


def test_rs_rejects_bad_arguments(B):
    import torch
    A, Bl = inputs.gemm_rs_inputs(2, 256, 64, 256, seed=1)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in Bl]
    out = [torch.empty(128, 256, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ws = torch.empty(16, dtype=torch.float32, device="cuda")   # far too small
    sig = B.Signals(B.tl_gemm_rs_num_flags(2, 256, 256))
    with pytest.raises(B.TLError) as e:
        B.tl_gemm_rs(dA, dB, out, ws, sig, 1)
    assert e.value.code == B.TL_ERR_INVALID and "workspace" in str(e.value)


@pytest.mark.slow
def test_rs_llm_full_size_sampled(B):
    c = inputs.CONFIGS["rs_llm"]
    R, M, K_r, N = c["R"], c["M"], c["K_r"], c["N"]
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=0)
    r = run_rs(B, A, Bl)
    assert r["status"] == (0, -1)
    check_flags(r)
    assert r["trace"].cpu().tolist()[:r["items"]] == expected_trace(R, M, N)
    rng = np.random.default_rng(2)
    rows = np.concatenate([rng.integers(0, M, 2500), [0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 2500), [N - 1, 0]])
    want = oracle.gemm_rs.gemm_rs_at(A, Bl, rows, cols)
    Md = M // R
    full = [to_f64(o) for o in r["out"]]
    got = np.array([full[row // Md][row % Md, col] for row, col in zip(rows, cols)])
    check_bf16(got, want, "sampled")
    assert all(np.isfinite(f).all() for f in full)


@pytest.mark.slow
def test_rs_mid_size_sampled(B):
    # R=8, M=4096, K_r=1792, N=4096: 0.8 GB on the device, inputs larger than L2
    R, M, K_r, N = 8, 4096, 1792, 4096
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=11)
    r = run_rs(B, A, Bl)
    assert r["status"] == (0, -1)
    rng = np.random.default_rng(3)
    rows, cols = rng.integers(0, M, 1500), rng.integers(0, N, 1500)
    want = oracle.gemm_rs.gemm_rs_at(A, Bl, rows, cols)
    Md = M // R
    full = [to_f64(o) for o in r["out"]]
    check_bf16(np.array([full[row // Md][row % Md, col] for row, col in zip(rows, cols)]), want, "sampled")


def test_rs_ring_order_sums_from_the_next_rank(B):
    # P_0 = 1, P_1 = 2^24, P_2 = -2^24, P_3 = 0 in every element.  Destination d adds
    # ranks d+1, d+2, d+3, d; in fp32 (1 + 2^24) rounds to 2^24, so a row is 0 exactly
    # when 1 and 2^24 are both added before -2^24:
    #   d=0: 2^24, -2^24, 0, 1 -> 1     d=1: -2^24, 0, 1, 2^24 -> 1
    #   d=2: 0, 1, 2^24, -2^24 -> 0     d=3: 1, 2^24, -2^24, 0 -> 0
    R, M, K_r, N = 4, 1024, 8, 256
    vals = [(1.0, 1.0), (2.0 ** 12, 2.0 ** 12), (-(2.0 ** 12), 2.0 ** 12), (0.0, 0.0)]
    A, Bl = [], []
    for a, b in vals:
        Am = np.zeros((M, K_r), np.float32)
        Am[:, 0] = a
        Bm = np.zeros((K_r, N), np.float32)
        Bm[0, :] = b
        A.append(inputs.bf16_bits_from_f32(Am))
        Bl.append(inputs.bf16_bits_from_f32(Bm))
    r = run_rs(B, A, Bl, options=B.TL_RS_RING_ORDER)
    assert r["status"] == (0, -1)
    p = [np.float32(a * b) for a, b in vals]
    for d, want in enumerate([1.0, 1.0, 0.0, 0.0]):
        acc = None
        for i in range(R):
            x = p[(d + 1 + i) % R]
            acc = x if acc is None else np.float32(acc + x)
        assert float(acc) == want
        assert np.all(to_f64(r["out"][d]) == want), d
    check_flags(r)


@pytest.mark.parametrize("R,M,K_r,N,options", [(4, 1024, 256, 512, 1), (3, 300, 72, 264, 1), (4, 1024, 256, 512, 3),
                                               (8, 2048, 128, 264, 2)])
def test_rs_bf16_partials_and_ring_order_parity(B, R, M, K_r, N, options):
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=60 + R + options)
    r = run_rs(B, A, Bl, options=options)
    assert r["status"] == (0, -1)
    parts = "bf16" if options & B.TL_RS_BF16_PARTIALS else "f32"
    order = "ring" if options & B.TL_RS_RING_ORDER else "rank"
    want = oracle.gemm_rs.gemm_rs_variant(A, Bl, parts, order)
    mag = oracle.gemm_rs.partial_abs_sum(A, Bl)
    Md = M // R
    for d in range(R):
        got, o = to_f64(r["out"][d]), want[d]
        assert np.isfinite(got).all()
        if parts == "f32":
            check_bf16(got, o, f"out[{d}]")
            continue
        # a partial rounded to bf16 on the GPU (from an fp32 accumulation) may land one
        # bf16 step away from the exact partial rounded, a step being at most 2^-7 |P_r|;
        # the final rounding adds 2^-9 |o|
        bound = 2.0 ** -7 * mag[d * Md:(d + 1) * Md] + 2.0 ** -8 * np.abs(o) + 1e-3 * np.abs(o).max()
        assert np.all(np.abs(got - o) <= bound), f"out[{d}]: max excess {np.max(np.abs(got - o) - bound):.3e}"
        assert np.abs(got - o).max() / np.abs(o).max() <= 2e-2
    check_flags(r)


def test_rs_max_ranks(B):
    # the largest rank count, 32: four rows per reducer slice of a 128-row half tile;
    # one more rank is rejected before any launch
    R, M, K_r, N = 32, 1024, 32, 256
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=320)
    r = run_rs(B, A, Bl)
    check(B, A, Bl, r)
    A, Bl = inputs.gemm_rs_inputs(33, 33 * 8, 32, 256, seed=330)
    with pytest.raises(B.TLError) as e:
        run_rs(B, A, Bl)
    assert e.value.code == B.TL_ERR_UNSUPPORTED
