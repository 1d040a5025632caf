"""Plain GEMM (CTA-pair tcgen05 kernel) through the C ABI against the oracle
(an AllGather-GEMM over one shard is the plain product)."""
import numpy as np
import pytest

import oracle
from tests.helpers import check_bf16, check_f32, dev_bf16, to_bits, to_f64
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


def run_gemm(B, A, Bm, f32=True, ws=None):
    import torch
    M, K = A.shape
    N = Bm.shape[1]
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    C32 = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") if f32 else None
    sig = B.Signals(1)
    B.tl_gemm(dev_bf16(A), dev_bf16(Bm), C, sig, C_f32=C32, workspace=ws)
    assert B.tl_query_status(sig) == (0, -1)
    return C, C32


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (512, 512, 512), (300, 264, 136), (8, 8, 8), (1000, 1032, 520),
                                   (2048, 1792, 4096)])
def test_gemm_parity(B, M, N, K):
    A, Bm = inputs.ag_gemm_inputs(1, M, K, N, "normal", seed=M + N + K)
    C, C32 = run_gemm(B, A[0], Bm)
    want = oracle.ag_gemm.ag_gemm(A, Bm)
    check_bf16(to_f64(C), want, "C")
    check_f32(to_f64(C32), want, "C_f32")


@pytest.mark.parametrize("M,N,K,splits", [
    (1024, 1024, 8192, 4),   # 16 tiles, 128 k-blocks
    (300, 264, 2048, 4),     # 2 x 2 ragged tiles, 32 k-blocks
    (104, 104, 1000, 2),     # one tile, 16 k-blocks with a K tail
    (512, 512, 8192, 16),    # the most splits: 4 tiles x 16, half the splits sum no chunk
    (512, 264, 8192, 16),    # N tail: the second tile column has one chunk for 16 splits
])
def test_gemm_splitk_parity(B, M, N, K, splits):
    import torch
    n = B.tl_gemm_workspace_size(M, N, K)
    assert n == 1024 + -(-M // 256) * -(-N // 256) * splits * 256 * 256 * 4
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    A, Bm = inputs.ag_gemm_inputs(1, M, K, N, "normal", seed=M + N + K + 1)
    C, C32 = run_gemm(B, A[0], Bm, ws=ws)
    want = oracle.ag_gemm.ag_gemm(A, Bm)
    check_bf16(to_f64(C), want, "C")
    check_f32(to_f64(C32), want, "C_f32")
    # the counters reset themselves; a second call gives the same bits
    assert int(ws[:1024].count_nonzero()) == 0
    C2, _ = run_gemm(B, A[0], Bm, f32=False, ws=ws)
    np.testing.assert_array_equal(to_bits(C2), to_bits(C))


def test_gemm_identity_exact(B):
    A = inputs.uniform_bf16((512, 256), 3)
    eye = inputs.bf16_bits_from_f32(np.eye(256, dtype=np.float32))
    C, _ = run_gemm(B, A, eye, f32=False)
    np.testing.assert_array_equal(to_bits(C), A)


@pytest.mark.slow
def test_gemm_llm_shape_sampled(B):
    A, Bm = inputs.ag_gemm_inputs(1, 8192, 4096, 1792, "normal", seed=1)
    C, _ = run_gemm(B, A[0], Bm, f32=False)
    rng = np.random.default_rng(0)
    rows, cols = rng.integers(0, 8192, 3000), rng.integers(0, 1792, 3000)
    check_bf16(to_f64(C)[rows, cols], oracle.ag_gemm.ag_gemm_at(A, Bm, rows, cols), "C sampled")


def test_gemm_splitk_graph_replays(B):
    # a captured call runs again with the same arguments: the last split to depart
    # zeroes the counters, so every replay counts from zero and gives the same bits
    import torch
    M, N, K = 512, 512, 8192
    A, Bm = inputs.ag_gemm_inputs(1, M, K, N, "normal", seed=91)
    dA, dB = dev_bf16(A[0]), dev_bf16(Bm)
    ws = torch.zeros(B.tl_gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    sig = B.Signals(1)
    B.tl_gemm(dA, dB, C, sig, workspace=ws)  # sets the kernel's launch attributes before the capture
    torch.cuda.synchronize()
    want = to_bits(C).copy()
    check_bf16(to_f64(C), oracle.ag_gemm.ag_gemm(A, Bm), "C")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.tl_gemm(dA, dB, C, sig, workspace=ws)
    for _ in range(3):
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert B.tl_query_status(sig) == (0, -1)
        np.testing.assert_array_equal(to_bits(C), want)
        assert int(ws[:1024].count_nonzero()) == 0
