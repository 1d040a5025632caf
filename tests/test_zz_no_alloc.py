"""tl_gemm_rs_noalloc: GEMM-ReduceScatter for callers that cannot allocate
device memory (their runtime owns the allocator, or they may only pass the
buffers they already hold).  The entry point takes its scratch from a static
device array inside the library; these tests call it through the C ABI and
check it against the allocating entry point tl_gemm_rs on the same inputs.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test before it."""
import numpy as np
import pytest

from tests.helpers import check_bf16, dev_bf16, to_f64
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


def _reference_outputs(B, dA, dB, R, M, N):
    import torch
    out = [torch.empty(M // R, N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    ws = torch.empty(B.tl_gemm_rs_workspace_size(R, M, N) // 4, dtype=torch.float32, device="cuda")
    sig = B.Signals(B.tl_gemm_rs_num_flags(R, M, N))
    B.tl_gemm_rs(dA, dB, out, ws, sig, 1)
    assert B.tl_query_status(sig) == (0, -1)
    return out


@pytest.mark.parametrize("R,M,K_r,N", [(4, 1024, 256, 512), (3, 300, 72, 264)])
def test_noalloc_matches_allocating_entry_point_twice(B, R, M, K_r, N):
    import torch
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=40 + R)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in Bl]
    ref = [to_f64(o) for o in _reference_outputs(B, dA, dB, R, M, N)]
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for call in range(2):   # the second call runs on the scratch the first one left behind
        out = [torch.full((M // R, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        B.tl_gemm_rs_noalloc(dA, dB, out, epoch=call + 1, dev_status=status)
        torch.cuda.synchronize()
        assert status.cpu().tolist() == [0, 0, 0, 0]
        for d in range(R):
            check_bf16(to_f64(out[d]), ref[d], f"call {call} out[{d}]")


def test_noalloc_rejects_a_problem_beyond_the_static_scratch(B):
    import torch
    R, M, K_r, N = 8, 8192, 64, 4096           # needs ~1 GiB of receive slots
    A = [torch.zeros(M, K_r, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    Bl = [torch.zeros(K_r, N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    out = [torch.zeros(M // R, N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    with pytest.raises(B.TLError) as e:
        B.tl_gemm_rs_noalloc(A, Bl, out, epoch=1)
    assert e.value.code == B.TL_ERR_UNSUPPORTED and "static scratch" in str(e.value)
