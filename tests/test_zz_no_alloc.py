"""tl_gemm_rs_noalloc: GEMM-ReduceScatter for callers that cannot allocate
device memory (their runtime owns the allocator, or they may only pass the
buffers they already hold).  The entry point takes its scratch from a static
device array inside the library; these tests call it through the C ABI and
check it bit for bit against the allocating entry point tl_gemm_rs on the
same inputs, and against the oracle within the bf16 tolerance.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test before it."""
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


def _allocating_outputs(B, dA, dB, R, M, N):
    import torch
    out = [torch.empty(M // R, N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    ws = torch.empty(B.tl_gemm_rs_workspace_size(R, M, N) // 4, dtype=torch.float32, device="cuda")
    sig = B.Signals(B.tl_gemm_rs_num_flags(R, M, N))
    B.tl_gemm_rs(dA, dB, out, ws, sig, 1)
    assert B.tl_query_status(sig) == (0, -1)
    return out


@pytest.mark.parametrize("R,M,K_r,N", [(4, 1024, 256, 512), (3, 300, 72, 264)])
def test_noalloc_matches_allocating_entry_point_twice(B, R, M, K_r, N):
    """Two calls in a row on different inputs with the same epoch.  The static
    scratch still holds the first call's flags (set for that epoch) and its
    partials, so the second call is right only if the flags are cleared before
    it runs and it waits for its own partials.  Both entry points run the same
    kernel on the same grid, so the outputs must be bit-identical; they are also
    held to the oracle within the bf16 tolerance."""
    import torch
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for call in range(2):
        A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=40 + R + 17 * call)
        dA = [dev_bf16(a) for a in A]
        dB = [dev_bf16(b) for b in Bl]
        ref = _allocating_outputs(B, dA, dB, R, M, N)
        want = oracle.gemm_rs.gemm_rs(A, Bl)
        out = [torch.full((M // R, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        B.tl_gemm_rs_noalloc(dA, dB, out, epoch=1, dev_status=status)
        torch.cuda.synchronize()
        assert status.cpu().tolist() == [0, 0, 0, 0]
        for d in range(R):
            assert torch.equal(out[d].view(torch.int16), ref[d].view(torch.int16)), f"call {call} out[{d}]"
            check_bf16(to_f64(out[d]), want[d], f"call {call} out[{d}]")


def test_noalloc_rejects_a_problem_beyond_the_static_scratch(B):
    # R=32, 8192 rows per destination, N=32768: 8.4M flags do not fit in the
    # static scratch.  The call must refuse before touching any buffer, so one
    # small tensor stands in for every pointer.
    import ctypes
    import torch
    R, M, K_r, N = 32, 32 * 8192, 64, 32768
    t = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    ptrs = (ctypes.c_void_p * R)(*([t.data_ptr()] * R))
    pp = ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p))
    a = B.tl_gemm_rs_args(R=R, M=M, K_r=K_r, N=N, A=pp, B=pp, out=pp, workspace=None, workspace_bytes=0,
                          signals=None, epoch=1, options=0, timeout_ns=0, trace=None)
    rc = B.lib.tl_gemm_rs_noalloc(ctypes.byref(a), None, torch.cuda.current_stream().cuda_stream)
    assert rc == B.TL_ERR_UNSUPPORTED
    assert "static scratch" in B.tl_last_error()


def test_noalloc_rejects_workspace_or_signals(B):
    import torch
    A, Bl = inputs.gemm_rs_inputs(2, 256, 64, 256, seed=1)
    dA = [dev_bf16(a) for a in A]
    dB = [dev_bf16(b) for b in Bl]
    out = [torch.empty(128, 256, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    import ctypes
    pa, pb, po = B._ptr_array(dA), B._ptr_array(dB), B._ptr_array(out)
    ws = torch.empty(1 << 20, dtype=torch.float32, device="cuda")
    a = B.tl_gemm_rs_args(R=2, M=256, K_r=64, N=256, A=ctypes.cast(pa, ctypes.POINTER(ctypes.c_void_p)),
                          B=ctypes.cast(pb, ctypes.POINTER(ctypes.c_void_p)),
                          out=ctypes.cast(po, ctypes.POINTER(ctypes.c_void_p)), workspace=ws.data_ptr(),
                          workspace_bytes=ws.numel() * 4, signals=None, epoch=1, options=0, timeout_ns=0,
                          trace=None)
    assert B.lib.tl_gemm_rs_noalloc(ctypes.byref(a), None, None) == B.TL_ERR_INVALID
