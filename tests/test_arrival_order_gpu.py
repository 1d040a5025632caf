"""Race exposure: chunks forced to arrive out of the order their consumers take
them in (tl_test_hold_chunks), so a missing or misplaced wait would show up as
a wrong result instead of passing by luck.  Each case holds back the chunks the
consumers want first -- the AllGather-GEMM's shard self+1 (first in the
arrival-ordered swizzle), the MoE pull mode's first chunk of sorted rows, the
MoE push mode's self shard -- and must still give the oracle's results, the
gathered bytes bit for bit, the static consumer order, every flag set and no
timeout.  Every call also checks that it took at least the hold, so the hold
did take effect."""
import time

import numpy as np
import pytest

import oracle
from tests.helpers import to_bits
from tests.test_ag_gemm_gpu import check_all, run_ag
from tests.test_moe_gpu import check_moe, run_moe
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

HOLD_NS = 30_000_000  # 30 ms: far longer than any copy here, far below the 1 s waits


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    yield binding
    binding.tl_test_hold_chunks(0, 0, 0)


def held(B, first, count, fn):
    B.tl_test_hold_chunks(first, count, HOLD_NS)
    try:
        t0 = time.perf_counter()
        r = fn()
        dt = time.perf_counter() - t0
    finally:
        B.tl_test_hold_chunks(0, 0, 0)
    assert dt >= 0.9 * HOLD_NS * 1e-9, f"the held call took {dt * 1e3:.1f} ms"
    return r


@pytest.mark.parametrize("R,Ms,K,N,self_rank,mode", [(8, 256, 512, 512, 0, "push"), (8, 256, 512, 512, 5, "pull"),
                                                     (3, 100, 136, 264, 1, "push"), (4, 1024, 1024, 768, 2, "pull")])
def test_ag_gemm_first_consumed_shard_arrives_last(B, R, Ms, K, N, self_rank, mode):
    A, Bm = inputs.ag_gemm_inputs(R, Ms, K, N, "normal", seed=1300 + R + self_rank)
    m = B.TL_MODE_PUSH if mode == "push" else B.TL_MODE_PULL
    nflags, rpb = B.tl_ag_gemm_num_flags(R, Ms, K)
    bpr = nflags // R
    nxt = (self_rank + 1) % R
    r = held(B, nxt * bpr, bpr, lambda: run_ag(B, A, Bm, self_rank=self_rank, mode=m, trace=True, f32=True))
    check_all(B, A, Bm, r, self_rank)


def test_allgather_first_copied_shard_arrives_last(B):
    import torch
    R, Ms, K, self_rank = 8, 64, 1024, 3
    A = [inputs.normal_bf16((Ms, K), 1340 + r) for r in range(R)]
    G = torch.full((R * Ms, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    nflags, _ = B.tl_ag_gemm_num_flags(R, Ms, K, 8)
    sig = B.Signals(nflags)
    bpr = nflags // R
    dA = [inputs.to_torch_bf16(a).cuda() for a in A]

    def call():
        B.tl_allgather(dA, G, sig, 9, self_rank=self_rank, rows_per_barrier=8)
        return B.tl_query_status(sig)
    assert held(B, ((self_rank + 1) % R) * bpr, bpr, call) == (0, -1)
    np.testing.assert_array_equal(to_bits(G), oracle.ag_gemm.gathered(A))
    assert np.all(sig.read_flags() == 9)


@pytest.mark.parametrize("count", [1, 4])
def test_moe_pull_first_chunks_arrive_last(B, count):
    X, ids, W = inputs.moe_inputs(4, 128, 256, 264, 8, 2, 1.2, seed=1360 + count)
    r = held(B, 0, count, lambda: run_moe(B, X, ids, W, self_rank=1, mode=B.TL_MODE_PULL))
    check_moe(B, X, ids, W, r, self_rank=1)


def test_moe_push_self_shard_arrives_last(B):
    X, ids, W = inputs.moe_inputs(4, 128, 256, 264, 8, 2, 1.2, seed=1370)
    self_rank = 2
    nflags, rpb = B.tl_moe_num_flags(4, 128, 256, 2, 0, B.TL_MODE_PUSH)
    bpr = nflags // 4
    r = held(B, self_rank * bpr, bpr, lambda: run_moe(B, X, ids, W, self_rank=self_rank, mode=B.TL_MODE_PUSH))
    check_moe(B, X, ids, W, r, self_rank=self_rank)


def test_hold_longer_than_half_the_timeout_is_rejected(B):
    A, Bm = inputs.ag_gemm_inputs(2, 128, 256, 256, "normal", seed=1380)
    B.tl_test_hold_chunks(0, 1, 10_000_000)
    try:
        with pytest.raises(B.TLError) as e:
            run_ag(B, A, Bm, timeout_ns=15_000_000)
        assert e.value.code == B.TL_ERR_INVALID
    finally:
        B.tl_test_hold_chunks(0, 0, 0)
    with pytest.raises(B.TLError):
        B.tl_test_hold_chunks(0, 1, 200_000_000)  # above 100 ms
