"""The communication halves alone: AllGather with per-chunk signals and the
rank-ordered ReduceScatter, through the C ABI."""
import numpy as np
import pytest

import oracle
from oracle import bf16
from tests.helpers import check_bf16, dev_bf16, pinned_bf16, to_bits, to_f64
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


@pytest.mark.parametrize("R,Ms,K,self_rank,rpb", [(2, 128, 512, 0, 0), (3, 100, 136, 2, 7), (8, 1024, 4096, 5, 0),
                                                   (64, 8, 64, 40, 0)])
def test_allgather_bit_exact_and_flags(B, R, Ms, K, self_rank, rpb):
    import torch
    A = [inputs.normal_bf16((Ms, K), 70 + r) for r in range(R)]
    G = torch.full((R * Ms, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    nflags, _ = B.tl_ag_gemm_num_flags(R, Ms, K, rpb)
    sig = B.Signals(nflags)
    B.tl_allgather([dev_bf16(a) for a in A], G, sig, 3, self_rank=self_rank, rows_per_barrier=rpb)
    assert B.tl_query_status(sig) == (0, -1)
    np.testing.assert_array_equal(to_bits(G), oracle.ag_gemm.gathered(A))
    assert np.all(sig.read_flags() == 3)


@pytest.mark.parametrize("host_ranks", [[1, 2], [0, 1, 2, 3]])
def test_allgather_pinned_host_shards_bit_exact(B, host_ranks):
    # shards in pinned host memory are copied with plain loads; the result is the same gather
    import torch
    R, Ms, K = 4, 200, 392
    A = [inputs.normal_bf16((Ms, K), 110 + r) for r in range(R)]
    src = [pinned_bf16(a) if r in host_ranks else dev_bf16(a) for r, a in enumerate(A)]
    G = torch.full((R * Ms, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    nflags, _ = B.tl_ag_gemm_num_flags(R, Ms, K, 9)
    sig = B.Signals(nflags)
    B.tl_allgather(src, G, sig, 5, self_rank=1, rows_per_barrier=9)
    assert B.tl_query_status(sig) == (0, -1)
    np.testing.assert_array_equal(to_bits(G), oracle.ag_gemm.gathered(A))
    assert np.all(sig.read_flags() == 5)


def test_allgather_rejects_pageable_host_shard_without_launch(B):
    import torch
    A = [inputs.normal_bf16((64, 256), 120 + r) for r in range(2)]
    src = [dev_bf16(A[0]), inputs.to_torch_bf16(A[1])]  # second shard: pageable host memory
    G = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    nflags, _ = B.tl_ag_gemm_num_flags(2, 64, 256)
    sig = B.Signals(nflags)
    with pytest.raises(B.TLError) as e:
        B.tl_allgather(src, G, sig, 1)
    assert e.value.code == B.TL_ERR_UNSUPPORTED and "pageable" in str(e.value)
    assert np.all(sig.read_flags() == 0)


def test_allgather_pull_waits_for_source(B):
    import torch
    A = [inputs.normal_bf16((64, 256), 90 + r) for r in range(4)]
    nflags, _ = B.tl_ag_gemm_num_flags(4, 64, 256)
    sig, ready = B.Signals(nflags), B.Signals(nflags)
    G = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    B.tl_tile_notify(ready, 0, nflags, 1)
    B.tl_allgather([dev_bf16(a) for a in A], G, sig, 1, mode=B.TL_MODE_PULL, src_ready=ready)
    assert B.tl_query_status(sig) == (0, -1)
    np.testing.assert_array_equal(to_bits(G), oracle.ag_gemm.gathered(A))
    # epoch 2 with one source chunk left at epoch 1: that copy times out, the rest completes
    B.tl_tile_notify(ready, 0, nflags, 2)
    B.tl_tile_notify(ready, nflags - 1, 1, 1)
    B.tl_allgather([dev_bf16(a) for a in A], G, sig, 2, mode=B.TL_MODE_PULL, src_ready=ready, timeout_ns=20_000_000)
    code, where = B.tl_query_status(sig)
    assert code == B.TL_ERR_TIMEOUT and where == nflags - 1
    assert int(sig.read_flags()[nflags - 1]) == 1


def _rank_order_fp32_sum_bf16(parts):
    """The definition written out: fp32 sums in rank order, then one bf16 rounding."""
    acc = parts[0].astype(np.float32)
    for p in parts[1:]:
        acc = (acc + p.astype(np.float32)).astype(np.float32)
    return bf16.encode_rne(acc.astype(np.float64))


@pytest.mark.parametrize("R,M,N", [(2, 64, 64), (8, 1024, 512), (3, 300, 264)])
def test_reduce_scatter_bit_exact(B, R, M, N):
    import torch
    rng = np.random.default_rng(R + M)
    parts = [rng.standard_normal((M, N)).astype(np.float32) * (r + 1) for r in range(R)]
    dparts = [torch.from_numpy(p).cuda() for p in parts]
    out = [torch.full((M // R, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    B.tl_reduce_scatter(dparts, out)
    want = _rank_order_fp32_sum_bf16(parts)
    got = np.concatenate([to_bits(o) for o in out])
    np.testing.assert_array_equal(got, want)


def test_decomposed_gemm_rs_matches_oracle(B):
    # separate per-rank GEMMs with fp32 partials, then the ReduceScatter: the decomposed schedule
    import torch
    R, M, K_r, N = 4, 512, 256, 512
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=17)
    sig = B.Signals(1)
    parts = [torch.empty(M, N, dtype=torch.float32, device="cuda") for _ in range(R)]
    for r in range(R):
        B.tl_gemm(dev_bf16(A[r]), dev_bf16(Bl[r]), None, sig, C_f32=parts[r])
    out = [torch.empty(M // R, N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    B.tl_reduce_scatter(parts, out)
    assert B.tl_query_status(sig) == (0, -1)
    for d, w in enumerate(oracle.gemm_rs.gemm_rs(A, Bl)):
        check_bf16(to_f64(out[d]), w, f"out[{d}]")
