"""AllGather through a slow link with the flag-in-data (low-latency) protocol and
the separate-flag protocol it is compared with, through the C ABI.

`gathered` must equal the oracle's concatenation of the shards bit for bit;
every chunk flag must hold the call's epoch; the link buffer is pinned host
memory (the slow link) or device memory.  The host plays a sending rank by
writing that rank's link words itself, and a rank that nobody sends makes the
receiver's bounded poll run out (TL_ERR_TIMEOUT) without hanging the GPU."""
import numpy as np
import pytest

import oracle
from tests.helpers import dev_bf16, to_bits
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


def link_buffer(B, R, Ms, K, rpb, where):
    import torch
    n = B.tl_allgather_ll_link_bytes(R, Ms, K, rpb)
    t = torch.zeros(n, dtype=torch.uint8)
    return t.pin_memory() if where == "host" else t.cuda()


def nchunks(Ms, K, rpb):
    if rpb <= 0:
        rpb = max(1, min(Ms, 8192 // (2 * K)))
    return -(-Ms // min(rpb, Ms))


def run(B, A, link, epoch, *, protocol, self_rank=0, rpb=0, send_mask=None, timeout_ns=0):
    import torch
    R, (Ms, K) = len(A), A[0].shape
    G = torch.full((R * Ms, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    sig = B.Signals(R * nchunks(Ms, K, rpb))
    B.tl_allgather_ll([dev_bf16(a) for a in A], link, G, sig, epoch, self_rank=self_rank, protocol=protocol,
                      send_mask=send_mask, rows_per_barrier=rpb, timeout_ns=timeout_ns)
    return G, sig, B.tl_query_status(sig)


@pytest.mark.parametrize("protocol", [0, 1])
@pytest.mark.parametrize("where", ["host", "device"])
@pytest.mark.parametrize("R,Ms,K,self_rank,rpb", [(8, 1, 4096, 0, 0), (8, 16, 1024, 5, 0), (3, 37, 136, 2, 5),
                                                  (4, 256, 2048, 1, 0), (64, 2, 64, 40, 1)])
def test_allgather_ll_bit_exact(B, protocol, where, R, Ms, K, self_rank, rpb):
    A = [inputs.normal_bf16((Ms, K), 900 + r) for r in range(R)]
    link = link_buffer(B, R, Ms, K, rpb, where)
    G, sig, st = run(B, A, link, 7, protocol=protocol, self_rank=self_rank, rpb=rpb)
    assert st == (0, -1)
    np.testing.assert_array_equal(to_bits(G), oracle.ag_gemm.gathered(A))
    assert np.all(sig.read_flags() == 7)


@pytest.mark.parametrize("protocol", [0, 1])
def test_allgather_ll_reuses_its_link_buffer(B, protocol):
    # the second call finds the first call's words (an older epoch) in the link and
    # must wait for its own: new inputs, the same link buffer
    R, Ms, K = 8, 4, 512
    link = link_buffer(B, R, Ms, K, 0, "host")
    for call in range(3):
        A = [inputs.normal_bf16((Ms, K), 950 + 10 * call + r) for r in range(R)]
        G, sig, st = run(B, A, link, 20 + call, protocol=protocol, self_rank=call % R)
        assert st == (0, -1)
        np.testing.assert_array_equal(to_bits(G), oracle.ag_gemm.gathered(A))


@pytest.mark.parametrize("protocol", [0, 1])
def test_allgather_ll_host_is_the_sender_of_one_rank(B, protocol):
    # rank 2's link region is written by the host before the launch, in the
    # documented layout; the launch sends the other ranks and receives all of them
    R, Ms, K, epoch, rpb = 4, 6, 256, 31, 2
    A = [inputs.normal_bf16((Ms, K), 970 + r) for r in range(R)]
    link = link_buffer(B, R, Ms, K, rpb, "host")
    ln = link.numpy()
    shard_words = np.ascontiguousarray(A[2]).view(np.uint32).ravel()      # 4-byte data words, row-major
    w0 = 2 * Ms * K * 2 // 4                                              # first word of rank 2's rows
    if protocol == 0:
        packed = (np.uint64(epoch) << np.uint64(32)) | shard_words.astype(np.uint64)
        ln.view(np.uint64)[w0:w0 + shard_words.size] = packed
    else:
        ln.view(np.uint32)[w0:w0 + shard_words.size] = shard_words
        raw = R * Ms * K * 2
        for c in range(nchunks(Ms, K, rpb)):
            ln[raw + (2 * nchunks(Ms, K, rpb) + c) * 128:][:4].view(np.uint32)[0] = epoch
    G, sig, st = run(B, A, link, epoch, protocol=protocol, self_rank=0, rpb=rpb, send_mask=0b1011)
    assert st == (0, -1)
    np.testing.assert_array_equal(to_bits(G), oracle.ag_gemm.gathered(A))


@pytest.mark.parametrize("protocol", [0, 1])
def test_allgather_ll_unsent_rank_times_out(B, protocol):
    # nobody sends rank 3: the receiver's poll of its words runs out after the bound,
    # records TL_ERR_TIMEOUT with a chunk of rank 3, and the context stays usable
    R, Ms, K = 4, 8, 512
    A = [inputs.normal_bf16((Ms, K), 990 + r) for r in range(R)]
    link = link_buffer(B, R, Ms, K, 0, "host")
    _, _, st = run(B, A, link, 5, protocol=protocol, send_mask=0b0111, timeout_ns=20_000_000)
    code, where = st
    assert code == B.TL_ERR_TIMEOUT
    assert where // nchunks(Ms, K, 0) == 3
    G, sig, st = run(B, A, link, 6, protocol=protocol)
    assert st == (0, -1)
    np.testing.assert_array_equal(to_bits(G), oracle.ag_gemm.gathered(A))
