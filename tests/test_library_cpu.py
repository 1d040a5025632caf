"""The C-ABI library on a machine without a GPU: it loads, exports every entry
point include/tilelink.h declares, and its host-side bookkeeping (tile orders,
flag counts, argument validation) matches the oracle bit for bit."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        names += re.findall(r"\b(tl_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(B):
    names = declared_functions()
    assert "tl_ag_gemm" in names and "tl_tile_wait" in names
    missing = [n for n in names if not hasattr(B.lib, n)]
    assert not missing, missing
    assert sorted(B.EXPORTED) == names


def test_version(B):
    assert B.tl_version() == 1


def test_ag_tile_order_matches_oracle(B):
    import oracle
    for (R, s, Ms) in [(2, 0, 128), (8, 0, 1024), (8, 3, 1024), (3, 1, 100), (5, 4, 77), (1, 0, 300), (4, 2, 256)]:
        got = B.tl_ag_gemm_tile_order(R, s, Ms)
        Mt = -(-R * Ms // 256)
        want = [m for (m, n) in oracle.ag_gemm.consumer_order(R, s, Ms, 256, 256, 256)]
        assert got == want[:Mt] and len(got) == Mt


def test_ag_num_flags(B):
    assert B.tl_ag_gemm_num_flags(8, 1024, 4096) == (8 * 64, 16)   # default: about 128 KB of A per chunk
    assert B.tl_ag_gemm_num_flags(2, 128, 512) == (2 * 1, 128)
    assert B.tl_ag_gemm_num_flags(3, 100, 136, 16) == (3 * 7, 16)
    assert B.tl_ag_gemm_num_flags(2, 10, 8, 0)[1] == 10   # capped at the shard


def test_splitk_workspace_sizes(B):
    # 152 SMs = 76 CTA pairs; tiles are 256 x 256, k-blocks 64 deep.  The split S
    # is the largest <= 16 dividing the k-blocks with >= 8 k-blocks per split and
    # tiles * S <= 76; the workspace is 1 KB of counters plus tiles * S fp32 tiles.
    tile_bytes = 256 * 256 * 4
    # M=1024, N=1024: 16 tiles; K=8192: 128 k-blocks -> S=4 (16 * 4 = 64 <= 76)
    assert B.tl_gemm_workspace_size(1024, 1024, 8192, 152) == 1024 + 16 * 4 * tile_bytes
    assert B.tl_ag_gemm_workspace_size(8, 128, 8192, 1024, 152) == 1024 + 16 * 4 * tile_bytes
    # 32 tiles -> S=2
    assert B.tl_gemm_workspace_size(2048, 1024, 8192, 152) == 1024 + 32 * 2 * tile_bytes
    # ragged: 600 x 520 is 3 x 3 tiles; K=2048 is 32 k-blocks -> S=4 (S=8 would leave 4 k-blocks)
    assert B.tl_ag_gemm_workspace_size(2, 300, 2048, 520, 152) == 1024 + 9 * 4 * tile_bytes
    # K=1000: 16 k-blocks -> S=2 (16 / 2 = 8), even for one tile
    assert B.tl_gemm_workspace_size(104, 104, 1000, 152) == 1024 + 1 * 2 * tile_bytes
    # no split: tiles fill the pairs, or too few k-blocks, or bad shapes
    assert B.tl_gemm_workspace_size(8192, 1792, 4096, 152) == 0      # 224 tiles
    assert B.tl_gemm_workspace_size(4096, 1024, 8192, 152) == 0      # 64 tiles: S=2 would need 128 units
    assert B.tl_gemm_workspace_size(1024, 1024, 512, 152) == 0       # 8 k-blocks
    assert B.tl_gemm_workspace_size(0, 1024, 8192, 152) == 0
    assert B.tl_ag_gemm_workspace_size(0, 128, 8192, 1024, 152) == 0
    # fewer SMs, fewer splits: 20 SMs = 10 pairs, 4 tiles -> S=2
    assert B.tl_gemm_workspace_size(512, 512, 8192, 20) == 1024 + 4 * 2 * tile_bytes


def test_ag_attn_num_flags(B):
    # one K and one V flag per 128-token chunk of every rank's shard
    assert B.tl_ag_attn_num_flags(8, 8192) == 2 * 8 * 64
    assert B.tl_ag_attn_num_flags(3, 300) == 2 * 3 * 3
    assert B.tl_ag_attn_num_flags(8, 1) == 2 * 8
    assert B.tl_ag_attn_num_flags(0, 5) == -1 and B.tl_ag_attn_num_flags(2, 0) == -1


def test_ag_attn_rejects_null_and_empty_without_launch(B):
    a = B.tl_ag_attn_args(R=2, self_rank=0, S_shard=0, H=4, H_kv=2, head_dim=128, causal=0, scale=0.0, epoch=1)
    assert B.lib.tl_ag_attn(ctypes.byref(a), None) == B.TL_ERR_INVALID
    a.S_shard = 16
    assert B.lib.tl_ag_attn(ctypes.byref(a), None) == B.TL_ERR_INVALID  # NULL tensors
    assert B.lib.tl_ag_attn(None, None) == B.TL_ERR_INVALID


def test_invalid_arguments_fail_without_launch(B):
    with pytest.raises(B.TLError) as e:
        B.lib_call = B.lib.tl_ag_gemm(None, None)
        B._check(B.lib_call)
    assert e.value.code == B.TL_ERR_INVALID
    h = ctypes.c_void_p()
    assert B.lib.tl_signals_create(0, ctypes.byref(h)) == B.TL_ERR_INVALID
    assert "num_flags" in B.tl_last_error()


def test_ag_gemm_rejects_unknown_swizzle_without_launch(B):
    # argument checks run before any device query, so this needs no GPU
    ptrs = (ctypes.c_void_p * 2)(16, 32)
    a = B.tl_ag_gemm_args(R=2, self_rank=0, M_shard=128, K=256, N=256, mode=B.TL_MODE_PUSH, rows_per_barrier=0,
                          swizzle=7, A_shards=ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)), B=48,
                          gathered=64, C=80, C_f32=None, signals=96, src_ready=None, epoch=1, reserved1=0,
                          timeout_ns=0, trace=None)
    assert B.lib.tl_ag_gemm(ctypes.byref(a), None) == B.TL_ERR_INVALID
    assert "swizzle" in B.tl_last_error()


def test_gemm_rs_rejects_unknown_options_without_launch(B):
    ptrs = (ctypes.c_void_p * 2)(16, 32)
    pp = ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p))
    a = B.tl_gemm_rs_args(R=2, M=256, K_r=64, N=256, A=pp, B=pp, out=pp, workspace=48, workspace_bytes=1 << 30,
                          signals=64, epoch=1, options=8, timeout_ns=0, trace=None)
    assert B.lib.tl_gemm_rs(ctypes.byref(a), None) == B.TL_ERR_INVALID
    assert "options" in B.tl_last_error()


def test_splitk_workspace_alignment_checked_without_launch(B):
    # a split-K workspace must be 16-byte aligned; the check runs before any device query
    ptrs = (ctypes.c_void_p * 2)(16, 32)
    a = B.tl_ag_gemm_args(R=2, self_rank=0, M_shard=128, K=8192, N=256, mode=B.TL_MODE_PUSH, rows_per_barrier=0,
                          swizzle=0, A_shards=ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)), B=48,
                          gathered=64, C=80, C_f32=None, signals=96, src_ready=None, epoch=1, reserved1=0,
                          timeout_ns=0, trace=None, workspace=104, workspace_bytes=1 << 30)
    assert B.lib.tl_ag_gemm(ctypes.byref(a), None) == B.TL_ERR_INVALID
    assert "aligned" in B.tl_last_error()
    g = B.tl_gemm_args(M=256, N=256, K=8192, reserved0=0, A=16, B=32, C=48, C_f32=None, signals=64, timeout_ns=0,
                       workspace=72, workspace_bytes=1 << 30)
    assert B.lib.tl_gemm(ctypes.byref(g), None) == B.TL_ERR_INVALID
    assert "aligned" in B.tl_last_error()


def test_allgather_ll_link_bytes(B):
    # the larger of the two layouts: packed words (8 bytes per 4 data bytes), or the raw
    # data followed by one 128-byte flag slot per chunk
    assert B.tl_allgather_ll_link_bytes(8, 1024, 4096) == 2 * 8 * 1024 * 4096 * 2
    assert B.tl_allgather_ll_link_bytes(2, 1, 8) == max(2 * 2 * 16, 2 * 16 + 2 * 128)
    assert B.tl_allgather_ll_link_bytes(3, 37, 136, 5) == max(2 * 3 * 37 * 136 * 2, 3 * 37 * 136 * 2 + 3 * 8 * 128)
    assert B.tl_allgather_ll_link_bytes(0, 1, 8) == 0


def test_allgather_ll_rejects_bad_arguments_without_a_device(B):
    # argument errors come back before any device query or launch
    shard = (ctypes.c_void_p * 2)(16, 32)
    pp = ctypes.cast(shard, ctypes.POINTER(ctypes.c_void_p))

    def args(**kw):
        a = dict(R=2, self_rank=0, M_shard=4, K=64, protocol=0, rows_per_barrier=0, A_shards=pp, link=64,
                 link_bytes=1 << 20, gathered=128, signals=256, send_mask=3, epoch=1, reserved0=0, timeout_ns=0)
        a.update(kw)
        return B.tl_allgather_ll_args(**a)
    for kw, code in [(dict(K=60), B.TL_ERR_UNSUPPORTED), (dict(protocol=2), B.TL_ERR_INVALID),
                     (dict(epoch=0), B.TL_ERR_INVALID), (dict(link=None), B.TL_ERR_INVALID),
                     (dict(link_bytes=100), B.TL_ERR_INVALID), (dict(link=72), B.TL_ERR_INVALID),
                     (dict(self_rank=2), B.TL_ERR_INVALID), (dict(R=65), B.TL_ERR_INVALID)]:
        a = args(**kw)
        assert B.lib.tl_allgather_ll(ctypes.byref(a), None) == code, kw
    assert B.lib.tl_allgather_ll(None, None) == B.TL_ERR_INVALID


def test_moe_down_sizes(B):
    # the chain schedule's workspace: an fp32 running sum per output tile (max_tiles x
    # ceil(Hd/256) tiles of 256 x 256, 256-byte aligned), then Y [P, Hd] fp32; one flag per
    # pass and 128-row half of every output tile
    def max_tiles(P, E):
        return -(-P // 256) + E
    for (R, T_r, k, E, Hd) in [(8, 1024, 2, 32, 4096), (3, 100, 3, 6, 136), (1, 1, 1, 1, 8), (32, 4, 2, 64, 8)]:
        P = R * T_r * k
        tiles = max_tiles(P, E) * -(-Hd // 256)
        sums = tiles * 2 * 128 * 256 * 4
        assert B.tl_moe_down_workspace_size(R, T_r, k, E, Hd) == -(-sums // 256) * 256 + P * Hd * 4
        assert B.tl_moe_down_num_flags(R, T_r, k, E, Hd) == 2 * R * tiles
    assert B.tl_moe_down_workspace_size(0, 1, 1, 1, 8) == 0
    assert B.tl_moe_down_num_flags(1, 0, 1, 1, 8) == -1
