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
    assert B.tl_ag_gemm_num_flags(8, 1024, 4096) == (8 * 256, 4)
    assert B.tl_ag_gemm_num_flags(2, 128, 512) == (2 * 4, 32)
    assert B.tl_ag_gemm_num_flags(3, 100, 136, 16) == (3 * 7, 16)
    assert B.tl_ag_gemm_num_flags(2, 10, 8, 0)[1] == 10   # capped at the shard


def test_invalid_arguments_fail_without_launch(B):
    with pytest.raises(B.TLError) as e:
        B.lib_call = B.lib.tl_ag_gemm(None, None)
        B._check(B.lib_call)
    assert e.value.code == B.TL_ERR_INVALID
    h = ctypes.c_void_p()
    assert B.lib.tl_signals_create(0, ctypes.byref(h)) == B.TL_ERR_INVALID
    assert "num_flags" in B.tl_last_error()
