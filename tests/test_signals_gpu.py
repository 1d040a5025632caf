"""Signal primitives on the GPU: notify/wait ordering, epochs, bounded waits."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


def test_notify_then_wait_passes_and_flags_hold_value(B):
    s = B.Signals(100)
    B.tl_tile_notify(s, 10, 50, 7)
    B.tl_tile_wait(s, 10, 50, 7, timeout_ns=100_000_000)
    assert B.tl_query_status(s) == (0, -1)
    f = s.read_flags()
    assert np.all(f[10:60] == 7) and np.all(f[:10] == 0) and np.all(f[60:] == 0)
    # an older epoch is already reached; wrap-safe comparison
    B.tl_tile_wait(s, 10, 50, 5, timeout_ns=100_000_000)
    assert B.tl_query_status(s) == (0, -1)
    s.close()


def test_wait_on_unset_flag_times_out_and_context_stays_usable(B):
    import torch
    s = B.Signals(64)
    B.tl_tile_notify(s, 0, 64, 3)
    B.tl_tile_notify(s, 40, 1, 2)          # flag 40 lags behind epoch 3
    B.tl_tile_wait(s, 0, 64, 3, timeout_ns=20_000_000)
    code, where = B.tl_query_status(s)
    assert code == B.TL_ERR_TIMEOUT and where == 40
    assert B.tl_query_status(s) == (0, -1)  # cleared by the query
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0
    s.close()


def test_epoch_wraparound(B):
    s = B.Signals(4)
    B.tl_tile_notify(s, 0, 4, 0xFFFFFFFF)
    B.tl_tile_wait(s, 0, 4, 0xFFFFFFFE, timeout_ns=50_000_000)
    assert B.tl_query_status(s) == (0, -1)
    B.tl_tile_notify(s, 0, 4, 1)          # 1 is "after" 0xFFFFFFFF mod 2^32
    B.tl_tile_wait(s, 0, 4, 0xFFFFFFFF, timeout_ns=50_000_000)
    assert B.tl_query_status(s) == (0, -1)
    s.close()


def test_reset_zeroes_flags(B):
    s = B.Signals(8)
    B.tl_tile_notify(s, 0, 8, 9)
    B.tl_signals_reset(s)
    assert np.all(s.read_flags() == 0)
    s.close()
