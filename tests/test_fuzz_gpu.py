"""Seeded random shapes for the three fused calls against the oracle.

The shapes are drawn from one fixed seed, so every run checks the same cases:
rank counts 1-16, ragged row counts, K and N any multiple of 8, random caller
rank, push or pull, either swizzle, split-K workspaces where the call accepts
one, GEMM-RS's partial and order options, MoE with 1-40 experts and top-1 to
top-4.  Each case runs the same checks as the hand-picked parity tests
(gathered rows, flags, tile tables and traces bit-exact; outputs within the
bf16 tolerance of the float64 oracle)."""
import numpy as np
import pytest

import oracle
from tests.helpers import check_bf16, to_f64
from tests.test_ag_gemm_gpu import check_all, run_ag
from tests.test_gemm_rs_gpu import check as check_rs
from tests.test_gemm_rs_gpu import check_flags, run_rs
from tests.test_moe_gpu import check_moe, run_moe
from tile_centric_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

N_CASES = 10


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding
    return binding


def _cases(seed, draw):
    rng = np.random.default_rng(seed)
    return [draw(rng) for _ in range(N_CASES)]


def _ag_case(rng):
    R = int(rng.integers(1, 17))
    Ms = int(rng.integers(1, 1 + 2048 // R))
    K = 8 * int(rng.integers(1, 97))
    N = 8 * int(rng.integers(1, 81))
    return dict(R=R, Ms=Ms, K=K, N=N, self_rank=int(rng.integers(0, R)), pull=bool(rng.integers(0, 2)),
                rows=bool(rng.integers(0, 2)), rpb=int(rng.choice([0, 1, 3, 16, 64])), splitk=bool(rng.integers(0, 2)))


def _rs_case(rng):
    R = int(rng.integers(1, 17))
    M = R * int(rng.integers(1, 1 + 2048 // R))
    return dict(R=R, M=M, K_r=8 * int(rng.integers(1, 65)), N=8 * int(rng.integers(1, 81)),
                options=int(rng.integers(0, 4)))


def _moe_case(rng):
    E = int(rng.integers(1, 41))
    return dict(R=int(rng.integers(1, 9)), T_r=int(rng.integers(1, 257)), H=8 * int(rng.integers(1, 65)),
                N=8 * int(rng.integers(1, 61)), E=E, k=int(rng.integers(1, min(4, E) + 1)),
                pull=bool(rng.integers(0, 2)), rpb=int(rng.choice([0, 1, 5, 32])))


AG_CASES = _cases(1201, _ag_case)
RS_CASES = _cases(1202, _rs_case)
MOE_CASES = _cases(1203, _moe_case)


@pytest.mark.parametrize("c", AG_CASES, ids=[str(i) for i in range(N_CASES)])
def test_fuzz_ag_gemm(B, c):
    import torch
    A, Bm = inputs.ag_gemm_inputs(c["R"], c["Ms"], c["K"], c["N"], "normal", seed=3000 + c["R"] * 7 + c["Ms"])
    ws = None
    if c["splitk"]:
        n = B.tl_ag_gemm_workspace_size(c["R"], c["Ms"], c["K"], c["N"])
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda") if n else None
    r = run_ag(B, A, Bm, self_rank=c["self_rank"], mode=B.TL_MODE_PULL if c["pull"] else B.TL_MODE_PUSH,
               rpb=c["rpb"], trace=not c["rows"], swizzle=B.TL_SWIZZLE_ROWS if c["rows"] else B.TL_SWIZZLE_ARRIVAL,
               ws=ws)
    check_all(B, A, Bm, r, c["self_rank"])


@pytest.mark.parametrize("c", RS_CASES, ids=[str(i) for i in range(N_CASES)])
def test_fuzz_gemm_rs(B, c):
    R, M, K_r, N, options = c["R"], c["M"], c["K_r"], c["N"], c["options"]
    A, Bl = inputs.gemm_rs_inputs(R, M, K_r, N, seed=4000 + R * 11 + M)
    r = run_rs(B, A, Bl, options=options)
    if options == 0:
        check_rs(B, A, Bl, r)
        return
    assert r["status"] == (0, -1), r["status"]
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
        # the bound of the bf16-partials parity test: one bf16 step of each partial,
        # plus the final rounding
        bound = 2.0 ** -7 * mag[d * Md:(d + 1) * Md] + 2.0 ** -8 * np.abs(o) + 1e-3 * np.abs(o).max()
        assert np.all(np.abs(got - o) <= bound), f"out[{d}]: max excess {np.max(np.abs(got - o) - bound):.3e}"
    check_flags(r)


@pytest.mark.parametrize("c", MOE_CASES, ids=[str(i) for i in range(N_CASES)])
def test_fuzz_moe(B, c):
    X, ids, W = inputs.moe_inputs(c["R"], c["T_r"], c["H"], c["N"], c["E"], c["k"], 1.2,
                                  seed=5000 + c["R"] * 13 + c["T_r"])
    self_rank = (c["T_r"] * 7) % c["R"]
    r = run_moe(B, X, ids, W, self_rank=self_rank, rpb=c["rpb"], mode=B.TL_MODE_PULL if c["pull"] else B.TL_MODE_PUSH)
    check_moe(B, X, ids, W, r, self_rank)
