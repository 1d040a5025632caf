"""Host logic of the bench that needs no GPU: which step inputs count as weights
(kept resident in the end-to-end measurement) and the bytes copied in per step."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _fake_workload():
    """A Workload with the step's host tensors replaced by small stand-ins of known
    sizes, in the order the real one holds them."""
    w = object.__new__(bench.Workload)
    R, Rr, Rm, E = bench.AG["R"], bench.RS["R"], bench.MOE["R"], bench.MOE["E"]
    w.h_ag = [torch.empty(3, dtype=torch.bfloat16) for _ in range(R)] + [torch.empty(100, dtype=torch.bfloat16)]
    w.h_rs = [torch.empty(5, dtype=torch.bfloat16) for _ in range(Rr)] + \
        [torch.empty(1000, dtype=torch.bfloat16) for _ in range(Rr)]
    w.h_moe = [torch.empty(7, dtype=torch.bfloat16) for _ in range(Rm)] + \
        [torch.empty(10000, dtype=torch.bfloat16) for _ in range(E)] + [torch.empty(11, dtype=torch.int32)]
    return w


def test_weights_are_b_the_b_r_and_the_experts():
    w = _fake_workload()
    R, Rr, Rm, E = bench.AG["R"], bench.RS["R"], bench.MOE["R"], bench.MOE["E"]
    n = len(w.h_ag) + len(w.h_rs) + len(w.h_moe)
    got = [i for i in range(n) if w._weight(i)]
    want = [R] + [R + 1 + Rr + r for r in range(Rr)] + [R + 1 + 2 * Rr + Rm + e for e in range(E)]
    assert got == want


def test_h2d_bytes_with_and_without_weights():
    w = _fake_workload()
    R, Rr, Rm, E = bench.AG["R"], bench.RS["R"], bench.MOE["R"], bench.MOE["E"]
    acts = 2 * (3 * R + 5 * Rr + 7 * Rm) + 4 * 11
    weights = 2 * (100 + 1000 * Rr + 10000 * E)
    assert w.h2d_bytes(weights=False) == acts
    assert w.h2d_bytes() == acts + weights
