"""Oracle for the tile-centric AllGather-GEMM, GEMM-ReduceScatter, MoE
(AllGather + grouped GEMM, and the down-projection side) and AllGather-KV
attention path.

TEST INFRASTRUCTURE ONLY.  A plain, slow CPU restatement of what the path
computes, written from the TileLink talk summary ("TileLink: Generating
Efficient Compute-Communication Overlapping Kernels using Tile-Centric
Primitives") and the mathematics of the operations.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline leg and its
``--impl reference`` arm) may import it.  The library's product path never
imports, links or calls anything here, and this package imports nothing from
the library: the two share only the seeded input generators.

Arithmetic: bf16 inputs are decoded exactly to float64; products and sums are
float64 (numpy's matmul / dot serve as the dot-product step); bookkeeping is
integer Python.

Pins (see ``tests/test_oracle_pins.py``): every function here is checked
against something other than itself -- brute-force loops on tiny inputs,
closed forms, invariants, hand-worked fixtures under ``tests/golden/`` and,
for bf16 rounding, the float32 -> bfloat16 conversion of an independent
library.
"""
from . import bf16, ag_gemm, gemm_rs, moe, attention  # noqa: F401
