"""Host-side checks of the seeded input generators (no method arithmetic here)."""
import numpy as np
import torch

from tile_centric_gemm_gb300 import inputs


def test_bf16_packing_matches_torch_conversion():
    x = np.random.default_rng(1).standard_normal(100_000).astype(np.float32) * 3
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(inputs.bf16_bits_from_f32(x), want)


def test_generators_are_seeded_and_shaped():
    A1, B1 = inputs.ag_gemm_inputs(2, 128, 512, 256, "uniform", seed=0)
    A2, B2 = inputs.ag_gemm_inputs(2, 128, 512, 256, "uniform", seed=0)
    assert [a.shape for a in A1] == [(128, 512)] * 2 and B1.shape == (512, 256)
    assert all(np.array_equal(a, b) for a, b in zip(A1, A2)) and np.array_equal(B1, B2)
    assert not np.array_equal(A1[0], A1[1])
    v = inputs.to_torch_bf16(A1[0]).float()
    assert float(v.min()) >= -1.0 and float(v.max()) <= 1.0


def test_zipf_routing_distinct_and_skewed():
    ids = inputs.zipf_topk(8192, 32, 2, 1.2, seed=3000)
    assert ids.shape == (8192, 2) and ids.dtype == np.int32
    assert np.all(ids[:, 0] != ids[:, 1])
    counts = np.bincount(ids.ravel(), minlength=32)
    # finite Zipf(1.2) over 32 experts, top-2 without replacement: expert 0 takes
    # roughly a quarter of the 16384 rows and counts fall with the expert index
    assert 3500 < counts[0] < 5500
    assert counts[0] > counts[1] > counts[4] > counts[16]
    assert counts.min() > 0
