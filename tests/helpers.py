"""Shared test helpers: device tensors from seeded bf16 bits, and the parity
gates used by every GPU test.

Tolerances
----------
* The stated gate: max-norm relative error ||g - o||_inf / ||o||_inf <= 2e-2
  for bf16 outputs and <= 1e-3 for fp32 outputs.
* A tighter elementwise bound derived from the arithmetic, applied as well:
  bf16 outputs carry one round-to-nearest-even (relative error <= 2^-9) on top
  of an fp32 accumulation whose error stays below K * 2^-24 * ||o||_inf for the
  value ranges used here, so |g - o| <= 2^-8 |o| + 1e-3 ||o||_inf; fp32 outputs
  must satisfy |g - o| <= 1e-4 ||o||_inf.
"""
import numpy as np

BF16_NORM_TOL = 2e-2
F32_NORM_TOL = 1e-3


def dev_bf16(bits):
    from tile_centric_gemm_gb300 import inputs
    return inputs.to_torch_bf16(bits).cuda()


def pinned_bf16(bits):
    """bf16 bits -> a pinned host torch tensor (device-addressable: the slow-link stand-in)."""
    from tile_centric_gemm_gb300 import inputs
    return inputs.to_torch_bf16(bits).pin_memory()


def to_bits(t):
    """bf16 torch tensor -> uint16 numpy bits."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t):
    return t.detach().double().cpu().numpy()


def check_bf16(got_f64, want, name=""):
    got_f64 = np.asarray(got_f64, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got_f64.shape == want.shape, (name, got_f64.shape, want.shape)
    assert np.all(np.isfinite(got_f64)), f"{name}: non-finite output"
    ninf = float(np.max(np.abs(want))) if want.size else 0.0
    err = np.abs(got_f64 - want)
    if want.size == 0:
        return 0.0
    norm_rel = float(err.max() / max(ninf, 1e-300))
    assert norm_rel <= BF16_NORM_TOL, f"{name}: normwise rel err {norm_rel:.3e}"
    bound = 2.0 ** -8 * np.abs(want) + 1e-3 * ninf
    bad = err > bound
    assert not bad.any(), f"{name}: {int(bad.sum())} elements beyond elementwise bound, worst {float((err - bound).max()):.3e}"
    return norm_rel


def check_f32(got_f64, want, name=""):
    got_f64 = np.asarray(got_f64, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got_f64.shape == want.shape, (name, got_f64.shape, want.shape)
    assert np.all(np.isfinite(got_f64)), f"{name}: non-finite output"
    ninf = float(np.max(np.abs(want)))
    err = np.abs(got_f64 - want)
    norm_rel = float(err.max() / max(ninf, 1e-300))
    assert norm_rel <= F32_NORM_TOL, f"{name}: normwise rel err {norm_rel:.3e}"
    assert float(err.max()) <= 1e-4 * ninf, f"{name}: max err {float(err.max()):.3e} > 1e-4 * {ninf:.3e}"
    return norm_rel
