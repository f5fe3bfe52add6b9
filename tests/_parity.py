"""Helpers shared by the GPU parity tests (test infrastructure only).

Tolerance (floating point, random data), applied per element and globally:
  * |gpu - ref| <= max(2e-2, 1.05 * 2**-8 * (A + |ref|) + 1e-4) for every element,
    where A = sum_j w_j |v_j| (the oracle's attention output with |V| in place of V);
  * ||gpu - ref||_2 / ||ref||_2 <= 5e-3 over all shards.
The absolute bar 2e-2 and the relative-L2 bar 5e-3 are the stated targets.  The
second term of the per-element bar is the rounding bound of the arithmetic the
kernel must do in bf16: each probability is rounded to bf16 before the PV
product (relative error <= 2**-8, so the output moves by <= 2**-8 * A) and the
output is rounded to bf16 (<= 2**-8 * |ref|).  For N(0,1) inputs A is below 1
and the bar is exactly 2e-2; only the outlier-channel inputs (values up to ~40)
reach the rounding bound.
Integer/layout work is compared bit for bit.
"""
import numpy as np

ABS_TOL = 2e-2
REL_L2_TOL = 5e-3
ELEM_REL = 2.0 ** -8


def bits_to_torch(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def torch_to_f64(t):
    import torch
    return t.detach().to("cpu").to(torch.float64).numpy()


def abs_bits(bits):
    """bf16 bit patterns of |x| (sign bit cleared)."""
    return (np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)).astype(np.uint16)


def assert_close(got, ref, absmass, where=""):
    """``absmass`` = sum_j w_j |v_j| for every output element (same shape as ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    absmass = np.asarray(absmass, dtype=np.float64)
    assert got.shape == ref.shape == absmass.shape, (got.shape, ref.shape, absmass.shape)
    assert np.isfinite(got).all(), f"{where}: non-finite output"
    err = np.abs(got - ref)
    tol = np.maximum(ABS_TOL, 1.05 * ELEM_REL * (absmass + np.abs(ref)) + 1e-4)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{where}: {bad.sum()} elements out of tolerance; worst at {i}: "
                             f"gpu={got[i]} ref={ref[i]} err={err[i]:.3e} tol={tol[i]:.3e}")
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= REL_L2_TOL, f"{where}: relative L2 error {rel:.3e} > {REL_L2_TOL}"
    return float(err.max()), float(rel)
