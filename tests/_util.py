"""Shared helpers for the tests: error metrics and tolerances.

Tolerances: bf16 outputs must match the fp64 oracle within a max relative
error (||gpu - ref||_inf / ||ref||_inf) of 2e-2; fp32 statistics r, s, LSE and
loss within 1e-3; integer work exactly.
"""
import numpy as np
import torch

TOL_BF16 = 2e-2
TOL_F32 = 1e-3
# The RMSNorm-backward statistic s sums a row of products with heavy
# cancellation; the bf16 rounding of the GEMM operand it is built from (hg,
# dout, qkv) moves it ~1e-3 relative to the exact fp64 value. It meets 1e-3
# against the oracle's storage-rounded form, and this bound against the exact
# canonical form.
TOL_S_EXACT = 5e-3


def to64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to(torch.float64).cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def maxrel(got, ref) -> float:
    got = to64(got)
    ref = to64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    return float(np.max(np.abs(got - ref)) / max(float(np.max(np.abs(ref))), 1e-300))


def elementwise_rel(got, ref) -> float:
    """Largest elementwise relative error |gpu - ref| / max(|ref|, floor),
    with floor = 1e-3 * rms(ref) so that entries near zero do not dominate.
    Reported beside the max-norm metric; the bounds apply to the latter."""
    got = to64(got)
    ref = to64(ref)
    floor = 1e-3 * max(float(np.sqrt(np.mean(ref * ref))), 1e-300)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


def assert_close(name, got, ref, tol):
    e = maxrel(got, ref)
    print(f"{name}: max rel err {e:.3e} (tol {tol:g}); elementwise {elementwise_rel(got, ref):.3e}")
    assert e <= tol, f"{name}: max rel err {e:.3e} > {tol:g}"
    return e


def assert_stat_near_exact(name, got, exact, rounded):
    """A backward statistic (s, s_a, s_b) against the exact canonical value.
    The bf16 storage the method applies to the GEMM operands it is built
    from moves it away from the exact value by what the oracle's
    storage-rounded form shows at these very inputs; the GPU value may be no
    further from exact than that plus the fp32 tolerance (of the largest
    |exact|). Over many rows the max-relative error must also stay within
    TOL_S_EXACT. A single row is one heavily cancelling sum whose magnitude
    is no scale for the rounding, so that second bound is not applied to it."""
    got64, ex, rd = to64(got), to64(exact), to64(rounded)
    scale = max(float(np.max(np.abs(ex))), 1e-300)
    e_gpu = float(np.max(np.abs(got64 - ex)))
    e_st = float(np.max(np.abs(rd - ex)))
    print(f"{name}: |gpu - exact| {e_gpu / scale:.3e}, |rounded - exact| {e_st / scale:.3e} "
          f"(relative to max |exact|)")
    assert e_gpu <= e_st + TOL_F32 * scale, f"{name}: further from exact than storage rounding allows"
    if ex.size > 1:
        assert_close(name, got, exact, TOL_S_EXACT)
