"""Parity tolerances, stated once.

The bar for floating-point outputs: max|dO| <= 5e-3 and max|dLSE| <= 1e-3
against the fp64 oracle (bf16 inputs, fp32 accumulation).  When O is stored
as bf16, the rounding of the output itself adds up to half a bf16 ulp of the
exact value, so the bf16 check is |dO| <= 5e-3 + ulp_bf16(|O_ref|)/2.
"""
import numpy as np

O_TOL = 5e-3
LSE_TOL = 1e-3

# (workload, output, max|dO|, max|dLSE|) of every whole-output comparison at full
# size, printed at the end of the test session (tests/conftest.py)
PARITY_LOG = []


def log_parity(what: str, o_err: float, lse_err: float):
    PARITY_LOG.append((what, float(o_err), float(lse_err)))


def half_ulp_bf16(x):
    """Half of the bf16 spacing at |x| (bf16 keeps 8 significant bits)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def check_o(got, ref, bf16_out: bool, what: str = "O"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    tol = O_TOL + (half_ulp_bf16(ref) if bf16_out else 0.0)
    bad = err > tol
    if bad.any():
        idx = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} values out of tolerance; worst at {idx}: "
                             f"got {got[idx]!r} ref {ref[idx]!r} (max |d| {err.max():.3e})")
    return float(err.max()) if err.size else 0.0


def check_lse(got, ref, what: str = "LSE"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), f"{what}: -inf pattern differs"
    assert not np.isnan(got).any(), f"{what}: NaN"
    g = np.where(ninf_r, 0.0, got)
    r = np.where(ninf_r, 0.0, ref)
    err = np.abs(g - r)
    if err.size and err.max() > LSE_TOL:
        idx = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(f"{what}: max |d| {err.max():.3e} at {idx} (got {got[idx]!r} ref {ref[idx]!r})")
    return float(err.max()) if err.size else 0.0
