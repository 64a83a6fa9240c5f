"""Shared tolerances and comparison helpers for the parity tests.

Attention outputs must satisfy max|err| <= 8e-3 and mean|err| <= 1e-3 against
the fp64 oracle on the same quantised cache (the stated accuracy bar for the
bf16-rounded FP32 result).  Quantised cache bytes must match bit for bit.
"""
import numpy as np

ATTN_MAX_ABS = 8e-3
ATTN_MEAN_ABS = 1e-3


def attn_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    return float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0


def assert_attn_close(got, ref, what=""):
    mx, mean = attn_errors(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    assert mx <= ATTN_MAX_ABS and mean <= ATTN_MEAN_ABS, \
        f"{what}: max|err|={mx:.3e} (<= {ATTN_MAX_ABS}), mean|err|={mean:.3e} (<= {ATTN_MEAN_ABS})"
    return mx, mean


# bf16 keeps 8 significant bits, so round-to-nearest moves a value x by at most
# 2^-8 |x|.  The absolute bar above presumes outputs of magnitude <= 2 (where
# that rounding is <= 7.8e-3); an attention row over one or a few keys is a
# raw value row of magnitude up to ~4.5 for unit-normal data, and there the
# format's own rounding is the floor of what any kernel can reach.
BF16_HALF_ULP_REL = 2.0 ** -8


def assert_attn_close_bf16_floor(got, ref, what=""):
    """The attention bar with a per-element floor at bf16's rounding of the
    exact value: |err| <= max(8e-3, 2^-8 |ref|); mean |err| <= 1e-3."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = np.maximum(ATTN_MAX_ABS, BF16_HALF_ULP_REL * np.abs(ref))
    worst = float((err / bound).max()) if err.size else 0.0
    mean = float(err.mean()) if err.size else 0.0
    assert worst <= 1.0 and mean <= ATTN_MEAN_ABS, \
        f"{what}: max err/bound={worst:.3f} (<= 1), max|err|={float(err.max()):.3e}, mean|err|={mean:.3e}"
    return float(err.max()) if err.size else 0.0, mean
