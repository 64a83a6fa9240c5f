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
