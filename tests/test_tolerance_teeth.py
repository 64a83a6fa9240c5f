"""The parity tolerance can see the long-context accumulation failure.

The pages' 128K result (phantomic12 vLLM-blog summary, "ACCURACY AT LONG
CONTEXT": FP8 attention whose P.V contraction ran in a low-precision
accumulator lost the needle; two-level accumulation fixed it) is a swamping
failure: once the running sum is large, each new small term rounds away.
Here a deliberately degraded accumulator, written only for this test on the
CPU, sums p_t * v_t over 131,072 keys with its running value rounded to a few
mantissa bits after every add; the row sum of p stays exact, so this isolates
the P.V accumulator (the oracle's own acc_bits pin degrades both sums).  Values ~ N(0.25, 0.125) under near-flat
attention make the output (about 0.25, where bf16 output rounding stays well
inside the bar) depend on all keys.  At 10 or 14 bits the result misses the
fp64 oracle by far more than the 8e-3 / 1e-3 bar; with a 23-bit (FP32-width)
accumulator it stays inside.  tests/test_gpu_parity.py runs the CUDA path on
the same kind of data."""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import ATTN_MAX_ABS, ATTN_MEAN_ABS, attn_errors

L, D, H = 131072, 128, 2


def _round_bits(x, bits):
    """Round to `bits` explicit mantissa bits, ties to even (np.round)."""
    m, e = np.frexp(x)
    return np.ldexp(np.round(m * 2.0 ** (bits + 1)) / 2.0 ** (bits + 1), e)


@pytest.fixture(scope="module")
def case():
    g = torch.Generator().manual_seed(5)
    q = (torch.randn((1, H, D), generator=g) * 0.05).to(torch.bfloat16)
    k = (torch.randn((L, 1, D), generator=g) * 0.5).to(torch.bfloat16)
    v = (torch.randn((L, 1, D), generator=g) * 0.125 + 0.25).to(torch.bfloat16)
    ks, vs = workload.per_tensor_scale(k), workload.per_tensor_scale(v)
    kc = oracle.quantize_bf16(workload.bf16_bits(k), ks)
    vc = oracle.quantize_bf16(workload.bf16_bits(v), vs)
    sm = float(np.float32(1.0 / np.sqrt(D)))
    ref = oracle.decode_attention(workload.bf16_bits(q), kc, vc, np.array([L]), ks, vs, sm, 0,
                                  nthreads=oracle.max_threads())[0]
    kf = oracle.e4m3_decode(kc[:, 0]) * ks
    vf = oracle.e4m3_decode(vc[:, 0]) * vs
    s = (kf @ q.float().numpy()[0].astype(np.float64).T).T * sm
    p = np.exp(s - s.max(axis=1, keepdims=True))
    return ref, p, vf


def _degraded(p, vf, bits):
    acc = np.zeros((H, D))
    for t in range(L):
        acc = _round_bits(acc + p[:, t:t + 1] * vf[t], bits)
    return acc / p.sum(axis=1, keepdims=True)


def _within_bar(got, ref):
    mx, mean = attn_errors(got, ref)
    return mx <= ATTN_MAX_ABS and mean <= ATTN_MEAN_ABS


@pytest.mark.parametrize("bits", [10, 14])
def test_low_precision_accumulator_fails_the_bar(case, bits):
    ref, p, vf = case
    assert not _within_bar(_degraded(p, vf, bits), ref)


def test_fp32_width_accumulator_meets_the_bar(case):
    ref, p, vf = case
    assert _within_bar(_degraded(p, vf, 23), ref)
