"""The allocation-free decode entry point (fp8kv_paged_decode_noalloc).

Callers that cannot allocate device memory while they decode -- an engine whose
memory manager already reserved nearly all HBM for its own paged KV pool, host
code under a no-allocation rule, a binding with no CUDA allocator -- use this
entry point; the split-merge scratch then lives in the library's fixed device
array.  Its results must match the oracle and the workspace entry point's,
call after call, although the array keeps the previous call's contents.  A
problem whose scratch fits the array just barely runs; one just beyond it is
refused before anything is launched.

This file sorts last on purpose: it runs after every other test (and must also
pass on its own in a fresh process).
"""
import pytest
import torch

from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import assert_attn_close
from tests.gpu_harness import Paged, oracle_codes, oracle_out

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


def _f64(t):
    return t.float().cpu().numpy().astype("float64")


def _noalloc(pc, w, window, out):
    fk.fp8kv_paged_decode_noalloc(pc.q, pc.k_cache, pc.v_cache, pc.block_tables, pc.seq_lens,
                                  w.max_seq_len, w.k_scale, w.v_scale, w.sm_scale, window, out)
    torch.cuda.synchronize()


@pytest.mark.parametrize("base,lens,window", [
    ("llama31_8b_b8_20k", [1500, 37, 700, 0], 0),
    ("gemma4e2b_b16_8k32k", [3000, 513], 512),
])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_consecutive_calls(base, lens, window):
    shape = workload.small_shape(base, batch=len(lens), len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=11, lens=lens)
    pc = Paged(w)
    pc.append_all()
    ref, err = pc.decode(window=window)
    assert err == 0
    kc, vc = oracle_codes(w)
    exact = oracle_out(w, kc, vc, window)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        _noalloc(pc, w, window, out)
        assert_attn_close(_f64(out), exact, "noalloc call %d against the oracle" % call)
        assert_attn_close(_f64(out), _f64(ref), "noalloc call %d against the workspace call" % call)


def _boundary_batch(hq, hkv, d, L):
    """The largest batch (<= 512) whose decode scratch fits the fixed array."""
    lo, hi = 1, 512
    assert fk.fp8kv_paged_decode_workspace_size(lo, hq, hkv, d, L) <= SCRATCH_BYTES
    assert fk.fp8kv_paged_decode_workspace_size(hi, hq, hkv, d, L) > SCRATCH_BYTES
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if fk.fp8kv_paged_decode_workspace_size(mid, hq, hkv, d, L) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_at_the_scratch_limit_runs_and_one_more_sequence_is_refused():
    base = "llama31_8b_b8_20k"            # 32 q / 8 kv heads, d = 128
    s0 = workload.CONFIGS[base]
    L = 40
    B = _boundary_batch(s0.num_q_heads, s0.num_kv_heads, s0.head_dim, L)
    shape = workload.small_shape(base, batch=B, len_lo=L, len_hi=L)
    w = workload.make_workload(shape, seed=4, lens=[L] * B)
    pc = Paged(w)
    pc.append_all()
    kc, vc = oracle_codes(w)
    out = torch.full((B, s0.num_q_heads, s0.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    _noalloc(pc, w, 0, out)
    assert_attn_close(_f64(out), oracle_out(w, kc, vc, 0), "noalloc at the limit (batch %d)" % B)
    # one sequence more: refused, nothing launched
    q = torch.zeros((B + 1, s0.num_q_heads, s0.head_dim), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B + 1, pc.block_tables.shape[1]), dtype=torch.int32, device="cuda")
    sl = torch.full((B + 1,), L, dtype=torch.int32, device="cuda")
    out2 = torch.empty_like(q)
    with pytest.raises(fk.Fp8kvError) as e:
        fk.fp8kv_paged_decode_noalloc(q, pc.k_cache, pc.v_cache, bt, sl, w.max_seq_len, 1.0, 1.0, 0.1, 0, out2)
    assert e.value.code == 3  # FP8KV_ERR_WORKSPACE


def test_noalloc_rejects_problems_far_beyond_the_fixed_scratch():
    # 4096 sequences x 8 kv heads x 4 heads x 128 dims of fp32 partials is far
    # beyond the fixed 8 MiB array: refused before anything is launched.
    B, hq, hkv, d = 4096, 32, 8, 128
    q = torch.zeros((B, hq, d), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((4, hkv, 16, d), dtype=torch.uint8, device="cuda")
    bt = torch.zeros((B, 2), dtype=torch.int32, device="cuda")
    sl = torch.full((B,), 20, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(fk.Fp8kvError) as e:
        fk.fp8kv_paged_decode_noalloc(q, cache, cache, bt, sl, 32, 1.0, 1.0, 0.1, 0, out)
    assert e.value.code == 3  # FP8KV_ERR_WORKSPACE
