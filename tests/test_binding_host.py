"""The Python binding's argument checks, on the CPU: shapes that do not fit
together and tensors that are not on a CUDA device are refused before any
call reaches the library (no GPU needed)."""
import pytest
import torch

from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import build as fbuild
from fp8_kv_cache_fp8kv_gb300 import workload


@pytest.fixture(scope="module", autouse=True)
def lib():
    fbuild.build()
    return fk.load()


def _prefill_args(**kw):
    T, hq, hkv, d, B, nb = 40, 32, 8, 128, 2, 10
    a = dict(q=torch.zeros((T, hq, d), dtype=torch.bfloat16),
             k_cache=torch.zeros((nb, hkv, 16, d), dtype=torch.uint8),
             v_cache=torch.zeros((nb, hkv, 16, d), dtype=torch.uint8),
             block_tables=torch.zeros((B, 5), dtype=torch.int32),
             seq_lens=torch.zeros(B, dtype=torch.int32),
             q_starts=torch.zeros(B + 1, dtype=torch.int32),
             max_q_len=20, max_seq_len=80, k_scale=0.01, v_scale=0.01, sm_scale=0.088, window=0,
             out=torch.zeros((T, hq, d), dtype=torch.bfloat16),
             workspace=torch.zeros(1024, dtype=torch.uint8))
    a.update(kw)
    return a


@pytest.mark.parametrize("kw", [
    dict(out=torch.zeros((39, 32, 128), dtype=torch.bfloat16)),            # out rows != q rows
    dict(v_cache=torch.zeros((10, 8, 16, 64), dtype=torch.uint8)),         # caches disagree
    dict(q_starts=torch.zeros(2, dtype=torch.int32)),                      # q_starts must be [B + 1]
    dict(block_tables=torch.zeros((3, 5), dtype=torch.int32)),             # block_tables rows != B
])
def test_prefill_refuses_mismatched_shapes(kw):
    with pytest.raises(ValueError):
        fk.prepare_paged_prefill(**_prefill_args(**kw))


def test_prefill_refuses_host_tensors():
    with pytest.raises(TypeError):
        fk.prepare_paged_prefill(**_prefill_args())


def test_decode_refuses_mismatched_shapes_and_host_tensors():
    q = torch.zeros((2, 32, 128), dtype=torch.bfloat16)
    kc = torch.zeros((10, 8, 16, 128), dtype=torch.uint8)
    bt = torch.zeros((2, 5), dtype=torch.int32)
    sl = torch.zeros(2, dtype=torch.int32)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError):
        fk.fp8kv_paged_decode(q, kc, kc, bt, sl, 80, 0.01, 0.01, 0.088, 0,
                              torch.zeros((2, 32, 64), dtype=torch.bfloat16), ws)
    with pytest.raises(ValueError):
        fk.fp8kv_paged_decode(q, kc, kc, torch.zeros((3, 5), dtype=torch.int32), sl, 80, 0.01, 0.01, 0.088, 0,
                              torch.zeros_like(q), ws)
    with pytest.raises(TypeError):
        fk.fp8kv_paged_decode(q, kc, kc, bt, sl, 80, 0.01, 0.01, 0.088, 0, torch.zeros_like(q), ws)


def test_prefill_queries_are_seeded_and_packed():
    shape = workload.small_shape("llama31_8b_b8_20k", 3, 1, 1)
    w = workload.make_workload(shape, seed=1, lens=[50, 0, 20])
    q1, s1 = workload.prefill_queries(w, [10, 0, 20], seed=4)
    q2, s2 = workload.prefill_queries(w, [10, 0, 20], seed=4)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    assert tuple(q1.shape) == (30, 32, 128) and s1.tolist() == [0, 10, 10, 30]
    with pytest.raises(AssertionError):
        workload.prefill_queries(w, [51, 0, 0], seed=4)   # more query tokens than cached tokens
