"""Host-side logic without a GPU: byte accounting against the pages' worked
example, and the seeded workload generator's invariants."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import accounting, workload

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_bytes_per_token_reproduces_worked_example():
    ex = json.load(open(os.path.join(GOLD, "qwen3_32b_capacity.json")))
    L, H, d = ex["num_layers"], ex["num_kv_heads"], ex["head_dim"]
    assert accounting.bytes_per_token(L, H, d, 1) == ex["elements_per_token"] == ex["fp8_bytes_per_token"]
    bf = accounting.bytes_per_token(L, H, d, 2)
    assert bf == ex["bf16_bytes_per_token"]
    seq = ex["sequence_tokens"]
    assert round(seq * bf / 1e9, 2) == ex["bf16_gb_per_sequence"]
    # the page truncates 4.295 GB to 4.29
    assert math.floor(seq * ex["fp8_bytes_per_token"] / 1e7) / 100 == ex["fp8_gb_per_sequence"]
    usable = round(ex["hbm_gb"] * ex["gpu_memory_utilization"], 2)
    assert usable == ex["usable_gb"]
    budget = round(usable - ex["bf16_weights_gb"] - ex["overhead_gb"], 2)
    assert budget == ex["kv_budget_gb"]
    assert int(budget // ex["bf16_gb_per_sequence"]) == ex["bf16_sequences"]
    assert int(budget // ex["fp8_gb_per_sequence"]) == ex["fp8_sequences"]


@pytest.mark.parametrize("name", list(workload.CONFIGS))
def test_arithmetic_intensity_is_2g_for_fp8(name):
    s = workload.CONFIGS[name]
    lens = [s.len_hi] * s.batch
    kv_bytes = sum(2 * s.num_kv_heads * L * s.head_dim for L in lens)
    flops = accounting.decode_flops(lens, s.num_q_heads, s.head_dim)
    assert flops / kv_bytes == 2 * s.group
    # bf16 would read twice the bytes at the same flops: intensity g
    assert flops / (2 * kv_bytes) == s.group


def test_decode_bytes_counts_window_pages():
    # one sequence of 100 tokens, window 20: tokens 80..99 -> pages 5 and 6
    b = accounting.decode_bytes([100], 4, 2, 16, window=20)
    assert b == 2 * 2 * 20 * 16 + 2 * 4 * 16 * 2 + 4 * 2
    assert accounting.decode_bytes([0], 4, 2, 16) == 2 * 4 * 16 * 2


def test_generator_is_deterministic_and_consistent():
    s = workload.small_shape("llama31_8b_b8_20k", batch=3, len_lo=1, len_hi=70)
    a = workload.make_workload(s, seed=1)
    b = workload.make_workload(s, seed=1)
    c = workload.make_workload(s, seed=2)
    assert a.digest() == b.digest() != c.digest()
    # the block table is a permutation of the physical blocks
    used = []
    for i, L in enumerate(a.seq_lens.tolist()):
        nb = (L + 15) // 16
        used += a.block_tables[i, :nb].tolist()
    assert sorted(used) == list(range(a.num_blocks))
    # the slot mapping agrees with the table, token by token
    for i, L in enumerate(a.seq_lens.tolist()):
        for t in range(L):
            slot = int(a.slot_mapping[int(a.seq_starts[i]) + t])
            assert slot == int(a.block_tables[i, t // 16]) * 16 + t % 16
    assert len(set(a.slot_mapping.tolist())) == a.slot_mapping.numel()
    # scales are amax/448 in fp32
    assert a.k_scale == float(np.float32(a.k.abs().max().float().item() / 448))
    assert a.sm_scale == float(np.float32(1 / math.sqrt(128)))


def test_needle_dominates_after_quantisation():
    """The planted key beats the log-sum-exp of every other logit of each query
    head by the stated margin (checked on the decoded cache in fp64), and the
    oracle's output is then that key's value row."""
    s = workload.small_shape("llama33_70b_needle_128k", batch=1, len_lo=4096, len_hi=4096)
    w = workload.make_workload(s, seed=0)
    p = w.needle_pos
    assert 0 <= p <= 4096 - 2
    kc = oracle.quantize_bf16(workload.bf16_bits(w.k), w.k_scale)
    vc = oracle.quantize_bf16(workload.bf16_bits(w.v), w.v_scale)
    kh = oracle.e4m3_decode(kc) * w.k_scale
    vh = oracle.e4m3_decode(vc) * w.v_scale
    q = w.q.to(torch.float64).numpy()
    g = s.group
    for h in range(s.num_q_heads):
        sc = w.sm_scale * kh[:, h // g, :] @ q[0, h]
        others = np.delete(sc, p)
        lse = others.max() + np.log(np.exp(others - others.max()).sum())
        assert sc[p] - lse >= s.needle_margin
    out = oracle.decode_attention(workload.bf16_bits(w.q), kc, vc, w.seq_lens.numpy(),
                                  w.k_scale, w.v_scale, w.sm_scale, 0)
    for h in range(s.num_q_heads):
        assert np.allclose(out[0, h], vh[p, h // g], rtol=0, atol=1e-5)
