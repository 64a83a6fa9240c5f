"""GPU tests of the failure path: a bounded wait that runs out.

A test hook makes one stage of CTA 0 never arrive (nothing issues it), with a
short wait limit, so the waiting side gives up: the kernel writes
FP8KV_ERR_TIMEOUT into the workspace error word, lets its copies in flight
land and returns.  Nothing faults or hangs.  The checks: the error is
reported; a later call on the same workspace skips its work (the output is
left as it was); after fp8kv_workspace_init the same call is correct again
(oracle parity) and reports no error.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import assert_attn_close, assert_attn_close_bf16_floor
from tests.gpu_harness import Paged, oracle_out

pytestmark = pytest.mark.gpu

TIMEOUT = 5
LIMIT_NS = 2_000_000   # 2 ms


def _decode_setup():
    shape = workload.small_shape("llama31_8b_b8_20k", 3, 1, 1)
    w = workload.make_workload(shape, seed=11, lens=[3000, 517, 1301])
    p = Paged(w, seed=11)
    p.append_all()
    s = w.shape
    ws = fk.alloc_workspace(3, s.num_q_heads, s.num_kv_heads, s.head_dim, w.max_seq_len)
    return w, p, ws


def _decode(p, w, ws, out, engine):
    fk.fp8kv_paged_decode_engine(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, w.max_seq_len, w.k_scale,
                                 w.v_scale, w.sm_scale, 0, out, ws, engine)


@pytest.mark.parametrize("stall_stage", [0, 2])   # CTA 0 streams 4 stages of this workload
def test_decode_wait_runs_out_reports_timeout_and_poisons_the_workspace(stall_stage):
    w, p, ws = _decode_setup()
    s = w.shape
    out = torch.full((3, s.num_q_heads, s.head_dim), 7.0, dtype=torch.bfloat16, device="cuda")
    t0 = time.perf_counter()
    code = fk.debug_paged_decode_stall(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, w.max_seq_len,
                                       w.k_scale, w.v_scale, w.sm_scale, 0, out, ws, stall_stage, LIMIT_NS)
    assert code == 0
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0   # bounded: a few wait limits, not a hang
    # a later call on the same workspace skips its work: both engines
    for engine in (fk.ENGINE_TENSOR_CORES, fk.ENGINE_CUDA_CORES):
        out2 = torch.full_like(out, 3.0)
        _decode(p, w, ws, out2, engine)
        torch.cuda.synchronize()
        assert torch.all(out2 == 3.0), "a call after a timeout must not run"
    assert fk.fp8kv_read_error(ws) == TIMEOUT
    # re-initialised, the workspace works again, on both engines
    kc, vc = p.gathered_codes()
    ref = oracle_out(w, kc, vc, 0)
    for engine in (fk.ENGINE_CUDA_CORES, fk.ENGINE_TENSOR_CORES):
        fk.fp8kv_workspace_init(ws)
        out3 = torch.empty_like(out)
        _decode(p, w, ws, out3, engine)
        torch.cuda.synchronize()
        assert fk.fp8kv_read_error(ws) == 0
        assert_attn_close(out3.float().cpu().numpy(), ref, "after re-initialisation, engine %d" % engine)


def test_decode_stall_hook_without_a_stall_is_the_plain_call():
    w, p, ws = _decode_setup()
    s = w.shape
    out = torch.empty((3, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    assert fk.debug_paged_decode_stall(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, w.max_seq_len,
                                       w.k_scale, w.v_scale, w.sm_scale, 0, out, ws, 1000, LIMIT_NS) == 0
    torch.cuda.synchronize()
    assert fk.fp8kv_read_error(ws) == 0
    kc, vc = p.gathered_codes()
    assert_attn_close(out.float().cpu().numpy(), oracle_out(w, kc, vc, 0), "stage 1000 never reached")


def test_decode_stall_hook_rejects_bad_arguments():
    w, p, ws = _decode_setup()
    s = w.shape
    out = torch.empty((3, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    for stage, ns in ((-1, LIMIT_NS), (0, 0), (0, 600_000_000)):
        assert fk.debug_paged_decode_stall(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, w.max_seq_len,
                                           w.k_scale, w.v_scale, w.sm_scale, 0, out, ws, stage, ns) == 1


@pytest.mark.parametrize("head_dim_base", ["llama31_8b_b8_20k", "gptoss20b_b8_16k", "gemma4e2b_b16_8k32k"])
def test_prefill_wait_runs_out_reports_timeout(head_dim_base):
    lens = [700, 300, 129]
    q_lens = [200, 64, 129]
    shape = workload.small_shape(head_dim_base, len(lens), 1, 1, needle_margin=None)
    w = workload.make_workload(shape, seed=5, lens=lens)
    p = Paged(w, seed=5)
    p.append_all()
    q, qs = workload.prefill_queries(w, q_lens, seed=5)
    s = w.shape
    mq = max(q_lens)
    ws = fk.alloc_prefill_workspace(len(lens), mq, w.max_seq_len, s.num_q_heads, s.num_kv_heads, s.head_dim, 16, 0)
    out = torch.zeros(q.shape, dtype=torch.bfloat16, device="cuda")
    qd, qsd = q.cuda(), qs.cuda()
    t0 = time.perf_counter()
    code = fk.debug_paged_prefill_stall(qd, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, qsd, mq,
                                        w.max_seq_len, w.k_scale, w.v_scale, w.sm_scale, 0, out, ws, 1, LIMIT_NS)
    assert code == 0
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert fk.fp8kv_read_error(ws) == TIMEOUT      # reading clears the word
    # the next call on the workspace is correct and reports nothing
    out2 = torch.empty_like(out)
    fk.fp8kv_paged_prefill(qd, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, qsd, mq, w.max_seq_len, w.k_scale,
                           w.v_scale, w.sm_scale, 0, out2, ws)
    torch.cuda.synchronize()
    assert fk.fp8kv_read_error(ws) == 0
    kc, vc = p.gathered_codes()
    ref = oracle.prefill_attention(workload.bf16_bits(q), kc, vc, w.seq_lens.numpy(), np.asarray(q_lens), w.k_scale,
                                   w.v_scale, w.sm_scale, 0, nthreads=oracle.max_threads())
    assert_attn_close_bf16_floor(out2.float().cpu().numpy(), ref, "prefill after a timeout")
