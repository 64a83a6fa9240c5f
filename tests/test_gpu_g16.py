"""GPU parity at 16 query heads per kv head.  The default decode carries the 16
heads as two MMA n-tiles of one unit per kv head at d <= 128 (each page read
once); at d = 256 and on the CUDA-core engine each kv head runs as two units
of 8 query heads over the same pages.  Checked: the fused step bit-identical
to append-then-decode, per-head scales against the per-head oracle, the
allocation-free call bit-identical to the workspace call, and the prefill.
The decode itself, both engines, and the bf16 twin are covered with every
other head layout, and at full size by the g16_b4_32k workload."""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import assert_attn_close, assert_attn_close_bf16_floor
from tests.gpu_harness import Paged, oracle_codes, oracle_out

pytestmark = pytest.mark.gpu


def _shape(d=128, hkv=2, batch=3):
    return workload.LayerShape(f"g16_d{d}", 16 * hkv, hkv, d, batch, 1, 1, (0,))


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_g16_step_equals_append_then_decode(d):
    w = workload.make_workload(_shape(d), seed=31, lens=[700, 17, 1])
    kc, vc = oracle_codes(w)
    for win in (0, 40):
        sep = Paged(w, seed=win)
        sep.append_all()
        out_sep, err_sep = sep.decode(window=win)
        fused = Paged(w, seed=win)
        fused.append_history()
        out_f, err_f = fused.step(window=win)
        assert err_sep == 0 and err_f == 0
        assert torch.equal(fused.k_cache, sep.k_cache) and torch.equal(fused.v_cache, sep.v_cache)
        assert torch.equal(out_f, out_sep)
        assert_attn_close(_f64(out_f), oracle_out(w, kc, vc, win), f"g16 d={d} step window={win}")


def test_g16_per_head_scales_match_oracle():
    w = workload.make_workload(_shape(128, hkv=4), seed=32, lens=[900, 33, 160])
    s = w.shape
    mag = torch.tensor([2.0 ** -h for h in range(s.num_kv_heads)], dtype=torch.float32).view(1, -1, 1)
    k = (w.k.float() * mag).to(torch.bfloat16)
    v = (w.v.float() * mag).to(torch.bfloat16)
    ks = (k.float().abs().amax(dim=(0, 2)) / 448).to(torch.float32)
    vs = (v.float().abs().amax(dim=(0, 2)) / 448).to(torch.float32)
    shape = (w.num_blocks, s.num_kv_heads, 16, s.head_dim)
    kcache = torch.full(shape, 0x5A, dtype=torch.uint8, device="cuda")
    vcache = torch.full(shape, 0x5A, dtype=torch.uint8, device="cuda")
    fk.fp8kv_quant_append_per_head(k.cuda(), v.cuda(), w.slot_mapping.cuda(), kcache, vcache, ks.cuda(), vs.cuda())
    kcodes = oracle.quantize_bf16_per_head(workload.bf16_bits(k), ks.numpy())
    vcodes = oracle.quantize_bf16_per_head(workload.bf16_bits(v), vs.numpy())
    B = w.seq_lens.numel()
    for win in (0, 50):
        ws = fk.alloc_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, w.max_seq_len, 16, win)
        out = torch.empty((B, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        fk.fp8kv_paged_decode_per_head(w.q.cuda(), kcache, vcache, w.block_tables.cuda(), w.seq_lens.cuda(),
                                       w.max_seq_len, ks.cuda(), vs.cuda(), w.sm_scale, win, out, ws)
        torch.cuda.synchronize()
        assert fk.fp8kv_read_error(ws) == 0
        ref = oracle.decode_attention_per_head(workload.bf16_bits(w.q), kcodes, vcodes, w.seq_lens.numpy(),
                                               ks.numpy(), vs.numpy(), w.sm_scale, win,
                                               nthreads=oracle.max_threads())
        assert_attn_close(_f64(out), ref, f"g16 per-head window={win}")


def test_g16_noalloc_equals_workspace_call():
    w = workload.make_workload(_shape(128), seed=33, lens=[1200, 5, 300])
    pc = Paged(w)
    pc.append_all()
    out_ws, err = pc.decode(window=0)
    assert err == 0
    s = w.shape
    out_na = torch.empty_like(out_ws)
    fk.fp8kv_paged_decode_noalloc(pc.q, pc.k_cache, pc.v_cache, pc.block_tables, pc.seq_lens, w.max_seq_len,
                                  w.k_scale, w.v_scale, w.sm_scale, 0, out_na)
    torch.cuda.synchronize()
    assert torch.equal(out_na, out_ws)


@pytest.mark.parametrize("d", [64, 128])
def test_g16_prefill_matches_oracle(d):
    lens = [300, 95, 17]
    q_lens = [37, 95, 1]
    w = workload.make_workload(_shape(d), seed=34, lens=lens)
    p = Paged(w, seed=34)
    p.append_all()
    q, qs = workload.prefill_queries(w, q_lens, seed=34)
    s = w.shape
    for window in (0, 40):
        ws = fk.alloc_prefill_workspace(len(lens), max(q_lens), w.max_seq_len, s.num_q_heads, s.num_kv_heads,
                                        s.head_dim, 16, window)
        out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        fk.fp8kv_paged_prefill(q.cuda(), p.k_cache, p.v_cache, p.block_tables, p.seq_lens, qs.cuda(), max(q_lens),
                               w.max_seq_len, w.k_scale, w.v_scale, w.sm_scale, window, out, ws)
        torch.cuda.synchronize()
        assert fk.fp8kv_read_error(ws) == 0
        kc, vc = p.gathered_codes()
        ref = oracle.prefill_attention(workload.bf16_bits(q), kc, vc, w.seq_lens.numpy(), np.asarray(q_lens),
                                       w.k_scale, w.v_scale, w.sm_scale, window, nthreads=oracle.max_threads())
        assert_attn_close_bf16_floor(_f64(out), ref, f"g16 prefill d={d} window={window}")
