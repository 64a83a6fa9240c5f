"""GPU parity with one K and one V scale per kv head: cache codes bit-exact
against the oracle's per-head quantiser, attention against the per-head fp64
oracle, the fused step bit-identical to append-then-decode, and equal head
scales bit-identical to the per-tensor calls."""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import assert_attn_close

pytestmark = pytest.mark.gpu


def _per_head_workload(base, lens, seed):
    """A workload whose kv heads differ in magnitude by powers of two (exact
    in bf16), with per-head amax/448 scales.  V stays within |v| <= ~4 so the
    outputs stay where bf16 output rounding is inside the tolerance."""
    shape = workload.small_shape(base, batch=len(lens), len_lo=1, len_hi=1, needle_margin=None)
    w = workload.make_workload(shape, seed=seed, lens=lens)
    hkv = shape.num_kv_heads
    kmag = torch.tensor([2.0 ** ((3 * h) % 8 - 5) for h in range(hkv)], dtype=torch.float32).view(1, hkv, 1)
    vmag = torch.tensor([2.0 ** -(h % 5) for h in range(hkv)], dtype=torch.float32).view(1, hkv, 1)
    k = (w.k.float() * kmag).to(torch.bfloat16)
    v = (w.v.float() * vmag).to(torch.bfloat16)
    ks = (k.float().abs().amax(dim=(0, 2)) / 448).to(torch.float32)
    vs = (v.float().abs().amax(dim=(0, 2)) / 448).to(torch.float32)
    ks[ks == 0] = 1.0
    vs[vs == 0] = 1.0
    return w, k, v, ks, vs


def _caches(w, fill=0x5A):
    s = w.shape
    shape = (w.num_blocks, s.num_kv_heads, 16, s.head_dim)
    return (torch.full(shape, fill, dtype=torch.uint8, device="cuda"),
            torch.full(shape, fill, dtype=torch.uint8, device="cuda"))


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


CASES = [
    ("llama31_8b_b8_20k", [2999, 1234, 16, 4097], (0, 128)),
    ("gptoss20b_b8_16k", [1, 63, 64, 65, 700], (0, 7)),
    ("gemma4e2b_b16_8k32k", [17, 513, 3000], (0, 33)),
    ("llama33_70b_needle_128k", [3000, 40], (0,)),
]


@pytest.mark.parametrize("base,lens,windows", CASES)
def test_per_head_append_and_decode_match_oracle(base, lens, windows):
    w, k, v, ks, vs = _per_head_workload(base, lens, seed=17)
    s = w.shape
    kc, vc = _caches(w)
    fk.fp8kv_quant_append_per_head(k.cuda(), v.cuda(), w.slot_mapping.cuda(), kc, vc, ks.cuda(), vs.cuda())
    torch.cuda.synchronize()
    ref_k = oracle.quantize_bf16_per_head(workload.bf16_bits(k), ks.numpy())
    ref_v = oracle.quantize_bf16_per_head(workload.bf16_bits(v), vs.numpy())
    blk, off = w.slot_mapping // 16, w.slot_mapping % 16
    assert np.array_equal(kc.cpu()[blk, :, off, :].numpy(), ref_k)
    assert np.array_equal(vc.cpu()[blk, :, off, :].numpy(), ref_v)
    B = len(lens)
    for win in windows:
        ws = fk.alloc_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, w.max_seq_len, 16, win)
        out = torch.empty((B, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        fk.fp8kv_paged_decode_per_head(w.q.cuda(), kc, vc, w.block_tables.cuda(), w.seq_lens.cuda(), w.max_seq_len,
                                       ks.cuda(), vs.cuda(), w.sm_scale, win, out, ws)
        torch.cuda.synchronize()
        assert fk.fp8kv_read_error(ws) == 0
        ref = oracle.decode_attention_per_head(workload.bf16_bits(w.q), ref_k, ref_v, w.seq_lens.numpy(), ks.numpy(),
                                               vs.numpy(), w.sm_scale, win, nthreads=oracle.max_threads())
        assert_attn_close(_f64(out), ref, f"per-head {base} window={win}")


def test_per_head_step_equals_append_then_decode():
    w, k, v, ks, vs = _per_head_workload("llama31_8b_b8_20k", [900, 17, 1600], seed=18)
    s = w.shape
    B = 3
    rows = w.new_token_rows()
    keep = torch.ones(k.shape[0], dtype=torch.bool)
    keep[rows] = False
    kc1, vc1 = _caches(w)
    kc2, vc2 = _caches(w)
    ksd, vsd = ks.cuda(), vs.cuda()
    fk.fp8kv_quant_append_per_head(k.cuda(), v.cuda(), w.slot_mapping.cuda(), kc1, vc1, ksd, vsd)
    fk.fp8kv_quant_append_per_head(k[keep].cuda(), v[keep].cuda(), w.slot_mapping[keep].cuda(), kc2, vc2, ksd, vsd)
    ws1 = fk.alloc_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, w.max_seq_len)
    ws2 = fk.alloc_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, w.max_seq_len)
    o1 = torch.empty((B, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    bt, sl = w.block_tables.cuda(), w.seq_lens.cuda()
    fk.fp8kv_paged_decode_per_head(w.q.cuda(), kc1, vc1, bt, sl, w.max_seq_len, ksd, vsd, w.sm_scale, 0, o1, ws1)
    fk.fp8kv_decode_step_per_head(w.q.cuda(), k[rows].cuda(), v[rows].cuda(), kc2, vc2, bt, sl, w.max_seq_len,
                                  ksd, vsd, w.sm_scale, 0, o2, ws2)
    torch.cuda.synchronize()
    assert fk.fp8kv_read_error(ws1) == 0 and fk.fp8kv_read_error(ws2) == 0
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2) and torch.equal(o1, o2)


def test_equal_head_scales_reproduce_the_per_tensor_calls_bit_for_bit():
    shape = workload.small_shape("llama33_70b_needle_128k", batch=2, len_lo=1, len_hi=1, needle_margin=None)
    w = workload.make_workload(shape, seed=19, lens=[5000, 333])
    s = w.shape
    ks = torch.full((s.num_kv_heads,), w.k_scale, dtype=torch.float32, device="cuda")
    vs = torch.full((s.num_kv_heads,), w.v_scale, dtype=torch.float32, device="cuda")
    kc1, vc1 = _caches(w)
    kc2, vc2 = _caches(w)
    fk.fp8kv_quant_append(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda(), kc1, vc1, w.k_scale, w.v_scale)
    fk.fp8kv_quant_append_per_head(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda(), kc2, vc2, ks, vs)
    ws = fk.alloc_workspace(2, s.num_q_heads, s.num_kv_heads, s.head_dim, w.max_seq_len)
    o1 = torch.empty((2, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    bt, sl = w.block_tables.cuda(), w.seq_lens.cuda()
    fk.fp8kv_paged_decode(w.q.cuda(), kc1, vc1, bt, sl, w.max_seq_len, w.k_scale, w.v_scale, w.sm_scale, 0, o1, ws)
    fk.fp8kv_paged_decode_per_head(w.q.cuda(), kc2, vc2, bt, sl, w.max_seq_len, ks, vs, w.sm_scale, 0, o2, ws)
    torch.cuda.synchronize()
    assert fk.fp8kv_read_error(ws) == 0
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2) and torch.equal(o1, o2)
