"""GPU parity of the split merge of the tensor-core engine.

A (sequence, kv head) unit whose pages span several CTAs leaves one FP32
partial per CTA.  When the launch plan gives units few partials, the CTA
that completes a unit (the last to count its partial on the unit's workspace
counter) combines them, staging chunks of partials through shared memory;
otherwise a separate merge kernel does.  The cases here plan the launch for
many sequences at max_seq_len and then run one long sequence among short
ones, so the long sequence's units are split over hundreds of CTAs and the
in-grid merge takes many staging chunks.  Each case runs three times on one
workspace (the counters must be back at zero after every call) and is
compared element by element with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import assert_attn_close
from tests.gpu_harness import Paged, oracle_codes, oracle_out

pytestmark = pytest.mark.gpu

CASES = [
    # (layout, batch, long length, short length, max_seq_len of the plan); the
    # short sequences span 3 pages each (outputs of 1-token sequences are bare
    # value rows, whose bf16 rounding alone would fill the mean-error budget)
    ("gemma4e2b_b16_8k32k", 128, 2048, 48, 2048),   # d = 256, g = 8: 8 KB partials, ~80 per unit, ~8 chunks
    ("g16_b4_32k", 128, 2048, 48, 2048),            # g = 16 native (two MMA n-tiles per unit), 2 chunks
    ("gptoss20b_b8_16k", 64, 4096, 48, 4096),       # d = 64, six warps per CTA
    ("llama31_8b_b8_20k", 8, 20000, 48, 22000),     # the 8 x 20K plan with one long sequence
]


@pytest.mark.parametrize("base,batch,long_len,short_len,plan_len", CASES)
def test_merge_of_heavily_split_units_matches_oracle(base, batch, long_len, short_len, plan_len):
    shape = workload.small_shape(base, batch=batch, len_lo=1, len_hi=1, needle_margin=None)
    lens = [long_len] + [short_len] * (batch - 1)
    w = workload.make_workload(shape, seed=21, lens=lens)
    pc = Paged(w)
    pc.append_all()
    s = w.shape
    wide = torch.zeros((batch, -(-plan_len // 16)), dtype=torch.int32, device="cuda")
    wide[:, :w.max_blocks_per_seq] = pc.block_tables
    ws = fk.alloc_workspace(batch, s.num_q_heads, s.num_kv_heads, s.head_dim, plan_len)
    kc, vc = oracle_codes(w)
    ref = oracle_out(w, kc, vc, 0)
    outs = []
    for _ in range(3):
        out = torch.full((batch, s.num_q_heads, s.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
        fk.fp8kv_paged_decode(pc.q, pc.k_cache, pc.v_cache, wide, pc.seq_lens, plan_len, w.k_scale, w.v_scale,
                              w.sm_scale, 0, out, ws)
        torch.cuda.synchronize()
        assert fk.fp8kv_read_error(ws) == 0
        outs.append(out)
    got = outs[0].float().cpu().numpy().astype(np.float64)
    assert_attn_close(got, ref, f"{base} B={batch} long={long_len}")
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
