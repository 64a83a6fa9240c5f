"""GPU parity of the bf16-cache twin (fp8kv_paged_decode_bf16) against the
fp64 oracle over the same bf16 values: max|err| <= 8e-3, mean|err| <= 1e-3,
small cases with ragged tails and windows, every supported head layout
(d = 64, 128, 256), NaN garbage in unwritten slots, and the full-size 8x20K,
128K-needle and gemma-like (d = 256) layouts."""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import assert_attn_close

pytestmark = pytest.mark.gpu


class PagedBf16:
    def __init__(self, w, fill_bits=None, seed=0):
        s = w.shape
        self.w = w
        shape = (w.num_blocks, s.num_kv_heads, workload.BLOCK_SIZE, s.head_dim)
        if fill_bits is None:
            g = torch.Generator(device="cuda").manual_seed(seed + 7)
            # random finite bf16 garbage (|x| < 2^8) in every slot the workload does not write
            self.k_cache = (torch.rand(shape, generator=g, device="cuda") * 512 - 256).to(torch.bfloat16)
            self.v_cache = (torch.rand(shape, generator=g, device="cuda") * 512 - 256).to(torch.bfloat16)
        else:
            self.k_cache = torch.full(shape, 0, dtype=torch.int16, device="cuda").fill_(fill_bits).view(torch.bfloat16)
            self.v_cache = self.k_cache.clone()
        sm = w.slot_mapping.to("cuda")
        blk, off = sm // workload.BLOCK_SIZE, sm % workload.BLOCK_SIZE
        if w.k.shape[0]:
            self.k_cache[blk, :, off, :] = w.k.to("cuda")
            self.v_cache[blk, :, off, :] = w.v.to("cuda")
        self.q = w.q.to("cuda")
        self.block_tables = w.block_tables.to("cuda")
        self.seq_lens = w.seq_lens.to("cuda")

    def decode(self, window=0):
        s = self.w.shape
        B = self.q.shape[0]
        ws = fk.alloc_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, self.w.max_seq_len, 16, window)
        out = torch.empty((B, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        fk.fp8kv_paged_decode_bf16(self.q, self.k_cache, self.v_cache, self.block_tables, self.seq_lens,
                                   self.w.max_seq_len, self.w.sm_scale, window, out, ws)
        torch.cuda.synchronize()
        return out, fk.fp8kv_read_error(ws)


def oracle_bf16(w, window):
    return oracle.decode_attention_bf16(workload.bf16_bits(w.q), workload.bf16_bits(w.k), workload.bf16_bits(w.v),
                                        w.seq_lens.numpy(), w.sm_scale, window, nthreads=oracle.max_threads())


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("base,lens,windows", [
    ("llama31_8b_b1_4k", [1, 15, 16, 17, 33, 100, 0, 1000], (0, 1, 17)),
    ("llama31_8b_b8_20k", [2999, 1234, 16, 4097], (0, 128)),
    ("gptoss20b_b8_16k", [1, 63, 64, 65, 700, 2500], (0, 128, 7)),
    ("llama33_70b_needle_128k", [3000, 40], (0, 16)),
    ("gemma4e2b_b16_8k32k", [1, 17, 511, 512, 513, 3000], (0, 512, 33)),
])
def test_bf16_small_cases_match_oracle(base, lens, windows):
    shape = workload.small_shape(base, batch=len(lens), len_lo=1, len_hi=1, needle_margin=None)
    w = workload.make_workload(shape, seed=13, lens=lens)
    pc = PagedBf16(w)
    for win in windows:
        out, err = pc.decode(window=win)
        assert err == 0
        assert_attn_close(_f64(out), oracle_bf16(w, win), f"bf16 {base} window={win}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_bf16_every_supported_head_layout(d, g):
    hkv = 2
    shape = workload.LayerShape(f"b{d}_{g}", hkv * g, hkv, d, 3, 1, 1, (0,))
    w = workload.make_workload(shape, seed=g * 100 + d, lens=[777, 16, 35])
    pc = PagedBf16(w)
    for win in (0, 50):
        out, err = pc.decode(window=win)
        assert err == 0
        assert_attn_close(_f64(out), oracle_bf16(w, win), f"bf16 d={d} g={g} window={win}")


def test_bf16_unwritten_nan_slots_never_leak():
    shape = workload.small_shape("llama31_8b_b8_20k", batch=3, len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=14, lens=[33, 1, 250])
    pc = PagedBf16(w, fill_bits=-1)  # 0xFFFF: a NaN in every unwritten slot
    for win in (0, 3, 20):
        out, err = pc.decode(window=win)
        assert err == 0 and torch.isfinite(out.float()).all()
        assert_attn_close(_f64(out), oracle_bf16(w, win), f"bf16 nan-filled window={win}")


@pytest.mark.parametrize("name", ["llama31_8b_b8_20k", "llama33_70b_needle_128k", "gemma4e2b_b16_8k32k"])
def test_bf16_full_size_matches_oracle(name):
    w = workload.make_workload(name, seed=0)
    pc = PagedBf16(w)
    out, err = pc.decode()
    assert err == 0
    assert_attn_close(_f64(out), oracle_bf16(w, 0), f"bf16 {name}")
    if w.needle_pos is not None:
        vn = w.v[w.needle_pos].double().numpy()
        g = w.shape.group
        expect = np.stack([vn[h // g] for h in range(w.shape.num_q_heads)])
        assert_attn_close(_f64(out)[0], expect, f"bf16 {name} needle row")
