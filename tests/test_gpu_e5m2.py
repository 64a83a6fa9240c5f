"""GPU parity of the E5M2 cache: every bf16 pattern quantised bit-exactly,
attention against the fp64 oracle over E5M2 codes (small cases with ragged
tails and windows, every head layout, the full-size 8x20K and 128K-needle
layouts), and the fused step bit-identical to append-then-decode."""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import assert_attn_close

pytestmark = pytest.mark.gpu

E5M2_MAX = 57344.0


def _scale(x):
    s = float(np.float32(x.float().abs().max() / torch.tensor(E5M2_MAX)))
    return s if s > 0 else 1.0


def _is_nan_code(c):
    return ((c & 0x7C) == 0x7C) & ((c & 0x3) != 0)


@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.7])
def test_e5m2_append_every_bf16_pattern_bit_exact(scale):
    d, hkv = 128, 2
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    T = 65536 // (d * hkv)
    x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(T, hkv, d)
    nb = T // 16 + 3
    perm = torch.randperm(nb * 16, generator=torch.Generator().manual_seed(2))[:T].to(torch.int64)
    kc = torch.zeros((nb, hkv, 16, d), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    fk.fp8kv_quant_append_e5m2(x.cuda(), x.cuda(), perm.cuda(), kc, vc, scale, scale)
    torch.cuda.synchronize()
    got = kc.cpu()[perm // 16, :, perm % 16, :].numpy()
    ref = oracle.quantize_bf16_e5m2(workload.bf16_bits(x), scale)
    nan = np.isnan(x.float().numpy())
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(_is_nan_code(got[nan]))


class PagedE5M2:
    def __init__(self, w, history_only=False):
        s = w.shape
        self.w = w
        self.ks, self.vs = _scale(w.k), _scale(w.v)
        shape = (w.num_blocks, s.num_kv_heads, 16, s.head_dim)
        g = torch.Generator(device="cuda").manual_seed(5)
        self.kc = torch.randint(0, 256, shape, dtype=torch.uint8, device="cuda", generator=g)
        self.vc = torch.randint(0, 256, shape, dtype=torch.uint8, device="cuda", generator=g)
        keep = torch.ones(w.k.shape[0], dtype=torch.bool)
        if history_only:
            L = w.seq_lens.to(torch.int64)
            keep[w.new_token_rows()[L > 0]] = False
        if int(keep.sum()):
            fk.fp8kv_quant_append_e5m2(w.k[keep].cuda(), w.v[keep].cuda(), w.slot_mapping[keep].cuda(), self.kc,
                                       self.vc, self.ks, self.vs)
        self.q, self.bt, self.sl = w.q.cuda(), w.block_tables.cuda(), w.seq_lens.cuda()

    def _ws_out(self, window):
        s, B = self.w.shape, self.q.shape[0]
        ws = fk.alloc_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, self.w.max_seq_len, 16, window)
        return ws, torch.empty((B, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")

    def decode(self, window=0):
        ws, out = self._ws_out(window)
        fk.fp8kv_paged_decode_e5m2(self.q, self.kc, self.vc, self.bt, self.sl, self.w.max_seq_len, self.ks, self.vs,
                                   self.w.sm_scale, window, out, ws)
        torch.cuda.synchronize()
        return out, fk.fp8kv_read_error(ws)

    def step(self, window=0):
        w = self.w
        B = self.q.shape[0]
        kn = torch.zeros((B, w.shape.num_kv_heads, w.shape.head_dim), dtype=torch.bfloat16)
        vn = torch.zeros_like(kn)
        L = w.seq_lens.to(torch.int64)
        nz = L > 0
        kn[nz] = w.k[w.new_token_rows()[nz]]
        vn[nz] = w.v[w.new_token_rows()[nz]]
        ws, out = self._ws_out(window)
        fk.fp8kv_decode_step_e5m2(self.q, kn.cuda(), vn.cuda(), self.kc, self.vc, self.bt, self.sl, w.max_seq_len,
                                  self.ks, self.vs, w.sm_scale, window, out, ws)
        torch.cuda.synchronize()
        return out, fk.fp8kv_read_error(ws)

    def oracle(self, window):
        w = self.w
        kc = oracle.quantize_bf16_e5m2(workload.bf16_bits(w.k), self.ks)
        vc = oracle.quantize_bf16_e5m2(workload.bf16_bits(w.v), self.vs)
        return kc, vc, oracle.decode_attention_e5m2(workload.bf16_bits(w.q), kc, vc, w.seq_lens.numpy(), self.ks,
                                                    self.vs, w.sm_scale, window, nthreads=oracle.max_threads())


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("base,lens,windows", [
    ("llama31_8b_b1_4k", [1, 15, 16, 17, 33, 100, 0, 1000], (0, 17)),
    ("gptoss20b_b8_16k", [1, 63, 64, 65, 700], (0, 7)),
    ("gemma4e2b_b16_8k32k", [1, 17, 513, 3000], (0, 33)),
    ("llama33_70b_needle_128k", [3000, 40], (0,)),
])
def test_e5m2_small_cases_match_oracle(base, lens, windows):
    shape = workload.small_shape(base, batch=len(lens), len_lo=1, len_hi=1, needle_margin=None)
    w = workload.make_workload(shape, seed=23, lens=lens)
    pc = PagedE5M2(w)
    for win in windows:
        kc, vc, ref = pc.oracle(win)
        blk, off = w.slot_mapping // 16, w.slot_mapping % 16
        assert np.array_equal(pc.kc.cpu()[blk, :, off, :].numpy(), kc)
        assert np.array_equal(pc.vc.cpu()[blk, :, off, :].numpy(), vc)
        out, err = pc.decode(win)
        assert err == 0
        assert_attn_close(_f64(out), ref, f"e5m2 {base} window={win}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_e5m2_head_layouts(d, g):
    shape = workload.LayerShape(f"e{d}_{g}", 2 * g, 2, d, 3, 1, 1, (0,))
    w = workload.make_workload(shape, seed=g * 10 + d, lens=[777, 16, 35])
    pc = PagedE5M2(w)
    for win in (0, 50):
        out, err = pc.decode(win)
        assert err == 0
        assert_attn_close(_f64(out), pc.oracle(win)[2], f"e5m2 d={d} g={g} window={win}")


def test_e5m2_step_equals_append_then_decode():
    shape = workload.small_shape("llama31_8b_b8_20k", batch=4, len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=24, lens=[2999, 1, 16, 4097])
    full = PagedE5M2(w)
    part = PagedE5M2(w, history_only=True)
    o1, e1 = full.decode()
    o2, e2 = part.step()
    assert e1 == 0 and e2 == 0
    assert torch.equal(full.kc, part.kc) and torch.equal(full.vc, part.vc) and torch.equal(o1, o2)


@pytest.mark.parametrize("name", ["llama31_8b_b8_20k", "llama33_70b_needle_128k"])
def test_e5m2_full_size_matches_oracle(name):
    w = workload.make_workload(name, seed=0)
    pc = PagedE5M2(w)
    out, err = pc.decode()
    assert err == 0
    kc, vc, ref = pc.oracle(0)
    assert_attn_close(_f64(out), ref, f"e5m2 {name}")
    if w.needle_pos is not None:
        vh = oracle.e5m2_decode(vc[w.needle_pos]) * pc.vs
        g = w.shape.group
        expect = np.stack([vh[h // g] for h in range(w.shape.num_q_heads)])
        assert_attn_close(_f64(out)[0], expect, f"e5m2 {name} needle row")
