"""Shared GPU-test plumbing: put a seeded workload into a paged device cache
through fp8kv_quant_append, run fp8kv_paged_decode (or the fused
fp8kv_decode_step), and fetch what the oracle needs to check them."""
import numpy as np
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload


class Paged:
    def __init__(self, w: workload.Workload, fill_byte=None, device="cuda", extra_blocks=0,
                 seed=0):
        s = w.shape
        self.w = w
        self.num_blocks = w.num_blocks + extra_blocks
        shape = (self.num_blocks, s.num_kv_heads, workload.BLOCK_SIZE, s.head_dim)
        if fill_byte is None:
            g = torch.Generator(device=device).manual_seed(seed + 99)
            self.k_cache = torch.randint(0, 256, shape, dtype=torch.uint8, device=device, generator=g)
            self.v_cache = torch.randint(0, 256, shape, dtype=torch.uint8, device=device, generator=g)
        else:
            self.k_cache = torch.full(shape, fill_byte, dtype=torch.uint8, device=device)
            self.v_cache = torch.full(shape, fill_byte, dtype=torch.uint8, device=device)
        self.q = w.q.to(device)
        self.block_tables = w.block_tables.to(device)
        self.seq_lens = w.seq_lens.to(device)

    def append_all(self):
        w = self.w
        if w.k.shape[0] == 0:
            return
        fk.fp8kv_quant_append(w.k.to("cuda"), w.v.to("cuda"), w.slot_mapping.to("cuda"),
                              self.k_cache, self.v_cache, w.k_scale, w.v_scale)

    def append_history(self):
        """Append every token except each sequence's newest one."""
        w = self.w
        keep = torch.ones(w.k.shape[0], dtype=torch.bool)
        L = w.seq_lens.to(torch.int64)
        keep[w.new_token_rows()[L > 0]] = False
        if int(keep.sum()) == 0:
            return
        fk.fp8kv_quant_append(w.k[keep].to("cuda"), w.v[keep].to("cuda"), w.slot_mapping[keep].to("cuda"),
                              self.k_cache, self.v_cache, w.k_scale, w.v_scale)

    def new_rows(self):
        """bf16 [B, Hkv, D]: each sequence's newest K and V row (zeros where empty)."""
        w = self.w
        s = w.shape
        B = w.seq_lens.shape[0]
        kn = torch.zeros((B, s.num_kv_heads, s.head_dim), dtype=torch.bfloat16)
        vn = torch.zeros_like(kn)
        L = w.seq_lens.to(torch.int64)
        nz = L > 0
        kn[nz] = w.k[w.new_token_rows()[nz]]
        vn[nz] = w.v[w.new_token_rows()[nz]]
        return kn.to("cuda"), vn.to("cuda")

    def step(self, window=0, out=None):
        """One fused decode step over a cache holding the history only."""
        s = self.w.shape
        B = self.q.shape[0]
        mx = self.w.max_seq_len
        kn, vn = self.new_rows()
        ws = fk.alloc_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, mx, 16, window)
        out = torch.empty((B, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda") if out is None else out
        fk.fp8kv_decode_step(self.q, kn, vn, self.k_cache, self.v_cache, self.block_tables, self.seq_lens, mx,
                             self.w.k_scale, self.w.v_scale, self.w.sm_scale, window, out, ws)
        torch.cuda.synchronize()
        return out, fk.fp8kv_read_error(ws)

    def gathered_codes(self):
        """Cache codes of every logical token, [T, Hkv, D] (host)."""
        kc = self.k_cache.cpu()
        vc = self.v_cache.cpu()
        sm = self.w.slot_mapping
        blk, off = sm // workload.BLOCK_SIZE, sm % workload.BLOCK_SIZE
        return kc[blk, :, off, :].numpy(), vc[blk, :, off, :].numpy()

    def decode(self, window=0, max_seq_len=None, block_tables=None, out=None, engine=None):
        s = self.w.shape
        B = self.q.shape[0]
        mx = self.w.max_seq_len if max_seq_len is None else max_seq_len
        bt = self.block_tables if block_tables is None else block_tables
        ws = fk.alloc_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, mx, 16, window)
        out = torch.empty((B, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda") if out is None else out
        if engine is None:
            fk.fp8kv_paged_decode(self.q, self.k_cache, self.v_cache, bt, self.seq_lens, mx,
                                  self.w.k_scale, self.w.v_scale, self.w.sm_scale, window, out, ws)
        else:
            fk.fp8kv_paged_decode_engine(self.q, self.k_cache, self.v_cache, bt, self.seq_lens, mx,
                                         self.w.k_scale, self.w.v_scale, self.w.sm_scale, window, out, ws,
                                         engine)
        torch.cuda.synchronize()
        err = fk.fp8kv_read_error(ws)
        return out, err


def oracle_codes(w):
    kc = oracle.quantize_bf16(workload.bf16_bits(w.k), w.k_scale)
    vc = oracle.quantize_bf16(workload.bf16_bits(w.v), w.v_scale)
    return kc, vc


def oracle_out(w, kc, vc, window):
    return oracle.decode_attention(workload.bf16_bits(w.q), kc, vc, w.seq_lens.numpy(), w.k_scale,
                                   w.v_scale, w.sm_scale, window, nthreads=oracle.max_threads())
