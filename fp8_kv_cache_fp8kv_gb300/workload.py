"""Seeded synthetic decode workloads (input generation only).

This module draws the inputs that both the CUDA library and the CPU oracle
consume: bf16 queries and keys/values, context lengths, a shuffled paged block
table and its slot mapping, and the per-tensor scales.  It holds none of the
attention or quantisation arithmetic; the only numerics here shape inputs
(normal draws, the amax/448 scale choice the workloads prescribe, and the
linear solve that plants the long-context needle key).

Shapes follow the model layers the FP8 KV pages measure (phantomic12 summary
of the vLLM FP8 KV-cache blog, "DECODE COST" and "THROUGHPUT": Llama-3.1-8B,
gpt-oss-20b with a 128-token window, gemma-4-E2B with head_dim 256 and a
512-token window, Llama-3.3-70B at 128K for the needle test).  Synthetic
normal data stands in for the pages' serving traffic and their 128K
needle-in-a-haystack set, neither of which exists here.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import numpy as np
import torch

BLOCK_SIZE = 16
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    batch: int
    len_lo: int          # context lengths uniform in [len_lo, len_hi]
    len_hi: int
    windows: tuple       # windows this workload is run with (0 = full)
    kv_std: float = 1.0
    needle_margin: float | None = None

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


# The five decode workloads (and one g = 16 layer).  "~16K" for the
# gpt-oss-like layer is read as uniform in [14000, 18000], the same +-2000
# spread as the ~20K serving batch.
CONFIGS = {
    "llama31_8b_b1_4k": LayerShape("llama31_8b_b1_4k", 32, 8, 128, 1, 4096, 4096, (0,)),
    "llama31_8b_b8_20k": LayerShape("llama31_8b_b8_20k", 32, 8, 128, 8, 18000, 22000, (0,)),
    "gptoss20b_b8_16k": LayerShape("gptoss20b_b8_16k", 64, 8, 64, 8, 14000, 18000, (0, 128)),
    "gemma4e2b_b16_8k32k": LayerShape("gemma4e2b_b16_8k32k", 8, 1, 256, 16, 8192, 32768, (0, 512)),
    "llama33_70b_needle_128k": LayerShape("llama33_70b_needle_128k", 64, 8, 128, 1, 131072, 131072,
                                          (0,), kv_std=0.5, needle_margin=12.0),
    # not one of the five: 16 query heads per kv head, to measure that each
    # page is read once at g = 16
    "g16_b4_32k": LayerShape("g16_b4_32k", 64, 4, 128, 4, 28000, 36000, (0,)),
}


@dataclasses.dataclass
class Workload:
    shape: LayerShape
    seed: int
    q: torch.Tensor              # bf16 [B, Hq, d]
    k: torch.Tensor              # bf16 [total_tokens, Hkv, d], logical order
    v: torch.Tensor              # bf16 [total_tokens, Hkv, d]
    seq_lens: torch.Tensor       # int32 [B]  (includes the token appended this step)
    seq_starts: torch.Tensor     # int64 [B]  first logical token of each sequence
    block_tables: torch.Tensor   # int32 [B, max_blocks_per_seq], physical block ids
    slot_mapping: torch.Tensor   # int64 [total_tokens], physical slot of each token
    num_blocks: int
    k_scale: float               # fp32 value, amax(|K|)/448
    v_scale: float
    sm_scale: float              # fp32 value, 1/sqrt(d)
    needle_pos: int | None = None

    @property
    def block_size(self) -> int:
        return BLOCK_SIZE

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    def new_token_rows(self) -> torch.Tensor:
        """Logical row of each sequence's newest token (appended in the step)."""
        return self.seq_starts + self.seq_lens.to(torch.int64) - 1

    def digest(self) -> str:
        """SHA-256 over every input tensor's bytes (recorded with results)."""
        h = hashlib.sha256()
        for t in (self.q, self.k, self.v, self.seq_lens, self.block_tables, self.slot_mapping):
            h.update(t.contiguous().view(torch.uint8).numpy().tobytes())
        h.update(np.array([self.k_scale, self.v_scale, self.sm_scale], np.float32).tobytes())
        return h.hexdigest()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 view of a bf16 tensor (what the C oracle takes)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def per_tensor_scale(x: torch.Tensor) -> float:
    """amax(|x|)/448 as an fp32 value (the scale choice the workloads fix)."""
    amax = x.abs().max().to(torch.float32)
    s = (amax / torch.tensor(E4M3_MAX, dtype=torch.float32)).item()
    return float(np.float32(s)) if s > 0 else 1.0


def _paged_layout(seq_lens: torch.Tensor, gen: torch.Generator):
    B = int(seq_lens.numel())
    blocks_per_seq = [(int(L) + BLOCK_SIZE - 1) // BLOCK_SIZE for L in seq_lens.tolist()]
    num_blocks = max(1, sum(blocks_per_seq))
    max_blocks = max([1] + blocks_per_seq)
    perm = torch.randperm(num_blocks, generator=gen).to(torch.int32)
    tables = torch.zeros((B, max_blocks), dtype=torch.int32)
    starts = torch.zeros(B, dtype=torch.int64)
    slots = []
    base = 0
    tok = 0
    for b in range(B):
        nb = blocks_per_seq[b]
        tables[b, :nb] = perm[base:base + nb]
        L = int(seq_lens[b])
        starts[b] = tok
        idx = torch.arange(L, dtype=torch.int64)
        slots.append(tables[b, idx // BLOCK_SIZE].to(torch.int64) * BLOCK_SIZE + idx % BLOCK_SIZE)
        base += nb
        tok += L
    slot_mapping = torch.cat(slots) if slots else torch.zeros(0, dtype=torch.int64)
    return tables, starts, slot_mapping, num_blocks


def _plant_needle(q: torch.Tensor, k: torch.Tensor, shape: LayerShape, L: int, pos: int,
                  sm_scale: float) -> None:
    """Overwrites key row `pos` (batch 1) so that, for every query head h of each
    kv head, the needle's logit beats the log-sum-exp of all other logits by at
    least `needle_margin`.  Other logits obey |s| <= sm_scale*|q_h|*max|k_t|
    (Cauchy-Schwarz), so their log-sum-exp is at most that bound + ln(L-1);
    the needle key is the minimum-norm key meeting bound + ln(L-1) + margin
    for all g query heads at once (it lies in the span of the group's queries).
    """
    g, d = shape.group, shape.head_dim
    for hk in range(shape.num_kv_heads):
        Qg = q[0, hk * g:(hk + 1) * g, :].to(torch.float64).numpy()      # [g, d]
        keys = k[:L, hk, :].to(torch.float64)
        norms = torch.linalg.vector_norm(keys, dim=1)
        norms[pos] = 0.0
        kmax = float(norms.max())
        qn = np.linalg.norm(Qg, axis=1)
        target = (sm_scale * qn * kmax + math.log(max(L - 1, 1)) + shape.needle_margin) / sm_scale
        coef = np.linalg.solve(Qg @ Qg.T, target)
        k[pos, hk, :] = torch.from_numpy(Qg.T @ coef).to(torch.bfloat16)


def make_workload(name_or_shape, seed: int = 0, lens=None) -> Workload:
    """Draws one seeded workload.  `lens` overrides the context lengths (used
    for small parity cases that keep a config's head layout)."""
    shape = CONFIGS[name_or_shape] if isinstance(name_or_shape, str) else name_or_shape
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    B, Hq, Hkv, d = shape.batch, shape.num_q_heads, shape.num_kv_heads, shape.head_dim
    if lens is None:
        seq_lens = torch.randint(shape.len_lo, shape.len_hi + 1, (B,), generator=gen, dtype=torch.int64)
    else:
        seq_lens = torch.as_tensor(lens, dtype=torch.int64).reshape(-1)
        B = int(seq_lens.numel())
    seq_lens = seq_lens.to(torch.int32)
    total = int(seq_lens.to(torch.int64).sum())
    q = torch.randn((B, Hq, d), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    k = (torch.randn((total, Hkv, d), generator=gen, dtype=torch.float32) * shape.kv_std).to(torch.bfloat16)
    v = (torch.randn((total, Hkv, d), generator=gen, dtype=torch.float32) * shape.kv_std).to(torch.bfloat16)
    sm_scale = float(np.float32(1.0 / math.sqrt(d)))
    needle_pos = None
    if shape.needle_margin is not None and B == 1 and total >= 2:
        L = int(seq_lens[0])
        needle_pos = int(torch.randint(0, L - 1, (1,), generator=gen).item())
        _plant_needle(q, k, shape, L, needle_pos, sm_scale)
    tables, starts, slot_mapping, num_blocks = _paged_layout(seq_lens, gen)
    return Workload(shape=shape, seed=int(seed), q=q, k=k, v=v, seq_lens=seq_lens,
                    seq_starts=starts, block_tables=tables, slot_mapping=slot_mapping,
                    num_blocks=num_blocks, k_scale=per_tensor_scale(k),
                    v_scale=per_tensor_scale(v), sm_scale=sm_scale, needle_pos=needle_pos)


def small_shape(base: str, batch: int, len_lo: int, len_hi: int, **kw) -> LayerShape:
    """A config's head layout with other batch/length settings (parity cases)."""
    s = CONFIGS[base]
    return dataclasses.replace(s, name=f"{s.name}_small", batch=batch, len_lo=len_lo,
                               len_hi=len_hi, **kw)


def prefill_queries(w: Workload, q_lens, seed: int = 0):
    """Seeded queries for a prefill chunk: sequence b's last q_lens[b] tokens,
    packed sequence after sequence, bf16 [sum q_lens, Hq, d] ~ N(0, 1), with
    the int32 [B + 1] cumulative row offsets."""
    q_lens = torch.as_tensor(q_lens, dtype=torch.int64).reshape(-1)
    assert q_lens.numel() == w.seq_lens.numel() and bool((q_lens <= w.seq_lens.to(torch.int64)).all())
    gen = torch.Generator(device="cpu").manual_seed(int(seed) + 7)
    R = int(q_lens.sum())
    q = torch.randn((R, w.shape.num_q_heads, w.shape.head_dim), generator=gen,
                    dtype=torch.float32).to(torch.bfloat16)
    starts = torch.zeros(q_lens.numel() + 1, dtype=torch.int32)
    starts[1:] = torch.cumsum(q_lens, 0).to(torch.int32)
    return q, starts
