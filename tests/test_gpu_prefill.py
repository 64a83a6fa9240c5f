"""GPU parity of the chunked prefill over the E4M3 cache: every head layout
with ragged lengths and chunk sizes (one token, a ragged tail of a tile, whole
prompts), sliding windows, empty sequences, the full-size 8x20K serving batch
and the 128K needle with sampled rows, and the device-side argument checks."""
import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import BF16_HALF_ULP_REL, assert_attn_close_bf16_floor as assert_attn_close
from tests.gpu_harness import Paged

pytestmark = pytest.mark.gpu


def _ws(p: Paged, mq, window):
    s = p.w.shape
    return fk.alloc_prefill_workspace(p.q.shape[0], mq, p.w.max_seq_len, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                      16, window)


def _run(p: Paged, q, q_starts, window, max_q_len=None, block_tables=None, seq_lens=None, ws=None):
    w = p.w
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    qs = q_starts.cuda()
    mq = int((q_starts[1:] - q_starts[:-1]).max()) if max_q_len is None else max_q_len
    own_ws = ws is None
    ws = _ws(p, mq, window) if own_ws else ws
    fk.fp8kv_paged_prefill(q.cuda(), p.k_cache, p.v_cache,
                           p.block_tables if block_tables is None else block_tables,
                           p.seq_lens if seq_lens is None else seq_lens, qs, mq, w.max_seq_len,
                           w.k_scale, w.v_scale, w.sm_scale, window, out, ws)
    torch.cuda.synchronize()
    if own_ws:
        assert fk.fp8kv_read_error(ws) == 0
    return out.float().cpu().numpy()


def _oracle(p: Paged, q, q_lens, window):
    kc, vc = p.gathered_codes()
    w = p.w
    return oracle.prefill_attention(workload.bf16_bits(q), kc, vc, w.seq_lens.numpy(), np.asarray(q_lens),
                                    w.k_scale, w.v_scale, w.sm_scale, window, nthreads=oracle.max_threads())


LAYOUTS = ["llama31_8b_b8_20k", "gptoss20b_b8_16k", "gemma4e2b_b16_8k32k", "llama33_70b_needle_128k"]


@pytest.mark.parametrize("base", LAYOUTS)
@pytest.mark.parametrize("window", [0, 40])
def test_prefill_small_every_layout(base, window):
    lens = [1, 17, 300, 95, 0, 64, 129]
    q_lens = [1, 17, 37, 95, 0, 1, 64]          # whole prompts, one token, ragged tails of a tile
    shape = workload.small_shape(base, len(lens), 1, 1, needle_margin=None)
    w = workload.make_workload(shape, seed=3, lens=lens)
    p = Paged(w, seed=3)
    p.append_all()
    q, qs = workload.prefill_queries(w, q_lens, seed=3)
    got = _run(p, q, qs, window)
    ref = _oracle(p, q, q_lens, window)
    assert_attn_close(got, ref, f"{base} window={window}")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prefill_seeds_and_windows(seed):
    shape = workload.small_shape("llama31_8b_b8_20k", 3, 200, 700)
    w = workload.make_workload(shape, seed=seed)
    p = Paged(w, seed=seed)
    p.append_all()
    L = w.seq_lens.tolist()
    q_lens = [L[0], min(L[1], 130), 33]
    q, qs = workload.prefill_queries(w, q_lens, seed=seed)
    for window in (0, 16, 128, 5000):
        got = _run(p, q, qs, window)
        ref = _oracle(p, q, q_lens, window)
        assert_attn_close(got, ref, f"seed={seed} window={window}")


def test_prefill_window_one_is_value_of_own_token():
    """window = 1: each row attends only its own key, so the output is that
    token's decoded V times v_scale; the only error left is the rounding of
    that value to bf16 (at most 2^-8 of it, plus the fp32 product's 2^-24)."""
    shape = workload.small_shape("gptoss20b_b8_16k", 2, 50, 90)
    w = workload.make_workload(shape, seed=4)
    p = Paged(w, seed=4)
    p.append_all()
    q_lens = [20, 33]
    q, qs = workload.prefill_queries(w, q_lens, seed=4)
    got = _run(p, q, qs, 1).astype(np.float64)
    ref = _oracle(p, q, q_lens, 1)
    assert np.all(np.abs(got - ref) <= BF16_HALF_ULP_REL * (1 + 2.0 ** -16) * np.abs(ref))


def test_prefill_max_q_len_larger_than_needed_and_zero_chunks():
    """A grid sized for a longer chunk than any sequence has, and sequences
    with no new tokens between others, leave no row unwritten and write no
    row twice."""
    lens = [40, 0, 33, 16]
    q_lens = [40, 0, 0, 16]
    shape = workload.small_shape("llama31_8b_b8_20k", len(lens), 1, 1)
    w = workload.make_workload(shape, seed=6, lens=lens)
    p = Paged(w, seed=6)
    p.append_all()
    q, qs = workload.prefill_queries(w, q_lens, seed=6)
    got = _run(p, q, qs, 0, max_q_len=40)
    ref = _oracle(p, q, q_lens, 0)
    assert np.all(np.isfinite(got))
    assert_attn_close(got, ref, "zero chunks")


def _oracle_rows(p: Paged, codes, q, q_lens, b, i0, i1, window):
    """Oracle for chunk rows [i0, i1) of sequence b: they are the last i1 - i0
    query tokens of the sequence cut just after row i1 - 1's position."""
    w = p.w
    kc, vc = codes
    s0 = int(w.seq_starts.numpy()[b])
    L = int(w.seq_lens.numpy()[b])
    qs = np.concatenate([[0], np.cumsum(q_lens)])
    end = L - q_lens[b] + i1                    # tokens the cut sequence holds
    return oracle.prefill_attention(workload.bf16_bits(q[qs[b] + i0:qs[b] + i1]), kc[s0:s0 + end],
                                    vc[s0:s0 + end], [end], [i1 - i0], w.k_scale, w.v_scale, w.sm_scale, window,
                                    nthreads=oracle.max_threads())


def _tile_blocks(q_len, tile_tokens, whole_tiles):
    """Row blocks to check: the whole tiles listed, and the two rows on both
    sides of every tile boundary of the chunk."""
    blocks = [(t * tile_tokens, min(q_len, (t + 1) * tile_tokens)) for t in whole_tiles]
    for bnd in range(tile_tokens, q_len, tile_tokens):
        blocks.append((bnd - 2, bnd + 2))
    blocks.append((q_len - 1, q_len))
    return blocks


def test_prefill_full_size_serving_batch_tiles_and_boundaries():
    """8 sequences of ~20K tokens, the last 512 of each a prefill chunk.  A
    tile holds 128 (token, head) rows = 32 tokens at g = 4: the first and the
    last tile of two sequences are compared whole, and every tile boundary of
    every sequence on both sides."""
    w = workload.make_workload("llama31_8b_b8_20k", seed=0)
    p = Paged(w, seed=0)
    p.append_all()
    q_lens = [512] * 8
    q, qs = workload.prefill_queries(w, q_lens, seed=0)
    got = _run(p, q, qs, 0)
    codes = p.gathered_codes()
    tile_tokens = 128 // (w.shape.num_q_heads // w.shape.num_kv_heads)
    for b in range(8):
        whole = [0, 512 // tile_tokens - 1] if b in (0, 7) else []
        for i0, i1 in _tile_blocks(512, tile_tokens, whole):
            ref = _oracle_rows(p, codes, q, q_lens, b, i0, i1, 0)
            assert_attn_close(got[qs[b] + i0:qs[b] + i1], ref, "8x20K chunk 512, seq %d rows %d..%d" % (b, i0, i1))


def test_prefill_needle_128k_tiles_and_boundaries():
    """The 131,072-token needle layout with a 256-token chunk at the end; the
    chunk's last row carries the query the needle key was planted for, so
    that row must retrieve the needle from among 128K keys.  A tile holds 16
    tokens at g = 8: the first and the last tile are compared whole, with
    both sides of every tile boundary."""
    w = workload.make_workload("llama33_70b_needle_128k", seed=0)
    p = Paged(w, seed=0)
    p.append_all()
    q_lens = [256]
    q, qs = workload.prefill_queries(w, q_lens, seed=0)
    q[255] = w.q[0]
    got = _run(p, q, qs, 0)
    codes = p.gathered_codes()
    tile_tokens = 128 // (w.shape.num_q_heads // w.shape.num_kv_heads)
    for i0, i1 in _tile_blocks(256, tile_tokens, [0, 256 // tile_tokens - 1]):
        ref = _oracle_rows(p, codes, q, q_lens, 0, i0, i1, 0)
        assert_attn_close(got[i0:i1], ref, "128K chunk 256 rows %d..%d" % (i0, i1))


def test_prefill_reports_bad_block_id_and_lengths():
    """Device-side checks: a block id outside the cache reads block 0 and is
    reported; a chunk longer than its sequence is clamped and reported."""
    shape = workload.small_shape("llama31_8b_b8_20k", 2, 60, 60)
    w = workload.make_workload(shape, seed=8)
    p = Paged(w, seed=8)
    p.append_all()
    q_lens = [20, 20]
    q, qs = workload.prefill_queries(w, q_lens, seed=8)
    ws = _ws(p, 20, 0)
    bt = p.block_tables.clone()
    bt[1, 0] = p.num_blocks + 5
    got = _run(p, q, qs, 0, block_tables=bt, ws=ws)
    assert fk.fp8kv_read_error(ws) == 1
    ref = _oracle(p, q, q_lens, 0)
    assert_attn_close(got[:20], ref[:20], "sequence with valid pages")
    assert np.all(np.isfinite(got))
    short = p.seq_lens.clone()
    short[0] = 10                                  # 20 query rows but only 10 tokens
    _run(p, q, qs, 0, seq_lens=short, ws=ws)
    assert fk.fp8kv_read_error(ws) == 1
    _run(p, q, qs, 0, ws=ws)
    assert fk.fp8kv_read_error(ws) == 0


@pytest.mark.parametrize("base", ["llama31_8b_b8_20k", "gemma4e2b_b16_8k32k"])
def test_prefill_short_chunk_long_context_splits_the_keys(base):
    """Few query tiles over a long context: the key range of each tile is
    split over many CTAs and their FP32 partials are merged."""
    lens = [5000, 3100]
    q_lens = [16, 3]
    shape = workload.small_shape(base, len(lens), 1, 1)
    w = workload.make_workload(shape, seed=9, lens=lens)
    p = Paged(w, seed=9)
    p.append_all()
    s = w.shape
    n_ws = fk.fp8kv_paged_prefill_workspace_size(2, 16, w.max_seq_len, s.num_q_heads, s.num_kv_heads, s.head_dim)
    assert n_ws > 4096      # the plan splits: the workspace holds partials
    q, qs = workload.prefill_queries(w, q_lens, seed=9)
    for window in (0, 700):
        got = _run(p, q, qs, window)
        ref = _oracle(p, q, q_lens, window)
        assert_attn_close(got, ref, f"{base} split window={window}")


@pytest.mark.parametrize("base", ["llama31_8b_b8_20k", "gptoss20b_b8_16k", "gemma4e2b_b16_8k32k"])
@pytest.mark.parametrize("sm_scale", [-0.07, 0.0])
def test_prefill_negative_and_zero_softmax_scale(base, sm_scale):
    # the softmax scale is any finite number: a negative one reverses the
    # order of the scores, zero makes every attended key weigh the same
    lens = [700, 300, 129]
    q_lens = [200, 64, 129]                     # 200 tokens span several tiles at every g
    shape = workload.small_shape(base, len(lens), 1, 1, needle_margin=None)
    w = workload.make_workload(shape, seed=8, lens=lens)
    w.sm_scale = sm_scale
    p = Paged(w, seed=8)
    p.append_all()
    q, qs = workload.prefill_queries(w, q_lens, seed=8)
    for window in (0, 50):
        got = _run(p, q, qs, window)
        ref = _oracle(p, q, q_lens, window)
        assert_attn_close(got, ref, f"{base} sm_scale={sm_scale} window={window}")
