"""GPU parity: libfp8kv (through its C ABI) against the CPU oracle.

Cache codes must match bit for bit; attention outputs must meet
max|err| <= 8e-3 and mean|err| <= 1e-3 against the fp64 oracle evaluated on
the same codes.  Small cases span several pages, splits and ragged tails; the
full-size cases run every workload at the size and in the launch
configuration the benchmark times, comparing every output element.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import workload
from tests._tol import assert_attn_close
from tests.gpu_harness import Paged, oracle_codes, oracle_out

pytestmark = pytest.mark.gpu


def _as_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


# ------------------------------------------------------------ quant_append

@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.7, float(np.float32(2.75 / 448))])
def test_quant_append_every_bf16_pattern_bit_exact(scale):
    d, hkv = 128, 2
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    T = 65536 // (d * hkv)
    x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(T, hkv, d)
    y = torch.from_numpy(np.roll(bits, 12345).view(np.int16).copy()).view(torch.bfloat16).reshape(T, hkv, d)
    nb = T // 16 + 3
    perm = torch.randperm(nb * 16, generator=torch.Generator().manual_seed(1))[:T].to(torch.int64)
    kc = torch.zeros((nb, hkv, 16, d), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    fk.fp8kv_quant_append(x.cuda(), y.cuda(), perm.cuda(), kc, vc, scale, scale * 2)
    torch.cuda.synchronize()
    gk = kc.cpu()[perm // 16, :, perm % 16, :].numpy()
    gv = vc.cpu()[perm // 16, :, perm % 16, :].numpy()
    for got, src, s in ((gk, x, scale), (gv, y, scale * 2)):
        ref = oracle.quantize_bf16(workload.bf16_bits(src), s)
        srcf = src.float().numpy()
        nan = np.isnan(srcf)
        assert np.array_equal(got[~nan], ref[~nan])
        assert np.all((got[nan] & 0x7F) == 0x7F)


def test_quant_append_skips_padding_and_out_of_range_slots():
    d, hkv, nb = 64, 1, 4
    x = torch.randn((5, hkv, d)).to(torch.bfloat16)
    slots = torch.tensor([3, -1, nb * 16, 17, nb * 16 + 100], dtype=torch.int64)
    kc = torch.full((nb, hkv, 16, d), 0xAB, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    fk.fp8kv_quant_append(x.cuda(), x.cuda(), slots.cuda(), kc, vc, 0.01, 0.01)
    torch.cuda.synchronize()
    flat = kc.cpu().reshape(nb * 16, d)  # hkv == 1: slot index = row
    ref = oracle.quantize_bf16(workload.bf16_bits(x), 0.01).reshape(5, d)
    assert np.array_equal(flat[3].numpy(), ref[0]) and np.array_equal(flat[17].numpy(), ref[3])
    untouched = [r for r in range(nb * 16) if r not in (3, 17)]
    assert bool((flat[untouched] == 0xAB).all())


# ------------------------------------------------------------ decode, small cases

SMALL = [
    # (base config, lengths, windows)
    ("llama31_8b_b1_4k", [1, 15, 16, 17, 33, 100, 0, 1000], (0, 1, 5, 16, 17, 100)),
    ("llama31_8b_b8_20k", [2999, 1234, 16, 4097], (0, 128)),
    ("gptoss20b_b8_16k", [1, 63, 64, 65, 700, 2500], (0, 128, 7)),
    ("gemma4e2b_b16_8k32k", [1, 17, 511, 512, 513, 3000], (0, 512, 33)),
    ("llama33_70b_needle_128k", [3000, 40], (0, 16)),
]


ENGINES = [fk.ENGINE_TENSOR_CORES, fk.ENGINE_CUDA_CORES]


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("base,lens,windows", SMALL)
def test_decode_small_cases_match_oracle(base, lens, windows, engine):
    shape = workload.small_shape(base, batch=len(lens), len_lo=1, len_hi=1, needle_margin=None)
    w = workload.make_workload(shape, seed=3, lens=lens)
    pc = Paged(w)
    pc.append_all()
    kc, vc = oracle_codes(w)
    gk, gv = pc.gathered_codes()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    for win in windows:
        out, err = pc.decode(window=win, engine=engine)
        assert err == 0
        assert_attn_close(_as_f64(out), oracle_out(w, kc, vc, win), f"{base} window={win} engine={engine}")


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_decode_every_supported_head_layout(d, g, engine):
    hkv = 2
    shape = workload.LayerShape(f"t{d}_{g}", hkv * g, hkv, d, 3, 1, 1, (0,))
    w = workload.make_workload(shape, seed=g * 1000 + d, lens=[777, 16, 35])
    pc = Paged(w)
    pc.append_all()
    kc, vc = oracle_codes(w)
    for win in (0, 50):
        out, err = pc.decode(window=win, engine=engine)
        assert err == 0
        assert_attn_close(_as_f64(out), oracle_out(w, kc, vc, win), f"d={d} g={g} window={win} engine={engine}")


@pytest.mark.parametrize("engine", ENGINES)
def test_unwritten_nan_slots_never_leak(engine):
    # Every byte of the cache starts as the NaN code; only written slots may count.
    shape = workload.small_shape("llama31_8b_b8_20k", batch=3, len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=4, lens=[33, 1, 250])
    pc = Paged(w, fill_byte=0x7F, extra_blocks=4)
    pc.append_all()
    kc, vc = oracle_codes(w)
    for win in (0, 3, 20):
        out, err = pc.decode(window=win, engine=engine)
        assert err == 0 and torch.isfinite(out.float()).all()
        assert_attn_close(_as_f64(out), oracle_out(w, kc, vc, win), f"nan-filled window={win}")


def test_result_independent_of_physical_placement():
    shape = workload.small_shape("llama31_8b_b8_20k", batch=2, len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=5, lens=[1500, 333])
    a = Paged(w)
    a.append_all()
    out_a, _ = a.decode()
    # the same logical cache under the identity block table
    ident = torch.zeros_like(w.block_tables)
    slots = []
    base = 0
    for b, L in enumerate(w.seq_lens.tolist()):
        nb = (L + 15) // 16
        ident[b, :nb] = torch.arange(base, base + nb, dtype=torch.int32)
        t = torch.arange(L)
        slots.append((ident[b, t // 16].to(torch.int64) * 16 + t % 16))
        base += nb
    w2 = workload.Workload(**{**w.__dict__, "block_tables": ident, "slot_mapping": torch.cat(slots)})
    b_ = Paged(w2)
    b_.append_all()
    out_b, _ = b_.decode()
    assert torch.equal(out_a, out_b)


def test_split_plan_does_not_change_the_result():
    shape = workload.small_shape("llama33_70b_needle_128k", batch=2, len_lo=1, len_hi=1, needle_margin=None)
    w = workload.make_workload(shape, seed=6, lens=[5000, 4100])
    pc = Paged(w)
    pc.append_all()
    out1, _ = pc.decode()
    wide = torch.zeros((2, 4 * w.max_blocks_per_seq), dtype=torch.int32, device="cuda")
    wide[:, :w.max_blocks_per_seq] = pc.block_tables
    out2, _ = pc.decode(max_seq_len=4 * 16 * w.max_blocks_per_seq, block_tables=wide)
    kc, vc = oracle_codes(w)
    ref = oracle_out(w, kc, vc, 0)
    assert_attn_close(_as_f64(out1), ref, "plan 1")
    assert_attn_close(_as_f64(out2), ref, "plan 2")
    assert float((out1.float() - out2.float()).abs().max()) <= 2 ** -7


def test_repeated_calls_on_one_workspace_agree():
    """One workspace serves call after call, whichever engine ran last: the
    split partials of each call are written before they are read, and the
    error word stays clear, so repeated calls give identical outputs."""
    shape = workload.small_shape("llama33_70b_needle_128k", batch=3, len_lo=1, len_hi=1, needle_margin=None)
    w = workload.make_workload(shape, seed=9, lens=[6000, 1, 2500])
    pc = Paged(w)
    pc.append_all()
    s = w.shape
    ws = fk.alloc_workspace(3, s.num_q_heads, s.num_kv_heads, s.head_dim, w.max_seq_len)
    outs = []
    for engine in (None, None, fk.ENGINE_CUDA_CORES, None, fk.ENGINE_TENSOR_CORES, None):
        out = torch.empty((3, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        args = (pc.q, pc.k_cache, pc.v_cache, pc.block_tables, pc.seq_lens, w.max_seq_len, w.k_scale, w.v_scale,
                w.sm_scale, 0, out, ws)
        if engine is None:
            fk.fp8kv_paged_decode(*args)
        else:
            fk.fp8kv_paged_decode_engine(*args, engine)
        torch.cuda.synchronize()
        assert fk.fp8kv_read_error(ws) == 0
        if engine is None:
            outs.append(out)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    kc, vc = oracle_codes(w)
    assert_attn_close(_as_f64(outs[0]), oracle_out(w, kc, vc, 0), "repeated calls")


def test_out_of_range_block_id_is_reported_not_faulted():
    shape = workload.small_shape("llama31_8b_b8_20k", batch=1, len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=7, lens=[40])
    pc = Paged(w)
    pc.append_all()
    bad = pc.block_tables.clone()
    bad[0, 1] = pc.num_blocks + 5
    _, err = pc.decode(block_tables=bad)
    assert err == 1  # FP8KV_ERR_INVALID_ARG
    _, err2 = pc.decode()
    assert err2 == 0


# ------------------------------------------------------------ fused decode step

STEP_CASES = [
    ("llama31_8b_b1_4k", [1, 15, 16, 17, 33, 100, 0, 1000], (0, 1, 17)),
    ("llama31_8b_b8_20k", [2999, 1234, 16, 4097], (0, 128)),
    ("gptoss20b_b8_16k", [1, 63, 64, 65, 700], (0, 7)),
    ("gemma4e2b_b16_8k32k", [1, 17, 513, 3000], (0, 33)),
    ("llama33_70b_needle_128k", [3000, 40], (0,)),
]


@pytest.mark.parametrize("base,lens,windows", STEP_CASES)
def test_decode_step_equals_append_then_decode(base, lens, windows):
    """The fused step writes the same cache bytes and returns the same outputs,
    bit for bit, as the append kernel followed by the decode kernel."""
    shape = workload.small_shape(base, batch=len(lens), len_lo=1, len_hi=1, needle_margin=None)
    w = workload.make_workload(shape, seed=11, lens=lens)
    kc, vc = oracle_codes(w)
    for win in windows:
        sep = Paged(w, seed=win)
        sep.append_all()
        out_sep, err_sep = sep.decode(window=win)
        fused = Paged(w, seed=win)          # same garbage in unwritten slots
        fused.append_history()
        out_f, err_f = fused.step(window=win)
        assert err_sep == 0 and err_f == 0
        assert torch.equal(fused.k_cache, sep.k_cache) and torch.equal(fused.v_cache, sep.v_cache)
        assert torch.equal(out_f, out_sep), f"{base} window={win}"
        assert_attn_close(_as_f64(out_f), oracle_out(w, kc, vc, win), f"step {base} window={win}")


def test_decode_step_writes_only_the_newest_slot():
    shape = workload.small_shape("llama31_8b_b8_20k", batch=3, len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=12, lens=[40, 16, 0])
    pc = Paged(w, fill_byte=0xAB, extra_blocks=2)
    before_k, before_v = pc.k_cache.clone(), pc.v_cache.clone()
    _, err = pc.step()
    assert err == 0
    kc, vc = oracle_codes(w)
    sm = w.slot_mapping
    changed = {int(sm[r]) for r in w.new_token_rows()[w.seq_lens > 0].tolist()}
    for cache, before, codes in ((pc.k_cache, before_k, kc), (pc.v_cache, before_v, vc)):
        flat = cache.cpu().permute(0, 2, 1, 3).reshape(-1, shape.num_kv_heads, shape.head_dim)
        ref = before.cpu().permute(0, 2, 1, 3).reshape(-1, shape.num_kv_heads, shape.head_dim).clone()
        for r in w.new_token_rows()[w.seq_lens > 0].tolist():
            ref[int(sm[r])] = torch.from_numpy(codes[r])
        assert torch.equal(flat, ref)
    assert len(changed) == 2


# ------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("name", list(workload.CONFIGS))
def test_full_size_workloads_match_oracle(name):
    w = workload.make_workload(name, seed=0)
    pc = Paged(w)
    pc.append_all()
    kc, vc = oracle_codes(w)
    gk, gv = pc.gathered_codes()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    for win in w.shape.windows:
        out, err = pc.decode(window=win)
        assert err == 0
        ref = oracle_out(w, kc, vc, win)
        assert_attn_close(_as_f64(out), ref, f"{name} window={win}")
        if w.needle_pos is not None:
            vh = oracle.e4m3_decode(vc[w.needle_pos]) * w.v_scale
            g = w.shape.group
            expect = np.stack([vh[h // g] for h in range(w.shape.num_q_heads)])
            assert_attn_close(_as_f64(out)[0], expect, f"{name} needle row")
        # the CUDA-core engine on the same cache
        out_c, err_c = pc.decode(window=win, engine=fk.ENGINE_CUDA_CORES)
        assert err_c == 0
        assert_attn_close(_as_f64(out_c), ref, f"{name} window={win} cuda cores")
        if w.needle_pos is not None:
            assert_attn_close(_as_f64(out_c)[0], expect, f"{name} needle row, cuda cores")
        # the fused step the benchmark times: same bytes, same outputs
        fused = Paged(w)
        fused.append_history()
        out_f, err_f = fused.step(window=win)
        assert err_f == 0
        assert torch.equal(fused.k_cache, pc.k_cache) and torch.equal(fused.v_cache, pc.v_cache)
        assert torch.equal(out_f, out), f"{name} window={win} fused step"
        del fused


def test_inputs_written_by_the_previous_kernel_are_seen():
    """Both kernels may be launched before the previous work on the stream ends;
    they must still read the inputs that work produced (here the new K/V rows
    and q come out of torch kernels issued right before each call)."""
    shape = workload.small_shape("llama31_8b_b8_20k", batch=2, len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=8, lens=[900, 1300])
    pc = Paged(w, fill_byte=0)
    k_dev = torch.zeros_like(w.k, device="cuda")
    v_dev = torch.zeros_like(w.v, device="cuda")
    k_dev.copy_(w.k.to("cuda").float().mul_(1.0).to(torch.bfloat16))   # produced just before the append
    v_dev.copy_(w.v.to("cuda").float().mul_(1.0).to(torch.bfloat16))
    fk.fp8kv_quant_append(k_dev, v_dev, w.slot_mapping.to("cuda"), pc.k_cache, pc.v_cache, w.k_scale, w.v_scale)
    pc.q = w.q.to("cuda").float().mul_(1.0).to(torch.bfloat16)          # produced just before the decode
    out, err = pc.decode()
    assert err == 0
    kc, vc = oracle_codes(w)
    gk, gv = pc.gathered_codes()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    assert_attn_close(_as_f64(out), oracle_out(w, kc, vc, 0), "fresh inputs")


def test_long_contraction_with_nonzero_mean_values():
    """131,072 keys, values ~ N(0.25, 0.125), near-flat attention: every key
    contributes and a low-precision accumulator would swamp (the CPU test
    test_tolerance_teeth shows the bar catches that).  The decode must meet
    the bar against the fp64 oracle."""
    shape = workload.LayerShape("flat_128k", 8, 1, 128, 1, 131072, 131072, (0,), kv_std=0.5)
    w = workload.make_workload(shape, seed=5)
    w.q = (w.q.float() * 0.05).to(torch.bfloat16)
    w.v = (w.v.float() * 0.25 + 0.25).to(torch.bfloat16)
    w.v_scale = workload.per_tensor_scale(w.v)
    pc = Paged(w)
    pc.append_all()
    kc, vc = oracle_codes(w)
    for engine in ENGINES:
        out, err = pc.decode(window=0, engine=engine)
        assert err == 0
        assert_attn_close(_as_f64(out), oracle_out(w, kc, vc, 0), f"flat 128K engine={engine}")


def test_decode_step_from_host_buffers_matches_the_device_step():
    """fp8kv_decode_step_host: the step's inputs packed in one pinned host
    buffer, copied in, the step, the output copied out -- the same cache bytes
    and output as fp8kv_decode_step on device inputs."""
    shape = workload.small_shape("llama31_8b_b8_20k", batch=3, len_lo=1, len_hi=1)
    w = workload.make_workload(shape, seed=12, lens=[900, 33, 2000])
    s = w.shape
    ref_p = Paged(w, seed=12)
    ref_p.append_history()
    ref_out, err = ref_p.step()
    assert err == 0
    p = Paged(w, seed=12)
    p.append_history()
    kn, vn = p.new_rows()
    parts = [w.q.contiguous(), kn.cpu().contiguous(), vn.cpu().contiguous(), w.seq_lens.contiguous()]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(parts, offs):
        h_in[o:o + t.numel() * t.element_size()] = t.view(torch.uint8).reshape(-1)
    d_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    views = [d_in[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(parts, offs)]
    out = torch.empty((3, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    h_out = torch.full(out.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    ws = fk.alloc_workspace(3, s.num_q_heads, s.num_kv_heads, s.head_dim, w.max_seq_len)
    call = fk.prepare_decode_step_host(h_in, d_in, h_out, views[0], views[1], views[2], p.k_cache, p.v_cache,
                                       p.block_tables, views[3], w.max_seq_len, w.k_scale, w.v_scale, w.sm_scale, 0,
                                       out, ws)
    call()
    torch.cuda.current_stream().synchronize()
    assert fk.fp8kv_read_error(ws) == 0
    assert torch.equal(h_out, ref_out.cpu())
    assert torch.equal(p.k_cache, ref_p.k_cache) and torch.equal(p.v_cache, ref_p.v_cache)


@pytest.mark.parametrize("engine", [fk.ENGINE_TENSOR_CORES, fk.ENGINE_CUDA_CORES])
def test_batch_above_512_sequences_runs_as_several_launches(engine):
    """600 sequences: the library runs them as consecutive launches of at
    most 512 sequences on one workspace; every output must match the oracle."""
    B = 600
    shape = workload.small_shape("llama31_8b_b8_20k", batch=B, len_lo=1, len_hi=90)
    w = workload.make_workload(shape, seed=13)
    pc = Paged(w)
    pc.append_all()
    out, err = pc.decode(engine=engine)
    assert err == 0
    kc, vc = oracle_codes(w)
    assert_attn_close(_as_f64(out), oracle_out(w, kc, vc, 0), "600 sequences")
