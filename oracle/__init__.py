"""fp8kv oracle -- TEST INFRASTRUCTURE ONLY.

Plain CPU statement of the fp8 paged decode-attention path: a scalar E4M3
encoder/decoder and fp64 two-pass softmax attention over the decoded cache.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and never imports it; the two meet only through the seeded input generator.

Sources: gpusmith.com "FP8 KV Cache Quantization: Capacity Gains and Accuracy
Risk" (sections "What FP8 KV changes", "Scales and calibration", "Worked
capacity example"); particula.tech "KV Cache Quantization: What FP8 and q8_0
Cost in Accuracy" (opening section, FP32 accumulation); phantomic12 summary of
the vLLM FP8 KV-cache blog ("ACCURACY AT LONG CONTEXT", "DECODE COST").

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
the pages or the mathematics fix (parity is pinned for every function).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_quantize_bf16.restype = None
        lib.oracle_quantize_bf16.argtypes = [P, ctypes.c_int64, ctypes.c_float, P]
        lib.oracle_encode_f32.restype = None
        lib.oracle_encode_f32.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_decode_codes.restype = None
        lib.oracle_decode_codes.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_decode_attention.restype = ctypes.c_int
        lib.oracle_decode_attention.argtypes = [
            P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, P, ctypes.c_int64, P]
        lib.oracle_decode_attention_bf16.restype = ctypes.c_int
        lib.oracle_decode_attention_bf16.argtypes = [
            P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_float, ctypes.c_int, ctypes.c_int, P, ctypes.c_int64, P]
        lib.oracle_decode_attention_per_head.restype = ctypes.c_int
        lib.oracle_decode_attention_per_head.argtypes = [
            P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
            ctypes.c_float, ctypes.c_int, ctypes.c_int, P, ctypes.c_int64, P]
        lib.oracle_decode_codes_e5m2.restype = None
        lib.oracle_decode_codes_e5m2.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_encode_f32_e5m2.restype = None
        lib.oracle_encode_f32_e5m2.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_quantize_bf16_e5m2.restype = None
        lib.oracle_quantize_bf16_e5m2.argtypes = [P, ctypes.c_int64, ctypes.c_float, P]
        lib.oracle_decode_attention_e5m2.restype = ctypes.c_int
        lib.oracle_decode_attention_e5m2.argtypes = [
            P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_int, P, ctypes.c_int64, P]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e4m3_decode(codes) -> np.ndarray:
    """Exact fp64 value of each E4M3 code (NaN for 0x7F / 0xFF)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_decode_codes(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    """E4M3 code of each fp32 value: round-to-nearest-even, saturate at +-448."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_encode_f32(_ptr(v), v.size, _ptr(out))
    return out


def quantize_bf16(x_bits, scale: float) -> np.ndarray:
    """Cache codes for bf16 inputs (given as uint16 bit patterns):
    code = e4m3(fp32(x) / fp32(scale)), one IEEE fp32 divide then one rounding."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_quantize_bf16(_ptr(x), x.size, float(scale), _ptr(out))
    return out


def decode_attention(q_bits, k_codes, v_codes, seq_lens, k_scale, v_scale,
                     sm_scale, window=0, nthreads=1, acc_bits=0) -> np.ndarray:
    """fp64 decode attention.

    q_bits   uint16 [B, Hq, d] bf16 bit patterns
    k_codes  uint8  [total_tokens, Hkv, d] E4M3 codes, sequences concatenated
             in logical token order
    v_codes  uint8  same layout as k_codes
    seq_lens int    [B]
    Returns fp64 [B, Hq, d].  ``acc_bits > 0`` selects a deliberately broken
    accumulator (sums rounded to that many significand bits after each add),
    used only to show that the parity tests can see such a failure.
    """
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, d = q.shape
    Hkv = kc.shape[1]
    assert kc.shape[2] == d and vc.shape == kc.shape
    starts = np.zeros(B, dtype=np.int64)
    if B > 1:
        starts[1:] = np.cumsum(lens.astype(np.int64))[:-1]
    assert int(lens.sum()) <= kc.shape[0]
    max_len = int(max(1, lens.max() if B else 1))
    nthreads = max(1, int(nthreads))
    scratch = np.empty(nthreads * (max_len + d), dtype=np.float64)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    rc = _load().oracle_decode_attention(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(starts), _ptr(lens), B, Hq, Hkv, d,
        float(k_scale), float(v_scale), float(sm_scale), int(window),
        int(acc_bits), nthreads, _ptr(scratch), max_len, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_decode_attention: bad arguments")
    return out



def decode_attention_bf16(q_bits, k_bits, v_bits, seq_lens, sm_scale, window=0, nthreads=1) -> np.ndarray:
    """fp64 decode attention over a bf16 cache (the comparison baseline of the
    fp8 cache): q_bits uint16 [B, Hq, d]; k_bits, v_bits uint16 [total_tokens,
    Hkv, d] bf16 bit patterns, sequences concatenated in logical order."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kb = np.ascontiguousarray(k_bits, dtype=np.uint16)
    vb = np.ascontiguousarray(v_bits, dtype=np.uint16)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, d = q.shape
    Hkv = kb.shape[1]
    assert kb.shape[2] == d and vb.shape == kb.shape
    starts = np.zeros(B, dtype=np.int64)
    if B > 1:
        starts[1:] = np.cumsum(lens.astype(np.int64))[:-1]
    assert int(lens.sum()) <= kb.shape[0]
    max_len = int(max(1, lens.max() if B else 1))
    nthreads = max(1, int(nthreads))
    scratch = np.empty(nthreads * (max_len + d), dtype=np.float64)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    rc = _load().oracle_decode_attention_bf16(
        _ptr(q), _ptr(kb), _ptr(vb), _ptr(starts), _ptr(lens), B, Hq, Hkv, d,
        float(sm_scale), int(window), nthreads, _ptr(scratch), max_len, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_decode_attention_bf16: bad arguments")
    return out


def quantize_bf16_per_head(bits, scales) -> np.ndarray:
    """E4M3 codes of bf16 bits [T, Hkv, d] with one scale per kv head: each
    head's elements are quantised exactly as quantize_bf16 does with that
    head's scale."""
    x = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.uint8)
    for h in range(x.shape[1]):
        out[:, h, :] = quantize_bf16(np.ascontiguousarray(x[:, h, :]), float(scales[h])).reshape(x.shape[0], x.shape[2])
    return out


def decode_attention_per_head(q_bits, k_codes, v_codes, seq_lens, k_scales, v_scales, sm_scale, window=0,
                              nthreads=1) -> np.ndarray:
    """fp64 decode attention over an E4M3 cache with per-kv-head scales
    (k_scales, v_scales: [Hkv] fp32)."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scales, dtype=np.float32)
    vs = np.ascontiguousarray(v_scales, dtype=np.float32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, d = q.shape
    Hkv = kc.shape[1]
    assert kc.shape[2] == d and vc.shape == kc.shape and ks.shape == (Hkv,) and vs.shape == (Hkv,)
    starts = np.zeros(B, dtype=np.int64)
    if B > 1:
        starts[1:] = np.cumsum(lens.astype(np.int64))[:-1]
    assert int(lens.sum()) <= kc.shape[0]
    max_len = int(max(1, lens.max() if B else 1))
    nthreads = max(1, int(nthreads))
    scratch = np.empty(nthreads * (max_len + d), dtype=np.float64)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    rc = _load().oracle_decode_attention_per_head(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(starts), _ptr(lens), B, Hq, Hkv, d, _ptr(ks), _ptr(vs),
        float(sm_scale), int(window), nthreads, _ptr(scratch), max_len, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_decode_attention_per_head: bad arguments")
    return out


# ---------------------------------------------------------------- E5M2

def e5m2_decode(codes) -> np.ndarray:
    """Exact fp64 value of each E5M2 code (+-inf for 0x7C / 0xFC, NaN for the
    other exponent-31 codes)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_decode_codes_e5m2(_ptr(c), c.size, _ptr(out))
    return out


def e5m2_encode(values) -> np.ndarray:
    """E5M2 code of each fp32 value: round-to-nearest-even, saturate at +-57344."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_encode_f32_e5m2(_ptr(v), v.size, _ptr(out))
    return out


def quantize_bf16_e5m2(x_bits, scale: float) -> np.ndarray:
    """E5M2 cache codes of bf16 inputs: code = e5m2(fp32(x) / fp32(scale))."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_quantize_bf16_e5m2(_ptr(x), x.size, float(scale), _ptr(out))
    return out


def decode_attention_e5m2(q_bits, k_codes, v_codes, seq_lens, k_scale, v_scale, sm_scale, window=0,
                          nthreads=1) -> np.ndarray:
    """fp64 decode attention over an E5M2 cache (per-tensor scales)."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, d = q.shape
    Hkv = kc.shape[1]
    starts = np.zeros(B, dtype=np.int64)
    if B > 1:
        starts[1:] = np.cumsum(lens.astype(np.int64))[:-1]
    assert int(lens.sum()) <= kc.shape[0] and vc.shape == kc.shape
    max_len = int(max(1, lens.max() if B else 1))
    nthreads = max(1, int(nthreads))
    scratch = np.empty(nthreads * (max_len + d), dtype=np.float64)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    rc = _load().oracle_decode_attention_e5m2(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(starts), _ptr(lens), B, Hq, Hkv, d, float(k_scale), float(v_scale),
        float(sm_scale), int(window), nthreads, _ptr(scratch), max_len, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_decode_attention_e5m2: bad arguments")
    return out


# ---------------------------------------------------------------- prefill (chunked) attention

def prefill_attention(q_bits, k_codes, v_codes, seq_lens, q_lens, k_scale, v_scale, sm_scale, window=0,
                      nthreads=1) -> np.ndarray:
    """fp64 causal attention of a chunk of new query tokens over an E4M3 cache.

    q_bits   uint16 [sum(q_lens), Hq, d]: the queries of sequence b are its
             last q_lens[b] tokens, positions seq_lens[b] - q_lens[b] ..
             seq_lens[b] - 1, packed sequence after sequence
    k_codes, v_codes  uint8 [sum(seq_lens), Hkv, d], sequences concatenated in
             logical order (the chunk's own keys included)
    Query token at position p attends keys [max(0, p + 1 - window), p]
    (window <= 0: [0, p]); row by row this is the decode attention of a
    sequence of length p + 1, which is how it is computed here.
    """
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    lens = np.asarray(seq_lens, dtype=np.int64)
    qls = np.asarray(q_lens, dtype=np.int64)
    assert np.all(qls <= lens) and q.shape[0] == int(qls.sum())
    R, Hq, d = q.shape
    Hkv = kc.shape[1]
    starts_seq = np.zeros(len(lens), dtype=np.int64)
    if len(lens) > 1:
        starts_seq[1:] = np.cumsum(lens)[:-1]
    row_start = np.repeat(starts_seq, qls)
    row_len = np.concatenate([np.arange(L - n + 1, L + 1) for L, n in zip(lens, qls)]).astype(np.int32) \
        if R else np.zeros(0, np.int32)
    max_len = int(max(1, row_len.max() if R else 1))
    nthreads = max(1, int(nthreads))
    scratch = np.empty(nthreads * (max_len + d), dtype=np.float64)
    out = np.zeros((R, Hq, d), dtype=np.float64)
    if R == 0:
        return out
    rc = _load().oracle_decode_attention(
        _ptr(q.reshape(R, Hq, d)), _ptr(kc), _ptr(vc), _ptr(np.ascontiguousarray(row_start)),
        _ptr(np.ascontiguousarray(row_len)), R, Hq, Hkv, d, float(k_scale), float(v_scale), float(sm_scale),
        int(window), 0, nthreads, _ptr(scratch), max_len, _ptr(out))
    if rc != 0:
        raise ValueError("prefill_attention: bad arguments")
    return out
