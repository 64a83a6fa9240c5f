"""Thin ctypes binding over libfp8kv (argument marshalling only).

Each function carries the C entry point's name and forwards torch tensors'
device pointers and sizes to it; every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if the shared library is
missing or a call returns an error status, a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

_lib = None

STATUS = {0: "FP8KV_OK", 1: "FP8KV_ERR_INVALID_ARG", 2: "FP8KV_ERR_UNSUPPORTED",
          3: "FP8KV_ERR_WORKSPACE", 4: "FP8KV_ERR_CUDA", 5: "FP8KV_ERR_TIMEOUT"}


class Fp8kvError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %s (%d)" % (fn, STATUS.get(code, "?"), code))
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Loads libfp8kv.so (building it first only when asked)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError("libfp8kv.so is not built (%s); run __graft_entry__.build()" % path)
        _build.build()
    lib = ctypes.CDLL(path)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.fp8kv_status_string.restype = ctypes.c_char_p
    lib.fp8kv_status_string.argtypes = [I]
    lib.fp8kv_quant_append.restype = I
    lib.fp8kv_quant_append.argtypes = [P, P, P, I64, P, P, I64, I, I, I, F, F, P]
    lib.fp8kv_paged_decode_workspace_size.restype = SZ
    lib.fp8kv_paged_decode_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.fp8kv_workspace_init.restype = I
    lib.fp8kv_workspace_init.argtypes = [P, SZ, P]
    lib.fp8kv_read_error.restype = I
    lib.fp8kv_read_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    lib.fp8kv_paged_decode.restype = I
    lib.fp8kv_paged_decode.argtypes = [P, P, P, I64, P, I, P, I, I, I, I, I, I, F, F, F, I, P, P, SZ, P]
    lib.fp8kv_paged_decode_engine.restype = I
    lib.fp8kv_paged_decode_engine.argtypes = [P, P, P, I64, P, I, P, I, I, I, I, I, I, F, F, F, I, P, P, SZ, P, I]
    lib.fp8kv_paged_decode_bf16.restype = I
    lib.fp8kv_paged_decode_bf16.argtypes = [P, P, P, I64, P, I, P, I, I, I, I, I, I, F, I, P, P, SZ, P]
    lib.fp8kv_quant_append_per_head.restype = I
    lib.fp8kv_quant_append_per_head.argtypes = [P, P, P, I64, P, P, I64, I, I, I, P, P, P]
    lib.fp8kv_paged_decode_per_head.restype = I
    lib.fp8kv_paged_decode_per_head.argtypes = [P, P, P, I64, P, I, P, I, I, I, I, I, I, P, P, F, I, P, P, SZ, P]
    lib.fp8kv_decode_step_per_head.restype = I
    lib.fp8kv_decode_step_per_head.argtypes = [P, P, P, P, P, I64, P, I, P, I, I, I, I, I, I, P, P, F, I, P, P, SZ, P]
    lib.fp8kv_quant_append_e5m2.restype = I
    lib.fp8kv_quant_append_e5m2.argtypes = [P, P, P, I64, P, P, I64, I, I, I, F, F, P]
    lib.fp8kv_paged_decode_e5m2.restype = I
    lib.fp8kv_paged_decode_e5m2.argtypes = [P, P, P, I64, P, I, P, I, I, I, I, I, I, F, F, F, I, P, P, SZ, P]
    lib.fp8kv_decode_step_e5m2.restype = I
    lib.fp8kv_decode_step_e5m2.argtypes = [P, P, P, P, P, I64, P, I, P, I, I, I, I, I, I, F, F, F, I, P, P, SZ, P]
    lib.fp8kv_decode_step.restype = I
    lib.fp8kv_decode_step.argtypes = [P, P, P, P, P, I64, P, I, P, I, I, I, I, I, I, F, F, F, I, P, P, SZ, P]
    lib.fp8kv_decode_step_host.restype = I
    lib.fp8kv_decode_step_host.argtypes = [P, P, SZ, P] + [P, P, P, P, P, I64, P, I, P, I, I, I, I, I, I, F, F, F, I,
                                                           P, P, SZ, P]
    lib.fp8kv_paged_decode_noalloc.restype = I
    lib.fp8kv_paged_decode_noalloc.argtypes = [P, P, P, I64, P, I, P, I, I, I, I, I, I, F, F, F, I, P, P]
    U64 = ctypes.c_uint64
    lib.fp8kv_debug_paged_decode_stall.restype = I
    lib.fp8kv_debug_paged_decode_stall.argtypes = [P, P, P, I64, P, I, P, I, I, I, I, I, I, F, F, F, I, P, P, SZ, P,
                                                   I, U64]
    lib.fp8kv_debug_paged_prefill_stall.restype = I
    lib.fp8kv_debug_paged_prefill_stall.argtypes = [P, I64, P, P, I64, P, I, P, P, I, I, I, I, I, I, I, F, F, F, I, P,
                                                    P, SZ, P, I, U64]
    lib.fp8kv_paged_prefill_workspace_size.restype = SZ
    lib.fp8kv_paged_prefill_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    lib.fp8kv_paged_prefill.restype = I
    lib.fp8kv_paged_prefill.argtypes = [P, I64, P, P, I64, P, I, P, P, I, I, I, I, I, I, I, F, F, F, I, P, P, SZ, P]
    _lib = lib
    return lib


def header_symbols() -> list:
    """Function names declared in include/fp8kv.h."""
    hdr = os.path.join(_build.INCLUDE, "fp8kv.h")
    text = open(hdr).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # drop comments
    return sorted(set(re.findall(r"\b(fp8kv_[a-z0-9_]+)\s*\(", text)))


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn, code):
    if code != 0:
        raise Fp8kvError(fn, code)


def _dev(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def fp8kv_status_string(code: int) -> str:
    return load().fp8kv_status_string(int(code)).decode()


def fp8kv_quant_append(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None):
    """k_new, v_new: bf16 [T, Hkv, D]; slot_mapping: int64 [T];
    k_cache, v_cache: uint8 [num_blocks, Hkv, block_size, D]."""
    nb, hkv, bs, d = k_cache.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, hkv, d) or tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("k_new/v_new must be [T, Hkv, D] matching the cache")
    if tuple(v_cache.shape) != tuple(k_cache.shape) or slot_mapping.numel() != T:
        raise ValueError("cache or slot_mapping shape mismatch")
    code = load().fp8kv_quant_append(
        _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(slot_mapping, torch.int64, "slot_mapping"), T,
        _dev(k_cache, torch.uint8, "k_cache"), _dev(v_cache, torch.uint8, "v_cache"),
        nb, bs, hkv, d, float(k_scale), float(v_scale), _stream(stream))
    _check("fp8kv_quant_append", code)


def fp8kv_paged_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                      block_size=16, window=0) -> int:
    n = load().fp8kv_paged_decode_workspace_size(int(batch), int(num_q_heads), int(num_kv_heads),
                                                 int(head_dim), int(max_seq_len), int(block_size),
                                                 int(window))
    if n == 0:
        raise Fp8kvError("fp8kv_paged_decode_workspace_size", 1)
    return int(n)


def fp8kv_workspace_init(workspace, stream=None):
    _check("fp8kv_workspace_init", load().fp8kv_workspace_init(
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def fp8kv_read_error(workspace, stream=None) -> int:
    code = ctypes.c_uint32(0)
    _check("fp8kv_read_error", load().fp8kv_read_error(
        _dev(workspace, torch.uint8, "workspace"), ctypes.byref(code), _stream(stream)))
    return int(code.value)


def alloc_workspace(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, block_size=16,
                    window=0, device=None, stream=None):
    """Allocates (through torch) and zero-fills a workspace for these sizes."""
    n = fp8kv_paged_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                          block_size, window)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    fp8kv_workspace_init(ws, stream)
    return ws


def fp8kv_paged_decode(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                       sm_scale, window, out, workspace, stream=None):
    """q, out: bf16 [B, Hq, D]; caches uint8 [num_blocks, Hkv, bs, D];
    block_tables int32 [B, max_blocks]; seq_lens int32 [B]."""
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    code = load().fp8kv_paged_decode(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.uint8, "k_cache"),
        _dev(v_cache, torch.uint8, "v_cache"), nb, _dev(block_tables, torch.int32, "block_tables"),
        block_tables.shape[1], _dev(seq_lens, torch.int32, "seq_lens"), int(max_seq_len), B, hq, hkv,
        d, bs, float(k_scale), float(v_scale), float(sm_scale), int(window),
        _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream))
    _check("fp8kv_paged_decode", code)


# fp8kv_engine
ENGINE_DEFAULT, ENGINE_TENSOR_CORES, ENGINE_CUDA_CORES = 0, 1, 2


def fp8kv_paged_decode_engine(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                              sm_scale, window, out, workspace, engine, stream=None):
    """fp8kv_paged_decode with the contraction engine chosen explicitly
    (ENGINE_TENSOR_CORES or ENGINE_CUDA_CORES; ENGINE_DEFAULT = the library's)."""
    prepare_paged_decode(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale, sm_scale,
                         window, out, workspace, stream, engine=engine)()


def fp8kv_paged_decode_noalloc(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                               sm_scale, window, out, stream=None):
    """Same as fp8kv_paged_decode without a workspace: for callers that cannot
    allocate device memory, the library's fixed 8 MiB device array holds the
    split-merge scratch.  Calls that overlap on the GPU race on that array."""
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    code = load().fp8kv_paged_decode_noalloc(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.uint8, "k_cache"),
        _dev(v_cache, torch.uint8, "v_cache"), nb, _dev(block_tables, torch.int32, "block_tables"),
        block_tables.shape[1], _dev(seq_lens, torch.int32, "seq_lens"), int(max_seq_len), B, hq, hkv,
        d, bs, float(k_scale), float(v_scale), float(sm_scale), int(window),
        _dev(out, torch.bfloat16, "out"), _stream(stream))
    _check("fp8kv_paged_decode_noalloc", code)


class PreparedCall:
    """A validated C call with its marshalled arguments kept, for callers that
    issue the same call repeatedly (decode loops): each invocation is just the
    C function call.  The tensors must stay alive and unchanged in shape."""

    def __init__(self, name, fn, args):
        self.name, self.fn, self.args = name, fn, args

    def __call__(self):
        code = self.fn(*self.args)
        if code != 0:
            raise Fp8kvError(self.name, code)


def prepare_quant_append(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None):
    nb, hkv, bs, d = k_cache.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, hkv, d) or tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("k_new/v_new must be [T, Hkv, D] matching the cache")
    if tuple(v_cache.shape) != tuple(k_cache.shape) or slot_mapping.numel() != T:
        raise ValueError("cache or slot_mapping shape mismatch")
    lib = load()
    args = (_dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
            _dev(slot_mapping, torch.int64, "slot_mapping"), ctypes.c_int64(T),
            _dev(k_cache, torch.uint8, "k_cache"), _dev(v_cache, torch.uint8, "v_cache"),
            ctypes.c_int64(nb), ctypes.c_int(bs), ctypes.c_int(hkv), ctypes.c_int(d),
            ctypes.c_float(k_scale), ctypes.c_float(v_scale), _stream(stream))
    return PreparedCall("fp8kv_quant_append", lib.fp8kv_quant_append, args)


def prepare_paged_decode(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                         sm_scale, window, out, workspace, stream=None, engine=None):
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    lib = load()
    I = ctypes.c_int
    args = (_dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.uint8, "k_cache"),
            _dev(v_cache, torch.uint8, "v_cache"), ctypes.c_int64(nb),
            _dev(block_tables, torch.int32, "block_tables"), I(block_tables.shape[1]),
            _dev(seq_lens, torch.int32, "seq_lens"), I(max_seq_len), I(B), I(hq), I(hkv), I(d), I(bs),
            ctypes.c_float(k_scale), ctypes.c_float(v_scale), ctypes.c_float(sm_scale), I(window),
            _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"),
            ctypes.c_size_t(workspace.numel()), _stream(stream))
    if engine is None:
        return PreparedCall("fp8kv_paged_decode", lib.fp8kv_paged_decode, args)
    return PreparedCall("fp8kv_paged_decode_engine", lib.fp8kv_paged_decode_engine, args + (I(engine),))


def _decode_step_args(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                      sm_scale, window, out, workspace, stream):
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q, out and the caches")
    if tuple(k_new.shape) != (B, hkv, d) or tuple(v_new.shape) != (B, hkv, d):
        raise ValueError("k_new/v_new must be [B, Hkv, D]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    I = ctypes.c_int
    return (_dev(q, torch.bfloat16, "q"), _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
            _dev(k_cache, torch.uint8, "k_cache"), _dev(v_cache, torch.uint8, "v_cache"), ctypes.c_int64(nb),
            _dev(block_tables, torch.int32, "block_tables"), I(block_tables.shape[1]),
            _dev(seq_lens, torch.int32, "seq_lens"), I(max_seq_len), I(B), I(hq), I(hkv), I(d), I(bs),
            ctypes.c_float(k_scale), ctypes.c_float(v_scale), ctypes.c_float(sm_scale), I(window),
            _dev(out, torch.bfloat16, "out"), _dev(workspace, torch.uint8, "workspace"),
            ctypes.c_size_t(workspace.numel()), _stream(stream))


def fp8kv_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                      sm_scale, window, out, workspace, stream=None):
    """Append each sequence's newest K/V row (token seq_lens[b]-1), then decode:
    q, out bf16 [B, Hq, D]; k_new, v_new bf16 [B, Hkv, D]."""
    _check("fp8kv_decode_step", load().fp8kv_decode_step(*_decode_step_args(
        q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale, sm_scale,
        window, out, workspace, stream)))


def prepare_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                        sm_scale, window, out, workspace, stream=None):
    args = _decode_step_args(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale,
                             v_scale, sm_scale, window, out, workspace, stream)
    return PreparedCall("fp8kv_decode_step", load().fp8kv_decode_step, args)


def _host(t, name):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("%s must be a host tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def prepare_decode_step_host(h_in, d_in, h_out, q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                             max_seq_len, k_scale, v_scale, sm_scale, window, out, workspace, stream=None):
    """fp8kv_decode_step_host, marshalled once: h_in (host, pinned) is copied to
    d_in (device, same byte size) before the step; q, k_new, v_new and
    seq_lens are device views the caller placed inside d_in; out is copied to
    h_out (host, pinned, same shape as out) after it."""
    if h_in.numel() * h_in.element_size() != d_in.numel() * d_in.element_size():
        raise ValueError("h_in and d_in must have the same size in bytes")
    if tuple(h_out.shape) != tuple(out.shape) or h_out.dtype != out.dtype:
        raise ValueError("h_out must match out")
    if not d_in.is_cuda:
        raise TypeError("d_in must be a CUDA tensor")
    args = (_host(h_in, "h_in"), ctypes.c_void_p(d_in.data_ptr()), ctypes.c_size_t(d_in.numel() * d_in.element_size()),
            _host(h_out, "h_out")) + _decode_step_args(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                                                       max_seq_len, k_scale, v_scale, sm_scale, window, out,
                                                       workspace, stream)
    return PreparedCall("fp8kv_decode_step_host", load().fp8kv_decode_step_host, args)


def _decode_bf16_args(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, sm_scale, window, out,
                      workspace, stream):
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    I = ctypes.c_int
    return (_dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
            _dev(v_cache, torch.bfloat16, "v_cache"), ctypes.c_int64(nb),
            _dev(block_tables, torch.int32, "block_tables"), I(block_tables.shape[1]),
            _dev(seq_lens, torch.int32, "seq_lens"), I(max_seq_len), I(B), I(hq), I(hkv), I(d), I(bs),
            ctypes.c_float(sm_scale), I(window), _dev(out, torch.bfloat16, "out"),
            _dev(workspace, torch.uint8, "workspace"), ctypes.c_size_t(workspace.numel()), _stream(stream))


def fp8kv_paged_decode_bf16(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, sm_scale, window, out,
                            workspace, stream=None):
    """The bf16-cache twin of fp8kv_paged_decode: caches bf16
    [num_blocks, Hkv, 16, D], no scales."""
    _check("fp8kv_paged_decode_bf16", load().fp8kv_paged_decode_bf16(*_decode_bf16_args(
        q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, sm_scale, window, out, workspace, stream)))


def prepare_paged_decode_bf16(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, sm_scale, window, out,
                              workspace, stream=None):
    args = _decode_bf16_args(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, sm_scale, window, out,
                             workspace, stream)
    return PreparedCall("fp8kv_paged_decode_bf16", load().fp8kv_paged_decode_bf16, args)


# ---------------------------------------------------------------- per-kv-head scales

def fp8kv_quant_append_per_head(k_new, v_new, slot_mapping, k_cache, v_cache, k_scales, v_scales, stream=None):
    """fp8kv_quant_append with fp32 [Hkv] device scale arrays."""
    nb, hkv, bs, d = k_cache.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, hkv, d) or tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("k_new/v_new must be [T, Hkv, D] matching the cache")
    if k_scales.numel() != hkv or v_scales.numel() != hkv:
        raise ValueError("k_scales/v_scales must have num_kv_heads entries")
    _check("fp8kv_quant_append_per_head", load().fp8kv_quant_append_per_head(
        _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(slot_mapping, torch.int64, "slot_mapping"), ctypes.c_int64(T), _dev(k_cache, torch.uint8, "k_cache"),
        _dev(v_cache, torch.uint8, "v_cache"), ctypes.c_int64(nb), bs, hkv, d,
        _dev(k_scales, torch.float32, "k_scales"), _dev(v_scales, torch.float32, "v_scales"), _stream(stream)))


def _per_head_common(q, k_cache, v_cache, block_tables, seq_lens, k_scales, v_scales):
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    if k_scales.numel() != hkv or v_scales.numel() != hkv:
        raise ValueError("k_scales/v_scales must have num_kv_heads entries")
    return B, hq, d, nb, hkv, bs


def fp8kv_paged_decode_per_head(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scales, v_scales,
                                sm_scale, window, out, workspace, stream=None):
    """fp8kv_paged_decode with fp32 [Hkv] device scale arrays."""
    B, hq, d, nb, hkv, bs = _per_head_common(q, k_cache, v_cache, block_tables, seq_lens, k_scales, v_scales)
    I = ctypes.c_int
    _check("fp8kv_paged_decode_per_head", load().fp8kv_paged_decode_per_head(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.uint8, "k_cache"), _dev(v_cache, torch.uint8, "v_cache"),
        ctypes.c_int64(nb), _dev(block_tables, torch.int32, "block_tables"), I(block_tables.shape[1]),
        _dev(seq_lens, torch.int32, "seq_lens"), I(max_seq_len), I(B), I(hq), I(hkv), I(d), I(bs),
        _dev(k_scales, torch.float32, "k_scales"), _dev(v_scales, torch.float32, "v_scales"),
        ctypes.c_float(sm_scale), I(window), _dev(out, torch.bfloat16, "out"),
        _dev(workspace, torch.uint8, "workspace"), ctypes.c_size_t(workspace.numel()), _stream(stream)))


def fp8kv_decode_step_per_head(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scales,
                               v_scales, sm_scale, window, out, workspace, stream=None):
    """fp8kv_decode_step with fp32 [Hkv] device scale arrays."""
    B, hq, d, nb, hkv, bs = _per_head_common(q, k_cache, v_cache, block_tables, seq_lens, k_scales, v_scales)
    I = ctypes.c_int
    _check("fp8kv_decode_step_per_head", load().fp8kv_decode_step_per_head(
        _dev(q, torch.bfloat16, "q"), _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(k_cache, torch.uint8, "k_cache"), _dev(v_cache, torch.uint8, "v_cache"), ctypes.c_int64(nb),
        _dev(block_tables, torch.int32, "block_tables"), I(block_tables.shape[1]),
        _dev(seq_lens, torch.int32, "seq_lens"), I(max_seq_len), I(B), I(hq), I(hkv), I(d), I(bs),
        _dev(k_scales, torch.float32, "k_scales"), _dev(v_scales, torch.float32, "v_scales"),
        ctypes.c_float(sm_scale), I(window), _dev(out, torch.bfloat16, "out"),
        _dev(workspace, torch.uint8, "workspace"), ctypes.c_size_t(workspace.numel()), _stream(stream)))


# ---------------------------------------------------------------- E5M2 cache

def fp8kv_quant_append_e5m2(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None):
    """fp8kv_quant_append writing E5M2 codes."""
    call = prepare_quant_append(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream)
    _check("fp8kv_quant_append_e5m2", load().fp8kv_quant_append_e5m2(*call.args))


def fp8kv_paged_decode_e5m2(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale, sm_scale,
                            window, out, workspace, stream=None):
    """fp8kv_paged_decode over an E5M2 cache."""
    call = prepare_paged_decode(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                                sm_scale, window, out, workspace, stream)
    _check("fp8kv_paged_decode_e5m2", load().fp8kv_paged_decode_e5m2(*call.args))


def fp8kv_decode_step_e5m2(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale,
                           v_scale, sm_scale, window, out, workspace, stream=None):
    """fp8kv_decode_step over an E5M2 cache."""
    _check("fp8kv_decode_step_e5m2", load().fp8kv_decode_step_e5m2(*_decode_step_args(
        q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale, sm_scale,
        window, out, workspace, stream)))


def fp8kv_paged_prefill_workspace_size(batch, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                                       block_size=16, window=0) -> int:
    n = load().fp8kv_paged_prefill_workspace_size(int(batch), int(max_q_len), int(max_seq_len), int(num_q_heads),
                                                  int(num_kv_heads), int(head_dim), int(block_size), int(window))
    if n == 0:
        raise Fp8kvError("fp8kv_paged_prefill_workspace_size", 1)
    return int(n)


def alloc_prefill_workspace(batch, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size=16,
                            window=0, device=None, stream=None):
    """Allocates (through torch) and zero-fills a prefill workspace for these sizes."""
    n = fp8kv_paged_prefill_workspace_size(batch, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                                           block_size, window)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    fp8kv_workspace_init(ws, stream)
    return ws


def prepare_paged_prefill(q, k_cache, v_cache, block_tables, seq_lens, q_starts, max_q_len, max_seq_len, k_scale,
                          v_scale, sm_scale, window, out, workspace, stream=None):
    """q, out: bf16 [sum q_len, Hq, D] (the sequences' query rows packed in
    order); caches uint8 [num_blocks, Hkv, bs, D]; block_tables int32
    [B, max_blocks]; seq_lens int32 [B]; q_starts int32 [B + 1] (cumulative
    q_len); workspace: uint8, fp8kv_paged_prefill_workspace_size bytes."""
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    B = seq_lens.numel()
    if d2 != d or tuple(out.shape) != (T, hq, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or q_starts.numel() != B + 1:
        raise ValueError("block_tables must be [B, max_blocks] and q_starts [B + 1]")
    lib = load()
    I = ctypes.c_int
    args = (_dev(q, torch.bfloat16, "q"), ctypes.c_int64(T), _dev(k_cache, torch.uint8, "k_cache"),
            _dev(v_cache, torch.uint8, "v_cache"), ctypes.c_int64(nb),
            _dev(block_tables, torch.int32, "block_tables"), I(block_tables.shape[1]),
            _dev(seq_lens, torch.int32, "seq_lens"), _dev(q_starts, torch.int32, "q_starts"), I(max_q_len),
            I(max_seq_len), I(B), I(hq), I(hkv), I(d), I(bs), ctypes.c_float(k_scale), ctypes.c_float(v_scale),
            ctypes.c_float(sm_scale), I(window), _dev(out, torch.bfloat16, "out"),
            _dev(workspace, torch.uint8, "workspace"), ctypes.c_size_t(workspace.numel()), _stream(stream))
    return PreparedCall("fp8kv_paged_prefill", lib.fp8kv_paged_prefill, args)


def fp8kv_paged_prefill(q, k_cache, v_cache, block_tables, seq_lens, q_starts, max_q_len, max_seq_len, k_scale,
                        v_scale, sm_scale, window, out, workspace, stream=None):
    """Causal (optionally windowed) attention of each sequence's newest
    q_len tokens over its fp8 cache; see prepare_paged_prefill for shapes."""
    prepare_paged_prefill(q, k_cache, v_cache, block_tables, seq_lens, q_starts, max_q_len, max_seq_len, k_scale,
                          v_scale, sm_scale, window, out, workspace, stream)()


# ---------------------------------------------------------------- failure-path test hooks

def debug_paged_decode_stall(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale, sm_scale,
                             window, out, workspace, stall_stage, wait_limit_ns, stream=None) -> int:
    """fp8kv_debug_paged_decode_stall: the CUDA-core decode with stage
    `stall_stage` of CTA 0 never issued and every ring wait limited to
    wait_limit_ns.  Returns the launch status (the timeout itself is reported
    through the workspace error word)."""
    args = prepare_paged_decode(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, k_scale, v_scale,
                                sm_scale, window, out, workspace, stream).args
    return load().fp8kv_debug_paged_decode_stall(*args, ctypes.c_int(stall_stage), ctypes.c_uint64(wait_limit_ns))


def debug_paged_prefill_stall(q, k_cache, v_cache, block_tables, seq_lens, q_starts, max_q_len, max_seq_len, k_scale,
                              v_scale, sm_scale, window, out, workspace, stall_stage, wait_limit_ns,
                              stream=None) -> int:
    """fp8kv_debug_paged_prefill_stall: the prefill with the score MMAs of
    stage `stall_stage` of CTA (0, 0, 0) never issued and the MMA waits
    limited to wait_limit_ns.  Returns the launch status."""
    args = prepare_paged_prefill(q, k_cache, v_cache, block_tables, seq_lens, q_starts, max_q_len, max_seq_len,
                                 k_scale, v_scale, sm_scale, window, out, workspace, stream).args
    return load().fp8kv_debug_paged_prefill_stall(*args, ctypes.c_int(stall_stage), ctypes.c_uint64(wait_limit_ns))
