"""The C ABI without a GPU: the library builds, loads, exports every function
include/fp8kv.h declares, and rejects bad arguments with a status code before
touching the device."""
import ctypes

import pytest

from fp8_kv_cache_fp8kv_gb300 import binding as fk
from fp8_kv_cache_fp8kv_gb300 import build as fbuild


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fk.load()


def test_every_header_symbol_is_exported(lib):
    names = fk.header_symbols()
    assert {"fp8kv_quant_append", "fp8kv_paged_decode", "fp8kv_decode_step", "fp8kv_paged_decode_workspace_size",
            "fp8kv_workspace_init", "fp8kv_read_error", "fp8kv_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in fk.STATUS.items():
        assert fk.fp8kv_status_string(code) == name
    assert fk.fp8kv_status_string(99) == "FP8KV_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails validation first
MISALIGNED = ctypes.c_void_p(0x10001)


def _decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, nb=100, bt=FAKE, mb=8, sl=FAKE, msl=128, B=2, hq=32, hkv=8, d=128,
             bs=16, ks=0.01, vs=0.01, sm=0.088, win=0, out=FAKE, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return lib.fp8kv_paged_decode(a["q"], a["k"], a["v"], a["nb"], a["bt"], a["mb"], a["sl"], a["msl"],
                                  a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["ks"], a["vs"], a["sm"],
                                  a["win"], a["out"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2), (dict(d=512), 2), (dict(bs=32), 2), (dict(hq=256, hkv=8), 2),
    (dict(hq=30, hkv=8), 1), (dict(ks=0.0), 1), (dict(vs=float("nan")), 1), (dict(sm=float("inf")), 1),
    (dict(q=None), 1), (dict(out=None), 1), (dict(bt=None), 1), (dict(q=MISALIGNED), 1),
    (dict(k=MISALIGNED), 1), (dict(mb=4, msl=128), 1), (dict(B=-1), 1), (dict(nb=0), 1),
    (dict(nb=1 << 31), 2), (dict(B=70000), 1),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_decode_empty_batch_is_a_no_op(lib):
    assert _decode(lib, B=0, q=None, out=None) == 0


def _engine(lib, engine, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, nb=100, bt=FAKE, mb=8, sl=FAKE, msl=128, B=2, hq=32, hkv=8, d=128,
             bs=16, ks=0.01, vs=0.01, sm=0.088, win=0, out=FAKE, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return lib.fp8kv_paged_decode_engine(a["q"], a["k"], a["v"], a["nb"], a["bt"], a["mb"], a["sl"], a["msl"],
                                         a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["ks"], a["vs"], a["sm"],
                                         a["win"], a["out"], a["ws"], a["wsb"], None, engine)


@pytest.mark.parametrize("engine,kw,code", [
    (3, {}, 1), (-1, {}, 1), (1, dict(d=96), 2), (2, dict(d=96), 2), (2, dict(q=None), 1),
    (2, dict(ks=0.0), 1), (1, dict(B=0, q=None, out=None), 0), (2, dict(B=0, q=None, out=None), 0),
])
def test_engine_entry_validates(lib, engine, kw, code):
    assert _engine(lib, engine, **kw) == code


def _bf16(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, nb=100, bt=FAKE, mb=8, sl=FAKE, msl=128, B=2, hq=32, hkv=8, d=128,
             bs=16, sm=0.088, win=0, out=FAKE, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return lib.fp8kv_paged_decode_bf16(a["q"], a["k"], a["v"], a["nb"], a["bt"], a["mb"], a["sl"], a["msl"],
                                       a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["sm"], a["win"], a["out"],
                                       a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2), (dict(bs=32), 2), (dict(hq=256, hkv=8), 2), (dict(hq=30, hkv=8), 1),
    (dict(sm=float("nan")), 1), (dict(q=None), 1), (dict(k=MISALIGNED), 1), (dict(mb=4, msl=128), 1),
    (dict(B=0, q=None, out=None), 0),
])
def test_bf16_twin_validates(lib, kw, code):
    assert _bf16(lib, **kw) == code


def _step(lib, **kw):
    a = dict(q=FAKE, kn=FAKE, vn=FAKE, k=FAKE, v=FAKE, nb=100, bt=FAKE, mb=8, sl=FAKE, msl=128, B=2, hq=32, hkv=8,
             d=128, bs=16, ks=0.01, vs=0.01, sm=0.088, win=0, out=FAKE, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return lib.fp8kv_decode_step(a["q"], a["kn"], a["vn"], a["k"], a["v"], a["nb"], a["bt"], a["mb"], a["sl"],
                                 a["msl"], a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["ks"], a["vs"], a["sm"],
                                 a["win"], a["out"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(kn=None), 1), (dict(vn=None), 1), (dict(kn=MISALIGNED), 1), (dict(vn=MISALIGNED), 1),
    (dict(d=96), 2), (dict(ks=0.0), 1), (dict(q=None), 1), (dict(mb=4, msl=128), 1),
])
def test_decode_step_rejects_bad_arguments(lib, kw, code):
    assert _step(lib, **kw) == code


def test_decode_step_empty_batch_is_a_no_op(lib):
    assert _step(lib, B=0, q=None, kn=None, vn=None, out=None) == 0


def _decode_ph(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, nb=100, bt=FAKE, mb=8, sl=FAKE, msl=128, B=2, hq=32, hkv=8, d=128,
             bs=16, ks=FAKE, vs=FAKE, sm=0.088, win=0, out=FAKE, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return lib.fp8kv_paged_decode_per_head(a["q"], a["k"], a["v"], a["nb"], a["bt"], a["mb"], a["sl"], a["msl"],
                                           a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["ks"], a["vs"], a["sm"],
                                           a["win"], a["out"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(ks=None), 1), (dict(vs=None), 1), (dict(ks=ctypes.c_void_p(0x10002)), 1), (dict(d=96), 2),
    (dict(sm=float("inf")), 1), (dict(B=0, q=None, out=None, ks=None, vs=None), 0),
])
def test_per_head_decode_validates(lib, kw, code):
    assert _decode_ph(lib, **kw) == code


def test_per_head_append_validates(lib):
    f = lib.fp8kv_quant_append_per_head
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 10, 16, 8, 128, None, FAKE, None) == 1
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 10, 16, 8, 128, ctypes.c_void_p(0x10002), FAKE, None) == 1
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 10, 16, 8, 24, FAKE, FAKE, None) == 2
    assert f(None, None, None, 0, FAKE, FAKE, 10, 16, 8, 128, None, None, None) == 0


def _append(lib, **kw):
    a = dict(k=FAKE, v=FAKE, sm=FAKE, T=4, kc=FAKE, vc=FAKE, nb=10, bs=16, hkv=8, d=128, ks=0.5, vs=0.5)
    a.update(kw)
    return lib.fp8kv_quant_append(a["k"], a["v"], a["sm"], a["T"], a["kc"], a["vc"], a["nb"], a["bs"],
                                  a["hkv"], a["d"], a["ks"], a["vs"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=24), 2), (dict(d=2048), 2), (dict(ks=-1.0), 1), (dict(vs=float("inf")), 1),
    (dict(kc=None), 1), (dict(k=None), 1), (dict(sm=None), 1), (dict(k=MISALIGNED), 1),
    (dict(T=-3), 1), (dict(nb=0), 1), (dict(hkv=0), 1),
])
def test_append_rejects_bad_arguments(lib, kw, code):
    assert _append(lib, **kw) == code


def test_append_zero_tokens_is_a_no_op(lib):
    assert _append(lib, T=0, k=None, v=None, sm=None) == 0


def test_workspace_calls_validate(lib):
    assert lib.fp8kv_workspace_init(None, 16, None) == 1
    assert lib.fp8kv_workspace_init(MISALIGNED, 16, None) == 1
    assert lib.fp8kv_read_error(None, None, None) == 1
    assert lib.fp8kv_paged_decode_workspace_size(2, 30, 8, 128, 100, 16, 0) == 0
    assert lib.fp8kv_paged_decode_workspace_size(2, 32, 8, 96, 100, 16, 0) == 0


def _prefill(lib, **kw):
    a = dict(q=FAKE, T=64, k=FAKE, v=FAKE, nb=100, bt=FAKE, mb=8, sl=FAKE, qs=FAKE, mq=64, msl=128, B=2, hq=32,
             hkv=8, d=128, bs=16, ks=0.01, vs=0.01, sm=0.088, win=0, out=FAKE, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    return lib.fp8kv_paged_prefill(a["q"], a["T"], a["k"], a["v"], a["nb"], a["bt"], a["mb"], a["sl"], a["qs"],
                                   a["mq"], a["msl"], a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["ks"], a["vs"],
                                   a["sm"], a["win"], a["out"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2), (dict(d=512), 2), (dict(bs=32), 2), (dict(hq=256, hkv=8), 2),
    (dict(hq=30, hkv=8), 1), (dict(ks=0.0), 1), (dict(vs=float("nan")), 1), (dict(sm=float("inf")), 1),
    (dict(q=None), 1), (dict(out=None), 1), (dict(qs=None), 1), (dict(q=MISALIGNED), 1),
    (dict(v=MISALIGNED), 1), (dict(mb=4, msl=128), 1), (dict(mq=200), 1),
    (dict(mq=-1), 1), (dict(T=-1), 1), (dict(B=-1), 1), (dict(nb=0), 1), (dict(nb=1 << 31), 2),
    (dict(B=70000), 1),
    (dict(B=0, q=None, out=None), 0), (dict(mq=0, q=None), 0), (dict(T=0, out=None), 0),
])
def test_prefill_validates(lib, kw, code):
    assert _prefill(lib, **kw) == code


def test_prefill_workspace_size_rejects_bad_shapes(lib):
    f = lib.fp8kv_paged_prefill_workspace_size
    assert f(2, 64, 128, 32, 8, 96, 16, 0) == 0       # head_dim
    assert f(2, 200, 128, 32, 8, 128, 16, 0) == 0     # max_q_len > max_seq_len
    assert f(2, 64, 128, 30, 8, 128, 16, 0) == 0      # heads not a multiple
    assert f(2, 64, 128, 32, 8, 128, 32, 0) == 0      # block size
