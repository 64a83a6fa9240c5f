"""Pins the CPU oracle to facts fixed by the FP8 KV pages and by mathematics.

Nothing here compares the oracle with itself: every check is a printed value
(tests/golden/*.json, with its citation), a brute-force search, a closed form,
an invariant, or an independent library routine (torch's float8_e4m3fn casts,
torch.softmax in fp64).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests._tol import ATTN_MAX_ABS, ATTN_MEAN_ABS, attn_errors

GOLD = os.path.join(os.path.dirname(__file__), "golden")
ALL = np.arange(256, dtype=np.uint8)


def golden(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def torch_decode(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_encode(values):
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# ---------------------------------------------------------------- decoder

def test_decoder_printed_format_facts():
    fmt = golden("e4m3_format.json")
    dec = oracle.e4m3_decode(ALL)
    finite = dec[np.isfinite(dec)]
    assert finite.max() == fmt["e4m3_max_normal"] == dec[0x7E]
    assert finite.min() == -fmt["e4m3_max_normal"] == dec[0xFE]
    assert finite.max() != fmt["e4m3fnuz_max_not_ours"] and finite.max() != fmt["e5m2_max"]
    # 3 mantissa bits: every binade [2^e, 2^(e+1)) of normals holds 2^3 codes
    # (the top binade [256, 512) loses its last code to NaN: 7 codes)
    mag = np.abs(finite)
    for e in range(-6, 9):
        n = np.count_nonzero((mag >= 2.0 ** e) & (mag < 2.0 ** (e + 1)))
        per_sign = 2 ** fmt["e4m3_mantissa_bits"] - (1 if e == 8 else 0)
        assert n == 2 * per_sign
    # one byte per element
    assert np.dtype(np.uint8).itemsize == fmt["fp8_bytes_per_element"]
    assert torch.empty(0, dtype=torch.float8_e4m3fn).element_size() == fmt["fp8_bytes_per_element"]
    assert torch.empty(0, dtype=torch.bfloat16).element_size() == fmt["bf16_bytes_per_element"]


def test_decoder_structure():
    dec = oracle.e4m3_decode(ALL)
    nan = np.isnan(dec)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert dec[0x00] == 0.0 and not math.copysign(1.0, dec[0x00]) < 0
    assert dec[0x80] == 0.0 and math.copysign(1.0, dec[0x80]) < 0
    assert dec[0x01] == 2.0 ** -9          # smallest subnormal
    assert dec[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert dec[0x08] == 2.0 ** -6          # smallest normal
    assert dec[0x38] == 1.0                # exponent bias 7
    pos = dec[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)        # strictly monotone in code order
    assert np.count_nonzero(pos > 0) == 126
    for c in range(0x7F):
        assert dec[c | 0x80] == -dec[c]


def test_decoder_matches_torch_float8_e4m3fn():
    ours = oracle.e4m3_decode(ALL)
    lib = torch_decode(ALL)
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all()


# ---------------------------------------------------------------- encoder

def _brute_force_encode(x):
    """Nearest E4M3 value by exhaustive search; ties to the even code;
    |x| >= 448 saturates; sign kept."""
    dec = oracle.e4m3_decode(ALL)
    mags = dec[0x00:0x7F]                     # 0 .. 448, codes 0x00..0x7E
    out = np.empty(x.shape, dtype=np.uint8)
    for i, v in enumerate(x.astype(np.float64)):
        a = abs(v)
        if a >= 448.0:
            c = 0x7E
        else:
            d = np.abs(mags - a)
            best = np.flatnonzero(d == d.min())
            c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
        out[i] = c | (0x80 if math.copysign(1.0, v) < 0 else 0)
    return out


def test_encoder_roundtrip_every_code():
    dec = oracle.e4m3_decode(ALL)
    ok = ~np.isnan(dec)
    assert np.array_equal(oracle.e4m3_encode(dec[ok].astype(np.float32)), ALL[ok])


def test_encoder_midpoints_ties_to_even():
    dec = oracle.e4m3_decode(ALL)
    for c in range(0x00, 0x7E):
        lo, hi = dec[c], dec[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2        # exactly representable
        even = c if c % 2 == 0 else c + 1
        for sgn in (0, 0x80):
            m = -mid if sgn else mid
            assert oracle.e4m3_encode(np.array([m]))[0] == (even | sgn)
            up = np.nextafter(mid, np.float32(np.inf))
            dn = np.nextafter(mid, np.float32(0))
            assert oracle.e4m3_encode(np.array([-up if sgn else up]))[0] == ((c + 1) | sgn)
            assert oracle.e4m3_encode(np.array([-dn if sgn else dn]))[0] == (c | sgn)


def test_encoder_matches_brute_force_search():
    rng = np.random.default_rng(1234)
    n = 20000
    mag = np.float32(2.0) ** rng.uniform(-13, 10, n).astype(np.float32)
    x = (mag * np.where(rng.random(n) < 0.5, -1, 1)).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), _brute_force_encode(x))


def test_encoder_matches_torch_in_range():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * 60).astype(np.float32)
    x = x[np.abs(x) < 448]
    x = np.concatenate([x, np.float32(2.0) ** rng.uniform(-12, -5, 5000).astype(np.float32)])
    assert np.array_equal(oracle.e4m3_encode(x), torch_encode(x))


def test_encoder_saturation_and_special_values():
    f = np.float32
    cases = [  # a list, not a dict: 0.0 and -0.0 are equal keys
        (f(448.0), 0x7E), (f(448.5), 0x7E), (f(464.0), 0x7E), (f(1e30), 0x7E), (f(np.inf), 0x7E),
        (f(-448.0), 0xFE), (f(-1e9), 0xFE), (f(-np.inf), 0xFE),
        (f(0.0), 0x00), (f(-0.0), 0x80),
        (f(2.0 ** -10), 0x00),                 # tie between 0 and 2^-9 -> even (0)
        (f(-2.0 ** -10), 0x80),                # sign kept on underflow
        (f(2.0 ** -10 * (1 + 2.0 ** -20)), 0x01),
        (f(2.0 ** -12), 0x00),
        (f(240.0), 0x77),                      # not the fnuz maximum
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    assert list(oracle.e4m3_encode(x)) == [c[1] for c in cases]
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


# ------------------------------------------------------------- quantiser

def test_quantize_divides_in_fp32_then_rounds_once():
    # Inputs (bf16 x, fp32 scale) whose exact quotient lies just beyond an E4M3
    # midpoint but whose IEEE fp32 quotient IS the midpoint: a single fp32
    # divide then one RNE rounding picks the even code; rounding the exact
    # quotient would pick the other neighbour.
    cases = [(0xBE6A, 0x3FDC3C3C), (0xBDC3, 0x3FB78787), (0xBFBA, 0x3EAF0F0F)]
    dec = oracle.e4m3_decode(ALL)
    for xb, sb in cases:
        x = np.array([xb << 16], np.uint32).view(np.float32)[0]
        s = np.array([sb], np.uint32).view(np.float32)[0]
        q32 = np.float32(x) / np.float32(s)
        exact = Fraction(float(x)) / Fraction(float(s))
        mags = dec[0x00:0x7F]
        i = int(np.searchsorted(mags, abs(float(q32))))
        lo, hi = i - 1, i
        assert Fraction(float(abs(q32))) == (Fraction(mags[lo]) + Fraction(mags[hi])) / 2
        assert abs(exact) != abs(Fraction(float(q32)))
        even = lo if lo % 2 == 0 else hi
        sign = 0x80 if x < 0 else 0
        got = oracle.quantize_bf16(np.array([xb], np.uint16), float(s))[0]
        assert got == (even | sign)


def test_quantize_matches_fp32_division_and_torch_cast():
    rng = np.random.default_rng(5)
    x = torch.randn(50000, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    for s in (np.float32(1.0), np.float32(0.011160714), np.float32(rng.uniform(0.001, 3))):
        y = x.to(torch.float32).numpy() / s                       # IEEE fp32 divide
        ref = torch_encode(y)
        inr = np.abs(y) < 448
        got = oracle.quantize_bf16(bits, float(s))
        assert np.array_equal(got[inr], ref[inr])
        assert np.all(got[~inr] & 0x7F == 0x7E)


def test_quantize_scale_one_is_plain_cast():
    # All 65536 bf16 bit patterns: with scale 1.0 the quantiser is a cast.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    got = oracle.quantize_bf16(bits, 1.0)
    fin = np.isfinite(f)
    inr = fin & (np.abs(f) < 448)
    assert np.array_equal(got[inr], torch_encode(f[inr]))
    big = fin & ~inr
    assert np.all(got[big] == np.where(f[big] < 0, 0xFE, 0x7E))
    assert np.all(got[np.isnan(f)] == 0x7F)


# ------------------------------------------------------------- attention

def _rand_case(seed, lens, Hq, Hkv, d, kv_std=1.0):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    T = int(sum(lens))
    q = torch.randn((B, Hq, d), generator=g).to(torch.bfloat16)
    k = (torch.randn((T, Hkv, d), generator=g) * kv_std).to(torch.bfloat16)
    v = (torch.randn((T, Hkv, d), generator=g) * kv_std).to(torch.bfloat16)
    ks = float(np.float32(k.abs().max().float() / 448))
    vs = float(np.float32(v.abs().max().float() / 448))
    qb = q.view(torch.int16).numpy().view(np.uint16)
    kc = oracle.quantize_bf16(k.view(torch.int16).numpy().view(np.uint16), ks)
    vc = oracle.quantize_bf16(v.view(torch.int16).numpy().view(np.uint16), vs)
    return q, qb, kc, vc, ks, vs


def _torch_reference(q, kc, vc, lens, ks, vs, sm, window):
    """fp64 softmax attention through torch's own routines."""
    B, Hq, d = q.shape
    Hkv = kc.shape[1]
    g = Hq // Hkv
    kh = torch.from_numpy(torch_decode(kc)) * ks
    vh = torch.from_numpy(torch_decode(vc)) * vs
    out = torch.zeros((B, Hq, d), dtype=torch.float64)
    start = 0
    for b, L in enumerate(lens):
        if L > 0:
            lo = L - window if (window > 0 and L > window) else 0
            for h in range(Hq):
                K = kh[start + lo:start + L, h // g, :]
                V = vh[start + lo:start + L, h // g, :]
                s = sm * (K @ q[b, h].to(torch.float64))
                out[b, h] = torch.softmax(s, dim=0) @ V
        start += L
    return out.numpy()


@pytest.mark.parametrize("lens,Hq,Hkv,d,window", [
    ([37], 4, 4, 16, 0), ([1, 50, 17], 8, 2, 32, 0), ([64, 3], 8, 1, 64, 5),
    ([100, 100], 16, 4, 128, 33), ([0, 20], 4, 2, 16, 0),
])
def test_attention_matches_torch_fp64_softmax(lens, Hq, Hkv, d, window):
    q, qb, kc, vc, ks, vs = _rand_case(11, lens, Hq, Hkv, d)
    sm = float(np.float32(1 / math.sqrt(d)))
    got = oracle.decode_attention(qb, kc, vc, lens, ks, vs, sm, window)
    ref = _torch_reference(q, kc, vc, lens, ks, vs, sm, window)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_attention_single_key_and_window_one_return_that_value():
    lens = [1, 9]
    q, qb, kc, vc, ks, vs = _rand_case(2, lens, 4, 2, 32)
    vh = oracle.e4m3_decode(vc) * vs
    out = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.17, 0)
    for h in range(4):
        assert np.array_equal(out[0, h], vh[0, h // 2])
    out_w1 = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.17, 1)
    for h in range(4):
        assert np.array_equal(out_w1[1, h], vh[1 + 8, h // 2])


def test_attention_zero_query_and_identical_keys_give_mean():
    lens = [40]
    q, qb, kc, vc, ks, vs = _rand_case(3, lens, 2, 1, 16)
    vh = oracle.e4m3_decode(vc) * vs
    zq = np.zeros_like(qb)
    out = oracle.decode_attention(zq, kc, vc, lens, ks, vs, 0.25, 0)
    assert np.allclose(out[0, 0], vh[:, 0].mean(axis=0), rtol=0, atol=1e-14)
    kc_same = np.repeat(kc[:1], 40, axis=0)
    out2 = oracle.decode_attention(qb, kc_same, vc, lens, ks, vs, 0.25, 10)
    assert np.allclose(out2[0, 1], vh[30:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_attention_window_equals_truncated_sequence():
    lens = [70, 45]
    q, qb, kc, vc, ks, vs = _rand_case(4, lens, 8, 2, 32)
    W = 20
    win = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.2, W)
    keep = np.r_[70 - W:70, 70 + 45 - W:70 + 45]
    trunc = oracle.decode_attention(qb, kc[keep], vc[keep], [W, W], ks, vs, 0.2, 0)
    assert np.array_equal(win, trunc)
    full = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.2, 0)
    assert np.array_equal(oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.2, 70), full)
    assert not np.allclose(win, full)


def test_attention_gqa_head_mapping():
    lens = [30]
    Hq, Hkv = 8, 4
    q, qb, kc, vc, ks, vs = _rand_case(5, lens, Hq, Hkv, 16)
    base = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.3, 0)
    for j in range(Hkv):
        kc2, vc2 = kc.copy(), vc.copy()
        kc2[:, j, :] = np.roll(kc2[:, j, :], 3, axis=0)
        vc2[:, j, :] = vc2[::-1, j, :]
        o = oracle.decode_attention(qb, kc2, vc2, lens, ks, vs, 0.3, 0)
        changed = [h for h in range(Hq) if not np.array_equal(o[0, h], base[0, h])]
        assert changed == list(range(j * 2, j * 2 + 2))


def test_attention_scales_enter_where_defined():
    lens = [25]
    q, qb, kc, vc, ks, vs = _rand_case(6, lens, 4, 2, 32)
    a = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.125, 0)
    b = oracle.decode_attention(qb, kc, vc, lens, ks, vs * 2, 0.125, 0)
    assert np.array_equal(b, 2 * a)                   # out is linear in v_scale
    c = oracle.decode_attention(qb, kc, vc, lens, ks * 2, vs, 0.125, 0)
    e = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.25, 0)
    assert np.array_equal(c, e)                       # k_scale multiplies the score
    assert not np.allclose(a, c)


def test_attention_invariant_to_token_order():
    lens = [60]
    q, qb, kc, vc, ks, vs = _rand_case(7, lens, 4, 1, 64)
    perm = np.random.default_rng(0).permutation(60)
    a = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.125, 0)
    b = oracle.decode_attention(qb, kc[perm], vc[perm], lens, ks, vs, 0.125, 0)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-15)


def test_attention_empty_sequence_is_zero():
    lens = [0, 5, 0]
    q, qb, kc, vc, ks, vs = _rand_case(8, lens, 2, 1, 16)
    out = oracle.decode_attention(qb, kc, vc, lens, ks, vs, 0.25, 0)
    assert np.all(out[0] == 0) and np.all(out[2] == 0) and np.any(out[1] != 0)


def test_reduced_precision_accumulator_fails_at_128k_and_fp32_passes():
    """A 10-bit accumulator over a 131072-token P.V contraction (the failure
    the pages describe past 100K) must break the attention tolerance; a 24-bit
    (fp32-width) accumulator must meet it.  This shows the parity bar can see
    that failure."""
    L = 131072
    q, qb, kc, vc, ks, vs = _rand_case(9, [L], 4, 1, 128, kv_std=0.5)
    sm = float(np.float32(1 / math.sqrt(128)))
    n = oracle.max_threads()
    ref = oracle.decode_attention(qb, kc, vc, [L], ks, vs, sm, 0, nthreads=n)
    bad = oracle.decode_attention(qb, kc, vc, [L], ks, vs, sm, 0, nthreads=n, acc_bits=10)
    good = oracle.decode_attention(qb, kc, vc, [L], ks, vs, sm, 0, nthreads=n, acc_bits=24)
    mx_b, mean_b = attn_errors(bad, ref)
    assert mx_b > ATTN_MAX_ABS or mean_b > ATTN_MEAN_ABS
    mx_g, mean_g = attn_errors(good, ref)
    assert mx_g <= ATTN_MAX_ABS / 10 and mean_g <= ATTN_MEAN_ABS / 10


# ------------------------------------------------------------- the bf16 cache (comparison baseline)

def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("lens,Hq,Hkv,d,window", [
    ([37], 4, 4, 16, 0), ([1, 50, 17], 8, 2, 32, 0), ([64, 3], 8, 1, 64, 5), ([100, 0, 100], 16, 4, 128, 33),
])
def test_bf16_attention_matches_torch_fp64_softmax(lens, Hq, Hkv, d, window):
    g = torch.Generator().manual_seed(21)
    B, T = len(lens), int(sum(lens))
    q = torch.randn((B, Hq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((T, Hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((T, Hkv, d), generator=g).to(torch.bfloat16)
    sm = float(np.float32(1 / math.sqrt(d)))
    got = oracle.decode_attention_bf16(_bits(q), _bits(k), _bits(v), lens, sm, window)
    G = Hq // Hkv
    ref = np.zeros((B, Hq, d))
    start = 0
    for b, L in enumerate(lens):
        if L > 0:
            lo = L - window if (window > 0 and L > window) else 0
            for h in range(Hq):
                K = k[start + lo:start + L, h // G].double()
                V = v[start + lo:start + L, h // G].double()
                ref[b, h] = (torch.softmax(sm * (K @ q[b, h].double()), dim=0) @ V).numpy()
        start += L
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_bf16_and_fp8_attention_agree_on_values_both_hold_exactly():
    """K and V drawn from E4M3 values (exact in bf16): the fp8 oracle with
    scale 1 on their codes and the bf16 oracle on the values must agree
    bit for bit, since both compute the same fp64 sums of the same numbers."""
    rng = np.random.default_rng(5)
    lens, Hq, Hkv, d = [33, 70], 8, 2, 64
    T = sum(lens)
    codes_k = rng.integers(0, 256, size=(T, Hkv, d)).astype(np.uint8)
    codes_v = rng.integers(0, 256, size=(T, Hkv, d)).astype(np.uint8)
    for c in (codes_k, codes_v):
        c[(c & 0x7F) == 0x7F] = 0x00          # no NaN codes
    kf = oracle.e4m3_decode(codes_k).astype(np.float32)
    vf = oracle.e4m3_decode(codes_v).astype(np.float32)
    kb = (kf.view(np.uint32) >> 16).astype(np.uint16)   # exact: E4M3 values have 3 mantissa bits
    vb = (vf.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((kb.astype(np.uint32) << 16).view(np.float32), kf)
    q = _bits(torch.randn((2, Hq, d), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16))
    for window in (0, 9):
        a = oracle.decode_attention(q, codes_k, codes_v, lens, 1.0, 1.0, 0.125, window)
        b = oracle.decode_attention_bf16(q, kb, vb, lens, 0.125, window)
        assert np.array_equal(a, b)


def test_bf16_attention_single_key_returns_its_value():
    g = torch.Generator().manual_seed(8)
    v = torch.randn((1, 2, 16), generator=g).to(torch.bfloat16)
    k = torch.randn((1, 2, 16), generator=g).to(torch.bfloat16)
    q = torch.randn((1, 4, 16), generator=g).to(torch.bfloat16)
    out = oracle.decode_attention_bf16(_bits(q), _bits(k), _bits(v), [1], 0.3, 0)
    for h in range(4):
        assert np.array_equal(out[0, h], v[0, h // 2].double().numpy())


# ------------------------------------------------------------- per-kv-head scales

def _per_head_case(seed, lens, Hq, Hkv, d):
    g = torch.Generator().manual_seed(seed)
    B, T = len(lens), int(sum(lens))
    q = torch.randn((B, Hq, d), generator=g).to(torch.bfloat16)
    # heads of very different magnitude, so one scale per head matters
    mag = torch.tensor([2.0 ** (3 * h - 4) for h in range(Hkv)]).view(1, Hkv, 1)
    k = (torch.randn((T, Hkv, d), generator=g) * mag).to(torch.bfloat16)
    v = (torch.randn((T, Hkv, d), generator=g) * mag).to(torch.bfloat16)
    ks = (k.float().abs().amax(dim=(0, 2)) / 448).numpy().astype(np.float32)
    vs = (v.float().abs().amax(dim=(0, 2)) / 448).numpy().astype(np.float32)
    return q, k, v, ks, vs


def test_per_head_quantize_is_per_tensor_quantize_of_each_head():
    q, k, v, ks, vs = _per_head_case(31, [20, 7], 8, 4, 32)
    kb = _bits(k)
    codes = oracle.quantize_bf16_per_head(kb, ks)
    for h in range(4):
        assert np.array_equal(codes[:, h, :], oracle.quantize_bf16(np.ascontiguousarray(kb[:, h, :]), ks[h]))
    # equal scales: the per-tensor codes
    same = np.full(4, ks.max(), dtype=np.float32)
    assert np.array_equal(oracle.quantize_bf16_per_head(kb, same), oracle.quantize_bf16(kb, float(ks.max())))


@pytest.mark.parametrize("window", [0, 6])
def test_per_head_attention_equals_per_tensor_attention_of_each_head(window):
    """Each kv head (with its q group) through the per-tensor oracle, at that
    head's scales, gives exactly the per-head oracle's output for the group."""
    lens, Hq, Hkv, d = [25, 1, 40], 8, 4, 32
    q, k, v, ks, vs = _per_head_case(32, lens, Hq, Hkv, d)
    kc = oracle.quantize_bf16_per_head(_bits(k), ks)
    vc = oracle.quantize_bf16_per_head(_bits(v), vs)
    qb = _bits(q)
    got = oracle.decode_attention_per_head(qb, kc, vc, lens, ks, vs, 0.2, window)
    G = Hq // Hkv
    for h in range(Hkv):
        ref = oracle.decode_attention(np.ascontiguousarray(qb[:, h * G:(h + 1) * G]),
                                      np.ascontiguousarray(kc[:, h:h + 1]), np.ascontiguousarray(vc[:, h:h + 1]),
                                      lens, float(ks[h]), float(vs[h]), 0.2, window)
        assert np.array_equal(got[:, h * G:(h + 1) * G], ref)


def test_per_head_attention_with_equal_scales_is_the_per_tensor_attention():
    lens, Hq, Hkv, d = [30, 12], 8, 2, 16
    q, k, v, ks, vs = _per_head_case(33, lens, Hq, Hkv, d)
    kc = oracle.quantize_bf16(_bits(k), 0.05)
    vc = oracle.quantize_bf16(_bits(v), 0.07)
    a = oracle.decode_attention(_bits(q), kc, vc, lens, 0.05, 0.07, 0.3, 0)
    b = oracle.decode_attention_per_head(_bits(q), kc, vc, lens, np.full(Hkv, 0.05, np.float32),
                                         np.full(Hkv, 0.07, np.float32), 0.3, 0)
    assert np.array_equal(a, b)


# ------------------------------------------------------------- E5M2 (the other FP8 format)

def test_e5m2_decoder_printed_facts_and_structure():
    """2 mantissa bits and a maximum of 57,344 (gpusmith.com, "What FP8 KV
    changes"); IEEE-style specials; every finite value once per sign."""
    c = np.arange(256, dtype=np.uint8)
    d = oracle.e5m2_decode(c)
    fin = np.isfinite(d)
    assert d[fin].max() == 57344.0 and d[0x7B] == 57344.0 and d[0xFB] == -57344.0
    assert np.isinf(d[0x7C]) and d[0x7C] > 0 and np.isinf(d[0xFC]) and d[0xFC] < 0
    assert np.isnan(d[[0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]]).all()
    assert d[0x01] == 2.0 ** -16 and d[0x04] == 2.0 ** -14          # smallest subnormal / normal
    pos = d[:0x7C]
    assert np.all(np.diff(pos) > 0)                                   # monotone in code order
    assert np.array_equal(d[0x80:0xFC], -pos)
    # each binade [2^e, 2^(e+1)) holds exactly 4 values (2 mantissa bits)
    for e in range(-14, 16):
        n = np.count_nonzero((pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1)))
        assert n == 4, e


def test_e5m2_decoder_matches_torch_float8_e5m2():
    c = np.arange(256, dtype=np.uint8)
    d = oracle.e5m2_decode(c)
    t = torch.from_numpy(c.copy()).view(torch.float8_e5m2).double().numpy()
    assert np.array_equal(np.isnan(d), np.isnan(t))
    ok = ~np.isnan(d)
    assert np.array_equal(d[ok], t[ok])


def test_e5m2_encoder_roundtrip_midpoints_and_saturation():
    c = np.arange(256, dtype=np.uint8)
    d = oracle.e5m2_decode(c)
    fin = np.isfinite(d)
    assert np.array_equal(oracle.e5m2_encode(d[fin].astype(np.float32)), c[fin])
    # midpoints between neighbours go to the even code
    pos = np.sort(d[(d > 0) & fin])
    mid = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (pos[:-1] + pos[1:]) / 2)   # exact in fp32
    got = oracle.e5m2_encode(mid)
    lo = oracle.e5m2_encode(pos[:-1].astype(np.float32))
    hi = oracle.e5m2_encode(pos[1:].astype(np.float32))
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, hi))
    sat = np.array([57344.0, 60000.0, 61440.0, 1e30, np.inf, -61440.0, -np.inf], dtype=np.float32)
    assert list(oracle.e5m2_encode(sat)) == [0x7B] * 5 + [0xFB] * 2
    assert oracle.e5m2_encode(np.array([np.nan], np.float32))[0] == 0x7F
    assert list(oracle.e5m2_encode(np.array([0.0, -0.0, 2.0 ** -18, -2.0 ** -18], np.float32))) == [0, 0x80, 0, 0x80]


def test_e5m2_encoder_matches_brute_force_and_torch_in_range():
    rng = np.random.default_rng(9)
    y = (rng.standard_normal(20000) * np.exp2(rng.integers(-18, 16, 20000))).astype(np.float32)
    y = y[np.abs(y) < 57344]
    got = oracle.e5m2_encode(y)
    c = np.arange(256, dtype=np.uint8)
    d = oracle.e5m2_decode(c)
    fin = np.isfinite(d)
    vals, codes = d[fin], c[fin]
    # brute force: nearest finite value, ties to the even code
    dist = np.abs(y[:, None].astype(np.float64) - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = np.where(dist == best, codes[None, :].astype(np.int32), 999)
    even = np.where(cand % 2 == 0, cand, 999).min(axis=1)
    first = cand.min(axis=1)
    ties = (dist == best).sum(axis=1) > 1
    want = np.where(ties, even, first).astype(np.uint8)
    # zero: the sign of the input decides between 0x00 and 0x80
    zero = want == 0
    want[zero & (y < 0)] = 0x80
    assert np.array_equal(got, want)
    t = torch.from_numpy(y).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(got, t)


@pytest.mark.parametrize("window", [0, 5])
def test_e5m2_attention_matches_torch_fp64_softmax(window):
    lens, Hq, Hkv, d = [33, 1, 60], 8, 2, 32
    g = torch.Generator().manual_seed(41)
    q = torch.randn((3, Hq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((sum(lens), Hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((sum(lens), Hkv, d), generator=g).to(torch.bfloat16)
    ks = float(np.float32(k.float().abs().max() / 57344))
    vs = float(np.float32(v.float().abs().max() / 57344))
    kc = oracle.quantize_bf16_e5m2(_bits(k), ks)
    vc = oracle.quantize_bf16_e5m2(_bits(v), vs)
    # the quantiser is the encoder applied to the fp32 quotient
    assert np.array_equal(kc, oracle.e5m2_encode((k.float() / torch.tensor(ks, dtype=torch.float32)).numpy()))
    got = oracle.decode_attention_e5m2(_bits(q), kc, vc, lens, ks, vs, 0.25, window)
    kh = torch.from_numpy(oracle.e5m2_decode(kc)) * ks
    vh = torch.from_numpy(oracle.e5m2_decode(vc)) * vs
    G = Hq // Hkv
    ref = np.zeros_like(got)
    start = 0
    for b, L in enumerate(lens):
        lo = L - window if (window > 0 and L > window) else 0
        for h in range(Hq):
            K = kh[start + lo:start + L, h // G]
            V = vh[start + lo:start + L, h // G]
            ref[b, h] = (torch.softmax(0.25 * (K @ q[b, h].double()), dim=0) @ V).numpy()
        start += L
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- prefill (chunked) attention

@pytest.mark.parametrize("window", [0, 9])
def test_prefill_matches_torch_causal_softmax(window):
    lens, qlens, Hq, Hkv, d = [40, 17, 5], [12, 17, 1], 8, 2, 32
    g = torch.Generator().manual_seed(51)
    T = sum(lens)
    k = torch.randn((T, Hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((T, Hkv, d), generator=g).to(torch.bfloat16)
    q = torch.randn((sum(qlens), Hq, d), generator=g).to(torch.bfloat16)
    ks = float(np.float32(k.float().abs().max() / 448))
    vs = float(np.float32(v.float().abs().max() / 448))
    kc = oracle.quantize_bf16(_bits(k), ks)
    vc = oracle.quantize_bf16(_bits(v), vs)
    sm = float(np.float32(0.2))   # the oracle takes sm_scale as an fp32 value
    got = oracle.prefill_attention(_bits(q), kc, vc, lens, qlens, ks, vs, sm, window)
    kh = torch.from_numpy(oracle.e4m3_decode(kc)) * ks
    vh = torch.from_numpy(oracle.e4m3_decode(vc)) * vs
    G = Hq // Hkv
    ref = np.zeros_like(got)
    s0, r0 = 0, 0
    for L, n in zip(lens, qlens):
        pos = torch.arange(L)
        for i in range(n):
            p = L - n + i
            mask = pos <= p
            if window > 0:
                mask &= pos > p - window
            for h in range(Hq):
                K = kh[s0:s0 + L, h // G]
                V = vh[s0:s0 + L, h // G]
                s = sm * (K @ q[r0 + i, h].double())
                s = torch.where(mask, s, torch.tensor(float("-inf"), dtype=torch.float64))
                ref[r0 + i, h] = (torch.softmax(s, dim=0) @ V).numpy()
        s0 += L
        r0 += n
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_prefill_last_row_is_the_decode_and_first_key_row_is_its_value():
    lens, qlens = [30, 20], [30, 4]
    q, qb, kc, vc, ks, vs = _rand_case(52, lens, 4, 2, 16)
    # queries: one row per query token, taken from the decode case's random q
    rng = np.random.default_rng(3)
    qrows = rng.integers(0, 0x3F80, size=(sum(qlens), 4, 16)).astype(np.uint16)  # finite bf16 patterns
    out = oracle.prefill_attention(qrows, kc, vc, lens, qlens, ks, vs, 0.3, 0)
    dec = oracle.decode_attention(np.stack([qrows[qlens[0] - 1], qrows[-1]]), kc, vc, lens, ks, vs, 0.3, 0)
    assert np.array_equal(out[qlens[0] - 1], dec[0]) and np.array_equal(out[-1], dec[1])
    vh = oracle.e4m3_decode(vc) * vs
    for h in range(4):   # the first token of sequence 0 attends only itself
        assert np.array_equal(out[0, h], vh[0, h // 2])
