/*
 * fp8kv oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the fp8 paged
 * decode-attention path computes.  Only the test-suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load this code; the product
 * library never links it and shares no source, header, table or helper with
 * it.
 *
 * Sources (the four web pages on FP8 KV caches):
 *   - gpusmith.com, "FP8 KV Cache Quantization: Capacity Gains and Accuracy
 *     Risk", section "What FP8 KV changes" (E4M3: 3 mantissa bits, maximum
 *     normal 448; 1 byte per element) and section "Scales and calibration"
 *     (each K and V tensor is divided by a scale before it is cast; one scale
 *     per tensor).  The bit layout follows the format paper that page cites
 *     (Micikevicius et al., "FP8 Formats for Deep Learning"): S.EEEE.MMM,
 *     exponent bias 7, subnormals, no infinities, NaN = S.1111.111.
 *   - particula.tech, "KV Cache Quantization: What FP8 and q8_0 Cost in
 *     Accuracy", opening section (partial results belong in a real FP32
 *     register; the oracle goes further and uses fp64).
 *   - phantomic12 vLLM-blog summary, "ACCURACY AT LONG CONTEXT" (the
 *     Softmax(AttnScore)*V contraction runs over the context length) and
 *     "DECODE COST" (sliding windows of 128 and 512).
 *
 * Readings where the pages are silent:
 *   - Rounding to E4M3 is round-to-nearest, ties-to-even; finite magnitudes
 *     >= 448 and infinities saturate to +-448 (codes 0x7E / 0xFE); NaN maps to
 *     0x7F; the sign of zero and of an underflow is kept.
 *   - "Divided by a scale" is one IEEE fp32 division x/s, followed by one
 *     rounding to E4M3 (so the oracle divides in fp32, not in fp64).
 *   - A sliding window W > 0 keeps the last W keys including the current one:
 *     t in [max(0, L - W), L - 1].  W <= 0 means full attention.
 *   - Query head h reads key/value head h / g, g = Hq / Hkv.
 *   - seq_len 0 produces an all-zero output row.
 *
 * Everything is computed in fp64 from the decoded codes, as the plain
 * definition of softmax attention (two passes: maximum, then weighted sums).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact value of an E4M3 code (fp64).  Normal: (8 + m) * 2^(e - 10), which is
 * (1 + m/8) * 2^(e - 7); subnormal (e == 0): m * 2^-9. */
double oracle_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double n) {
    double fl = floor(n);
    double frac = n - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* E4M3 encoder: RNE, saturating to the largest finite value. */
uint8_t oracle_e4m3_encode(float y) {
    uint32_t bits;
    memcpy(&bits, &y, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    if (isnan(y)) return 0x7F;
    double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* includes +-inf */
    if (a == 0.0) return sign;
    /* a = f * 2^ex, f in [0.5, 1): the leading binade is 2^(ex - 1). */
    int ex;
    frexp(a, &ex);
    int E = ex - 1;
    if (E < -6) E = -6;            /* subnormal range shares the 2^-6 quantum */
    double quantum = ldexp(1.0, E - 3);
    double r = round_half_even(a / quantum); /* exact: quantum is a power of 2 */
    double v = r * quantum;                  /* representable E4M3 magnitude   */
    if (v == 0.0) return sign;
    if (v > 448.0) v = 448.0;                /* cannot happen for a < 448      */
    uint8_t code;
    if (v < ldexp(1.0, -6)) {
        code = (uint8_t)(v / ldexp(1.0, -9)); /* subnormal: m * 2^-9 */
    } else {
        int vex;
        frexp(v, &vex);
        int Ev = vex - 1;                                   /* v in [2^Ev, 2^(Ev+1)) */
        int m = (int)(v / ldexp(1.0, Ev - 3)) - 8;          /* 0..7 */
        code = (uint8_t)(((Ev + 7) << 3) | m);
    }
    return (uint8_t)(sign | code);
}

/*
 * E5M2 (the other FP8 format; gpusmith.com, "What FP8 KV changes": 2 mantissa
 * bits, maximum 57,344).  Layout after the same format paper: S.EEEEE.MM,
 * exponent bias 15, subnormals m * 2^-16, IEEE-style specials (exponent 31:
 * mantissa 0 = infinity, otherwise NaN).
 */
double oracle_e5m2_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 2) & 0x1F;
    int m = c & 0x3;
    double v;
    if (e == 31) return m == 0 ? (s ? -INFINITY : INFINITY) : NAN;
    if (e == 0)
        v = ldexp((double)m, -16);
    else
        v = ldexp((double)(4 + m), e - 17);
    return s ? -v : v;
}

/* E5M2 encoder: RNE, saturating finite magnitudes >= 57344 and infinities to
 * +-57344 (0x7B / 0xFB); NaN maps to 0x7F; the sign of zero and of an
 * underflow is kept. */
uint8_t oracle_e5m2_encode(float y) {
    uint32_t bits;
    memcpy(&bits, &y, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    if (isnan(y)) return 0x7F;
    double a = fabs((double)y);
    if (a >= 57344.0) return (uint8_t)(sign | 0x7B);
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);
    int E = ex - 1;                 /* a in [2^E, 2^(E+1)) */
    if (E < -14) E = -14;           /* subnormals share the 2^-16 quantum */
    double quantum = ldexp(1.0, E - 2);
    double v = round_half_even(a / quantum) * quantum;
    if (v == 0.0) return sign;
    uint8_t code;
    if (v < ldexp(1.0, -14)) {
        code = (uint8_t)(v / ldexp(1.0, -16));
    } else {
        int vex;
        frexp(v, &vex);
        int Ev = vex - 1;
        int m = (int)(v / ldexp(1.0, Ev - 2)) - 4;     /* 0..3 */
        code = (uint8_t)(((Ev + 15) << 2) | m);
    }
    return (uint8_t)(sign | code);
}

/* Quantise-on-append into E5M2: code = e5m2(fp32(x) / scale). */
void oracle_quantize_bf16_e5m2(const uint16_t* x, int64_t n, float scale, uint8_t* out);

void oracle_decode_codes_e5m2(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e5m2_decode(c[i]);
}

static float bf16_bits_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Quantise-on-append: code = e4m3(fp32(x) / scale), with an fp32 IEEE divide. */
void oracle_quantize_bf16(const uint16_t* x, int64_t n, float scale, uint8_t* out) {
    /* every element is independent; threads only split the index range */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) {
        float xf = bf16_bits_to_float(x[i]);
        float y = xf / scale;
        out[i] = oracle_e4m3_encode(y);
    }
}

void oracle_quantize_bf16_e5m2(const uint16_t* x, int64_t n, float scale, uint8_t* out) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) {
        float xf = bf16_bits_to_float(x[i]);
        float y = xf / scale;
        out[i] = oracle_e5m2_encode(y);
    }
}

void oracle_encode_f32_e5m2(const float* y, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e5m2_encode(y[i]);
}

void oracle_encode_f32(const float* y, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(y[i]);
}

void oracle_decode_codes(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}

/* Rounds v to `bits` significand bits (nearest, ties to even); used only by the
 * reduced-precision accumulator below. */
static double round_to_bits(double v, int bits) {
    if (v == 0.0 || !isfinite(v)) return v;
    int ex;
    frexp(v, &ex);
    double q = ldexp(1.0, ex - bits);
    double n = fabs(v) / q;
    double r = round_half_even(n) * q;
    return v < 0 ? -r : r;
}

/*
 * Where the cached K and V of one sequence live: E4M3 codes with their
 * per-tensor scales (the fp8 cache), or bf16 values (the bf16 cache that the
 * fp8 one is compared against).  Element i of token t, kv head hk is at
 * t * Hkv * d + hk * d + i.
 */
typedef struct {
    const uint8_t* kc;   /* E4M3 codes, or NULL */
    const uint8_t* vc;
    const uint16_t* kb;  /* bf16 bits, used when kc is NULL */
    const uint16_t* vb;
    const double* dec;   /* decoded value of each of the 256 codes */
    double k_scale, v_scale;        /* per-tensor scales ... */
    const float* k_head_scales;     /* ... or one per kv head ([Hkv]) when not NULL */
    const float* v_head_scales;
    int Hkv, d;
} kv_store;

static double kv_key(const kv_store* s, int64_t idx) {
    if (!s->kc) return (double)bf16_bits_to_float(s->kb[idx]);
    const double sc = s->k_head_scales ? (double)s->k_head_scales[(idx / s->d) % s->Hkv] : s->k_scale;
    return s->dec[s->kc[idx]] * sc;
}

static double kv_value(const kv_store* s, int64_t idx) {
    if (!s->vc) return (double)bf16_bits_to_float(s->vb[idx]);
    const double sc = s->v_head_scales ? (double)s->v_head_scales[(idx / s->d) % s->Hkv] : s->v_scale;
    return s->dec[s->vc[idx]] * sc;
}

/*
 * One query head of decode attention over a contiguous (logical-order) run of
 * cached tokens; the store points at token 0 of the sequence.
 * acc_bits <= 0: fp64 accumulation (the oracle proper).  acc_bits > 0: the
 * exp-weighted sums are rounded to acc_bits significand bits after every add,
 * a deliberately broken variant that models an imprecise accumulator.
 */
static void attend_one_head(const uint16_t* qh, const kv_store* kv,
                            int64_t L, int window, int Hkv, int hk, int d,
                            double sm_scale, int acc_bits, double* sigma,
                            double* num, double* out) {
    int64_t lo = 0;
    if (window > 0 && L > window) lo = L - window;
    int64_t stride = (int64_t)Hkv * d;
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    if (L <= 0) return;
    /* pass 1: scores and their maximum */
    double mx = -INFINITY;
    for (int64_t t = lo; t < L; ++t) {
        const int64_t kr = t * stride + (int64_t)hk * d;
        double s = 0.0;
        for (int i = 0; i < d; ++i)
            s += (double)bf16_bits_to_float(qh[i]) * kv_key(kv, kr + i);
        s *= sm_scale;
        sigma[t - lo] = s;
        if (s > mx) mx = s;
    }
    /* pass 2: exp-weighted sums */
    double den = 0.0;
    for (int i = 0; i < d; ++i) num[i] = 0.0;
    for (int64_t t = lo; t < L; ++t) {
        double w = exp(sigma[t - lo] - mx);
        const int64_t vr = t * stride + (int64_t)hk * d;
        if (acc_bits > 0) {
            den = round_to_bits(den + w, acc_bits);
            for (int i = 0; i < d; ++i)
                num[i] = round_to_bits(num[i] + w * kv_value(kv, vr + i), acc_bits);
        } else {
            den += w;
            for (int i = 0; i < d; ++i) num[i] += w * kv_value(kv, vr + i);
        }
    }
    for (int i = 0; i < d; ++i) out[i] = num[i] / den;
}

/* Decode attention for a batch over either store (the two entry points below). */
static int attention_batch(const uint16_t* q, const uint8_t* kc, const uint8_t* vc, const uint16_t* kb,
                           const uint16_t* vb, const int64_t* seq_start, const int32_t* seq_lens,
                           int B, int Hq, int Hkv, int d,
                           float k_scale, float v_scale, const float* k_head_scales, const float* v_head_scales,
                           float sm_scale, int window, int acc_bits, int nthreads, double* scratch,
                           int64_t max_len, double* out, int e5m2) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || nthreads <= 0) return -1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > max_len) return -1;
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = e5m2 ? oracle_e5m2_decode((uint8_t)c) : oracle_e4m3_decode((uint8_t)c);
    int g = Hq / Hkv;
    int64_t units = (int64_t)B * Hq;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        int b = (int)(u / Hq), h = (int)(u % Hq);
        double* sigma = scratch + (int64_t)tid * (max_len + d);
        double* num = sigma + max_len;
        const int64_t off = seq_start[b] * (int64_t)Hkv * d;
        kv_store kv = {kc ? kc + off : NULL, vc ? vc + off : NULL, kb ? kb + off : NULL, vb ? vb + off : NULL,
                       dec, (double)k_scale, (double)v_scale, k_head_scales, v_head_scales, Hkv, d};
        attend_one_head(q + ((int64_t)b * Hq + h) * d, &kv, seq_lens[b], window, Hkv, h / g, d,
                        (double)sm_scale, acc_bits, sigma, num, out + ((int64_t)b * Hq + h) * d);
    }
    return 0;
}

/*
 * Decode attention for a batch over an E4M3 cache.
 *   q        bf16 bits [B, Hq, d]
 *   kc, vc   E4M3 codes [total_tokens, Hkv, d]; sequence b occupies tokens
 *            [seq_start[b], seq_start[b] + seq_lens[b]) in logical order
 *   out      fp64 [B, Hq, d]
 *   scratch  fp64, at least nthreads * (max_len + d) elements
 * Returns 0 on success, -1 on bad arguments.
 */
int oracle_decode_attention(const uint16_t* q, const uint8_t* kc, const uint8_t* vc,
                            const int64_t* seq_start, const int32_t* seq_lens,
                            int B, int Hq, int Hkv, int d,
                            float k_scale, float v_scale, float sm_scale, int window,
                            int acc_bits, int nthreads, double* scratch,
                            int64_t max_len, double* out) {
    if (!kc || !vc) return -1;
    return attention_batch(q, kc, vc, NULL, NULL, seq_start, seq_lens, B, Hq, Hkv, d, k_scale, v_scale, NULL, NULL,
                           sm_scale, window, acc_bits, nthreads, scratch, max_len, out, 0);
}

/* The same attention over an E5M2 cache (per-tensor scales). */
int oracle_decode_attention_e5m2(const uint16_t* q, const uint8_t* kc, const uint8_t* vc,
                                 const int64_t* seq_start, const int32_t* seq_lens,
                                 int B, int Hq, int Hkv, int d,
                                 float k_scale, float v_scale, float sm_scale, int window,
                                 int nthreads, double* scratch, int64_t max_len, double* out) {
    if (!kc || !vc) return -1;
    return attention_batch(q, kc, vc, NULL, NULL, seq_start, seq_lens, B, Hq, Hkv, d, k_scale, v_scale, NULL, NULL,
                           sm_scale, window, 0, nthreads, scratch, max_len, out, 1);
}

/*
 * The same attention over an E4M3 cache with one K and one V scale per kv
 * head (k_scales, v_scales: [Hkv]); code c of kv head h stands for
 * decode(c) * scales[h].
 */
int oracle_decode_attention_per_head(const uint16_t* q, const uint8_t* kc, const uint8_t* vc,
                                     const int64_t* seq_start, const int32_t* seq_lens,
                                     int B, int Hq, int Hkv, int d,
                                     const float* k_scales, const float* v_scales, float sm_scale, int window,
                                     int nthreads, double* scratch, int64_t max_len, double* out) {
    if (!kc || !vc || !k_scales || !v_scales) return -1;
    return attention_batch(q, kc, vc, NULL, NULL, seq_start, seq_lens, B, Hq, Hkv, d, 1.0f, 1.0f, k_scales,
                           v_scales, sm_scale, window, 0, nthreads, scratch, max_len, out, 0);
}

/*
 * The same attention over a bf16 cache (kb, vb: bf16 bits [total_tokens, Hkv,
 * d]); no scales.
 */
int oracle_decode_attention_bf16(const uint16_t* q, const uint16_t* kb, const uint16_t* vb,
                                 const int64_t* seq_start, const int32_t* seq_lens,
                                 int B, int Hq, int Hkv, int d, float sm_scale, int window,
                                 int nthreads, double* scratch, int64_t max_len, double* out) {
    if (!kb || !vb) return -1;
    return attention_batch(q, NULL, NULL, kb, vb, seq_start, seq_lens, B, Hq, Hkv, d, 1.0f, 1.0f, NULL, NULL,
                           sm_scale, window, 0, nthreads, scratch, max_len, out, 0);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
