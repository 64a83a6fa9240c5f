// Paged fp8 (E4M3) decode attention for sm_103a.
//
// What it computes: single-query grouped-query softmax attention over a paged
// KV cache stored as E4M3 codes with per-tensor K and V scales, the fp8 cache
// read directly with dequantisation fused into the attention (gpusmith.com,
// "FP8 KV Cache Quantization: Capacity Gains and Accuracy Risk", sections
// "What FP8 KV changes" and "Attention backend interactions"), with scores,
// softmax and P.V accumulated in real FP32 registers however long the context
// (particula.tech, "KV Cache Quantization: What FP8 and q8_0 Cost in
// Accuracy", opening section; phantomic12 vLLM-blog summary, "ACCURACY AT
// LONG CONTEXT": the P.V contraction runs over the context length), and an
// optional sliding window (same summary, "DECODE COST": windows 128, 512).
//
// How (persistent CTAs over a flattened, evenly split page list):
//  * All g query heads of a kv head are handled together, so every cache byte
//    is read from HBM once.  Decode attention is bandwidth-bound (2g flop per
//    fp8 byte), so the kernel is built around streaming pages at HBM speed.
//  * The attended pages of every (sequence, kv head) unit are laid end to end
//    and cut into one equal contiguous range per CTA (2 CTAs per SM), so all
//    CTAs finish together whatever the mix of sequence lengths.  A CTA walks
//    the units its range overlaps ("segments").
//  * Tensor-core engine (the default, stream_decode_kernel): no producer
//    warps.  Each of the 4 warps of a CTA (6 at d = 64) takes one contiguous
//    share of every segment and streams it with 16-byte cp.async copies
//    (evict-first L2 policy) into a private ring of 3 stages (2 at d = 64
//    and d = 256), up to two stages ahead of the one it computes (one with
//    a two-stage ring); its block ids are consecutive entries of
//    one block-table row, read 32 at a time one window ahead.  Copies end by
//    themselves, so there is no barrier handshake and no wait to bound.  In a
//    decode step (fp8kv_decode_step) the warp whose share holds a unit's last
//    page first quantises the sequence's newest K and V rows into it, fences,
//    and only then copies it.  Many warps issuing small copies streamed the
//    random 2 KB pages faster than two TMA-issuing producer warps per CTA.
//  * CUDA-core engine (comparison only, paged_decode_kernel): two producer
//    warps stream the pages with TMA tensor copies into a ring guarded by
//    mbarriers (every wait bounded), four consumer warps own every fourth
//    stage.
//  * Per stage a consumer warp converts codes to f16 (exact) and runs the
//    score contraction S^T = K Q^T and the value contraction O^T += V^T P^T on
//    the tensor cores (mma m16n8k16, fp32 accumulators): the g <= 8 query
//    heads form the n=8 side.  The stage's P.V tile is then added into
//    separate FP32 registers (O = O*alpha + tile), so the long contraction is
//    summed in IEEE FP32, not inside the MMA.  The CUDA-core engine instead
//    sums FP32 fma chains of exact f16 products; it is slower at every
//    supported g and is used only when asked for.
//  * The softmax max/sum use warp shuffles; P is rounded to f16 for the MMA.
//  * At the end of a segment the CTA's warps merge through shared memory; a
//    unit split over several CTAs leaves FP32 partials.  When the plan gives
//    units few partials, each such CTA of the tensor-core engine counts its
//    partial on a per-unit counter in the workspace, and the CTA whose partial
//    completes the count combines the unit's partials at the end of its range
//    (one launch per call).  Otherwise, and always in the CUDA-core engine, a
//    small merge kernel combines them, launched as a programmatic dependent:
//    it derives the split from the lengths while the decode grid finishes,
//    then waits for that grid and reads the partials.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fp8kv.h"
#include "trace.cuh"
#include "partition.cuh"
#include "ptx.cuh"
#include "walk.cuh"

namespace fp8kv {

constexpr int kBS = 16;                    // tokens per page (block_size)
constexpr int kNCW = 4;                    // consumer warps per CTA
constexpr int kNPW = 2;                    // producer warps: one issues K copies, one V copies
constexpr int kThreads = (kNCW + kNPW) * 32;
constexpr int kStageHalf = 4096;           // K bytes (and V bytes) per stage
constexpr int kStageBytes = 2 * kStageHalf;
constexpr int kCtasPerSm = 2;
constexpr int kMaxBatch = 512;             // sequences per launch; larger batches run in chunks
constexpr int kMaxMergeSplits = 1024;      // CTAs per launch are capped at this (the merge keeps one weight each)
constexpr int kMinPagesPerCta = 16;
constexpr int kMaxG = 16;                  // query heads per kv head at most (partial (max, sum) entries per slot)
constexpr uint64_t kWaitLimitNs = 500000000ull;  // 0.5 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
    const uint16_t* q;          // bf16 [B, Hq, D]
    const uint16_t* k_new;      // bf16 [B, Hkv, D] newest rows to append first, or null
    const uint16_t* v_new;
    uint8_t* k_cache;           // the caches (written only when appending)
    uint8_t* v_cache;
    float k_scale_raw;          // per-tensor scales (the append divides by them)
    float v_scale_raw;
    const float* k_scales;      // [Hkv] per-kv-head scales, or null for the per-tensor ones
    const float* v_scales;
    float sm_scale;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    uint16_t* out;              // bf16 [B, Hq, D]
    uint32_t* err;              // workspace error word
    int decode_ctas;            // grid size of the decode kernel (the merge recomputes its split)
    float2* part_ml;            // [B*Hkv + ctas][kMaxG] (max, sum) in log2 units
    float* part_o;              // [B*Hkv + ctas][G][D]  unnormalised partial outputs
    int32_t* split_cnt;         // [B*Hkv] partials written so far per split unit (tensor-core engine);
                                // zero between calls: the CTA that completes a unit resets it
    int inline_merge;           // 1: the CTA that completes a split unit merges it; 0: the merge kernel does
    int64_t num_blocks;
    int max_blocks_per_seq;
    int max_seq_len;
    int batch;
    int num_q_heads;
    int num_kv_heads;           // units per sequence: the cache's kv heads << kv_shift
    int kv_shift;               // 1 when g = 16 runs as two units of 8 query heads per cache head
    int window;
    float score_scale;          // sm_scale * k_scale * log2(e)
    float v_scale;
    // Failure-path test hook of the CUDA-core engine (fp8kv_debug_paged_decode_stall):
    // the K producer of CTA 0 never issues stage stall_stage (-1: none), and
    // the ring waits give up after wait_ns (normally kWaitLimitNs).
    uint64_t wait_ns;
    int stall_stage;
};

// Geometry of one head dimension D with ES-byte elements (1: E4M3 codes,
// 2: bf16 for the bf16 twin).  Pages, boxes, stages and per-thread loads are
// in bytes; k-steps and m-tiles in elements.
template <int D, int ES = 1>
struct Geo {
    static constexpr int RB = D * ES;                   // bytes of one token row of one head
    static constexpr int PAGE = kBS * RB;               // bytes of one K (or V) page
    static constexpr int SH = PAGE > kStageHalf ? PAGE : kStageHalf;  // K bytes (and V bytes) per stage
    static constexpr int SB = 2 * SH;                   // bytes per stage
    static constexpr int PPS = SH / PAGE;               // pages per stage: 4, 2, 1
    static constexpr int HALVES = RB >= 128 ? RB / 128 : 1;
    static constexpr int ROWB = RB >= 128 ? 128 : RB;   // bytes per smem row of one TMA box
    static constexpr int BOX = kBS * ROWB;              // bytes of one TMA box
    static constexpr int DBOX = ROWB / ES;              // elements per box row
    static constexpr int KS = D / 16;                   // k-steps of the score MMA
    static constexpr int MT = D / 16;                   // m-tiles of the value MMA
    static constexpr int KW = ROWB / 4;                 // K bytes a thread reads per row per box
    static constexpr int KSH = KW / (4 * ES);           // k-steps per box
    static constexpr int VW = ROWB / 8;                 // V bytes a thread reads per token per box
    static constexpr int VWD = VW / ES;                 // ... in elements
    static constexpr int MTH = VWD / 2;                 // m-tiles per box
    static constexpr int XW = MT * 4 + 4;               // per-lane words exchanged in the warp merge
    static constexpr int STAGES = XW > 40 ? 8 : 12;     // ring slots (a multiple of kNCW)
    static_assert(PPS >= 1 && PPS * PAGE == SH, "stage must hold whole pages");
    static_assert(STAGES % kNCW == 0, "every consumer warp owns whole ring slots");
    static_assert(32 % PPS == 0, "a 32-page block-id batch holds whole stages");
    static_assert(KSH * HALVES == KS && MTH * HALVES == MT, "boxes cover the head dimension");
};

// The CUDA-core consumers also keep the segment's f16 queries ([G][D]) and
// their shifts ([8]) in shared memory.
template <int D, int G>
constexpr size_t smem_bytes() {
    return 1024 + Geo<D>::STAGES * kStageBytes + 2 * Geo<D>::XW * 32 * sizeof(float) +
           4 * Geo<D>::STAGES * sizeof(uint64_t) + (2 * kMaxBatch + 1 + 4 + 32 * kNPW) * sizeof(int32_t) + 16 +
           G * D * sizeof(uint16_t) + 8 * sizeof(int);
}

// Byte offset of (row r, byte o) inside one TMA box written with the 128-byte
// (rows of 128 B) or 64-byte (rows of 64 B) swizzle: the 16-byte chunk index
// is XORed with address bits 7.. of the row start.
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int r, int o) {
    if constexpr (ROWB == 128)
        return r * 128 + ((((o >> 4) ^ (r & 7)) << 4) | (o & 15));
    else
        return r * 64 + ((((o >> 4) ^ ((r >> 1) & 3)) << 4) | (o & 15));
}

// The streaming kernel's own layout of a staged page (its cp.async copies and
// its fragment loads are the only users, so it need not match TMA's): rows of
// 128 bytes as swz<128>; rows of 64 bytes (d = 64) go in pairs into 128-byte
// lines whose eight 16-byte chunks are XOR-permuted per line, the halves
// swapped on every other line.  Measured on the gpt-oss-like step: 0.2 us
// faster than swz<64>.  Its 8-byte value loads still take 4 wavefronts instead
// of 2 (a half-warp reads pieces of four rows, two of them in the same half
// of their lines); a permutation that makes them conflict-free (chunk bits
// 2, 1, 0 flipped by line bits 0, 1, 2) measured 0.14 us slower, so the
// shared-memory wavefronts are not what bounds this kernel.
template <int ROWB>
__device__ __forceinline__ uint32_t sswz(int r, int o) {
    if constexpr (ROWB == 128) {
        return swz<128>(r, o);
    } else {
        const int line = r >> 1;
        const int c = ((r & 1) << 2) | (o >> 4);
        const int g = ((line & 1) << 2) | ((line >> 1) & 3);
        return static_cast<uint32_t>(line * 128 + ((c ^ g) << 4) + (o & 15));
    }
}

__device__ __forceinline__ void report(uint32_t* err, uint32_t code) { atomicCAS(err, 0u, code); }

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kNCW * 32) : "memory"); }

// Named barrier 1 over the first NW warps of the CTA.
template <int NW>
__device__ __forceinline__ void consumer_sync_n() { asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory"); }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Per-sequence geometry: the attended keys of a length-L sequence are
// [first_token, L); they occupy pages first_token/16 .. (L-1)/16.
__device__ __forceinline__ int clamp_len(int L, int max_len) { return L < 0 ? 0 : (L > max_len ? max_len : L); }
__device__ __forceinline__ int first_token(int L, int window) { return (window > 0 && L > window) ? L - window : 0; }
__device__ __forceinline__ int attended_pages(int L, int window) {
    return L > 0 ? (L - 1) / kBS - first_token(L, window) / kBS + 1 : 0;
}

// Block id of page `lane` of a batch; an id outside [0, num_blocks) is
// reported and returned as -1 (its page is then read from block 0 and never
// written).
__device__ __forceinline__ int load_block_id(const int32_t* row, int lane, int count, int64_t num_blocks,
                                             uint32_t* err) {
    int id = 0;
    if (lane < count) {
        id = __ldg(row + lane);
        if (id < 0 || id >= num_blocks) {
            report(err, FP8KV_ERR_INVALID_ARG);
            id = -1;
        }
    }
    return id;
}

// One new K or V row (D bf16 values) held by a warp: lane l owns elements
// [l*D/32, (l+1)*D/32).
template <int D>
struct NewRow {
    uint32_t w[D / 64];
};

template <int D>
__device__ __forceinline__ void load_new_row(NewRow<D>& r, const uint16_t* src_row, int lane) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(src_row + lane * (D / 32));
#pragma unroll
    for (int i = 0; i < D / 64; ++i) r.w[i] = __ldg(p + i);
}

// Quantise-on-append of the warp's row: code = E4M3_satfinite(fp32(x) / scale)
// with one IEEE divide and one RNE conversion (the same arithmetic as the
// quant_append kernel), stored at dst_row.
template <int D, bool E5M2 = false>
__device__ __forceinline__ void store_new_row(const NewRow<D>& r, uint8_t* dst_row, int lane, float scale) {
    uint16_t c[D / 64];
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
        const float e0 = __uint_as_float(r.w[i] << 16), e1 = __uint_as_float(r.w[i] & 0xFFFF0000u);
        c[i] = E5M2 ? f32x2_to_e5m2x2_satfinite(__fdiv_rn(e0, scale), __fdiv_rn(e1, scale))
                    : f32x2_to_e4m3x2_satfinite(__fdiv_rn(e0, scale), __fdiv_rn(e1, scale));
    }
    uint8_t* dst = dst_row + lane * (D / 32);
    if constexpr (D == 64) {
        *reinterpret_cast<uint16_t*>(dst) = c[0];
    } else if constexpr (D == 128) {
        *reinterpret_cast<uint32_t*>(dst) = static_cast<uint32_t>(c[0]) | (static_cast<uint32_t>(c[1]) << 16);
    } else {
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(static_cast<uint32_t>(c[0]) | (static_cast<uint32_t>(c[1]) << 16),
                       static_cast<uint32_t>(c[2]) | (static_cast<uint32_t>(c[3]) << 16));
    }
}

// Query fragments of one (sequence, kv head): the B operand of the score MMA,
// pre-scaled per head by a power of two so the f16 copy is exact (largest |q|
// in [2^14, 2^15)); cs[j] scales the raw score of head 2*tig+j back and into
// log2 units.
// Four FP8 codes (one 32-bit word, code 0 in the low byte) -> two f16x2:
// codes 0,1 in lo and 2,3 in hi; exact for both formats.
template <bool E5M2>
__device__ __forceinline__ void codes4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    if constexpr (E5M2)
        e5m2x4_to_f16x2x2(w, lo, hi);
    else
        e4m3x4_to_f16x2x2(w, lo, hi);
}

// Score multiplier (sm_scale * k_scale * log2 e, multiplied in that order as
// the host does for the per-tensor scale) and V scale of kv head hk.
__device__ __forceinline__ float unit_score_scale(const DecodeArgs& a, int hk) {
    return a.k_scales ? (a.sm_scale * __ldg(a.k_scales + (hk >> a.kv_shift))) * kLog2e : a.score_scale;
}

__device__ __forceinline__ float unit_v_scale(const DecodeArgs& a, int hk) {
    return a.v_scales ? __ldg(a.v_scales + (hk >> a.kv_shift)) : a.v_scale;
}

template <int D, int G>
__device__ __forceinline__ void load_query(const DecodeArgs& a, int b, int hk, int gid, int tig,
                                           uint32_t (&qf)[Geo<D>::KS][2], float (&cs)[2], int h0 = 0) {
    using Gm = Geo<D>;
    uint32_t qw[Gm::HALVES][Gm::KSH][2];
    float qmax = 0.f;
#pragma unroll
    for (int hh = 0; hh < Gm::HALVES; ++hh) {
#pragma unroll
        for (int c = 0; c < Gm::KW / 8; ++c) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h0 + gid < G)
                v = __ldg(reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(b) * a.num_q_heads + hk * G + h0 + gid) * D +
                                                         hh * 128 + tig * Gm::KW) + c);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qw[hh][c * 2 + e / 2][e % 2] = w4[e];
                qmax = fmaxf(qmax, fmaxf(fabsf(bf16_to_f32(w4[e] & 0xFFFF)), fabsf(bf16_to_f32(w4[e] >> 16))));
            }
        }
    }
    qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
    qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
    int shift = 0;
    if (qmax > 0.f) {
        const int e = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFF) - 127;
        shift = max(-100, min(100, 14 - e));
    }
    const float up = __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
#pragma unroll
    for (int hh = 0; hh < Gm::HALVES; ++hh)
#pragma unroll
        for (int kk = 0; kk < Gm::KSH; ++kk)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t w = qw[hh][kk][e];
                qf[hh * Gm::KSH + kk][e] = pack_f16x2(bf16_to_f32(w & 0xFFFF) * up, bf16_to_f32(w >> 16) * up);
            }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int sh = __shfl_sync(0xffffffffu, shift, (2 * tig + j) * 4);
        cs[j] = unit_score_scale(a, hk) * __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
    }
}

// bf16 twin: the g query rows of kv head hk as bf16 B fragments of the score
// MMA (no scaling: the cache is bf16 too), in the k order that matches how a
// thread reads its K bytes: MMA k = 2*tig + e and 2*tig + 8 + e of k-step kk
// of box hh are elements hh*64 + tig*16 + 4*kk + e and ... + 2 + e.
template <int D, int G>
__device__ __forceinline__ void load_query_bf16(const DecodeArgs& a, int b, int hk, int gid, int tig,
                                                uint32_t (&qf)[Geo<D, 2>::KS][2], float (&cs)[2], int h0 = 0) {
    using Gm = Geo<D, 2>;
#pragma unroll
    for (int hh = 0; hh < Gm::HALVES; ++hh) {
        uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
        if (h0 + gid < G) {
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + (static_cast<int64_t>(b) * a.num_q_heads + hk * G + h0 + gid) * D + hh * Gm::DBOX + tig * 16);
            v0 = __ldg(src);
            v1 = __ldg(src + 1);
        }
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int kk = 0; kk < Gm::KSH; ++kk) {
            qf[hh * Gm::KSH + kk][0] = w[2 * kk];
            qf[hh * Gm::KSH + kk][1] = w[2 * kk + 1];
        }
    }
    cs[0] = cs[1] = a.score_scale;
}

// The V bytes one thread feeds to the value MMA from one box of a page:
// token rows 2*tig, 2*tig+1, 2*tig+8, 2*tig+9, VW bytes each at column
// gid*VW.  Rows outside [lo, L) (or a page past the stage's last) read as
// zero codes, so stale NaN codes never meet a zero probability.
template <int D, int ES>
__device__ __forceinline__ void load_v_box(const uint8_t* box, int gid, int tig, int t0, int lo, int L, bool page_ok,
                                           uint32_t (&v)[4][Geo<D, ES>::VW / 4]) {
    using Gm = Geo<D, ES>;
    const bool edge = t0 < lo || t0 + kBS > L;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int row = 2 * tig + (r & 1) + 8 * (r >> 1);
        if (page_ok) {
            if constexpr (Gm::VW == 16) {
                const uint4 x = *reinterpret_cast<const uint4*>(box + sswz<Gm::ROWB>(row, gid * 16));
                v[r][0] = x.x; v[r][1] = x.y; v[r][2] = x.z; v[r][3] = x.w;
            } else {
                const uint2 x = *reinterpret_cast<const uint2*>(box + sswz<Gm::ROWB>(row, gid * 8));
                v[r][0] = x.x; v[r][1] = x.y;
            }
        }
        if (!page_ok || (edge && (t0 + row < lo || t0 + row >= L))) {
#pragma unroll
            for (int ww = 0; ww < Gm::VW / 4; ++ww) v[r][ww] = 0u;
        }
    }
}

// Folds state (m2, l2, o2) into (m, l, o): the FP32 softmax-merge identity.
template <int MT>
__device__ __forceinline__ void combine(float (&m)[2], float (&l)[2], float (&o)[MT][4], const float (&m2)[2],
                                        const float (&l2)[2], const float (&o2)[MT][4]) {
    float f1[2], f2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float M = fmaxf(m[j], m2[j]);
        const float Mu = M == -INFINITY ? 0.f : M;
        f1[j] = fast_exp2(m[j] - Mu);
        f2[j] = fast_exp2(m2[j] - Mu);
        l[j] = l[j] * f1[j] + l2[j] * f2[j];
        m[j] = M;
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] = o[mt][0] * f1[0] + o2[mt][0] * f2[0];
        o[mt][1] = o[mt][1] * f1[1] + o2[mt][1] * f2[1];
        o[mt][2] = o[mt][2] * f1[0] + o2[mt][2] * f2[0];
        o[mt][3] = o[mt][3] * f1[1] + o2[mt][3] * f2[1];
    }
}

template <int MT>
__device__ __forceinline__ void publish(float* x, int lane, const float (&m)[2], const float (&l)[2],
                                        const float (&o)[MT][4]) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) x[(mt * 4 + r) * 32 + lane] = o[mt][r];
    x[(MT * 4 + 0) * 32 + lane] = m[0];
    x[(MT * 4 + 1) * 32 + lane] = m[1];
    x[(MT * 4 + 2) * 32 + lane] = l[0];
    x[(MT * 4 + 3) * 32 + lane] = l[1];
}

template <int MT>
__device__ __forceinline__ void absorb(const float* x, int lane, float (&m)[2], float (&l)[2], float (&o)[MT][4]) {
    float m2[2], l2[2], o2[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) o2[mt][r] = x[(mt * 4 + r) * 32 + lane];
    m2[0] = x[(MT * 4 + 0) * 32 + lane];
    m2[1] = x[(MT * 4 + 1) * 32 + lane];
    l2[0] = x[(MT * 4 + 2) * 32 + lane];
    l2[1] = x[(MT * 4 + 3) * 32 + lane];
    combine<MT>(m, l, o, m2, l2, o2);
}

// ---------------------------------------------------------------- CUDA-core consumers
//
// The same split-context flash-decoding step with both contractions on the
// CUDA cores: every score and every P.V sum is an FP32 fma chain of exact f16
// products (K, V and P are f16-exact: E4M3 codes, the f16-rounded
// probabilities; q is the same power-of-two-scaled f16 copy the tensor-core
// consumers use).  Scores: lane = token (D = 256: two lanes per token, one per
// 128-dim half), q broadcast from shared memory.  P.V: lane = D/32 output
// dims, the stage's probabilities broadcast from shared memory.
template <int D, int G>
struct SimtGeo {
    using Gm = Geo<D>;
    static constexpr int TS = Gm::PPS * kBS;              // tokens per stage: 64, 32, 16
    static constexpr int TPL = TS >= 32 ? TS / 32 : 1;     // tokens per lane in the score pass
    static constexpr int DSPLIT = TS >= 32 ? 1 : 32 / TS;  // lanes sharing one token (D = 256: 2)
    static constexpr int DPL = D / 32;                     // output dims per lane in the value pass
    static constexpr int CH = Gm::ROWB / 16;               // 16-byte chunks per box row
    static constexpr int XW = G * DPL + 2;                 // words per lane in the warp merge
    static constexpr int PSM = TS * G * 2;                 // bytes of one warp's f16 probabilities
    static_assert(XW <= Gm::XW, "merge state fits the exchange buffer");
    static_assert(kNCW * PSM <= 2 * Gm::XW * 32 * 4, "probabilities fit the exchange buffer");
    static_assert(DSPLIT == 1 || DSPLIT == Gm::HALVES, "split lanes cover one 128-dim box each");
};

template <int N>
__device__ __forceinline__ void load_f16s(const uint8_t* p, uint16_t (&h)[N]) {
    if constexpr (N == 1) {
        h[0] = *reinterpret_cast<const uint16_t*>(p);
    } else if constexpr (N == 2) {
        const uint32_t x = *reinterpret_cast<const uint32_t*>(p);
        h[0] = x & 0xFFFF; h[1] = x >> 16;
    } else if constexpr (N == 4) {
        const uint2 x = *reinterpret_cast<const uint2*>(p);
        h[0] = x.x & 0xFFFF; h[1] = x.x >> 16; h[2] = x.y & 0xFFFF; h[3] = x.y >> 16;
    } else {
        const uint4 x = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) { h[2 * i] = w[i] & 0xFFFF; h[2 * i + 1] = w[i] >> 16; }
    }
}

template <int N>
__device__ __forceinline__ void store_f16s(uint8_t* p, const float (&v)[N]) {
    if constexpr (N == 1) {
        const __half h = __float2half_rn(v[0]);
        *reinterpret_cast<uint16_t*>(p) = *reinterpret_cast<const uint16_t*>(&h);
    } else if constexpr (N == 2) {
        *reinterpret_cast<uint32_t*>(p) = pack_f16x2(v[0], v[1]);
    } else if constexpr (N == 4) {
        *reinterpret_cast<uint2*>(p) = make_uint2(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]));
    } else {
        *reinterpret_cast<uint4*>(p) = make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]),
                                                  pack_f16x2(v[4], v[5]), pack_f16x2(v[6], v[7]));
    }
}

template <int G, int DPL>
__device__ __forceinline__ void simt_combine(float (&m)[G], float (&l)[G], float (&o)[G][DPL], const float (&m2)[G],
                                             const float (&l2)[G], const float (&o2)[G][DPL]) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const float M = fmaxf(m[j], m2[j]);
        const float Mu = M == -INFINITY ? 0.f : M;
        const float f1 = fast_exp2(m[j] - Mu), f2 = fast_exp2(m2[j] - Mu);
        l[j] = l[j] * f1 + l2[j] * f2;
        m[j] = M;
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[j][d] = o[j][d] * f1 + o2[j][d] * f2;
    }
}

// Lane-major exchange of a warp's (m, l, o); m and l are warp-uniform and go
// one head per lane.
template <int G, int DPL>
__device__ __forceinline__ void simt_publish(float* x, int lane, const float (&m)[G], const float (&l)[G],
                                             const float (&o)[G][DPL]) {
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int d = 0; d < DPL; ++d) x[(j * DPL + d) * 32 + lane] = o[j][d];
#pragma unroll
    for (int j = 0; j < G; ++j)
        if (lane == j) {
            x[(G * DPL) * 32 + j] = m[j];
            x[(G * DPL + 1) * 32 + j] = l[j];
        }
}

template <int G, int DPL>
__device__ __forceinline__ void simt_absorb(const float* x, int lane, float (&m)[G], float (&l)[G],
                                            float (&o)[G][DPL]) {
    float m2[G], l2[G], o2[G][DPL];
#pragma unroll
    for (int j = 0; j < G; ++j) {
#pragma unroll
        for (int d = 0; d < DPL; ++d) o2[j][d] = x[(j * DPL + d) * 32 + lane];
        m2[j] = x[(G * DPL) * 32 + j];
        l2[j] = x[(G * DPL + 1) * 32 + j];
    }
    simt_combine<G, DPL>(m, l, o, m2, l2, o2);
}

// Byte offset, inside one V page, of the D/32 codes lane `lane` reads from a
// row whose swizzle phase is k (the row's address bits 7-9 for 128-byte rows,
// 7-8 for 64-byte rows), minus the row start.
template <int D>
__device__ __forceinline__ int simt_v_offset(int lane, int k) {
    using Gm = Geo<D>;
    const int o = D == 256 ? (lane % 16) * 8 : lane * (D / 32);   // offset inside the box row
    const int box = D == 256 ? (lane / 16) * Gm::BOX : 0;
    return box + ((((o >> 4) ^ k) << 4) | (o & 15));
}

// One token of the P.V pass: o[j][d] += P[j] * V[d] for the lane's D/32 dims.
template <int D, int G>
__device__ __forceinline__ void simt_pv_row(const uint8_t* vrow, const uint8_t* prow, float (&o)[G][D / 32]) {
    constexpr int DPL = D / 32;
    uint32_t vh[DPL / 2];
    if constexpr (DPL == 2) {
        vh[0] = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(vrow));
    } else if constexpr (DPL == 4) {
        e4m3x4_to_f16x2x2(*reinterpret_cast<const uint32_t*>(vrow), vh[0], vh[1]);
    } else {
        const uint2 c8 = *reinterpret_cast<const uint2*>(vrow);
        e4m3x4_to_f16x2x2(c8.x, vh[0], vh[1]);
        e4m3x4_to_f16x2x2(c8.y, vh[2], vh[3]);
    }
    uint16_t ph[G];
    load_f16s<G>(prow, ph);
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int k = 0; k < DPL / 2; ++k) fma_f16x2_f16_f32(o[j][2 * k], o[j][2 * k + 1], vh[k], ph[j]);
}

// Shared state of one CTA that the consumer warps read.
struct CtaView {
    uint8_t* ring;
    float* xbuf;
    uint64_t* full_bar;   // [S] K half of a slot landed; V: full_bar + S
    uint64_t* empty_bar;  // [S] K half of a slot consumed; V: empty_bar + S
    const int32_t* pre;
    const int32_t* lens;
    volatile int* flag;
    uint16_t* qsm;   // [G][D] f16 scaled queries of the current segment
    int* qsh;        // [G] their power-of-two shifts
    int64_t s, e;
    Partition part;
    int c;
};

template <int D, int G>
__device__ __forceinline__ void simt_consumers(const DecodeArgs& a, const CtaView& v, int warp, int lane) {
    using Gm = Geo<D>;
    using Sg = SimtGeo<D, G>;
    constexpr int S = Gm::STAGES;
    constexpr int DPL = Sg::DPL;
    const int B = a.batch, Hkv = a.num_kv_heads;
    uint8_t* psm = reinterpret_cast<uint8_t*>(v.xbuf) + warp * Sg::PSM;  // this warp's probabilities
    float m[G], l[G], o[G][DPL], cs[G];
    constexpr int NK = Gm::ROWB == 128 ? 8 : 4;  // swizzle phases of a box row
    int vo[NK];
#pragma unroll
    for (int k = 0; k < NK; ++k) vo[k] = simt_v_offset<D>(lane, k);
    int st_base = 0;
    Walker w;
    walk_start(w, v.pre, B, Hkv, v.s);
    while (true) {
        const int64_t seg_end = min(v.e, w.base + w.n);
        const int lp0 = static_cast<int>(w.g - w.base);
        const int np_seg = static_cast<int>(seg_end - w.g);
        const int nst = (np_seg + Gm::PPS - 1) / Gm::PPS;
        const int L = v.lens[w.b];
        const int lo = first_token(L, a.window);
        const int pg_first = lo / kBS + lp0;

        // ---- the segment's queries -> scaled f16 in shared memory (one warp per head)
        for (int j = warp; j < G; j += kNCW) {
            const uint16_t* src = a.q + (static_cast<int64_t>(w.b) * a.num_q_heads + w.hk * G + j) * D + lane * DPL;
            float x[DPL];
            if constexpr (DPL == 2) {
                const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(src));
                x[0] = bf16_to_f32(u & 0xFFFF); x[1] = bf16_to_f32(u >> 16);
            } else if constexpr (DPL == 4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
                x[0] = bf16_to_f32(u.x & 0xFFFF); x[1] = bf16_to_f32(u.x >> 16);
                x[2] = bf16_to_f32(u.y & 0xFFFF); x[3] = bf16_to_f32(u.y >> 16);
            } else {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
                const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) { x[2 * i] = bf16_to_f32(ww[i] & 0xFFFF); x[2 * i + 1] = bf16_to_f32(ww[i] >> 16); }
            }
            float qmax = 0.f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) qmax = fmaxf(qmax, fabsf(x[d]));
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
            int shift = 0;
            if (qmax > 0.f) {
                const int ex = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFF) - 127;
                shift = max(-100, min(100, 14 - ex));
            }
            const float up = __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
#pragma unroll
            for (int d = 0; d < DPL; ++d) x[d] *= up;
            store_f16s<DPL>(reinterpret_cast<uint8_t*>(v.qsm + j * D + lane * DPL), x);
            if (lane == 0) v.qsh[j] = shift;
        }
        if (seg_end < v.e) {  // warm L2 with the next segment's queries
            Walker nw = w;
            walk_next(nw, v.pre, Hkv);
            if (lane < G * D * 2 / 128)
                prefetch_l2(reinterpret_cast<const uint8_t*>(a.q + (static_cast<int64_t>(nw.b) * a.num_q_heads + nw.hk * G) * D) +
                            lane * 128);
        }
        consumer_sync();
#pragma unroll
        for (int j = 0; j < G; ++j) {
            cs[j] = unit_score_scale(a, w.hk) * __uint_as_float(static_cast<uint32_t>(127 - v.qsh[j]) << 23);
            m[j] = -INFINITY;
            l[j] = 0.f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[j][d] = 0.f;
        }

        for (int i = (warp - st_base % kNCW + kNCW) % kNCW; i < nst; i += kNCW) {
            const int st = st_base + i;
            const int slot = st % S;
            if (v.flag[1]) break;
            if (!mbar_wait_bounded(&v.full_bar[slot], (st / S) & 1, a.wait_ns)) {
                report(a.err, FP8KV_ERR_TIMEOUT);
                v.flag[1] = 1;
                break;
            }
            const int p0 = i * Gm::PPS;
            const int np = min(Gm::PPS, np_seg - p0);
            const uint8_t* kst = v.ring + slot * kStageBytes;
            const uint8_t* vst = kst + kStageHalf;
            const int tok_base = (pg_first + p0) * kBS;

            // ---- scores: s[t][j] = sum_d K[t][d] q_j[d]
            float sc[Sg::TPL][G];
            {
                const int hb = Sg::DSPLIT == 1 ? 0 : lane / Sg::TS;
                float acc[Sg::TPL][G][2];
#pragma unroll
                for (int t = 0; t < Sg::TPL; ++t)
#pragma unroll
                    for (int j = 0; j < G; ++j) acc[t][j][0] = acc[t][j][1] = 0.f;
#pragma unroll
                for (int cc = 0; cc < Sg::CH; ++cc) {
                    uint4 x[Sg::TPL];
#pragma unroll
                    for (int t = 0; t < Sg::TPL; ++t) {
                        const int tl = Sg::DSPLIT == 1 ? t * 32 + lane : lane % Sg::TS;
                        const uint8_t* box = kst + (tl / kBS) * Gm::PAGE + hb * Gm::BOX;
                        x[t] = *reinterpret_cast<const uint4*>(box + swz<Gm::ROWB>(tl % kBS, 16 * cc));
                    }
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        const uint16_t* qj = v.qsm + j * D + hb * 128 + 16 * cc;
                        const uint4 qa = *reinterpret_cast<const uint4*>(qj);
                        const uint4 qb = *reinterpret_cast<const uint4*>(qj + 8);
#pragma unroll
                        for (int t = 0; t < Sg::TPL; ++t) {
                            uint32_t k0, k1, k2, k3, k4, k5, k6, k7;
                            e4m3x4_to_f16x2x2(x[t].x, k0, k1);
                            e4m3x4_to_f16x2x2(x[t].y, k2, k3);
                            e4m3x4_to_f16x2x2(x[t].z, k4, k5);
                            e4m3x4_to_f16x2x2(x[t].w, k6, k7);
                            fma_f16x2_f32(acc[t][j][0], acc[t][j][1], k0, qa.x);
                            fma_f16x2_f32(acc[t][j][0], acc[t][j][1], k1, qa.y);
                            fma_f16x2_f32(acc[t][j][0], acc[t][j][1], k2, qa.z);
                            fma_f16x2_f32(acc[t][j][0], acc[t][j][1], k3, qa.w);
                            fma_f16x2_f32(acc[t][j][0], acc[t][j][1], k4, qb.x);
                            fma_f16x2_f32(acc[t][j][0], acc[t][j][1], k5, qb.y);
                            fma_f16x2_f32(acc[t][j][0], acc[t][j][1], k6, qb.z);
                            fma_f16x2_f32(acc[t][j][0], acc[t][j][1], k7, qb.w);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < Sg::TPL; ++t)
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        float sv = acc[t][j][0] + acc[t][j][1];
                        if constexpr (Sg::DSPLIT == 2) sv += __shfl_xor_sync(0xffffffffu, sv, 16);
                        sc[t][j] = sv;
                    }
            }

            __syncwarp();
            if (lane == 0) mbar_arrive(&v.empty_bar[slot]);  // the K half is free again

            // ---- mask, scale to log2 units, stage maximum
            float mx[G];
#pragma unroll
            for (int j = 0; j < G; ++j) mx[j] = -INFINITY;
#pragma unroll
            for (int t = 0; t < Sg::TPL; ++t) {
                const int tl = Sg::DSPLIT == 1 ? t * 32 + lane : lane % Sg::TS;
                const int tok = tok_base + tl;
                const bool valid = tl < np * kBS && tok >= lo && tok < L;
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    sc[t][j] = valid ? sc[t][j] * cs[j] : -INFINITY;
                    mx[j] = fmaxf(mx[j], sc[t][j]);
                }
            }
            float alpha[G], muse[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], off));
                const float mn = fmaxf(m[j], mx[j]);
                muse[j] = mn == -INFINITY ? 0.f : mn;
                alpha[j] = fast_exp2(m[j] - muse[j]);
                m[j] = mn;
            }

            // ---- probabilities -> f16 in this warp's shared slice; each lane's
            // share of l moves to the new maximum first
#pragma unroll
            for (int j = 0; j < G; ++j) l[j] *= alpha[j];
            __syncwarp();  // the previous stage's readers are done with the slice
#pragma unroll
            for (int t = 0; t < Sg::TPL; ++t) {
                const int tl = Sg::DSPLIT == 1 ? t * 32 + lane : lane % Sg::TS;
                float pr[G];
#pragma unroll
                for (int j = 0; j < G; ++j) pr[j] = fast_exp2(sc[t][j] - muse[j]);
                if (Sg::DSPLIT == 1 || lane < Sg::TS) {
#pragma unroll
                    for (int j = 0; j < G; ++j) l[j] += pr[j];
                    store_f16s<G>(psm + tl * G * 2, pr);
                }
            }
            __syncwarp();

            // ---- P.V: o[j][d] += sum_t P[t][j] V[t][d] over the stage's valid tokens
            if (!mbar_wait_bounded(&v.full_bar[S + slot], (st / S) & 1, a.wait_ns)) {
                report(a.err, FP8KV_ERR_TIMEOUT);
                v.flag[1] = 1;
                break;
            }
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[j][d] *= alpha[j];
            const int t_lo = max(lo - tok_base, 0);
            const int t_hi = min(L - tok_base, np * kBS);
            if (t_lo == 0 && t_hi == np * kBS) {
                // every token of the stage attended: fully unrolled rows with
                // the swizzled lane offsets taken from vo[]
#pragma unroll
                for (int p = 0; p < Gm::PPS; ++p) {
                    if (p < np) {
#pragma unroll
                        for (int r = 0; r < kBS; ++r)
                            simt_pv_row<D, G>(vst + p * Gm::PAGE + r * Gm::ROWB + vo[Gm::ROWB == 128 ? (r & 7) : ((r >> 1) & 3)],
                                              psm + (p * kBS + r) * G * 2, o);
                    }
                }
            } else {
#pragma unroll 2
                for (int t = t_lo; t < t_hi; ++t) {
                    const int r = t % kBS;
                    simt_pv_row<D, G>(vst + (t / kBS) * Gm::PAGE + r * Gm::ROWB +
                                          simt_v_offset<D>(lane, Gm::ROWB == 128 ? (r & 7) : ((r >> 1) & 3)),
                                      psm + t * G * 2, o);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&v.empty_bar[S + slot]);
        }
        st_base += nst;

#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) l[j] += __shfl_xor_sync(0xffffffffu, l[j], off);

        // ---- merge the four warps' states into warp 0 (the exchange buffer
        // also holds the probability slices: every warp leaves its stages first)
        consumer_sync();
        if (warp >= 2) simt_publish<G, DPL>(v.xbuf + (warp - 2) * Sg::XW * 32, lane, m, l, o);
        consumer_sync();
        if (warp < 2) simt_absorb<G, DPL>(v.xbuf + warp * Sg::XW * 32, lane, m, l, o);
        consumer_sync();
        if (warp == 1) simt_publish<G, DPL>(v.xbuf, lane, m, l, o);
        consumer_sync();
        if (warp == 0) simt_absorb<G, DPL>(v.xbuf, lane, m, l, o);

        // ---- emit (as the tensor-core consumers do)
        const int u = w.b * Hkv + w.hk;
        const int c_first = cta_of(v.part, w.base);
        const int c_last = cta_of(v.part, w.base + w.n - 1);
        const int k_u = c_last - c_first + 1;
        if (warp == 0) {
            if (k_u == 1) {
                uint16_t* out_u = a.out + (static_cast<int64_t>(w.b) * a.num_q_heads + w.hk * G) * D + lane * DPL;
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float sc_out = l[j] > 0.f ? unit_v_scale(a, w.hk) / l[j] : 0.f;
                    uint32_t pk[DPL / 2];
#pragma unroll
                    for (int k = 0; k < DPL / 2; ++k)
                        pk[k] = static_cast<uint32_t>(f32_to_bf16(o[j][2 * k] * sc_out)) |
                                (static_cast<uint32_t>(f32_to_bf16(o[j][2 * k + 1] * sc_out)) << 16);
                    if constexpr (DPL == 2) *reinterpret_cast<uint32_t*>(out_u + j * D) = pk[0];
                    else if constexpr (DPL == 4) *reinterpret_cast<uint2*>(out_u + j * D) = make_uint2(pk[0], pk[1]);
                    else *reinterpret_cast<uint4*>(out_u + j * D) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            } else {
                const int64_t slot_idx = static_cast<int64_t>(u) + v.c;
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    float* po = a.part_o + (slot_idx * G + j) * D + lane * DPL;
#pragma unroll
                    for (int d = 0; d < DPL; d += 2) *reinterpret_cast<float2*>(po + d) = make_float2(o[j][d], o[j][d + 1]);
                    if (lane == 0) a.part_ml[slot_idx * kMaxG + j] = make_float2(m[j], l[j]);
                }
            }
        }
        consumer_sync();  // warp 0 is done with the exchange buffer
        if (seg_end >= v.e) break;
        walk_next(w, v.pre, Hkv);
    }
}

// The CUDA-core engine: TMA producers, an mbarrier-guarded ring, CUDA-core
// consumers (simt_consumers).  E4M3 cache, per-tensor or per-head scales.
template <int D, int G>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeArgs a) {
    using Gm = Geo<D>;
    constexpr int S = Gm::STAGES;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned ring (the swizzle pattern is a function of address
    // bits 4..9); offsetting the shared array keeps the address space known.
    uint8_t* ring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* xbuf = reinterpret_cast<float*>(ring + S * kStageBytes);  // [2][XW][32]
    // Each ring slot holds a K half and a V half with a barrier pair each:
    // full_bar[s] / full_bar[S + s] complete when the K / V copies land,
    // empty_bar[s] / empty_bar[S + s] when the consumer is done with them, so
    // the K half returns to its producer as soon as the scores are computed.
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(xbuf + 2 * Gm::XW * 32);  // [2][S]
    uint64_t* empty_bar = full_bar + 2 * S;                                     // [2][S]
    int32_t* pre = reinterpret_cast<int32_t*>(empty_bar + 2 * S);    // [kMaxBatch + 1] page prefix
    int32_t* lens = pre + kMaxBatch + 1;                             // [kMaxBatch] clamped lengths
    volatile int* flag = reinterpret_cast<volatile int*>(lens + kMaxBatch);  // [1] abort
    int32_t* ids = lens + kMaxBatch + 4;                             // [kNPW][32] block ids per producer
    uint16_t* qsm = reinterpret_cast<uint16_t*>(                     // CUDA-core consumers: [G][D] f16 q
        ring + ((reinterpret_cast<uint8_t*>(ids + 32 * kNPW) - ring + 15) & ~static_cast<intptr_t>(15)));
    int* qsh = reinterpret_cast<int*>(qsm + G * D);                  // [8] q shifts

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Set-up that reads no input: the ring barriers (shared memory) and the
    // tensor-map descriptors (kernel parameters).
    if (tid == 0) {
        for (int st0 = 0; st0 < 2 * S; ++st0) {
            mbar_init(&full_bar[st0], 1);
            mbar_init(&empty_bar[st0], 1);
        }
        flag[1] = 0;
        fence_barrier_init();
    }
    if (warp == kNCW && lane == 0) prefetch_tmap(&tmK);
    if (warp == kNCW + 1 && lane == 0) prefetch_tmap(&tmV);
    // This grid may have started before the previous one on the stream
    // finished (programmatic launch): wait for it before reading any input,
    // since that grid may have produced them (q, lengths, tables, the cache).
    griddep_wait();
    // The merge kernel that follows may start now: it reads the lengths (final,
    // since every CTA of this grid is past its wait) and waits for this grid's
    // completion before reading anything this grid writes.
    griddep_launch_dependents();
    const int B = a.batch, Hkv = a.num_kv_heads, C = gridDim.x, c = blockIdx.x;

    // ---- attended pages per sequence and their exclusive prefix; the error
    // word is read alongside (a CTA of an earlier call that gave up a wait
    // fails every later call until the workspace is re-initialised)
    if (warp == 0) {
        uint32_t prev_err = 0;
        if (lane == 0) prev_err = *reinterpret_cast<volatile uint32_t*>(a.err);
        int run = 0;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int b = b0 + lane;
            int n = 0;
            if (b < B) {
                const int Lraw = __ldg(a.seq_lens + b);
                if (Lraw < 0 || Lraw > a.max_seq_len) report(a.err, FP8KV_ERR_INVALID_ARG);
                lens[b] = clamp_len(Lraw, a.max_seq_len);
                n = attended_pages(lens[b], a.window);
            }
            int x = n;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            if (b < B) pre[b] = run + x - n;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) {
            pre[B] = run;
            flag[2] = prev_err == FP8KV_ERR_TIMEOUT;
        }
    }
    __syncthreads();
    if (flag[2]) return;

    const int64_t P = static_cast<int64_t>(Hkv) * pre[B];
    // sequences with nothing to attend (length 0) produce zeros
    for (int b = c; b < B; b += C) {
        if (pre[b + 1] == pre[b]) {
            uint16_t* ob = a.out + static_cast<int64_t>(b) * a.num_q_heads * D;
            for (int i = tid; i < a.num_q_heads * D; i += kThreads) ob[i] = 0;
        }
    }
    const int Ce = static_cast<int>(P < C ? P : C);  // CTAs with work: every one gets >= 1 page
    if (c >= Ce) return;
    const Partition part = make_partition(P, Ce);
    const int64_t s = range_start(part, c);
    const int64_t e = range_start(part, c + 1);

    if (warp >= kNCW) {
        // ------------------------------------------------------------ producers
        // Two producer warps walk the same pages: the first issues the K
        // copies (and posts each stage's byte count), the second the V copies,
        // so their issue latencies overlap.  In each, lane 0 alone issues;
        // once per 32 pages the warp hands it the next 32 block ids through
        // shared memory and loads the 32 after those while lane 0 works.
        const int pw = warp - kNCW;
        const CUtensorMap* tm = pw == 0 ? &tmK : &tmV;
        int32_t* my_ids = ids + pw * 32;
        const uint64_t pol = l2_policy_evict_first();
        int st = 0;
        bool ok = true;
        // Batches of up to 32 pages never straddle a segment; the ids of the
        // batch after the current one (in the same or the next segment) are
        // loaded while lane 0 issues the current one.
        //
        // With a row to append (a decode step), the producer that owns a
        // unit's last page first writes that sequence's newest K (or V) row
        // into the page, orders the write before its own copies
        // (fence.proxy.async), and only then issues the page.
        const bool appending = a.k_new != nullptr;
        const uint16_t* new_rows = pw == 0 ? a.k_new : a.v_new;
        uint8_t* cache = pw == 0 ? a.k_cache : a.v_cache;
        const float scale_raw = pw == 0 ? a.k_scale_raw : a.v_scale_raw;  // per-tensor; per head below
        const float* head_scales = pw == 0 ? a.k_scales : a.v_scales;
        Walker w;
        walk_start(w, pre, B, Hkv, s);
        auto seg_pages = [&](const Walker& x) { return static_cast<int>(min(e, x.base + x.n) - x.g); };
        auto seg_row = [&](const Walker& x) {
            return a.block_tables + static_cast<int64_t>(x.b) * a.max_blocks_per_seq +
                   first_token(lens[x.b], a.window) / kBS + (x.g - x.base);
        };
        auto seg_reaches_end = [&](const Walker& x) { return min(e, x.base + x.n) == x.base + x.n; };
        int np_seg = seg_pages(w);
        const int32_t* row = seg_row(w);
        int p0 = 0;
        int nxt = load_block_id(row, lane, np_seg, a.num_blocks, a.err);
        int seg_b = w.b, seg_hk = w.hk;
        bool seg_last = appending && seg_reaches_end(w);
        NewRow<D> nrow;
        // the cache (and the new rows) have Hkv >> kv_shift heads; unit hk reads head hk >> kv_shift
        const int kvs = a.kv_shift, Hc = Hkv >> kvs;
        if (seg_last) load_new_row<D>(nrow, new_rows + (static_cast<int64_t>(w.b) * Hc + (w.hk >> kvs)) * D, lane);
        bool more = true;
        while (ok && more) {
            const int cur = nxt;
            const int hk = seg_hk;
            const int nb = min(32, np_seg - p0);
            const bool batch_has_last = seg_last && p0 + nb == np_seg;
            const int batch_b = seg_b;
            const NewRow<D> batch_row = nrow;
            __syncwarp();  // lane 0 is done with the previous batch
            my_ids[lane] = cur;
            p0 += 32;
            if (p0 >= np_seg) {
                if (min(e, w.base + w.n) >= e) {
                    more = false;
                } else {
                    walk_next(w, pre, Hkv);
                    np_seg = seg_pages(w);
                    row = seg_row(w);
                    p0 = 0;
                    seg_b = w.b;
                    seg_hk = w.hk;
                    seg_last = appending && seg_reaches_end(w);
                    if (seg_last)
                        load_new_row<D>(nrow, new_rows + (static_cast<int64_t>(w.b) * Hc + (w.hk >> kvs)) * D, lane);
                }
            }
            nxt = more ? load_block_id(row + p0, lane, np_seg - p0, a.num_blocks, a.err) : 0;
            __syncwarp();
            if (batch_has_last) {
                const int id = my_ids[nb - 1];
                if (id >= 0) {
                    const int L = lens[batch_b];
                    // with two units per cache head both write the same bytes: identical values
                    uint8_t* dst_row = cache + ((static_cast<int64_t>(id) * Hc + (hk >> kvs)) * kBS + (L - 1) % kBS) * D;
                    store_new_row<D>(batch_row, dst_row, lane,
                                           head_scales ? __ldg(head_scales + (hk >> kvs)) : scale_raw);
                    fence_proxy_async_global();
                }
                __syncwarp();
            }
            if (lane == 0) {
                for (int q = 0; q < nb && ok; q += Gm::PPS) {
                    const int np = min(Gm::PPS, nb - q);
                    const int slot = st % S;
                    if (flag[1] || (st >= S && !mbar_wait_bounded(&empty_bar[pw * S + slot], ((st / S) & 1) ^ 1,
                                                                   a.wait_ns))) {
                        report(a.err, FP8KV_ERR_TIMEOUT);
                        flag[1] = 1;
                        ok = false;
                        break;
                    }
                    if (c == 0 && pw == 0 && st == a.stall_stage) {  // test hook: this stage never arrives
                        ++st;
                        continue;
                    }
                    // this producer's half of the stage (K or V)
                    mbar_arrive_expect_tx(&full_bar[pw * S + slot], static_cast<uint32_t>(np * Gm::PAGE));
                    uint8_t* dst = ring + slot * kStageBytes + pw * kStageHalf;
                    for (int p = 0; p < np; ++p) {
                        const int id = max(my_ids[q + p], 0);
#pragma unroll
                        for (int h = 0; h < Gm::HALVES; ++h)
                            tma_load_4d(dst + p * Gm::PAGE + h * Gm::BOX, tm, &full_bar[pw * S + slot], h * 128, 0,
                                        hk >> kvs, id, pol);
                    }
                    ++st;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        // The CTA must not exit with copies in flight, and consumers that gave
        // up a wait no longer wait for them: before leaving, the producer waits
        // (with the normal limit) for the last ring's worth of stages it
        // issued.  Normally those have landed or are about to.
        if (lane == 0) {
            for (int t = st > S ? st - S : 0; t < st; ++t)
                if (!(c == 0 && pw == 0 && t == a.stall_stage))  // a stage the test hook skipped has no copies
                    mbar_wait_bounded(&full_bar[pw * S + t % S], (t / S) & 1, kWaitLimitNs);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const CtaView v{ring, xbuf, full_bar, empty_bar, pre, lens, flag, qsm, qsh, s, e, part, c};
    simt_consumers<D, G>(a, v, warp, lane);
}

// ---------------------------------------------------------------- streaming decode (per-warp rings)
//
// The same split-context flash-decoding step with a different copy pipeline:
// there are no producer warps.  Every consumer warp streams its own pages
// with 16-byte cp.async copies into a private ring of R stages in shared
// memory, R-1 stages ahead of the stage it computes.  Each warp takes one
// contiguous share of every segment of its CTA (the segment's pages cut into
// NW equal runs), so its block ids are consecutive entries of one block-table
// row; they are read 32 at a time, one window ahead.  Copies complete by
// themselves (no barrier handshake, no bounded waits); the warps of a CTA
// meet only at segment ends, to merge their partial softmax states.

// One stage: the np (<= PPS) pages of K at kst and V at vst, holding tokens
// [tok_base, tok_base + 16*np) of a sequence attended on [lo, L), folded into
// the running state (m, l, o) of the warp.  The query heads sit on the MMA's
// n side, 8 per n-tile: NT = 2 n-tiles carry g = 16 heads, and the converted
// K and V fragments feed both tiles' MMAs, so each page is read once.
template <int D, int ES, bool E5M2, int NT>
__device__ __forceinline__ void tc_stage(const uint8_t* kst, const uint8_t* vst, int np, int tok_base, int lo, int L,
                                         int gid, int tig, const uint32_t (&qf)[NT][Geo<D, ES>::KS][2],
                                         const float (&cs)[NT][2], float (&m)[NT][2], float (&l)[NT][2],
                                         float (&o)[NT][Geo<D, ES>::MT][4]) {
    using Gm = Geo<D, ES>;
    constexpr bool kEarlyV = Gm::MT == 8 && NT == 1;
    // ---- (d = 128) the stage's V fragments into registers first, so their
    // shared-memory latency overlaps the score math
    uint32_t vr[kEarlyV ? Gm::PPS : 1][kEarlyV ? Gm::HALVES : 1][4][Gm::VW / 4];
    if constexpr (kEarlyV) {
#pragma unroll
        for (int p = 0; p < Gm::PPS; ++p)
#pragma unroll
            for (int hh = 0; hh < Gm::HALVES; ++hh)
                load_v_box<D, ES>(vst + p * Gm::PAGE + hh * Gm::BOX, gid, tig, tok_base + p * kBS, lo, L, p < np,
                                  vr[p][hh]);
    }

    // ---- scores S^T[token][head] = K Q^T, two accumulator chains per page
    // and n-tile (even and odd k-steps) to halve the dependent MMA latency
    float sc[Gm::PPS][NT][4];
#pragma unroll
    for (int p = 0; p < Gm::PPS; ++p) {
        float s1[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int r = 0; r < 4; ++r) sc[p][t][r] = s1[t][r] = 0.f;
        if (p < np) {
#pragma unroll
            for (int hh = 0; hh < Gm::HALVES; ++hh) {
                const uint8_t* box = kst + p * Gm::PAGE + hh * Gm::BOX;
                uint32_t w0[Gm::KW / 4], w1[Gm::KW / 4];
#pragma unroll
                for (int cc = 0; cc < Gm::KW / 16; ++cc) {
                    const uint4 x = *reinterpret_cast<const uint4*>(box + sswz<Gm::ROWB>(gid, tig * Gm::KW + 16 * cc));
                    const uint4 y = *reinterpret_cast<const uint4*>(box + sswz<Gm::ROWB>(gid + 8, tig * Gm::KW + 16 * cc));
                    w0[4 * cc + 0] = x.x; w0[4 * cc + 1] = x.y; w0[4 * cc + 2] = x.z; w0[4 * cc + 3] = x.w;
                    w1[4 * cc + 0] = y.x; w1[4 * cc + 1] = y.y; w1[4 * cc + 2] = y.z; w1[4 * cc + 3] = y.w;
                }
#pragma unroll
                for (int kk = 0; kk < Gm::KSH; ++kk) {
                    const int ks = hh * Gm::KSH + kk;
                    uint32_t af[4];
                    if constexpr (ES == 1) {
                        codes4_to_f16x2x2<E5M2>(w0[kk], af[0], af[2]);
                        codes4_to_f16x2x2<E5M2>(w1[kk], af[1], af[3]);
                    } else {
                        af[0] = w0[2 * kk];
                        af[2] = w0[2 * kk + 1];
                        af[1] = w1[2 * kk];
                        af[3] = w1[2 * kk + 1];
                    }
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        float(&acc)[4] = (ks & 1) ? s1[t] : sc[p][t];
                        if constexpr (ES == 1)
                            mma_16816(acc, af, qf[t][ks][0], qf[t][ks][1], acc);
                        else
                            mma_16816_bf16(acc, af, qf[t][ks][0], qf[t][ks][1], acc);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int r = 0; r < 4; ++r) sc[p][t][r] += s1[t][r];
    }

    // ---- mask, scale to log2 units, stage maximum
    float mx[NT][2];
    const bool interior = tok_base >= lo && tok_base + np * kBS <= L && np == Gm::PPS;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        mx[t][0] = mx[t][1] = -INFINITY;
#pragma unroll
        for (int p = 0; p < Gm::PPS; ++p)
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int tok = tok_base + p * kBS + gid + 8 * e2;
                const bool valid = interior || ((p < np) && tok >= lo && tok < L);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float x = valid ? sc[p][t][2 * e2 + j] * cs[t][j] : -INFINITY;
                    sc[p][t][2 * e2 + j] = x;
                    mx[t][j] = fmaxf(mx[t][j], x);
                }
            }
    }
    float alpha[NT][2], muse[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mx[t][j] = fmaxf(mx[t][j], __shfl_xor_sync(0xffffffffu, mx[t][j], 4));
            mx[t][j] = fmaxf(mx[t][j], __shfl_xor_sync(0xffffffffu, mx[t][j], 8));
            mx[t][j] = fmaxf(mx[t][j], __shfl_xor_sync(0xffffffffu, mx[t][j], 16));
            const float mn = fmaxf(m[t][j], mx[t][j]);
            muse[t][j] = mn == -INFINITY ? 0.f : mn;
            alpha[t][j] = fast_exp2(m[t][j] - muse[t][j]);
            m[t][j] = mn;
        }

    // ---- probabilities -> f16 (bf16 for the bf16 twin) B fragments of the value MMA
    uint32_t pb[Gm::PPS][NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        float lsum[2] = {0.f, 0.f};
#pragma unroll
        for (int p = 0; p < Gm::PPS; ++p) {
            const float p00 = fast_exp2(sc[p][t][0] - muse[t][0]);
            const float p01 = fast_exp2(sc[p][t][1] - muse[t][1]);
            const float p10 = fast_exp2(sc[p][t][2] - muse[t][0]);
            const float p11 = fast_exp2(sc[p][t][3] - muse[t][1]);
            lsum[0] += p00 + p10;
            lsum[1] += p01 + p11;
            if constexpr (ES == 1) {
                pb[p][t][0] = movmatrix_trans(pack_f16x2(p00, p01));
                pb[p][t][1] = movmatrix_trans(pack_f16x2(p10, p11));
            } else {
                pb[p][t][0] = movmatrix_trans(pack_bf16x2(p00, p01));
                pb[p][t][1] = movmatrix_trans(pack_bf16x2(p10, p11));
            }
        }
        l[t][0] = l[t][0] * alpha[t][0] + lsum[0];
        l[t][1] = l[t][1] * alpha[t][1] + lsum[1];
    }

    // ---- P.V tile of this stage: O^T[dim][head] = V^T P^T
    float ot[NT][Gm::MT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) ot[t][mt][0] = ot[t][mt][1] = ot[t][mt][2] = ot[t][mt][3] = 0.f;
#pragma unroll
    for (int p = 0; p < Gm::PPS; ++p) {
        if (p < np) {
#pragma unroll
            for (int hh = 0; hh < Gm::HALVES; ++hh) {
                uint32_t v[4][Gm::VW / 4];
                if constexpr (kEarlyV) {
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int ww = 0; ww < Gm::VW / 4; ++ww) v[r][ww] = vr[p][hh][r][ww];
                } else {
                    load_v_box<D, ES>(vst + p * Gm::PAGE + hh * Gm::BOX, gid, tig, tok_base + p * kBS, lo, L, true, v);
                }
#pragma unroll
                for (int mtl = 0; mtl < Gm::MTH; ++mtl) {
                    uint32_t af[4];
                    if constexpr (ES == 1) {
                        const uint32_t sel = (mtl & 1) ? 0x7362u : 0x5140u;
                        const uint32_t x01 = byte_perm(v[0][mtl >> 1], v[1][mtl >> 1], sel);
                        const uint32_t x23 = byte_perm(v[2][mtl >> 1], v[3][mtl >> 1], sel);
                        codes4_to_f16x2x2<E5M2>(x01, af[0], af[1]);
                        codes4_to_f16x2x2<E5M2>(x23, af[2], af[3]);
                    } else {
                        af[0] = byte_perm(v[0][mtl], v[1][mtl], 0x5410u);
                        af[1] = byte_perm(v[0][mtl], v[1][mtl], 0x7632u);
                        af[2] = byte_perm(v[2][mtl], v[3][mtl], 0x5410u);
                        af[3] = byte_perm(v[2][mtl], v[3][mtl], 0x7632u);
                    }
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        float(&acc)[4] = ot[t][hh * Gm::MTH + mtl];
                        if constexpr (ES == 1)
                            mma_16816(acc, af, pb[p][t][0], pb[p][t][1], acc);
                        else
                            mma_16816_bf16(acc, af, pb[p][t][0], pb[p][t][1], acc);
                    }
                }
            }
        }
    }

    // ---- fold the tile into the FP32 accumulators
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
            o[t][mt][0] = fmaf(o[t][mt][0], alpha[t][0], ot[t][mt][0]);
            o[t][mt][1] = fmaf(o[t][mt][1], alpha[t][1], ot[t][mt][1]);
            o[t][mt][2] = fmaf(o[t][mt][2], alpha[t][0], ot[t][mt][2]);
            o[t][mt][3] = fmaf(o[t][mt][3], alpha[t][1], ot[t][mt][3]);
        }
}

// Combines the k_u partials of unit u (slots u + c_first ...) into its output
// rows, with all NTHR threads of the CTA.  The partials come from other CTAs
// of the grid, so they are read through L2: the unit's slots are contiguous,
// and chunks of them are copied into `stage` (shared memory the streaming no
// longer needs) by 16-byte cp.async copies issued all at once; thread i then
// folds (query head, 4 dims) items i, i + NTHR, ... over the chunk (max, then
// rescale and accumulate).
template <int D, int G, int NTHR, int STAGE_BYTES>
__device__ __forceinline__ void merge_unit(const DecodeArgs& a, int u, int c_first, int k_u, int tid,
                                           uint8_t* stage) {
    constexpr int NG = D / 4;                      // float4 groups per head
    constexpr int ITEMS = G * NG;
    constexpr int IT = (ITEMS + NTHR - 1) / NTHR;  // items per thread
    constexpr int OB = G * D * 4;                  // bytes of one partial's outputs
    constexpr int MB = kMaxG * 8;                  // bytes of one partial's (max, sum) entries
    constexpr int cap = STAGE_BYTES / (OB + MB);   // partials per chunk
    static_assert(cap >= 1, "the staging area holds at least one partial");
    const int Hkv = a.num_kv_heads, b = u / Hkv, hk = u - b * Hkv;
    const int64_t s0 = static_cast<int64_t>(u) + c_first;
    const float4* so = reinterpret_cast<const float4*>(stage);             // [cap][G][NG]
    const float2* sml = reinterpret_cast<const float2*>(stage + cap * OB);  // [cap][kMaxG]
    const uint32_t so_s = smem_u32(stage), sml_s = smem_u32(stage + cap * OB);
    float M[IT], Lh[IT];
    float4 acc[IT];
#pragma unroll
    for (int j = 0; j < IT; ++j) {
        M[j] = -INFINITY;
        Lh[j] = 0.f;
        acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k0 = 0; k0 < k_u; k0 += cap) {
        const int kc = min(cap, k_u - k0);
        const uint8_t* go = reinterpret_cast<const uint8_t*>(a.part_o + (s0 + k0) * G * D);
        const uint8_t* gml = reinterpret_cast<const uint8_t*>(a.part_ml + (s0 + k0) * kMaxG);
        for (int i = tid; i < kc * (OB / 16); i += NTHR) cp_async_16(so_s + i * 16, go + i * 16);
        for (int i = tid; i < kc * (MB / 16); i += NTHR) cp_async_16(sml_s + i * 16, gml + i * 16);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
#pragma unroll
        for (int j = 0; j < IT; ++j) {
            const int it = tid + j * NTHR;
            if (it < ITEMS) {
                const int h = it / NG, g4 = it - (it / NG) * NG;
                float Mb = M[j];
                for (int k = 0; k < kc; ++k) Mb = fmaxf(Mb, sml[k * kMaxG + h].x);
                const float Mbu = Mb == -INFINITY ? 0.f : Mb;
                const float r = fast_exp2(M[j] - Mbu);
                float4 x = acc[j];
                float lx = Lh[j] * r;
                x.x *= r; x.y *= r; x.z *= r; x.w *= r;
                for (int k = 0; k < kc; ++k) {
                    const float2 ml = sml[k * kMaxG + h];
                    const float f = fast_exp2(ml.x - Mbu);
                    const float4 v = so[(k * G + h) * NG + g4];
                    x.x += f * v.x; x.y += f * v.y; x.z += f * v.z; x.w += f * v.w;
                    lx += f * ml.y;
                }
                acc[j] = x;
                Lh[j] = lx;
                M[j] = Mb;
            }
        }
        __syncthreads();  // the chunk is consumed before the next one lands
    }
    const float vsc = unit_v_scale(a, hk);
#pragma unroll
    for (int j = 0; j < IT; ++j) {
        const int it = tid + j * NTHR;
        if (it < ITEMS) {
            const int h = it / NG, g4 = it - (it / NG) * NG;
            const float sc_out = Lh[j] > 0.f ? vsc / Lh[j] : 0.f;
            uint16_t* out = a.out + (static_cast<int64_t>(b) * a.num_q_heads + hk * G + h) * D;
            const uint32_t lo2 =
                f32_to_bf16(acc[j].x * sc_out) | (static_cast<uint32_t>(f32_to_bf16(acc[j].y * sc_out)) << 16);
            const uint32_t hi2 =
                f32_to_bf16(acc[j].z * sc_out) | (static_cast<uint32_t>(f32_to_bf16(acc[j].w * sc_out)) << 16);
            *reinterpret_cast<uint2*>(out + g4 * 4) = make_uint2(lo2, hi2);
        }
    }
}

// Warps and ring depth of the streaming kernel.  Two CTAs share an SM
// (228 KB of shared memory, 64K registers).  At d = 256 the larger merge
// buffers leave room for two ring stages per warp, elsewhere three.  At
// d = 64 (g <= 8, whose registers allow it) 6 warps with two stages each
// measured 7% faster than 4 warps with three: more warps issuing copies.
// The bf16 cache at d = 256 has 8 KB pages: a stage is one page of K and one
// of V (16 KB), and three warps with two stages each fit.
template <int D, int ES, int G>
struct StreamCfg {
    static constexpr bool kWide = D == 64 && ES == 1 && G <= 8;
    static constexpr bool kBigPage = Geo<D, ES>::SH > kStageHalf;            // bf16 at d = 256: 8 KB pages
    static constexpr int NW = kWide ? 6 : kBigPage ? 3 : 4;                  // warps per CTA
    static constexpr int R = (Geo<D, ES>::XW > 40 || kWide) ? 2 : 3;         // ring stages per warp
    static constexpr int NBUF = NW / 2;                                      // merge exchange buffers
    static constexpr int CPP = Geo<D, ES>::PAGE / 512;                       // 16-byte copies per lane per page
};

template <int D, int ES, int G>
constexpr size_t stream_smem_bytes() {
    using Sc = StreamCfg<D, ES, G>;
    return 128 + static_cast<size_t>(Sc::NW) * Sc::R * Geo<D, ES>::SB + Sc::NBUF * Geo<D, ES>::XW * 32 * sizeof(float) +
           (2 * kMaxBatch + 1 + 8) * sizeof(int32_t);
}

// Dynamic shared memory one of kCtasPerSm resident CTAs may take (228 KB per
// SM, 1 KB of it reserved per CTA).
constexpr size_t kSmemPerCta = (228u * 1024u) / kCtasPerSm - 1024u;

template <int D, int G, int ES, bool E5M2>
__global__ void __launch_bounds__(StreamCfg<D, ES, G>::NW * 32, kCtasPerSm)
    stream_decode_kernel(const DecodeArgs a) {
    using Gm = Geo<D, ES>;
    using Sc = StreamCfg<D, ES, G>;
    constexpr int NW = Sc::NW, R = Sc::R, CPP = Sc::CPP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* rings = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    float* xbuf = reinterpret_cast<float*>(rings + NW * R * Gm::SB);                 // [NBUF][XW][32]
    int32_t* pre = reinterpret_cast<int32_t*>(xbuf + Sc::NBUF * Gm::XW * 32);         // [kMaxBatch + 1]
    int32_t* lens = pre + kMaxBatch + 1;                                              // [kMaxBatch]
    volatile int* flag = reinterpret_cast<volatile int*>(lens + kMaxBatch);            // [1] earlier timeout
    int32_t* mlist = lens + kMaxBatch + 1;  // [0]: units this CTA completes; then (u, c_first, k_u) each

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // This grid may have started before the previous one on the stream
    // finished (programmatic launch): wait for it before reading any input.
    griddep_wait();
    // The next grid on the stream may start its set-up now; it waits for
    // this grid's completion before it reads anything this grid writes.
    griddep_launch_dependents();
    const int B = a.batch, Hkv = a.num_kv_heads, C = gridDim.x, c = blockIdx.x;

    // ---- attended pages per sequence and their exclusive prefix; the error
    // word is read alongside (a call that gave up a wait fails every later
    // call on the workspace until it is re-initialised)
    if (warp == 0) {
        uint32_t prev_err = 0;
        if (lane == 0) prev_err = *reinterpret_cast<volatile uint32_t*>(a.err);
        int run = 0;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int b = b0 + lane;
            int n = 0;
            if (b < B) {
                const int Lraw = __ldg(a.seq_lens + b);
                if (Lraw < 0 || Lraw > a.max_seq_len) report(a.err, FP8KV_ERR_INVALID_ARG);
                lens[b] = clamp_len(Lraw, a.max_seq_len);
                n = attended_pages(lens[b], a.window);
            }
            int x = n;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            if (b < B) pre[b] = run + x - n;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) {
            pre[B] = run;
            flag[0] = prev_err == FP8KV_ERR_TIMEOUT;
            mlist[0] = 0;
        }
    }
    __syncthreads();
    if (flag[0]) return;

    const int64_t P = static_cast<int64_t>(Hkv) * pre[B];
    for (int b = c; b < B; b += C) {  // sequences with nothing to attend produce zeros
        if (pre[b + 1] == pre[b]) {
            uint16_t* ob = a.out + static_cast<int64_t>(b) * a.num_q_heads * D;
            for (int i = tid; i < a.num_q_heads * D; i += NW * 32) ob[i] = 0;
        }
    }
    const int Ce = static_cast<int>(P < C ? P : C);
    if (c >= Ce) return;
    const Partition part = make_partition(P, Ce);
    const int64_t s = range_start(part, c);
    const int64_t e = range_start(part, c + 1);

    // ---- this warp's ring and its per-lane copy offsets: lane l copies the
    // 16-byte chunks l, l+32, ... of a page, stored at their swizzled place
    uint8_t* ring = rings + warp * R * Gm::SB;
    const uint32_t ring_s = smem_u32(ring);
    uint32_t soff[CPP];
#pragma unroll
    for (int i = 0; i < CPP; ++i) {
        const int byte = (lane + 32 * i) * 16;
        const int r = byte / Gm::RB, b = byte % Gm::RB;
        soff[i] = (b / Gm::ROWB) * Gm::BOX + sswz<Gm::ROWB>(r, b % Gm::ROWB);
    }
    const uint64_t pol = l2_policy_evict_first();
    const bool appending = ES == 1 && a.k_new != nullptr;
    const int kvs = a.kv_shift, Hc = Hkv >> kvs;

    // ---- issue side: a cursor over this warp's pages in windows of up to 32
    // pages that never straddle a segment (walk.cuh).  Lane l holds the block
    // id of page start + l of the window; the window after the current one is
    // read one window ahead, with the newest K/V rows when it holds a unit's
    // last page and this is a decode step.
    struct Win {
        WinPos pos;
        int id;     // lane-held block id
        bool last;  // the window holds its unit's last page, which gets the new rows first
        NewRow<D> krow, vrow;
    };
    auto load_win = [&](Win& x) {
        x.id = 0;
        x.last = false;
        if (!x.pos.valid) return;
        const int32_t* row = a.block_tables + static_cast<int64_t>(x.pos.w.b) * a.max_blocks_per_seq +
                             first_token(lens[x.pos.w.b], a.window) / kBS + (x.pos.w.g - x.pos.w.base);
        x.id = load_block_id(row + x.pos.start, lane, x.pos.n, a.num_blocks, a.err);
        x.last = appending && window_holds_unit_end(x.pos, e);
        if (x.last) {
            const int64_t nr = static_cast<int64_t>(x.pos.w.b) * Hc + (x.pos.w.hk >> kvs);
            load_new_row<D>(x.krow, a.k_new + nr * D, lane);
            load_new_row<D>(x.vrow, a.v_new + nr * D, lane);
        }
    };
    Win cur, nxt;
    {
        Walker w0;
        walk_start(w0, pre, B, Hkv, s);
        cur.pos = first_window_from(w0, true, pre, Hkv, e, warp, NW);
        load_win(cur);
        nxt.pos = next_window(cur.pos, pre, Hkv, e, warp, NW);
        load_win(nxt);
    }
    int cpos = 0;   // pages of the current window already issued
    int ist = 0;    // stages issued
    // Issues this warp's next stage (up to PPS pages of K and V) into ring
    // slot ist % R, or an empty copy group once its pages are exhausted.
    auto issue_stage = [&]() {
        if (cur.pos.valid) {
            const int n = min(Gm::PPS, cur.pos.n - cpos);
            const uint32_t slot = ring_s + (ist % R) * Gm::SB;
            for (int p = 0; p < n; ++p) {
                const int id = __shfl_sync(0xffffffffu, cur.id, cpos + p);
                const int64_t page = static_cast<int64_t>(max(id, 0)) * Hc + (cur.pos.w.hk >> kvs);
                const uint8_t* ksrc = a.k_cache + page * Gm::PAGE;
                const uint8_t* vsrc = a.v_cache + page * Gm::PAGE;
                if (cur.last && cur.pos.start + cpos + p == cur.pos.hi - 1 && id >= 0) {
                    // the unit's last page: write the sequence's newest K and
                    // V rows into it first (the same quantisation as the
                    // append kernel), then copy it
                    const int L = lens[cur.pos.w.b];
                    const int64_t roff = static_cast<int64_t>((L - 1) % kBS) * D;
                    const float ksc = a.k_scales ? __ldg(a.k_scales + (cur.pos.w.hk >> kvs)) : a.k_scale_raw;
                    const float vsc = a.v_scales ? __ldg(a.v_scales + (cur.pos.w.hk >> kvs)) : a.v_scale_raw;
                    store_new_row<D, E5M2>(cur.krow, a.k_cache + page * Gm::PAGE + roff, lane, ksc);
                    store_new_row<D, E5M2>(cur.vrow, a.v_cache + page * Gm::PAGE + roff, lane, vsc);
                    __threadfence();
                    __syncwarp();
                }
#pragma unroll
                for (int i = 0; i < CPP; ++i) {
                    cp_async_16(slot + p * Gm::PAGE + soff[i], ksrc + (lane + 32 * i) * 16, pol);
                    cp_async_16(slot + Gm::SH + p * Gm::PAGE + soff[i], vsrc + (lane + 32 * i) * 16, pol);
                }
            }
            cpos += n;
            if (cpos == cur.pos.n) {
                cur = nxt;
                cpos = 0;
                nxt.pos = next_window(cur.pos, pre, Hkv, e, warp, NW);
                load_win(nxt);
            }
        }
        cp_async_commit();
        ++ist;
    };
#pragma unroll
    for (int i = 0; i < R - 1; ++i) issue_stage();

    // ---- compute side: the segments of the CTA's range in order; in each,
    // this warp's share stage by stage, then the CTA's warps merge
    const int gid = lane >> 2, tig = lane & 3;
    constexpr int NT = G > 8 ? 2 : 1;  // n-tiles of 8 query heads
    uint32_t qf[NT][Gm::KS][2];
    float cs[NT][2];
    float m[NT][2], l[NT][2];
    float o[NT][Gm::MT][4];
    int kst = 0;  // stages computed
    Walker w;
    walk_start(w, pre, B, Hkv, s);
    while (true) {
        const int64_t seg_end = min(e, w.base + w.n);
        const int lp0 = static_cast<int>(w.g - w.base);
        int q0, q1;
        warp_share(w, e, warp, NW, q0, q1);
        const int L = lens[w.b];
        const int lo = first_token(L, a.window);
        const int pg_first = lo / kBS + lp0;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if constexpr (ES == 1)
                load_query<D, G>(a, w.b, w.hk, gid, tig, qf[t], cs[t], 8 * t);
            else
                load_query_bf16<D, G>(a, w.b, w.hk, gid, tig, qf[t], cs[t], 8 * t);
            m[t][0] = m[t][1] = -INFINITY;
            l[t][0] = l[t][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < Gm::MT; ++mt) o[t][mt][0] = o[t][mt][1] = o[t][mt][2] = o[t][mt][3] = 0.f;
        }

        for (int p0 = q0; p0 < q1; p0 += Gm::PPS) {
            issue_stage();
            cp_async_wait<R - 1>();
            __syncwarp();
            const uint8_t* kst_p = ring + (kst % R) * Gm::SB;
            tc_stage<D, ES, E5M2, NT>(kst_p, kst_p + Gm::SH, min(Gm::PPS, q1 - p0), (pg_first + p0) * kBS, lo, L,
                                      gid, tig, qf, cs, m, l, o);
            __syncwarp();  // every lane is done with the slot before it is refilled
            ++kst;
        }

#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                l[t][j] += __shfl_xor_sync(0xffffffffu, l[t][j], 4);
                l[t][j] += __shfl_xor_sync(0xffffffffu, l[t][j], 8);
                l[t][j] += __shfl_xor_sync(0xffffffffu, l[t][j], 16);
            }

        // ---- merge the warps' states into warp 0 (tree through smem), one
        // n-tile after the other through the same buffers
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int n = NW; n > 1; n -= n / 2) {
                const int h = n / 2;
                if (warp >= n - h && warp < n)
                    publish<Gm::MT>(xbuf + (warp - (n - h)) * Gm::XW * 32, lane, m[t], l[t], o[t]);
                consumer_sync_n<NW>();
                if (warp < h) absorb<Gm::MT>(xbuf + warp * Gm::XW * 32, lane, m[t], l[t], o[t]);
                consumer_sync_n<NW>();
            }

        // ---- emit: the whole unit in this CTA -> output; else a partial
        const int u = w.b * Hkv + w.hk;
        const int c_first = cta_of(part, w.base);
        const int c_last = cta_of(part, w.base + w.n - 1);
        if (warp == 0) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (c_first == c_last) {
                    uint16_t* out_u = a.out + (static_cast<int64_t>(w.b) * a.num_q_heads + w.hk * G) * D;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int h = 8 * t + 2 * tig + j;
                        const float sc_out = l[t][j] > 0.f ? unit_v_scale(a, w.hk) / l[t][j] : 0.f;
                        if (h < G) {
#pragma unroll
                            for (int mt = 0; mt < Gm::MT; ++mt) {
                                // dimensions dim and dim + 1 together (one 4-byte store)
                                const int dim = (mt / Gm::MTH) * Gm::DBOX + Gm::VWD * gid + 2 * (mt % Gm::MTH);
                                *reinterpret_cast<uint32_t*>(out_u + h * D + dim) =
                                    static_cast<uint32_t>(f32_to_bf16(o[t][mt][j] * sc_out)) |
                                    (static_cast<uint32_t>(f32_to_bf16(o[t][mt][2 + j] * sc_out)) << 16);
                            }
                        }
                    }
                } else {
                    const int64_t slot_idx = static_cast<int64_t>(u) + c;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int h = 8 * t + 2 * tig + j;
                        if (h < G) {
                            float* po = a.part_o + (slot_idx * G + h) * D;
#pragma unroll
                            for (int mt = 0; mt < Gm::MT; ++mt)
#pragma unroll
                                for (int e2 = 0; e2 < 2; ++e2)
                                    po[(mt / Gm::MTH) * Gm::DBOX + Gm::VWD * gid + 2 * (mt % Gm::MTH) + e2] = o[t][mt][2 * e2 + j];
                            if (gid == 0) a.part_ml[slot_idx * kMaxG + h] = make_float2(m[t][j], l[t][j]);
                        }
                    }
                }
            }
            if (c_first != c_last && a.inline_merge) {
                // Publish the partial, then count it.  The CTA that brings the
                // count to k_u merges the unit once its own range is done (a
                // range holds at most two split units: its first and its last
                // segment).
                __threadfence();
                __syncwarp();
                if (lane == 0) {
                    const int k_u = c_last - c_first + 1;
                    if (atomicAdd(a.split_cnt + u, 1) == k_u - 1) {
                        a.split_cnt[u] = 0;  // every partial is in: ready for the next call
                        __threadfence();
                        const int i = mlist[0];
                        mlist[1 + 3 * i] = u;
                        mlist[2 + 3 * i] = c_first;
                        mlist[3 + 3 * i] = k_u;
                        mlist[0] = i + 1;
                    }
                }
            }
        }
        if (seg_end >= e) break;
        walk_next(w, pre, Hkv);
    }
    cp_async_wait<0>();

    // ---- the units this CTA completed: combine their partials into the output
    // (the rings and the exchange buffers, contiguous, stage the partials)
    __syncthreads();
    const int nm = mlist[0];
    for (int i = 0; i < nm; ++i)
        merge_unit<D, G, NW * 32, NW * R * Gm::SB + Sc::NBUF * Gm::XW * 32 * static_cast<int>(sizeof(float))>(
            a, mlist[1 + 3 * i], mlist[2 + 3 * i], mlist[3 + 3 * i], tid, rings);
}

// Combines the partials of every (sequence, kv head) unit that was split over
// several CTAs, when the decode grid does not (see merge_inline): one CTA per
// (unit, query head of the group).  Its 4 * D threads split the unit's
// partials into 16 slices (8 loads in flight per thread, one online
// softmax-merge pass), then combine the slices in shared memory.  It starts as
// a programmatic dependent of the decode grid and waits for that grid's
// completion before reading.
template <int D>
__host__ __device__ constexpr int merge_threads() { return 4 * D; }

template <int D, int G>
__global__ void __launch_bounds__(merge_threads<D>()) merge_kernel(const DecodeArgs a) {
    constexpr int kMergeThreads = merge_threads<D>();
    constexpr int NG = D / 4;                // float4 groups per head: 16, 32, 64
    constexpr int KS = kMergeThreads / NG;   // slices of the partial list: 16
    __shared__ float sm_m[KS][NG], sm_l[KS][NG];
    __shared__ float4 sm_o[KS][NG];
    griddep_launch_dependents();  // the next call's set-up may overlap this merge
    const int u = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int g4 = tid % NG, ks = tid / NG;
    // Where this unit's partials are: the decode grid's page split, recomputed
    // from the lengths while that grid finishes (they are final: the decode
    // CTAs trigger this grid only after their own wait).
    __shared__ long long red[2][kMergeThreads / 32];
    const int Hkv = a.num_kv_heads, b = u / Hkv, hk = u - b * Hkv;
    long long before = 0, total = 0;
    for (int i = tid; i < a.batch; i += kMergeThreads) {
        const int n = attended_pages(clamp_len(__ldg(a.seq_lens + i), a.max_seq_len), a.window);
        total += n;
        before += i < b ? n : 0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, off);
        total += __shfl_xor_sync(0xffffffffu, total, off);
    }
    if ((tid & 31) == 0) {
        red[0][tid >> 5] = before;
        red[1][tid >> 5] = total;
    }
    __syncthreads();
    before = total = 0;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) {
        before += red[0][w];
        total += red[1][w];
    }
    const int nb = attended_pages(clamp_len(__ldg(a.seq_lens + b), a.max_seq_len), a.window);
    int k_u = 0, c_first = 0;
    if (nb > 0) {
        const int64_t P = static_cast<int64_t>(Hkv) * total;
        const Partition part = make_partition(P, static_cast<int>(P < a.decode_ctas ? P : a.decode_ctas));
        const int64_t base = static_cast<int64_t>(Hkv) * before + static_cast<int64_t>(hk) * nb;
        c_first = cta_of(part, base);
        k_u = cta_of(part, base + nb - 1) - c_first + 1;
    }
    // Every CTA waits, even one with nothing to merge: this grid must not
    // complete (and release the next grid on the stream) before the decode
    // grid has.
    griddep_wait();
    if (k_u <= 1) return;  // empty (zeros), or written directly by its only CTA
    // a decode CTA gave up a wait (in this call or an earlier one on this
    // workspace): the partials are incomplete, and the error word says so
    if (*reinterpret_cast<volatile uint32_t*>(a.err) == FP8KV_ERR_TIMEOUT) return;
    const int64_t s0 = static_cast<int64_t>(u) + c_first;
    float M = -INFINITY, Lh = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = ks; k0 < k_u; k0 += 8 * KS) {
        float2 ml[8];
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int k = k0 + j * KS;
            if (k < k_u) {
                ml[j] = a.part_ml[(s0 + k) * kMaxG + h];
                v[j] = *(reinterpret_cast<const float4*>(a.part_o + ((s0 + k) * G + h) * D) + g4);
            } else {
                ml[j] = make_float2(-INFINITY, 0.f);
                v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float Mb = M;
#pragma unroll
        for (int j = 0; j < 8; ++j) Mb = fmaxf(Mb, ml[j].x);
        const float Mbu = Mb == -INFINITY ? 0.f : Mb;
        const float r = fast_exp2(M - Mbu);
        acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
        Lh *= r;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float f = fast_exp2(ml[j].x - Mbu);
            acc.x += f * v[j].x; acc.y += f * v[j].y; acc.z += f * v[j].z; acc.w += f * v[j].w;
            Lh += f * ml[j].y;
        }
        M = Mb;
    }
    sm_m[ks][g4] = M;
    sm_l[ks][g4] = Lh;
    sm_o[ks][g4] = acc;
    __syncthreads();
    if (ks != 0) return;
    float Mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < KS; ++j) Mt = fmaxf(Mt, sm_m[j][g4]);
    const float Mtu = Mt == -INFINITY ? 0.f : Mt;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float Lt = 0.f;
#pragma unroll
    for (int j = 0; j < KS; ++j) {
        const float f = fast_exp2(sm_m[j][g4] - Mtu);
        o.x += f * sm_o[j][g4].x; o.y += f * sm_o[j][g4].y; o.z += f * sm_o[j][g4].z; o.w += f * sm_o[j][g4].w;
        Lt += f * sm_l[j][g4];
    }
    const float sc_out = Lt > 0.f ? unit_v_scale(a, hk) / Lt : 0.f;
    uint16_t* out = a.out + (static_cast<int64_t>(b) * a.num_q_heads + hk * G + h) * D;
    const uint32_t lo2 = f32_to_bf16(o.x * sc_out) | (static_cast<uint32_t>(f32_to_bf16(o.y * sc_out)) << 16);
    const uint32_t hi2 = f32_to_bf16(o.z * sc_out) | (static_cast<uint32_t>(f32_to_bf16(o.w * sc_out)) << 16);
    *reinterpret_cast<uint2*>(out + g4 * 4) = make_uint2(lo2, hi2);
}

// ---------------------------------------------------------------- host side

struct Plan {
    int batch;  // sequences per launch (batches above kMaxBatch run in chunks)
    int ctas;   // CTAs per launch
};

Plan make_plan(int batch, int num_kv_heads, int D, int max_seq_len, int window, int sms) {
    (void)D;
    Plan p{std::max(1, std::min(batch, kMaxBatch)), 1};
    if (max_seq_len <= 0) return p;
    const int64_t all_pages = (max_seq_len + kBS - 1) / kBS;
    int64_t max_pages = all_pages;
    if (window > 0 && window < max_seq_len) max_pages = std::min<int64_t>(all_pages, (window + kBS - 1) / kBS + 1);
    const int64_t pmax = static_cast<int64_t>(p.batch) * num_kv_heads * max_pages;
    const int64_t want = (pmax + kMinPagesPerCta - 1) / kMinPagesPerCta;
    p.ctas = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(std::min<int64_t>(want, static_cast<int64_t>(sms) * kCtasPerSm), kMaxMergeSplits)));
    return p;
}

// Who merges the split units of a tensor-core launch.  The CTA that completes
// a unit merges it when the unit's partials are few (one SM reads them all
// through L2: about 25 GB/s measured); otherwise the merge kernel, whose CTAs
// (one per unit and query head) spread the reading over many SMs.  The
// partials per unit are estimated from the plan with every sequence at
// max_seq_len: a unit of n pages meets at most ceil(n / pages per CTA) + 1
// CTAs.  Shorter sequences only change the speed of the chosen merge.
constexpr int64_t kInlineMergeBytes = 16 << 10;

bool merge_inline(const Plan& p, int batch, int units_per_seq, int G, int D, int max_seq_len, int window) {
    if (p.ctas <= 1 || max_seq_len <= 0) return true;
    const int64_t all_pages = (max_seq_len + kBS - 1) / kBS;
    int64_t n = all_pages;
    if (window > 0 && window < max_seq_len) n = std::min<int64_t>(all_pages, (window + kBS - 1) / kBS + 1);
    const int64_t total = static_cast<int64_t>(batch) * units_per_seq * n;
    const int64_t per_cta = std::max<int64_t>(1, total / p.ctas);
    const int64_t k_est = std::min<int64_t>(p.ctas, (n + per_cta - 1) / per_cta + 1);
    return k_est * G * D * static_cast<int64_t>(sizeof(float)) <= kInlineMergeBytes;
}

struct WsLayout {
    size_t cnt, ml, o, total;  // byte offsets of the split counters, the partial (max, sum), the partial outputs
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int batch, int num_q_heads, int num_kv_heads, int D, const Plan& p) {
    (void)batch;
    const size_t units = static_cast<size_t>(p.batch) * num_kv_heads;
    const size_t slots = units + p.ctas;
    const int G = num_q_heads / num_kv_heads;
    WsLayout w;
    w.cnt = 256;  // after the header (the error word)
    w.ml = w.cnt + align256(units * sizeof(int32_t));
    w.o = w.ml + align256(slots * kMaxG * sizeof(float2));
    w.total = w.o + align256(slots * G * D * sizeof(float));
    return w;
}

// SM count of the current device (queried once per device).
int device_sms(int* sms) {
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *sms = c;
            return 0;
        }
    }
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) cache[dev].store(*sms, std::memory_order_relaxed);
    return 0;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// The cache as a 4-D tensor {D, 16 tokens, kv heads, blocks} of bytes; one box
// is one page (or one 128-byte-wide half of a D=256 page).
bool encode_cache_map(CUtensorMap* m, const void* base, int64_t num_blocks, int Hkv, int D) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(kBS),
                                static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(kBS) * D,
                                   static_cast<cuuint64_t>(kBS) * D * Hkv};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(D >= 128 ? 128 : D), static_cast<cuuint32_t>(kBS), 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw = D >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoding a tensor map is pure host work on its arguments; the last few
// (pointer, shape) -> map results are kept so repeated decode calls over the
// same cache skip it.
bool make_cache_map(CUtensorMap* m, const void* base, int64_t num_blocks, int Hkv, int D) {
    struct Entry {
        const void* base;
        int64_t num_blocks;
        int Hkv, D;
        CUtensorMap map;
    };
    constexpr int kEntries = 8;
    static std::mutex mu;
    static Entry entries[kEntries];
    static int used = 0, next = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry& e = entries[i];
            if (e.base == base && e.num_blocks == num_blocks && e.Hkv == Hkv && e.D == D) {
                *m = e.map;
                return true;
            }
        }
    }
    if (!encode_cache_map(m, base, num_blocks, Hkv, D)) return false;
    std::lock_guard<std::mutex> lock(mu);
    Entry& e = entries[next];
    e.base = base;
    e.num_blocks = num_blocks;
    e.Hkv = Hkv;
    e.D = D;
    e.map = *m;
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return true;
}

template <int D, int G>
cudaError_t launch(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeArgs& a, int ctas,
                   cudaStream_t stream) {
    // The shared-memory opt-in is per device; remember which devices have it.
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit == 0 || !(done_mask.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(paged_decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_bytes<D, G>()));
        if (e != cudaSuccess) return e;
        done_mask.fetch_or(bit, std::memory_order_release);
    }
    // Both grids may start before the previous work on the stream ends; each
    // waits (griddepcontrol.wait) before touching what that work wrote.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes<D, G>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, G>, mk, mv, a);
    if (e != cudaSuccess || ctas == 1) return e;  // one CTA: every unit is written directly
    cudaLaunchConfig_t mcfg = {};
    mcfg.gridDim = dim3(a.batch * a.num_kv_heads, G);
    mcfg.blockDim = dim3(merge_threads<D>());
    mcfg.dynamicSmemBytes = 0;
    mcfg.stream = stream;
    mcfg.attrs = attr;
    mcfg.numAttrs = 1;
    return cudaLaunchKernelEx(&mcfg, merge_kernel<D, G>, a);
}

template <int D, int G, int ES = 1, bool E5M2 = false>
cudaError_t launch_stream(const DecodeArgs& a, int ctas, cudaStream_t stream) {
    static_assert(stream_smem_bytes<D, ES, G>() <= kSmemPerCta, "two CTAs must fit on one SM");
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit == 0 || !(done_mask.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(stream_decode_kernel<D, G, ES, E5M2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(stream_smem_bytes<D, ES, G>()));
        if (e != cudaSuccess) return e;
        done_mask.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(StreamCfg<D, ES, G>::NW * 32);
    cfg.dynamicSmemBytes = stream_smem_bytes<D, ES, G>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, stream_decode_kernel<D, G, ES, E5M2>, a);
    if (e != cudaSuccess || ctas == 1 || a.inline_merge) return e;  // merged inside the decode grid
    cudaLaunchConfig_t mcfg = {};
    mcfg.gridDim = dim3(a.batch * a.num_kv_heads, G);
    mcfg.blockDim = dim3(merge_threads<D>());
    mcfg.dynamicSmemBytes = 0;
    mcfg.stream = stream;
    mcfg.attrs = attr;
    mcfg.numAttrs = 1;
    return cudaLaunchKernelEx(&mcfg, merge_kernel<D, G>, a);
}

template <int D, int ES = 1, bool E5M2 = false>
cudaError_t launch_stream_g(int G, const DecodeArgs& a, int ctas, cudaStream_t s) {
    switch (G) {
        case 1: return launch_stream<D, 1, ES, E5M2>(a, ctas, s);
        case 2: return launch_stream<D, 2, ES, E5M2>(a, ctas, s);
        case 4: return launch_stream<D, 4, ES, E5M2>(a, ctas, s);
        case 8: return launch_stream<D, 8, ES, E5M2>(a, ctas, s);
        case 16:
            if constexpr (D <= 128) return launch_stream<D, 16, ES, E5M2>(a, ctas, s);
            else return cudaErrorInvalidValue;  // g = 16 at d = 256 runs as two units of 8 (head_map)
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_g(int G, const CUtensorMap& mk, const CUtensorMap& mv, const DecodeArgs& a, int ctas,
                     cudaStream_t s) {
    switch (G) {
        case 1: return launch<D, 1>(mk, mv, a, ctas, s);
        case 2: return launch<D, 2>(mk, mv, a, ctas, s);
        case 4: return launch<D, 4>(mk, mv, a, ctas, s);
        case 8: return launch<D, 8>(mk, mv, a, ctas, s);
        default: return cudaErrorInvalidValue;
    }
}

// The contraction engine a call uses when the caller leaves it open.
bool default_is_cuda_cores(int /*head_dim*/, int /*G*/) { return false; }

bool supported(int head_dim, int block_size, int G) {
    return (head_dim == 64 || head_dim == 128 || head_dim == 256) && block_size == kBS &&
           (G == 1 || G == 2 || G == 4 || G == 8 || G == 16);
}

// How the kernels see the heads.  The streaming kernel at d <= 128 carries
// g = 16 natively (two MMA n-tiles of 8 heads on the same K and V fragments:
// each page is read once).  At d = 256, and on the CUDA-core engine, g = 16
// runs as two units of 8 query heads per cache head (each reads the head's
// pages): two n-tiles' accumulators do not fit beside the rest there.
struct HeadMap {
    int units_per_seq;  // kv-head units per sequence
    int g;              // query heads per unit
    int shift;          // unit -> cache head: hk >> shift
};

HeadMap head_map(int num_q_heads, int num_kv_heads, int head_dim, bool simt) {
    const int G = num_q_heads / num_kv_heads;
    if (G == 16 && (simt || head_dim > 128)) return {2 * num_kv_heads, 8, 1};
    return {num_kv_heads, G, 0};
}

}  // namespace fp8kv

using namespace fp8kv;

extern "C" size_t fp8kv_paged_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                                    int max_seq_len, int block_size, int window) {
    if (batch < 0 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0 || max_seq_len < 0)
        return 0;
    if (!supported(head_dim, block_size, num_q_heads / num_kv_heads)) return 0;
    int sms = 0;
    if (device_sms(&sms) != 0) return 0;
    // enough for either engine (their head mappings differ at g = 16)
    size_t total = 0;
    for (const bool simt : {false, true}) {
        const HeadMap hm = head_map(num_q_heads, num_kv_heads, head_dim, simt);
        const Plan p = make_plan(batch, hm.units_per_seq, head_dim, max_seq_len, window, sms);
        total = std::max(total, ws_layout(batch, hm.units_per_seq * hm.g, hm.units_per_seq, head_dim, p).total);
    }
    return total;
}

namespace {

// Host-side staging around a decode call: the inputs copied in before it, the
// output copied out after it (fp8kv_decode_step_host).
struct HostStage {
    const void* h_in;
    void* d_in;
    size_t in_bytes;
    void* h_out;
};

// The failure-path test hook's settings (fp8kv_debug_paged_decode_stall).
struct StallHook {
    int stall_stage;
    uint64_t wait_ns;
};

fp8kv_status decode_impl(const void* q, const void* k_new, const void* v_new, const uint8_t* k_cache,
                         const uint8_t* v_cache, int64_t num_blocks, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len, int batch,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size, float k_scale,
                         float v_scale, float sm_scale, int window, void* out, void* workspace,
                         size_t workspace_bytes, void* stream, int engine, int es = 1,
                         const float* k_scales = nullptr, const float* v_scales = nullptr, bool e5m2 = false,
                         const HostStage* hs = nullptr, const StallHook* dbg = nullptr) {
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (batch < 0 || batch > 65535 || num_kv_heads < 1 || num_kv_heads > 65535 || num_q_heads < 1 ||
        num_q_heads % num_kv_heads != 0 || max_seq_len < 0 || num_blocks < 1 || max_blocks_per_seq < 0)
        return FP8KV_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !(k_scale > 0) || !std::isfinite(v_scale) || !(v_scale > 0) ||
        !std::isfinite(sm_scale))
        return FP8KV_ERR_INVALID_ARG;
    if (!supported(head_dim, block_size, num_q_heads / num_kv_heads)) return FP8KV_ERR_UNSUPPORTED;
    if (engine != FP8KV_ENGINE_DEFAULT && engine != FP8KV_ENGINE_TENSOR_CORES && engine != FP8KV_ENGINE_CUDA_CORES)
        return FP8KV_ERR_INVALID_ARG;
    const bool simt = engine == FP8KV_ENGINE_CUDA_CORES ||
                      (engine == FP8KV_ENGINE_DEFAULT && default_is_cuda_cores(head_dim, num_q_heads / num_kv_heads));
    const HeadMap hm = head_map(num_q_heads, num_kv_heads, head_dim, simt);
    const int G = hm.g;
    if (num_blocks >= (INT64_C(1) << 31) || num_blocks * num_kv_heads >= (INT64_C(1) << 31))
        return FP8KV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_blocks_per_seq) * block_size < max_seq_len) return FP8KV_ERR_INVALID_ARG;
    // total (sequence, kv head, page) triples of one launch must stay far inside int64 index math
    if (static_cast<int64_t>(std::min(batch, kMaxBatch)) * num_kv_heads * ((max_seq_len + kBS - 1) / kBS + 1) >=
        (INT64_C(1) << 40))
        return FP8KV_ERR_UNSUPPORTED;
    if (batch == 0) return FP8KV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return FP8KV_ERR_INVALID_ARG;
    if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(out)) return FP8KV_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return FP8KV_ERR_INVALID_ARG;
    if (k_new && (!a16(k_new) || !a16(v_new))) return FP8KV_ERR_INVALID_ARG;
    if ((k_scales == nullptr) != (v_scales == nullptr)) return FP8KV_ERR_INVALID_ARG;
    if (k_scales && ((reinterpret_cast<uintptr_t>(k_scales) & 3u) || (reinterpret_cast<uintptr_t>(v_scales) & 3u)))
        return FP8KV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return FP8KV_ERR_INVALID_ARG;
    int sms = 0;
    if (device_sms(&sms) != 0) return FP8KV_ERR_CUDA;
    const WsLayout w = ws_layout(batch, num_q_heads, hm.units_per_seq, head_dim,
                                 make_plan(batch, hm.units_per_seq, head_dim, max_seq_len, window, sms));
    if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FP8KV_ERR_WORKSPACE;

    CUtensorMap mk, mv;  // the CUDA-core engine's TMA view of the caches (rows of head_dim bytes)
    if (simt && (!make_cache_map(&mk, k_cache, num_blocks, num_kv_heads, head_dim) ||
                 !make_cache_map(&mv, v_cache, num_blocks, num_kv_heads, head_dim)))
        return FP8KV_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (hs && hs->in_bytes > 0 &&
        cudaMemcpyAsync(hs->d_in, hs->h_in, hs->in_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return FP8KV_ERR_CUDA;
    // A host output buffer that the device can address (page-locked memory,
    // mapped under unified addressing) receives the result directly from the
    // kernels' stores, across the host link; otherwise the result goes to
    // `out` and is copied to h_out after the step.
    bool direct_out = false;
    if (hs && hs->h_out) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, hs->h_out) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
            pa.devicePointer != nullptr && a16(pa.devicePointer)) {
            out = pa.devicePointer;
            direct_out = true;
        } else {
            (void)cudaGetLastError();  // not a registered host buffer: copy instead
        }
    }
    // Batches above kMaxBatch sequences run as consecutive launches on the
    // stream, reusing the workspace.
    for (int b0 = 0; b0 < batch; b0 += kMaxBatch) {
        const int nb = std::min(kMaxBatch, batch - b0);
        const Plan p = make_plan(nb, hm.units_per_seq, head_dim, max_seq_len, window, sms);
        DecodeArgs a;
        a.q = static_cast<const uint16_t*>(q) + static_cast<int64_t>(b0) * num_q_heads * head_dim;
        a.k_new = k_new ? static_cast<const uint16_t*>(k_new) + static_cast<int64_t>(b0) * num_kv_heads * head_dim
                        : nullptr;
        a.v_new = v_new ? static_cast<const uint16_t*>(v_new) + static_cast<int64_t>(b0) * num_kv_heads * head_dim
                        : nullptr;
        a.k_cache = const_cast<uint8_t*>(k_cache);
        a.v_cache = const_cast<uint8_t*>(v_cache);
        a.k_scale_raw = k_scale;
        a.v_scale_raw = v_scale;
        a.k_scales = k_scales;
        a.v_scales = v_scales;
        a.sm_scale = sm_scale;
        a.block_tables = block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq;
        a.seq_lens = seq_lens + b0;
        a.out = static_cast<uint16_t*>(out) + static_cast<int64_t>(b0) * num_q_heads * head_dim;
        a.err = reinterpret_cast<uint32_t*>(ws);
        a.decode_ctas = p.ctas;
        a.part_ml = reinterpret_cast<float2*>(ws + w.ml);
        a.part_o = reinterpret_cast<float*>(ws + w.o);
        a.split_cnt = reinterpret_cast<int32_t*>(ws + w.cnt);
        a.inline_merge = !simt && merge_inline(p, nb, hm.units_per_seq, G, head_dim, max_seq_len, window);
        a.num_blocks = num_blocks;
        a.max_blocks_per_seq = max_blocks_per_seq;
        a.max_seq_len = max_seq_len;
        a.batch = nb;
        a.num_q_heads = num_q_heads;
        a.num_kv_heads = hm.units_per_seq;
        a.kv_shift = hm.shift;
        a.window = window > 0 ? window : 0;
        a.score_scale = sm_scale * k_scale * kLog2e;
        a.v_scale = v_scale;
        a.wait_ns = dbg ? dbg->wait_ns : kWaitLimitNs;
        a.stall_stage = dbg ? dbg->stall_stage : -1;
        cudaError_t e;
        if (!simt) {
            if (es == 2)
                e = head_dim == 64 ? launch_stream_g<64, 2>(G, a, p.ctas, s)
                    : head_dim == 128 ? launch_stream_g<128, 2>(G, a, p.ctas, s)
                                      : launch_stream_g<256, 2>(G, a, p.ctas, s);
            else if (e5m2)
                e = head_dim == 64 ? launch_stream_g<64, 1, true>(G, a, p.ctas, s)
                    : head_dim == 128 ? launch_stream_g<128, 1, true>(G, a, p.ctas, s)
                                      : launch_stream_g<256, 1, true>(G, a, p.ctas, s);
            else
                e = head_dim == 64 ? launch_stream_g<64>(G, a, p.ctas, s)
                    : head_dim == 128 ? launch_stream_g<128>(G, a, p.ctas, s)
                                      : launch_stream_g<256>(G, a, p.ctas, s);
        } else {
            e = head_dim == 64 ? launch_g<64>(G, mk, mv, a, p.ctas, s)
                : head_dim == 128 ? launch_g<128>(G, mk, mv, a, p.ctas, s)
                                  : launch_g<256>(G, mk, mv, a, p.ctas, s);
        }
        if (e != cudaSuccess) return FP8KV_ERR_CUDA;
    }
    if (hs && !direct_out &&
        cudaMemcpyAsync(hs->h_out, out, static_cast<size_t>(batch) * num_q_heads * head_dim * 2,
                        cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return FP8KV_ERR_CUDA;
    return FP8KV_OK;
}

}  // namespace

extern "C" fp8kv_status fp8kv_paged_decode(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                           int64_t num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                                           const int32_t* seq_lens, int max_seq_len, int batch, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size, float k_scale,
                                           float v_scale, float sm_scale, int window, void* out, void* workspace,
                                           size_t workspace_bytes, void* stream) {
    FP8KV_TRACE("fp8kv_paged_decode");
    return decode_impl(q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq,
                       seq_lens, max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, k_scale,
                       v_scale, sm_scale, window, out, workspace, workspace_bytes, stream, FP8KV_ENGINE_DEFAULT);
}

extern "C" fp8kv_status fp8kv_paged_decode_engine(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                                  int64_t num_blocks, const int32_t* block_tables,
                                                  int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                                  int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                                  int block_size, float k_scale, float v_scale, float sm_scale,
                                                  int window, void* out, void* workspace, size_t workspace_bytes,
                                                  void* stream, int engine) {
    FP8KV_TRACE("fp8kv_paged_decode_engine");
    return decode_impl(q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq,
                       seq_lens, max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, k_scale,
                       v_scale, sm_scale, window, out, workspace, workspace_bytes, stream, engine);
}

extern "C" fp8kv_status fp8kv_paged_decode_bf16(const void* q, const void* k_cache, const void* v_cache,
                                                int64_t num_blocks, const int32_t* block_tables,
                                                int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                                int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                                int block_size, float sm_scale, int window, void* out,
                                                void* workspace, size_t workspace_bytes, void* stream) {
    FP8KV_TRACE("fp8kv_paged_decode_bf16");
    return decode_impl(q, nullptr, nullptr, static_cast<const uint8_t*>(k_cache), static_cast<const uint8_t*>(v_cache),
                       num_blocks, block_tables, max_blocks_per_seq, seq_lens, max_seq_len, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, 1.0f, 1.0f, sm_scale, window, out, workspace,
                       workspace_bytes, stream, FP8KV_ENGINE_TENSOR_CORES, 2);
}

extern "C" fp8kv_status fp8kv_paged_decode_per_head(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                                    int64_t num_blocks, const int32_t* block_tables,
                                                    int max_blocks_per_seq, const int32_t* seq_lens,
                                                    int max_seq_len, int batch, int num_q_heads, int num_kv_heads,
                                                    int head_dim, int block_size, const float* k_scales,
                                                    const float* v_scales, float sm_scale, int window, void* out,
                                                    void* workspace, size_t workspace_bytes, void* stream) {
    FP8KV_TRACE("fp8kv_paged_decode_per_head");
    if (batch > 0 && (!k_scales || !v_scales)) return FP8KV_ERR_INVALID_ARG;
    return decode_impl(q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq,
                       seq_lens, max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, 1.0f, 1.0f,
                       sm_scale, window, out, workspace, workspace_bytes, stream, FP8KV_ENGINE_DEFAULT, 1, k_scales,
                       v_scales);
}

extern "C" fp8kv_status fp8kv_decode_step_per_head(const void* q, const void* k_new, const void* v_new,
                                                   uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                                                   const int32_t* block_tables, int max_blocks_per_seq,
                                                   const int32_t* seq_lens, int max_seq_len, int batch,
                                                   int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                                   const float* k_scales, const float* v_scales, float sm_scale,
                                                   int window, void* out, void* workspace, size_t workspace_bytes,
                                                   void* stream) {
    FP8KV_TRACE("fp8kv_decode_step_per_head");
    if (batch > 0 && (!k_new || !v_new || !k_scales || !v_scales)) return FP8KV_ERR_INVALID_ARG;
    return decode_impl(q, k_new, v_new, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                       max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, 1.0f, 1.0f, sm_scale,
                       window, out, workspace, workspace_bytes, stream, FP8KV_ENGINE_DEFAULT, 1, k_scales, v_scales);
}

extern "C" fp8kv_status fp8kv_paged_decode_e5m2(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                                int64_t num_blocks, const int32_t* block_tables,
                                                int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                                int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                                int block_size, float k_scale, float v_scale, float sm_scale,
                                                int window, void* out, void* workspace, size_t workspace_bytes,
                                                void* stream) {
    FP8KV_TRACE("fp8kv_paged_decode_e5m2");
    return decode_impl(q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq,
                       seq_lens, max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, k_scale,
                       v_scale, sm_scale, window, out, workspace, workspace_bytes, stream, FP8KV_ENGINE_TENSOR_CORES,
                       1, nullptr, nullptr, true);
}

extern "C" fp8kv_status fp8kv_decode_step_e5m2(const void* q, const void* k_new, const void* v_new,
                                               uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                                               const int32_t* block_tables, int max_blocks_per_seq,
                                               const int32_t* seq_lens, int max_seq_len, int batch,
                                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                               float k_scale, float v_scale, float sm_scale, int window, void* out,
                                               void* workspace, size_t workspace_bytes, void* stream) {
    FP8KV_TRACE("fp8kv_decode_step_e5m2");
    if (batch > 0 && (!k_new || !v_new)) return FP8KV_ERR_INVALID_ARG;
    return decode_impl(q, k_new, v_new, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                       max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, k_scale, v_scale,
                       sm_scale, window, out, workspace, workspace_bytes, stream, FP8KV_ENGINE_TENSOR_CORES, 1,
                       nullptr, nullptr, true);
}

extern "C" fp8kv_status fp8kv_decode_step(const void* q, const void* k_new, const void* v_new, uint8_t* k_cache,
                                          uint8_t* v_cache, int64_t num_blocks, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                          int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                          float k_scale, float v_scale, float sm_scale, int window, void* out,
                                          void* workspace, size_t workspace_bytes, void* stream) {
    FP8KV_TRACE("fp8kv_decode_step");
    if (batch > 0 && (!k_new || !v_new)) return FP8KV_ERR_INVALID_ARG;
    return decode_impl(q, k_new, v_new, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                       max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, k_scale, v_scale,
                       sm_scale, window, out, workspace, workspace_bytes, stream, FP8KV_ENGINE_DEFAULT);
}

extern "C" fp8kv_status fp8kv_decode_step_host(const void* h_in, void* d_in, size_t in_bytes, void* h_out,
                                               const void* q, const void* k_new, const void* v_new,
                                               uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                                               const int32_t* block_tables, int max_blocks_per_seq,
                                               const int32_t* seq_lens, int max_seq_len, int batch,
                                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                               float k_scale, float v_scale, float sm_scale, int window, void* out,
                                               void* workspace, size_t workspace_bytes, void* stream) {
    FP8KV_TRACE("fp8kv_decode_step_host");
    if (batch > 0 && (!k_new || !v_new)) return FP8KV_ERR_INVALID_ARG;
    if ((in_bytes > 0 && (!h_in || !d_in)) || (batch > 0 && !h_out)) return FP8KV_ERR_INVALID_ARG;
    if (batch == 0) {  // nothing to attend: only the inputs move
        if (in_bytes > 0 && cudaMemcpyAsync(d_in, h_in, in_bytes, cudaMemcpyHostToDevice,
                                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return FP8KV_ERR_CUDA;
        return FP8KV_OK;
    }
    const HostStage hs{h_in, d_in, in_bytes, h_out};
    return decode_impl(q, k_new, v_new, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                       max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, k_scale, v_scale,
                       sm_scale, window, out, workspace, workspace_bytes, stream, FP8KV_ENGINE_DEFAULT, 1, nullptr,
                       nullptr, false, &hs);
}

extern "C" fp8kv_status fp8kv_debug_paged_decode_stall(const void* q, const uint8_t* k_cache,
                                                       const uint8_t* v_cache, int64_t num_blocks,
                                                       const int32_t* block_tables, int max_blocks_per_seq,
                                                       const int32_t* seq_lens, int max_seq_len, int batch,
                                                       int num_q_heads, int num_kv_heads, int head_dim,
                                                       int block_size, float k_scale, float v_scale, float sm_scale,
                                                       int window, void* out, void* workspace,
                                                       size_t workspace_bytes, void* stream, int stall_stage,
                                                       uint64_t wait_limit_ns) {
    FP8KV_TRACE("fp8kv_debug_paged_decode_stall");
    if (stall_stage < 0 || wait_limit_ns == 0 || wait_limit_ns > kWaitLimitNs) return FP8KV_ERR_INVALID_ARG;
    const StallHook dbg{stall_stage, wait_limit_ns};
    return decode_impl(q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                       max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, k_scale, v_scale,
                       sm_scale, window, out, workspace, workspace_bytes, stream, FP8KV_ENGINE_CUDA_CORES, 1, nullptr,
                       nullptr, false, nullptr, &dbg);
}

// ---------------------------------------------------------------- allocation-free variant
//
// Some callers cannot allocate device memory at the point where they decode:
// a serving engine that reserved nearly all HBM up front for its own paged-KV
// pool (so a late cudaMalloc fails or fragments that pool), host code running
// under a no-allocation rule (a fixed-budget or real-time loop, a plugin inside
// a framework that owns every device buffer), or a language binding with no
// CUDA allocator at hand.  For them the split-merge scratch lives in a
// fixed-size device array that is part of the library image itself.

namespace fp8kv {

// 8 MiB covers every workload shape exercised here: the largest, 16
// sequences of up to 32K tokens at head_dim 256 with 8 query heads per kv
// head, needs (16 units + 304 CTAs) x 8 heads x 256 dims x 4 B = 2.6 MB of
// partials.  Every device that loads the library holds this array until the
// process exits.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of the array on the current device, looked up once per device
// (host code only sees a host-side stand-in for the symbol).
static void* static_scratch_address() {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace fp8kv

extern "C" fp8kv_status fp8kv_paged_decode_noalloc(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                                   int64_t num_blocks, const int32_t* block_tables,
                                                   int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                                   int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                                   int block_size, float k_scale, float v_scale, float sm_scale,
                                                   int window, void* out, void* stream) {
    FP8KV_TRACE("fp8kv_paged_decode_noalloc");
    if (batch < 0 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0 || max_seq_len < 0)
        return FP8KV_ERR_INVALID_ARG;
    if (!supported(head_dim, block_size, num_q_heads / num_kv_heads)) return FP8KV_ERR_UNSUPPORTED;
    if (batch == 0) return FP8KV_OK;
    int sms = 0;
    if (device_sms(&sms) != 0) return FP8KV_ERR_CUDA;
    const HeadMap hm = head_map(num_q_heads, num_kv_heads, head_dim, false);  // the default engine's
    const Plan p = make_plan(batch, hm.units_per_seq, head_dim, max_seq_len, window, sms);
    const WsLayout w = ws_layout(batch, num_q_heads, hm.units_per_seq, head_dim, p);
    if (w.total > kStaticScratchBytes) return FP8KV_ERR_WORKSPACE;  // problem too large for the fixed array
    void* scratch = static_scratch_address();
    if (scratch == nullptr) return FP8KV_ERR_CUDA;
    // The array keeps the previous call's contents: the error word and the
    // split counters must start at zero.
    if (cudaMemsetAsync(scratch, 0, w.ml, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8KV_ERR_CUDA;
    return fp8kv_paged_decode(q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                              max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, k_scale, v_scale,
                              sm_scale, window, out, scratch, kStaticScratchBytes, stream);
}

extern "C" fp8kv_status fp8kv_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    FP8KV_TRACE("fp8kv_workspace_init");
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FP8KV_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FP8KV_OK
               : FP8KV_ERR_CUDA;
}

extern "C" fp8kv_status fp8kv_read_error(void* workspace, uint32_t* code, void* stream) {
    FP8KV_TRACE("fp8kv_read_error");
    if (!workspace || !code) return FP8KV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t zero = 0;
    if (cudaMemcpyAsync(code, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return FP8KV_ERR_CUDA;
    if (cudaMemcpyAsync(workspace, &zero, sizeof(uint32_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return FP8KV_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA;
}

extern "C" const char* fp8kv_status_string(fp8kv_status status) {
    switch (status) {
        case FP8KV_OK: return "FP8KV_OK";
        case FP8KV_ERR_INVALID_ARG: return "FP8KV_ERR_INVALID_ARG";
        case FP8KV_ERR_UNSUPPORTED: return "FP8KV_ERR_UNSUPPORTED";
        case FP8KV_ERR_WORKSPACE: return "FP8KV_ERR_WORKSPACE";
        case FP8KV_ERR_CUDA: return "FP8KV_ERR_CUDA";
        case FP8KV_ERR_TIMEOUT: return "FP8KV_ERR_TIMEOUT";
        default: return "FP8KV_ERR_UNKNOWN";
    }
}
