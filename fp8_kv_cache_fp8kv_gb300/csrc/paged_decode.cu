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
// How (one CTA = one (split of the context, kv head, sequence)):
//  * All g query heads of a kv head share the CTA, so every cache byte is read
//    from HBM once.  Decode attention is bandwidth-bound (2g flop per fp8
//    byte), so the kernel is built around streaming pages at HBM speed.
//  * One producer warp streams K and V pages with TMA tensor copies (128-byte
//    or 64-byte swizzle, evict-first L2 policy) into a ring of shared-memory
//    stages guarded by mbarriers.  Four consumer warps each own every fourth
//    stage and keep their own online-softmax state.
//  * Per stage a consumer warp converts codes to f16 (exact) and runs the
//    score contraction S^T = K Q^T and the value contraction O^T += V^T P^T on
//    the tensor cores (mma m16n8k16, fp32 accumulators): with g <= 8 the
//    query heads form the n=8 side, so no tensor-core work is padded for g=8.
//    FP32 CUDA cores alone cannot keep up with HBM at g=8 on this part (2g
//    flop per byte at ~7 TB/s exceeds their FMA rate).  The stage's P.V tile
//    is then added into separate FP32 registers (O = O*alpha + tile), so the
//    long contraction is summed in IEEE FP32, not inside the MMA.
//  * The softmax max/sum use warp shuffles; P is rounded to f16 for the MMA.
//  * Warps are merged in shared memory; splits of one (sequence, kv head) are
//    merged in FP32 by the last CTA to finish (an atomic counter in the
//    workspace; no CTA ever waits for another).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fp8kv.h"
#include "ptx.cuh"

namespace fp8kv {

constexpr int kBS = 16;                    // tokens per page (block_size)
constexpr int kNCW = 4;                    // consumer warps per CTA
constexpr int kThreads = (kNCW + 1) * 32;  // + one producer warp
constexpr int kStages = 12;                // ring slots; a multiple of kNCW
constexpr int kStageHalf = 4096;           // K bytes (and V bytes) per stage
constexpr int kStageBytes = 2 * kStageHalf;
constexpr int kMaxPagesPerSplit = 512;
constexpr int kCtasPerSm = 2;
constexpr uint64_t kWaitLimitNs = 500000000ull;  // 0.5 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
    const uint16_t* q;          // bf16 [B, Hq, D]
    const int32_t* block_tables;
    const int32_t* seq_lens;
    uint16_t* out;              // bf16 [B, Hq, D]
    uint32_t* err;              // workspace error word
    int32_t* counters;          // [B*Hkv]
    float2* part_ml;            // [B*Hkv, max_splits, 8]  (max, sum) in log2 units
    float* part_o;              // [B*Hkv, max_splits, G, D]
    int64_t num_blocks;
    int max_blocks_per_seq;
    int max_seq_len;
    int num_q_heads;
    int num_kv_heads;
    int pages_per_split;
    int max_splits;
    int window;
    float score_scale;          // sm_scale * k_scale * log2(e)
    float v_scale;
};

template <int D>
struct Geo {
    static constexpr int PAGE = kBS * D;                // bytes of one K (or V) page
    static constexpr int PPS = kStageHalf / PAGE;       // pages per stage: 4, 2, 1
    static constexpr int HALVES = D >= 128 ? D / 128 : 1;
    static constexpr int ROWB = D >= 128 ? 128 : D;     // bytes per smem row of one TMA box
    static constexpr int BOX = kBS * ROWB;              // bytes of one TMA box
    static constexpr int KS = D / 16;                   // k-steps of the score MMA
    static constexpr int MT = D / 16;                   // m-tiles of the value MMA
    static constexpr int KW = ROWB / 4;                 // K bytes a thread reads per row per box
    static constexpr int KSH = KW / 4;                  // k-steps per box
    static constexpr int VW = ROWB / 8;                 // V bytes a thread reads per token per box
    static constexpr int MTH = VW / 2;                  // m-tiles per box
    static_assert(PPS >= 1 && PPS * PAGE == kStageHalf, "stage must hold whole pages");
};

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

__device__ __forceinline__ void report(uint32_t* err, uint32_t code) { atomicCAS(err, 0u, code); }

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kNCW * 32) : "memory"); }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeArgs a) {
    using Gm = Geo<D>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned ring (the swizzle pattern is a function of address
    // bits 4..9); offsetting the shared array keeps the address space known.
    uint8_t* ring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(ring + kStages * kStageBytes);
    uint64_t* empty_bar = full_bar + kStages;
    int32_t* blk = reinterpret_cast<int32_t*>(empty_bar + kStages);
    int* flag = blk + kMaxPagesPerSplit;

    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // A previous CTA gave up a wait: skip the work, the call is already failed.
    if (*reinterpret_cast<volatile uint32_t*>(a.err) == FP8KV_ERR_TIMEOUT) return;
    int L = a.seq_lens[b];
    if (L < 0 || L > a.max_seq_len) {  // outside the caller's contract: clamp and report
        if (split == 0 && hk == 0 && threadIdx.x == 0) report(a.err, FP8KV_ERR_INVALID_ARG);
        L = L < 0 ? 0 : a.max_seq_len;
    }
    const int lo = (a.window > 0 && L > a.window) ? L - a.window : 0;
    const int first_pg = lo / kBS;
    const int n_pages = L > 0 ? (L - 1) / kBS - first_pg + 1 : 0;
    const int nsplit = n_pages > 0 ? (n_pages + a.pages_per_split - 1) / a.pages_per_split : 1;
    if (split >= nsplit) return;
    const int hq0 = hk * G;
    uint16_t* out_bh = a.out + (static_cast<int64_t>(b) * a.num_q_heads + hq0) * D;
    if (n_pages == 0) {
        for (int i = tid; i < G * D; i += kThreads) out_bh[i] = 0;
        return;
    }
    const int pg_begin = first_pg + split * a.pages_per_split;
    const int npg = min(a.pages_per_split, first_pg + n_pages - pg_begin);
    const int n_stages = (npg + Gm::PPS - 1) / Gm::PPS;

    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq + pg_begin;
    for (int i = tid; i < npg; i += kThreads) {
        int id = __ldg(bt + i);
        if (id < 0 || id >= a.num_blocks) {
            report(a.err, FP8KV_ERR_INVALID_ARG);
            id = 0;
        }
        blk[i] = id;
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kNCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            const uint64_t pol = l2_policy_evict_first();
            int issued = 0;
            for (int st = 0; st < n_stages; ++st) {
                const int slot = st % kStages;
                if (st >= kStages &&
                    !mbar_wait_bounded(&empty_bar[slot], ((st / kStages) & 1) ^ 1, kWaitLimitNs)) {
                    report(a.err, FP8KV_ERR_TIMEOUT);
                    break;
                }
                const int p0 = st * Gm::PPS;
                const int np = min(Gm::PPS, npg - p0);
                mbar_arrive_expect_tx(&full_bar[slot], static_cast<uint32_t>(np * 2 * Gm::PAGE));
                uint8_t* kst = ring + slot * kStageBytes;
                uint8_t* vst = kst + kStageHalf;
                for (int p = 0; p < np; ++p) {
                    const int id = blk[p0 + p];
#pragma unroll
                    for (int h = 0; h < Gm::HALVES; ++h) {
                        tma_load_4d(kst + p * Gm::PAGE + h * Gm::BOX, &tmK, &full_bar[slot], h * 128, 0, hk, id, pol);
                        tma_load_4d(vst + p * Gm::PAGE + h * Gm::BOX, &tmV, &full_bar[slot], h * 128, 0, hk, id, pol);
                    }
                }
                issued = st + 1;
            }
            // Only after a failed wait can copies still be in flight while
            // consumers have stopped waiting: drain them (bounded) before exit.
            if (issued < n_stages) {
                for (int st = issued > kStages ? issued - kStages : 0; st < issued; ++st)
                    mbar_wait_bounded(&full_bar[st % kStages], (st / kStages) & 1, kWaitLimitNs);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int gid = lane >> 2, tig = lane & 3;

    // Query fragments (B operand of the score MMA), pre-scaled per head by a
    // power of two so the f16 copy is exact; the score is scaled back later.
    uint32_t qf[Gm::KS][2];
    float cs[2];
    {
        uint32_t qw[Gm::HALVES][Gm::KSH][2];
        float qmax = 0.f;
#pragma unroll
        for (int hh = 0; hh < Gm::HALVES; ++hh) {
#pragma unroll
            for (int c = 0; c < Gm::KW / 8; ++c) {  // KW dims = 2*KW bytes of bf16 = KW/8 uint4
                uint4 v = make_uint4(0, 0, 0, 0);
                if (gid < G)
                    v = __ldg(reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(b) * a.num_q_heads + hq0 + gid) * D +
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
        // shift so that the largest |q| of the head lands in [2^14, 2^15)
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
            cs[j] = a.score_scale * __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
        }
    }

    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};
    float o[Gm::MT][4];
#pragma unroll
    for (int mt = 0; mt < Gm::MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int st = warp; st < n_stages; st += kNCW) {
        const int slot = st % kStages;
        if (!mbar_wait_bounded(&full_bar[slot], (st / kStages) & 1, kWaitLimitNs)) {
            report(a.err, FP8KV_ERR_TIMEOUT);
            break;
        }
        const int p0 = st * Gm::PPS;
        const int np = min(Gm::PPS, npg - p0);
        const uint8_t* kst = ring + slot * kStageBytes;
        const uint8_t* vst = kst + kStageHalf;
        const int tok_base = (pg_begin + p0) * kBS;

        // ---- scores S^T[token][head] = K Q^T
        float s[Gm::PPS][4];
#pragma unroll
        for (int p = 0; p < Gm::PPS; ++p) {
            s[p][0] = s[p][1] = s[p][2] = s[p][3] = 0.f;
            if (p < np) {
#pragma unroll
                for (int hh = 0; hh < Gm::HALVES; ++hh) {
                    const uint8_t* box = kst + p * Gm::PAGE + hh * Gm::BOX;
                    uint32_t w0[Gm::KSH], w1[Gm::KSH];
#pragma unroll
                    for (int c = 0; c < Gm::KW / 16; ++c) {
                        const uint4 x = *reinterpret_cast<const uint4*>(box + swz<Gm::ROWB>(gid, tig * Gm::KW + 16 * c));
                        const uint4 y = *reinterpret_cast<const uint4*>(box + swz<Gm::ROWB>(gid + 8, tig * Gm::KW + 16 * c));
                        w0[4 * c + 0] = x.x; w0[4 * c + 1] = x.y; w0[4 * c + 2] = x.z; w0[4 * c + 3] = x.w;
                        w1[4 * c + 0] = y.x; w1[4 * c + 1] = y.y; w1[4 * c + 2] = y.z; w1[4 * c + 3] = y.w;
                    }
#pragma unroll
                    for (int kk = 0; kk < Gm::KSH; ++kk) {
                        uint32_t af[4];
                        e4m3x4_to_f16x2x2(w0[kk], af[0], af[2]);
                        e4m3x4_to_f16x2x2(w1[kk], af[1], af[3]);
                        mma_16816(s[p], af, qf[hh * Gm::KSH + kk][0], qf[hh * Gm::KSH + kk][1], s[p]);
                    }
                }
            }
        }

        // ---- mask, scale to log2 units, stage maximum
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int p = 0; p < Gm::PPS; ++p)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tok = tok_base + p * kBS + gid + 8 * e;
                const bool valid = (p < np) && tok >= lo && tok < L;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float t = valid ? s[p][2 * e + j] * cs[j] : -INFINITY;
                    s[p][2 * e + j] = t;
                    mx[j] = fmaxf(mx[j], t);
                }
            }
        float alpha[2], muse[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
            const float mn = fmaxf(m[j], mx[j]);
            muse[j] = mn == -INFINITY ? 0.f : mn;
            alpha[j] = fast_exp2(m[j] - muse[j]);
            m[j] = mn;
        }

        // ---- probabilities -> f16 B fragments of the value MMA
        uint32_t pb[Gm::PPS][2];
        float lsum[2] = {0.f, 0.f};
#pragma unroll
        for (int p = 0; p < Gm::PPS; ++p) {
            const float p00 = fast_exp2(s[p][0] - muse[0]);
            const float p01 = fast_exp2(s[p][1] - muse[1]);
            const float p10 = fast_exp2(s[p][2] - muse[0]);
            const float p11 = fast_exp2(s[p][3] - muse[1]);
            lsum[0] += p00 + p10;
            lsum[1] += p01 + p11;
            pb[p][0] = movmatrix_trans(pack_f16x2(p00, p01));
            pb[p][1] = movmatrix_trans(pack_f16x2(p10, p11));
        }
        l[0] = l[0] * alpha[0] + lsum[0];
        l[1] = l[1] * alpha[1] + lsum[1];

        // ---- P.V tile of this stage: O^T[dim][head] = V^T P^T
        float ot[Gm::MT][4];
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) ot[mt][0] = ot[mt][1] = ot[mt][2] = ot[mt][3] = 0.f;
#pragma unroll
        for (int p = 0; p < Gm::PPS; ++p) {
            if (p < np) {
                const int t0 = tok_base + p * kBS;
                const bool edge = t0 < lo || t0 + kBS > L;
#pragma unroll
                for (int hh = 0; hh < Gm::HALVES; ++hh) {
                    const uint8_t* box = vst + p * Gm::PAGE + hh * Gm::BOX;
                    uint32_t v[4][Gm::VW / 4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int row = 2 * tig + (r & 1) + 8 * (r >> 1);
                        if constexpr (Gm::VW == 16) {
                            const uint4 x = *reinterpret_cast<const uint4*>(box + swz<Gm::ROWB>(row, gid * 16));
                            v[r][0] = x.x; v[r][1] = x.y; v[r][2] = x.z; v[r][3] = x.w;
                        } else {
                            const uint2 x = *reinterpret_cast<const uint2*>(box + swz<Gm::ROWB>(row, gid * 8));
                            v[r][0] = x.x; v[r][1] = x.y;
                        }
                        if (edge) {
                            const int tok = t0 + row;
                            if (tok < lo || tok >= L) {
#pragma unroll
                                for (int w = 0; w < Gm::VW / 4; ++w) v[r][w] = 0u;  // never let stale NaN codes meet p = 0
                            }
                        }
                    }
#pragma unroll
                    for (int mtl = 0; mtl < Gm::MTH; ++mtl) {
                        const uint32_t sel = (mtl & 1) ? 0x7362u : 0x5140u;
                        const uint32_t x01 = byte_perm(v[0][mtl >> 1], v[1][mtl >> 1], sel);
                        const uint32_t x23 = byte_perm(v[2][mtl >> 1], v[3][mtl >> 1], sel);
                        uint32_t af[4];
                        e4m3x4_to_f16x2x2(x01, af[0], af[1]);
                        e4m3x4_to_f16x2x2(x23, af[2], af[3]);
                        mma_16816(ot[hh * Gm::MTH + mtl], af, pb[p][0], pb[p][1], ot[hh * Gm::MTH + mtl]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);

        // ---- fold the tile into the FP32 accumulators
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
            o[mt][0] = fmaf(o[mt][0], alpha[0], ot[mt][0]);
            o[mt][1] = fmaf(o[mt][1], alpha[1], ot[mt][1]);
            o[mt][2] = fmaf(o[mt][2], alpha[0], ot[mt][2]);
            o[mt][3] = fmaf(o[mt][3], alpha[1], ot[mt][3]);
        }
    }

#pragma unroll
    for (int j = 0; j < 2; ++j) {
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 4);
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 8);
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 16);
    }

    // ---------------------------------------------------------------- merge warps
    consumer_sync();  // every consumer is done with the ring: reuse it
    float* Ow = reinterpret_cast<float*>(ring);   // [kNCW][8][D]
    float* mw = Ow + kNCW * 8 * D;                // [kNCW][8]
    float* lw = mw + kNCW * 8;
#pragma unroll
    for (int mt = 0; mt < Gm::MT; ++mt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int dim = (mt / Gm::MTH) * 128 + Gm::VW * gid + 2 * (mt % Gm::MTH) + e;
#pragma unroll
            for (int j = 0; j < 2; ++j) Ow[(warp * 8 + 2 * tig + j) * D + dim] = o[mt][2 * e + j];
        }
    if (gid == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mw[warp * 8 + 2 * tig + j] = m[j];
            lw[warp * 8 + 2 * tig + j] = l[j];
        }
    }
    consumer_sync();

    const int bh = b * a.num_kv_heads + hk;
    const int64_t part = static_cast<int64_t>(bh) * a.max_splits + split;
    for (int idx = tid; idx < G * D; idx += kNCW * 32) {
        const int h = idx / D, i = idx - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) M = fmaxf(M, mw[w * 8 + h]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float O = 0.f, Lh = 0.f;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) {
            const float f = fast_exp2(mw[w * 8 + h] - Mu);
            O += Ow[(w * 8 + h) * D + i] * f;
            Lh += lw[w * 8 + h] * f;
        }
        if (nsplit == 1) {
            out_bh[idx] = f32_to_bf16(Lh > 0.f ? O * a.v_scale / Lh : 0.f);
        } else {
            a.part_o[part * G * D + idx] = O;
            if (i == 0) a.part_ml[part * 8 + h] = make_float2(M, Lh);
        }
    }
    if (nsplit == 1) return;

    // ---------------------------------------------------------------- merge splits
    __threadfence();
    consumer_sync();
    if (tid == 0) {
        const int old = atomicAdd(&a.counters[bh], 1);
        *flag = (old == nsplit - 1);
    }
    consumer_sync();
    if (!*flag) return;
    __threadfence();
    const int64_t base = static_cast<int64_t>(bh) * a.max_splits;
    for (int idx = tid; idx < G * D; idx += kNCW * 32) {
        const int h = idx / D;
        float M = -INFINITY;
        for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(&a.part_ml[(base + sp) * 8 + h].x));
        const float Mu = M == -INFINITY ? 0.f : M;
        float O = 0.f, Lh = 0.f;
        for (int sp = 0; sp < nsplit; ++sp) {
            const float2 ml = __ldcg(&a.part_ml[(base + sp) * 8 + h]);
            const float f = fast_exp2(ml.x - Mu);
            O += __ldcg(&a.part_o[(base + sp) * G * D + idx]) * f;
            Lh += ml.y * f;
        }
        out_bh[idx] = f32_to_bf16(Lh > 0.f ? O * a.v_scale / Lh : 0.f);
    }
    if (tid == 0) a.counters[bh] = 0;  // ready for the next call
}

// ---------------------------------------------------------------- host side

struct Plan {
    int pages_per_split;
    int max_splits;
};

int stage_pages(int D) { return kStageHalf / (kBS * D); }

Plan make_plan(int batch, int num_kv_heads, int D, int max_seq_len, int window, int sms) {
    Plan p{1, 1};
    if (max_seq_len <= 0) return p;
    const int all_pages = (max_seq_len + kBS - 1) / kBS;
    int max_pages = all_pages;
    if (window > 0 && window < max_seq_len) max_pages = std::min(all_pages, (window + kBS - 1) / kBS + 1);
    const int64_t units = static_cast<int64_t>(batch) * num_kv_heads;
    const int64_t target = static_cast<int64_t>(sms) * kCtasPerSm * 2;
    int64_t splits = std::max<int64_t>(1, (target + units - 1) / units);
    const int sp = stage_pages(D);
    int pps = static_cast<int>((max_pages + splits - 1) / splits);
    pps = std::max(sp, (pps + sp - 1) / sp * sp);
    if (pps > kMaxPagesPerSplit) pps = kMaxPagesPerSplit;
    p.pages_per_split = pps;
    p.max_splits = (max_pages + pps - 1) / pps;
    return p;
}

struct WsLayout {
    size_t counters, ml, o, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int batch, int num_q_heads, int num_kv_heads, int D, const Plan& p) {
    const size_t units = static_cast<size_t>(batch) * num_kv_heads;
    const int G = num_q_heads / num_kv_heads;
    WsLayout w;
    w.counters = 256;
    w.ml = w.counters + align256(units * sizeof(int32_t));
    w.o = w.ml + align256(units * p.max_splits * 8 * sizeof(float2));
    w.total = w.o + align256(units * p.max_splits * G * D * sizeof(float));
    return w;
}

int device_sms(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
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
bool make_cache_map(CUtensorMap* m, const void* base, int64_t num_blocks, int Hkv, int D) {
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

constexpr size_t smem_bytes() {
    return 1024 + kStages * kStageBytes + 2 * kStages * sizeof(uint64_t) + kMaxPagesPerSplit * sizeof(int32_t) + 64;
}

template <int D, int G>
cudaError_t launch(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeArgs& a, int batch, int Hkv,
                   cudaStream_t stream) {
    // The shared-memory opt-in is per device; remember which devices have it.
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit == 0 || !(done_mask.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(paged_decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_bytes()));
        if (e != cudaSuccess) return e;
        done_mask.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.max_splits, Hkv, batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes();
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, G>, mk, mv, a);
}

template <int D>
cudaError_t launch_g(int G, const CUtensorMap& mk, const CUtensorMap& mv, const DecodeArgs& a, int batch, int Hkv,
                     cudaStream_t s) {
    switch (G) {
        case 1: return launch<D, 1>(mk, mv, a, batch, Hkv, s);
        case 2: return launch<D, 2>(mk, mv, a, batch, Hkv, s);
        case 4: return launch<D, 4>(mk, mv, a, batch, Hkv, s);
        case 8: return launch<D, 8>(mk, mv, a, batch, Hkv, s);
        default: return cudaErrorInvalidValue;
    }
}

bool supported(int head_dim, int block_size, int G) {
    return (head_dim == 64 || head_dim == 128 || head_dim == 256) && block_size == kBS &&
           (G == 1 || G == 2 || G == 4 || G == 8);
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
    const Plan p = make_plan(batch, num_kv_heads, head_dim, max_seq_len, window, sms);
    return ws_layout(batch, num_q_heads, num_kv_heads, head_dim, p).total;
}

extern "C" fp8kv_status fp8kv_paged_decode(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                           int64_t num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                                           const int32_t* seq_lens, int max_seq_len, int batch, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size, float k_scale,
                                           float v_scale, float sm_scale, int window, void* out, void* workspace,
                                           size_t workspace_bytes, void* stream) {
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (batch < 0 || batch > 65535 || num_kv_heads < 1 || num_kv_heads > 65535 || num_q_heads < 1 ||
        num_q_heads % num_kv_heads != 0 || max_seq_len < 0 || num_blocks < 1 || max_blocks_per_seq < 0)
        return FP8KV_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !(k_scale > 0) || !std::isfinite(v_scale) || !(v_scale > 0) ||
        !std::isfinite(sm_scale))
        return FP8KV_ERR_INVALID_ARG;
    const int G = num_q_heads / num_kv_heads;
    if (!supported(head_dim, block_size, G)) return FP8KV_ERR_UNSUPPORTED;
    if (num_blocks >= (INT64_C(1) << 31) || num_blocks * num_kv_heads >= (INT64_C(1) << 31))
        return FP8KV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_blocks_per_seq) * block_size < max_seq_len) return FP8KV_ERR_INVALID_ARG;
    if (batch == 0) return FP8KV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return FP8KV_ERR_INVALID_ARG;
    if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(out)) return FP8KV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return FP8KV_ERR_INVALID_ARG;
    int sms = 0;
    if (device_sms(&sms) != 0) return FP8KV_ERR_CUDA;
    const Plan p = make_plan(batch, num_kv_heads, head_dim, max_seq_len, window, sms);
    const WsLayout w = ws_layout(batch, num_q_heads, num_kv_heads, head_dim, p);
    if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FP8KV_ERR_WORKSPACE;

    CUtensorMap mk, mv;
    if (!make_cache_map(&mk, k_cache, num_blocks, num_kv_heads, head_dim) ||
        !make_cache_map(&mv, v_cache, num_blocks, num_kv_heads, head_dim))
        return FP8KV_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecodeArgs a;
    a.q = static_cast<const uint16_t*>(q);
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = static_cast<uint16_t*>(out);
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.counters = reinterpret_cast<int32_t*>(ws + w.counters);
    a.part_ml = reinterpret_cast<float2*>(ws + w.ml);
    a.part_o = reinterpret_cast<float*>(ws + w.o);
    a.num_blocks = num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.max_seq_len = max_seq_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.pages_per_split = p.pages_per_split;
    a.max_splits = p.max_splits;
    a.window = window > 0 ? window : 0;
    a.score_scale = sm_scale * k_scale * kLog2e;
    a.v_scale = v_scale;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (head_dim) {
        case 64: e = launch_g<64>(G, mk, mv, a, batch, num_kv_heads, s); break;
        case 128: e = launch_g<128>(G, mk, mv, a, batch, num_kv_heads, s); break;
        default: e = launch_g<256>(G, mk, mv, a, batch, num_kv_heads, s); break;
    }
    return e == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA;
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

// 8 MiB covers every workload shape exercised here (the largest, 16 x 32K
// tokens at head_dim 256, needs about 5 MiB).  Every device that loads the
// library holds this array until the process exits.
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
    if (batch < 0 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0 || max_seq_len < 0)
        return FP8KV_ERR_INVALID_ARG;
    if (!supported(head_dim, block_size, num_q_heads / num_kv_heads)) return FP8KV_ERR_UNSUPPORTED;
    if (batch == 0) return FP8KV_OK;
    int sms = 0;
    if (device_sms(&sms) != 0) return FP8KV_ERR_CUDA;
    const Plan p = make_plan(batch, num_kv_heads, head_dim, max_seq_len, window, sms);
    const WsLayout w = ws_layout(batch, num_q_heads, num_kv_heads, head_dim, p);
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
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FP8KV_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FP8KV_OK
               : FP8KV_ERR_CUDA;
}

extern "C" fp8kv_status fp8kv_read_error(void* workspace, uint32_t* code, void* stream) {
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
