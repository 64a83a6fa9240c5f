// Chunked-prefill attention over the paged fp8 (E4M3) KV cache, for sm_103a.
//
// What it computes: the new query tokens of each sequence (the last q_len of
// its seq_len tokens, already appended to the cache) attend causally over the
// sequence's cached keys, optionally within a sliding window: query position
// p reads keys [max(0, p + 1 - window), p].  This is the prefill pass that
// reads the same fp8 cache as decode (gpusmith.com, "FP8 KV Cache
// Quantization: Capacity Gains and Accuracy Risk", "Attention backend
// interactions"; phantomic12 vLLM-blog summary, "ACCURACY AT LONG CONTEXT":
// the P.V contraction runs over the context, so partial sums live in real
// FP32 registers).
//
// How: one CTA per (tile of 32 query rows, kv head, sequence).  A query row is
// a (token, query head) pair of the kv head's group; each of the 4 warps owns
// 8 rows, the n side of the m16n8k16 MMA, exactly as the decode kernel uses
// its g heads.  The tile's key pages (from the first row's window start to
// the last row's position) stream through a double-buffered shared-memory
// page (cp.async, the 128-byte swizzle of a TMA box, so fragment loads are
// conflict-free).  Per page and warp: S^T = K Q^T (keys on the m side), the
// causal/window mask, an online softmax per row in log2 units, P rounded to
// f16, the page's O^T = V^T P^T tile in fresh accumulators, then folded into
// FP32 registers (O = O * alpha + tile).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fp8kv.h"
#include "ptx.cuh"

namespace fp8kv {
namespace prefill {

constexpr int kBS = 16;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = 8;
constexpr int kRows = kWarps * kRowsPerWarp;  // query rows per CTA
constexpr float kLog2e = 1.4426950408889634f;

struct Args {
    const uint16_t* q;           // bf16 [sum q_len, Hq, D], packed by sequence
    const uint8_t* k_cache;      // E4M3 [num_blocks, Hkv, 16, D]
    const uint8_t* v_cache;
    const int32_t* block_tables; // [B, max_blocks_per_seq]
    const int32_t* seq_lens;     // [B]
    const int32_t* q_starts;     // [B + 1] cumulative query-row offsets
    uint16_t* out;               // bf16 [sum q_len, Hq, D]
    uint32_t* err;               // error word (first word of a decode workspace), or null
    int64_t num_blocks;
    int64_t num_q_tokens;        // rows of q and out
    int max_blocks_per_seq;
    int max_seq_len;
    int max_q_len;
    int num_q_heads;
    int num_kv_heads;
    int window;
    float score_scale;           // sm_scale * k_scale * log2(e)
    float v_scale;
};

// Byte offset of (row r, byte o) inside a 16-row box with rows of ROWB bytes,
// 128-byte (or 64-byte) swizzle: the layout a TMA box lands in.
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int r, int o) {
    if constexpr (ROWB == 128)
        return r * 128 + ((((o >> 4) ^ (r & 7)) << 4) | (o & 15));
    else
        return r * 64 + ((((o >> 4) ^ ((r >> 1) & 3)) << 4) | (o & 15));
}

template <int D>
struct Geo {
    static constexpr int ROWB = D >= 128 ? 128 : D;  // bytes per box row
    static constexpr int HALVES = D >= 128 ? D / 128 : 1;
    static constexpr int BOX = kBS * ROWB;
    static constexpr int PAGE = kBS * D;
    static constexpr int KS = D / 16;                // k-steps of the score MMA
    static constexpr int MT = D / 16;                // m-tiles of the value MMA
    static constexpr int KW = ROWB / 4;              // K bytes a thread reads per row per box
    static constexpr int KSH = KW / 4;               // k-steps per box
    static constexpr int VW = ROWB / 8;              // V bytes a thread reads per key per box
    static constexpr int MTH = VW / 2;               // m-tiles per box
};

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void report(uint32_t* err, uint32_t code) {
    if (err) atomicCAS(err, 0u, code);
}

// Page `pg` of (sequence row `bt`, kv head hk) into the smem page (K and V).
// A block id outside [0, num_blocks) reads block 0 and is reported.
template <int D>
__device__ __forceinline__ void load_page(const Args& a, const int32_t* bt, int hk, int pg, uint8_t* ks, uint8_t* vs) {
    using Gm = Geo<D>;
    int id = __ldg(bt + pg);
    if (id < 0 || id >= a.num_blocks) {
        if (threadIdx.x == 0) report(a.err, FP8KV_ERR_INVALID_ARG);
        id = 0;
    }
    const int64_t base = (static_cast<int64_t>(id) * a.num_kv_heads + hk) * Gm::PAGE;
    constexpr int kChunks = Gm::PAGE / 16;
    for (int i = threadIdx.x; i < kChunks; i += kThreads) {
        const int r = i / (D / 16), c = i % (D / 16);
        const int h = (c * 16) / Gm::ROWB, o = (c * 16) % Gm::ROWB;
        const uint32_t dst = h * Gm::BOX + swz<Gm::ROWB>(r, o);
        cp_async16(ks + dst, a.k_cache + base + r * D + c * 16);
        cp_async16(vs + dst, a.v_cache + base + r * D + c * 16);
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) paged_prefill_kernel(const Args a) {
    using Gm = Geo<D>;
    __shared__ __align__(1024) uint8_t sk[2][Gm::PAGE];
    __shared__ __align__(1024) uint8_t sv[2][Gm::PAGE];
    griddep_wait();                // inputs may come from the previous grid on the stream
    griddep_launch_dependents();
    const int b = blockIdx.z, hk = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const int q0 = __ldg(a.q_starts + b);
    const int L_in = __ldg(a.seq_lens + b);
    const int L = L_in < 0 ? 0 : (L_in > a.max_seq_len ? a.max_seq_len : L_in);
    const int n_in = __ldg(a.q_starts + b + 1) - q0;   // query tokens of this sequence
    int n = n_in < 0 ? 0 : min(n_in, min(L, a.max_q_len));
    if (q0 < 0 || q0 + static_cast<int64_t>(n) > a.num_q_tokens) n = 0;   // never touch rows outside q / out
    if (L != L_in || n != n_in) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) report(a.err, FP8KV_ERR_INVALID_ARG);
    }
    const int rows = n * G;
    const int R0 = blockIdx.x * kRows;
    if (R0 >= rows) return;
    const int p_first = L - n + R0 / G;                                  // position of the tile's first token
    const int p_last = L - n + (min(R0 + kRows, rows) - 1) / G;
    const int lo_first = (a.window > 0 && p_first + 1 > a.window) ? p_first + 1 - a.window : 0;
    const int pg0 = lo_first / kBS, pg1 = p_last / kBS;
    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;

    // ---- this warp's 8 query rows as f16 B fragments (power-of-two pre-scale
    // per row so the f16 copy of the bf16 value is exact), as in decode
    const int rw = R0 + warp * kRowsPerWarp;   // first row of the warp
    uint32_t qf[Gm::KS][2];
    float cs[2];
    {
        const int myrow = rw + gid;            // the row whose q this lane's B fragment column holds
        const bool ok = myrow < rows;
        const int tok = ok ? myrow / G : 0, hq = hk * G + (ok ? myrow % G : 0);
        const uint16_t* qrow = a.q + (static_cast<int64_t>(q0 + tok) * a.num_q_heads + hq) * D;
        uint32_t qw[Gm::HALVES][Gm::KSH][2];
        float qmax = 0.f;
#pragma unroll
        for (int hh = 0; hh < Gm::HALVES; ++hh)
#pragma unroll
            for (int c = 0; c < Gm::KW / 8; ++c) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (ok) v = __ldg(reinterpret_cast<const uint4*>(qrow + hh * 128 + tig * Gm::KW) + c);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    qw[hh][c * 2 + e / 2][e % 2] = w4[e];
                    qmax = fmaxf(qmax, fmaxf(fabsf(bf16_to_f32(w4[e] & 0xFFFF)), fabsf(bf16_to_f32(w4[e] >> 16))));
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
            cs[j] = a.score_scale * __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
        }
    }
    // positions and window starts of this lane's two accumulator rows (2*tig, 2*tig+1)
    int pq[2], lq[2];
    bool rv[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int r = rw + 2 * tig + j;
        rv[j] = r < rows;
        pq[j] = L - n + (rv[j] ? r / G : 0);
        lq[j] = (a.window > 0 && pq[j] + 1 > a.window) ? pq[j] + 1 - a.window : 0;
    }

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[Gm::MT][4];
#pragma unroll
    for (int mt = 0; mt < Gm::MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    load_page<D>(a, bt, hk, pg0, sk[0], sv[0]);
    cp_async_commit();
    for (int pg = pg0; pg <= pg1; ++pg) {
        const int buf = (pg - pg0) & 1;
        if (pg < pg1) load_page<D>(a, bt, hk, pg + 1, sk[buf ^ 1], sv[buf ^ 1]);
        cp_async_commit();
        cp_async_wait_1();             // this page has landed (the next may still be in flight)
        __syncthreads();
        const uint8_t* kst = sk[buf];
        const uint8_t* vst = sv[buf];
        const int t0 = pg * kBS;

        // ---- scores S^T[key][row] = K Q^T
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int hh = 0; hh < Gm::HALVES; ++hh) {
            const uint8_t* box = kst + hh * Gm::BOX;
            uint32_t w0[Gm::KW / 4], w1[Gm::KW / 4];
#pragma unroll
            for (int cc = 0; cc < Gm::KW / 16; ++cc) {
                const uint4 x = *reinterpret_cast<const uint4*>(box + swz<Gm::ROWB>(gid, tig * Gm::KW + 16 * cc));
                const uint4 y = *reinterpret_cast<const uint4*>(box + swz<Gm::ROWB>(gid + 8, tig * Gm::KW + 16 * cc));
                w0[4 * cc + 0] = x.x; w0[4 * cc + 1] = x.y; w0[4 * cc + 2] = x.z; w0[4 * cc + 3] = x.w;
                w1[4 * cc + 0] = y.x; w1[4 * cc + 1] = y.y; w1[4 * cc + 2] = y.z; w1[4 * cc + 3] = y.w;
            }
#pragma unroll
            for (int kk = 0; kk < Gm::KSH; ++kk) {
                uint32_t af[4];
                e4m3x4_to_f16x2x2(w0[kk], af[0], af[2]);
                e4m3x4_to_f16x2x2(w1[kk], af[1], af[3]);
                mma_16816(sc, af, qf[hh * Gm::KSH + kk][0], qf[hh * Gm::KSH + kk][1], sc);
            }
        }

        // ---- causal / window mask, scale to log2 units, page maximum per row
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
            const int key = t0 + gid + 8 * e2;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const bool valid = rv[j] && key <= pq[j] && key >= lq[j];
                const float t = valid ? sc[2 * e2 + j] * cs[j] : -INFINITY;
                sc[2 * e2 + j] = t;
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
        const float p00 = fast_exp2(sc[0] - muse[0]), p01 = fast_exp2(sc[1] - muse[1]);
        const float p10 = fast_exp2(sc[2] - muse[0]), p11 = fast_exp2(sc[3] - muse[1]);
        l[0] = l[0] * alpha[0] + (p00 + p10);
        l[1] = l[1] * alpha[1] + (p01 + p11);
        const uint32_t pb0 = movmatrix_trans(pack_f16x2(p00, p01));
        const uint32_t pb1 = movmatrix_trans(pack_f16x2(p10, p11));

        // ---- P.V tile of this page: O^T[dim][row] = V^T P^T; keys that no row
        // of the tile attends read as zero codes (stale NaN codes never meet p = 0)
        const int kmin = lo_first, kmax = p_last;
        float ot[Gm::MT][4];
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) ot[mt][0] = ot[mt][1] = ot[mt][2] = ot[mt][3] = 0.f;
#pragma unroll
        for (int hh = 0; hh < Gm::HALVES; ++hh) {
            const uint8_t* box = vst + hh * Gm::BOX;
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
                const int key = t0 + row;
                if (key < kmin || key > kmax) {
#pragma unroll
                    for (int ww = 0; ww < Gm::VW / 4; ++ww) v[r][ww] = 0u;
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
                mma_16816(ot[hh * Gm::MTH + mtl], af, pb0, pb1, ot[hh * Gm::MTH + mtl]);
            }
        }
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
            o[mt][0] = fmaf(o[mt][0], alpha[0], ot[mt][0]);
            o[mt][1] = fmaf(o[mt][1], alpha[1], ot[mt][1]);
            o[mt][2] = fmaf(o[mt][2], alpha[0], ot[mt][2]);
            o[mt][3] = fmaf(o[mt][3], alpha[1], ot[mt][3]);
        }
        __syncthreads();               // every warp is done with this buffer before it is refilled
    }
    cp_async_wait_0();

    // ---- normalise and write this lane's two rows
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 4);
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 8);
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 16);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int r = rw + 2 * tig + j;
        if (r >= rows) continue;
        const float sc_out = l[j] > 0.f ? a.v_scale / l[j] : 0.f;
        uint16_t* orow = a.out + (static_cast<int64_t>(q0 + r / G) * a.num_q_heads + hk * G + r % G) * D;
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt)
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int dim = (mt / Gm::MTH) * 128 + Gm::VW * gid + 2 * (mt % Gm::MTH) + e2;
                orow[dim] = f32_to_bf16(o[mt][2 * e2 + j] * sc_out);
            }
    }
}

template <int D>
cudaError_t launch_g(int G, const Args& a, dim3 grid, cudaStream_t s) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (G) {
        case 1: return cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, 1>, a);
        case 2: return cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, 2>, a);
        case 4: return cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, 4>, a);
        case 8: return cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, 8>, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace prefill
}  // namespace fp8kv

extern "C" fp8kv_status fp8kv_paged_prefill(const void* q, int64_t num_q_tokens, const uint8_t* k_cache, const uint8_t* v_cache,
                                            int64_t num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                                            const int32_t* seq_lens, const int32_t* q_starts, int max_q_len,
                                            int max_seq_len, int batch, int num_q_heads, int num_kv_heads,
                                            int head_dim, int block_size, float k_scale, float v_scale,
                                            float sm_scale, int window, void* out, void* workspace,
                                            void* stream) {
    using namespace fp8kv::prefill;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (batch < 0 || batch > 65535 || num_kv_heads < 1 || num_kv_heads > 65535 || num_q_heads < 1 ||
        num_q_heads % num_kv_heads != 0 || max_seq_len < 0 || max_q_len < 0 || max_q_len > max_seq_len ||
        num_blocks < 1 || max_blocks_per_seq < 0 || num_q_tokens < 0)
        return FP8KV_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !(k_scale > 0) || !std::isfinite(v_scale) || !(v_scale > 0) ||
        !std::isfinite(sm_scale))
        return FP8KV_ERR_INVALID_ARG;
    const int G = num_q_heads / num_kv_heads;
    if (!(head_dim == 64 || head_dim == 128 || head_dim == 256) || block_size != kBS ||
        !(G == 1 || G == 2 || G == 4 || G == 8))
        return FP8KV_ERR_UNSUPPORTED;
    if (num_blocks >= (INT64_C(1) << 31) || num_blocks * num_kv_heads >= (INT64_C(1) << 31))
        return FP8KV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_blocks_per_seq) * block_size < max_seq_len) return FP8KV_ERR_INVALID_ARG;
    if (batch == 0 || max_q_len == 0 || num_q_tokens == 0) return FP8KV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !q_starts || !out) return FP8KV_ERR_INVALID_ARG;
    if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(out)) return FP8KV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(q_starts) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 3u))
        return FP8KV_ERR_INVALID_ARG;
    const int64_t tiles = (static_cast<int64_t>(max_q_len) * G + kRows - 1) / kRows;
    if (tiles > INT32_MAX) return FP8KV_ERR_UNSUPPORTED;
    Args a;
    a.q = static_cast<const uint16_t*>(q);
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.q_starts = q_starts;
    a.out = static_cast<uint16_t*>(out);
    a.num_blocks = num_blocks;
    a.num_q_tokens = num_q_tokens;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.max_seq_len = max_seq_len;
    a.max_q_len = max_q_len;
    a.err = static_cast<uint32_t*>(workspace);
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.window = window > 0 ? window : 0;
    a.score_scale = sm_scale * k_scale * kLog2e;
    a.v_scale = v_scale;
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(num_kv_heads), static_cast<unsigned>(batch));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (head_dim) {
        case 64: e = launch_g<64>(G, a, grid, s); break;
        case 128: e = launch_g<128>(G, a, grid, s); break;
        default: e = launch_g<256>(G, a, grid, s); break;
    }
    return e == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA;
}
