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
// How: a unit is (tile of 128 query rows, kv head, sequence); a query row is
// a (token, query head) pair of the kv head's group.  Three kernels on the
// 5th-generation tensor cores (tcgen05.mma from swizzled f16 tiles in shared
// memory, S in tensor memory, one row per thread (TMEM lane) for the online
// softmax):
//  * paged_prefill_ws_kernel (d = 64 and 128, chunks of two or more tiles):
//    two tiles per CTA, 128-key stages, and warp roles -- converter warps,
//    one MMA-issuing thread, a softmax warpgroup per tile -- that overlap
//    through mbarriers.  P goes to tensor memory as the value MMA's A
//    operand, and the tensor cores carry O across stages in FP32;
//  * paged_prefill_ws1_kernel (d = 256): one tile per CTA with the same kind
//    of roles; each stage's P.V tile, computed in fresh FP32 accumulators, is
//    folded into an FP32 accumulator in tensor memory (O = O * alpha + tile,
//    IEEE FMA);
//  * paged_prefill_tc_kernel (single-tile chunks at d = 64 and 128): one
//    tile per CTA, its four warps taking each stage's steps in turn, the
//    fold into registers.
// See the comments above them.  When the units are too few to fill the GPU,
// each unit's key range is split over several CTAs whose FP32 partials (row
// maximum, row sum, unnormalised output) a second kernel merges (split plan:
// prefill_plan.h).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "fp8kv.h"
#include "trace.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"
#include "prefill_plan.h"

namespace fp8kv {

int device_sms(int* sms);  // SM count of the current device (paged_decode.cu)

namespace prefill {

constexpr int kBS = 16;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsTC = 128;            // query rows per unit of the tcgen05 kernel (one per TMEM lane)
constexpr size_t kHeader = 256;         // error word, then the partials
constexpr float kLog2e = 1.4426950408889634f;

struct Args {
    const uint16_t* q;           // bf16 [num_q_tokens, Hq, D], packed by sequence
    const uint8_t* k_cache;      // E4M3 [num_blocks, Hkv, 16, D]
    const uint8_t* v_cache;
    const int32_t* block_tables; // [B, max_blocks_per_seq]
    const int32_t* seq_lens;     // [B]
    const int32_t* q_starts;     // [B + 1] cumulative query-row offsets
    uint16_t* out;               // bf16 [num_q_tokens, Hq, D]
    uint32_t* err;               // error word
    float* part_o;               // [units][splits][rows][D] unnormalised FP32 outputs
    float2* part_ml;             // [units][splits][rows] (row maximum in log2 units, row sum)
    int64_t num_blocks;
    int64_t num_q_tokens;
    int max_blocks_per_seq;
    int max_seq_len;
    int max_q_len;
    int num_q_heads;
    int num_kv_heads;
    int tiles;                   // query tiles per (sequence, kv head)
    int rows;                    // query rows per tile (kRowsTC)
    int splits;                  // CTAs per unit
    int window;
    float score_scale;           // sm_scale * k_scale * log2(e)
    float v_scale;
    // Failure-path test hook of the tcgen05 kernel (fp8kv_debug_paged_prefill_stall):
    // CTA (0, 0, 0) never issues the score MMAs of stage stall_stage (-1: none),
    // and the MMA waits give up after wait_ns (normally 0.5 s).
    uint64_t wait_ns;
    int stall_stage;
};

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void report(uint32_t* err, uint32_t code) { atomicCAS(err, 0u, code); }

// What one (tile, kv head, sequence) covers: its query rows and the key
// range the rows attend, from the device-side lengths (clamped; an entry
// outside the documented bounds is reported when `report_errors`).
struct Unit {
    int q0;          // first packed query row of the sequence
    int L;           // keys in the cache
    int n;           // query tokens of the sequence
    int rows;        // n * G
    int R0;          // first row of the tile
    int kmin, kmax;  // keys the tile attends (inclusive)
};

template <int G>
__device__ __forceinline__ bool make_unit(const Args& a, int b, int tile, bool report_errors, Unit& u) {
    u.q0 = __ldg(a.q_starts + b);
    const int L_in = __ldg(a.seq_lens + b);
    u.L = L_in < 0 ? 0 : min(L_in, a.max_seq_len);
    const int n_in = __ldg(a.q_starts + b + 1) - u.q0;
    int n = n_in < 0 ? 0 : min(n_in, min(u.L, a.max_q_len));
    if (u.q0 < 0 || u.q0 + static_cast<int64_t>(n) > a.num_q_tokens) n = 0;  // never touch rows outside q / out
    if (report_errors && (u.L != L_in || n != n_in)) report(a.err, FP8KV_ERR_INVALID_ARG);
    u.n = n;
    u.rows = n * G;
    u.R0 = tile * a.rows;
    if (u.R0 >= u.rows) return false;
    const int p_first = u.L - n + u.R0 / G;
    u.kmax = u.L - n + (min(u.R0 + a.rows, u.rows) - 1) / G;
    u.kmin = (a.window > 0 && p_first + 1 > a.window) ? p_first + 1 - a.window : 0;
    return true;
}

// ---------------------------------------------------------------------------
// The one-tile prefill kernel, on the 5th-generation tensor cores (tcgen05):
// single-tile chunks at d = 64 and 128 (written for d = 256 too).
//
// A unit is 128 query rows; thread t of the 4 warps owns row t, which is
// TMEM lane t of both accumulators.  Per stage of 64 keys (4 pages):
//   1. the stage's fp8 K and V pages (cp.async into a 2-slot staging ring)
//      are converted into f16 operand tiles, K as 64 keys x d and V
//      transposed as d x 64 keys, both K-major with the 128-byte swizzle
//      (the Q tile, 128 rows x d, is built once);
//   2. one thread issues S = Q K^T (M = 128, N = 64: d/16 MMAs of K = 16)
//      into TMEM columns [0, 64) and commits it to an mbarrier;
//   3. each thread loads its row of S, masks it, runs the online softmax in
//      log2 units and writes its row of P (f16) over the K tile, which the
//      finished score MMAs no longer need;
//   4. one thread issues O_tile = P V (M = 128, N = d: 4 MMAs) into TMEM
//      columns [64, 64 + d);
//   5. each thread loads its row of O_tile and folds it into FP32 registers,
//      O = O * alpha + O_tile: the two-level accumulation.
// At d = 256 a row's 256 FP32 outputs do not fit in registers beside its
// scores: the accumulator lives in TMEM columns [256, 512) (zeroed at the
// start), and steps 4-5 run twice per stage, for output dimensions [0, 128)
// and [128, 256), through the same 128 O_tile columns.  The fold is then a
// tcgen05.ld of the tile and of the accumulator, the FMA, and a tcgen05.st
// back.  The operand tiles take 192 KB of shared memory: one CTA per SM.
// Every tcgen05.ld/st is warp-collective: all threads execute them, also
// those whose row lies past the tile's last.
namespace tcg {
constexpr int kKeys = 64;                       // keys per stage
constexpr int kPages = kKeys / kBS;             // 4 pages per stage
constexpr uint64_t kWaitNs = 500000000ull;      // bounded waits on the MMA barriers
}  // namespace tcg

template <int D>
struct TcGeo {
    static constexpr int NB = D / 64;                             // 128-byte atom columns of a d-wide f16 row
    static constexpr int QT = 0;                                  // Q tile: NB blocks x 128 rows x 128 B
    static constexpr int KT = QT + NB * 128 * 128;                // K tile: NB blocks x 64 keys x 128 B; P aliases it
    static constexpr int KP = NB * tcg::kKeys * 128 > 128 * 128 ? NB * tcg::kKeys * 128 : 128 * 128;
    static constexpr int VT = KT + KP;                            // V^T tile: d rows x 128 B
    static constexpr int STG = VT + D * 128;                      // staging: 2 slots x (K, V: 64 keys x d bytes)
    static constexpr int SLOT = 2 * tcg::kKeys * D;
    static constexpr int SMEM = STG + 2 * SLOT;                   // 192 KB at d = 256, 96 KB at 128, 56 KB at 64
    // TMEM: S at [0, 64), O_tile at [64, 64 + min(d, 128)); at d = 256 the
    // FP32 output accumulator (d columns) at [256, 512)
    static constexpr uint32_t COLS = D == 256 ? 512 : (D == 128 ? 256 : 128);
    static constexpr int ON = D == 256 ? 128 : D;                 // N of one P.V MMA group
    static constexpr uint32_t OACC = 256;                         // d = 256: accumulator columns
    static constexpr int CPR = D / 16;                            // 16-byte chunks per staged key row
    static constexpr int VPASS = D == 256 ? 2 : 1;                // passes of the V^T conversion
};

// Staged key row k, 16-byte chunk c: the XOR keeps the conversions' reads free
// of bank conflicts (8 consecutive keys per K read; 8 keys 8 apart per V read).
// (At d = 256 a key row is 256 bytes: the XOR of the low 3 chunk bits keeps
// each 128-byte half's chunks apart in the same way.)
template <int D>
__device__ __forceinline__ uint32_t stg_k(int k, int c) {
    if constexpr (D >= 128) return k * D + ((c ^ (k & 7)) << 4);
    else return k * 64 + ((c ^ ((k >> 1) & 3)) << 4);
}
template <int D>
__device__ __forceinline__ uint32_t stg_v(int k, int c) {
    if constexpr (D >= 128) return k * D + ((c ^ ((k >> 3) & 7)) << 4);
    else return k * 64 + ((c ^ ((k >> 3) & 3)) << 4);
}
// The same address for a key k = 8 kb + i of key block kb.
template <int D>
__device__ __forceinline__ uint32_t stg_v_kb(int k, int kb, int c) {
    if constexpr (D >= 128) return k * D + ((c ^ kb) << 4);
    else return k * 64 + ((c ^ (kb & 3)) << 4);
}

// Pages [pg, pg + np) of (block-table row bt, kv head hk) into staging slot
// `dst` (K rows, then V rows).  A block id outside [0, num_blocks) reads
// block 0 and is reported.
template <int D>
__device__ __forceinline__ void load_stage_tc(const Args& a, const int32_t* bt, int hk, int pg, int np, uint32_t dst,
                                              int tid = threadIdx.x) {
    using Tg = TcGeo<D>;
    constexpr int kChunks = kBS * Tg::CPR;      // 16-byte chunks per page
    for (int i = tid; i < np * kChunks; i += 128) {
        const int p = i / kChunks, ci = i % kChunks;
        int id = __ldg(bt + pg + p);
        if (id < 0 || id >= a.num_blocks) {
            if (ci == 0) report(a.err, FP8KV_ERR_INVALID_ARG);
            id = 0;
        }
        const int64_t base = (static_cast<int64_t>(id) * a.num_kv_heads + hk) * (kBS * D);
        const int r = ci / Tg::CPR, c = ci % Tg::CPR, k = p * kBS + r;
        cp_async16(dst + stg_k<D>(k, c), a.k_cache + base + r * D + c * 16);
        cp_async16(dst + tcg::kKeys * D + stg_v<D>(k, c), a.v_cache + base + r * D + c * 16);
    }
}

// One stage's operand tiles, by 128 threads (thread index ct): the staged
// fp8 K rows of the stage's 64 keys into the f16 K tile at kt (64 keys x d,
// K-major, 128-byte swizzle) and the staged V rows, transposed, into the f16
// V^T tile at vt (d rows x 64 keys).  Keys outside [kmin, kmax] or past the
// stage's np pages become zeros in V^T (their scores are masked).
template <int D, int KS = tcg::kKeys * 128>   // KS: bytes between the K tile's 128-byte atom columns
__device__ __forceinline__ void convert_stage_k(const uint8_t* stg, uint8_t* kt, int ct) {
    // K: thread ct converts CH staged chunks (16 dims each) of key ct & 63
    {
        constexpr int CH = D / 32;                        // 8 at d = 256, 4 at 128, 2 at 64
        const int k = ct & 63, part = ct >> 6;
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            const int c = part * CH + i;                   // staged chunk: dims 16c .. 16c + 15
            const uint4 x = *reinterpret_cast<const uint4*>(stg + stg_k<D>(k, c));
            uint32_t f[8];
            e4m3x4_to_f16x2x2(x.x, f[0], f[1]);
            e4m3x4_to_f16x2x2(x.y, f[2], f[3]);
            e4m3x4_to_f16x2x2(x.z, f[4], f[5]);
            e4m3x4_to_f16x2x2(x.w, f[6], f[7]);
            const int j = 2 * (c & 3);                     // f16 chunk within the 64-dim block c / 4
            uint8_t* dst = kt + (c >> 2) * KS + k * 128;
            *reinterpret_cast<uint4*>(dst + ((j ^ (k & 7)) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<uint4*>(dst + (((j + 1) ^ (k & 7)) << 4)) = make_uint4(f[4], f[5], f[6], f[7]);
        }
    }
}

template <int D>
__device__ __forceinline__ void convert_stage_v(const uint8_t* stg, uint8_t* vt, int ct, int t0, int np, int kmin,
                                                int kmax) {
    using Tg = TcGeo<D>;
    // V^T: thread ct (ct < d) converts keys [8kb, 8kb + 8) x dims [8db, 8db + 8)
#pragma unroll
    for (int vp = 0; vp < Tg::VPASS; ++vp)
        if (D >= 128 || ct < D) {
            const int kb = ct & 7, db = (ct >> 3) + 16 * vp;
            uint32_t w[8][2];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = 8 * kb + i, key = t0 + k;
                uint2 x = make_uint2(0, 0);
                if (k < np * kBS && key >= kmin && key <= kmax)
                    x = *reinterpret_cast<const uint2*>(stg + tcg::kKeys * D + stg_v_kb<D>(k, kb, db >> 1) +
                                                        8 * (db & 1));
                w[i][0] = x.x;
                w[i][1] = x.y;
            }
            uint32_t vt4[8][4];   // [dim][key pair]
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2)
#pragma unroll
                for (int hw = 0; hw < 2; ++hw) {
                    e4m3x4_to_f16x2x2(byte_perm(w[2 * i2][hw], w[2 * i2 + 1][hw], 0x5140u), vt4[4 * hw + 0][i2],
                                      vt4[4 * hw + 1][i2]);
                    e4m3x4_to_f16x2x2(byte_perm(w[2 * i2][hw], w[2 * i2 + 1][hw], 0x7362u), vt4[4 * hw + 2][i2],
                                      vt4[4 * hw + 3][i2]);
                }
#pragma unroll
            for (int dd = 0; dd < 8; ++dd)
                *reinterpret_cast<uint4*>(vt + (8 * db + dd) * 128 + ((kb ^ dd) << 4)) =
                    make_uint4(vt4[dd][0], vt4[dd][1], vt4[dd][2], vt4[dd][3]);
        }
}

template <int D>
__device__ __forceinline__ void convert_stage(const uint8_t* stg, uint8_t* kt, uint8_t* vt, int ct, int t0, int np,
                                              int kmin, int kmax) {
    convert_stage_k<D>(stg, kt, ct);
    convert_stage_v<D>(stg, vt, ct, t0, np, kmin, kmax);
}

template <int D, int G>
__global__ void __launch_bounds__(128) paged_prefill_tc_kernel(const Args a) {
    using Tg = TcGeo<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tmem_base;
    uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(sm);
    const int t = threadIdx.x, warp = t >> 5;
    if (t == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    griddep_wait();                // inputs may come from the previous grid on the stream
    griddep_launch_dependents();
    const int b = blockIdx.z, hk = blockIdx.y;
    const int tile = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
    Unit u;
    if (!make_unit<G>(a, b, tile, blockIdx.x == 0 && hk == 0 && t == 0, u)) return;

    // ---- this split's key pages; the first stage's copies start now
    const int pg0 = u.kmin / kBS, np_all = u.kmax / kBS - pg0 + 1;
    const int sp0 = pg0 + static_cast<int>(static_cast<int64_t>(split) * np_all / a.splits);
    const int sp1 = pg0 + static_cast<int>(static_cast<int64_t>(split + 1) * np_all / a.splits);
    const int nst = (sp1 - sp0 + tcg::kPages - 1) / tcg::kPages;
    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
    if (nst > 0) load_stage_tc<D>(a, bt, hk, sp0, min(tcg::kPages, sp1 - sp0), sb + Tg::STG);
    cp_async_commit();

    // ---- this thread's query row into the Q tile as f16, pre-scaled by a
    // power of two so that the copy of the bf16 values is exact
    const int r = u.R0 + t;
    const bool rv = r < u.rows;
    float cs;
    int pq, lq;
    {
        // 16-byte chunks of the bf16 row (8 values each), in passes of at
        // most 16 chunks (d = 256 reads its row twice: maximum, then copy)
        constexpr int NC = D / 8, PC = NC > 16 ? 16 : NC, NP = NC / PC;
        const int tok = rv ? r / G : 0, hq = hk * G + (rv ? r % G : 0);
        const uint4* qrow = reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(u.q0 + tok) * a.num_q_heads + hq) * D);
        uint4 qv[PC];
        float qmax = 0.f;
#pragma unroll
        for (int ps = 0; ps < NP; ++ps)
#pragma unroll
            for (int c = 0; c < PC; ++c) {
                qv[c] = rv ? __ldg(qrow + ps * PC + c) : make_uint4(0, 0, 0, 0);
                const uint32_t w4[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    qmax = fmaxf(qmax, fmaxf(fabsf(bf16_to_f32(w4[e] & 0xFFFF)), fabsf(bf16_to_f32(w4[e] >> 16))));
            }
        int shift = 0;
        if (qmax > 0.f) {
            const int e = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFF) - 127;
            shift = max(-100, min(100, 14 - e));
        }
        const float up = __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
#pragma unroll
        for (int ps = 0; ps < NP; ++ps)
#pragma unroll
            for (int cc = 0; cc < PC; ++cc) {
                const int c = ps * PC + cc;
                if (NP > 1) qv[cc] = rv ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
                const uint32_t w4[4] = {qv[cc].x, qv[cc].y, qv[cc].z, qv[cc].w};
                uint32_t f[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    f[e] = pack_f16x2(bf16_to_f32(w4[e] & 0xFFFF) * up, bf16_to_f32(w4[e] >> 16) * up);
                *reinterpret_cast<uint4*>(sm + Tg::QT + (c >> 3) * 16384 + t * 128 + (((c & 7) ^ (t & 7)) << 4)) =
                    make_uint4(f[0], f[1], f[2], f[3]);
            }
        cs = a.score_scale * __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
        pq = u.L - u.n + (rv ? r / G : 0);
        lq = (a.window > 0 && pq + 1 > a.window) ? pq + 1 - a.window : 0;
    }
    // the warp's first position and its last valid row's window start: a
    // stage of keys in [wlo1, wpos0] is attended in full by every row of the warp
    const int wr0 = u.R0 + warp * 32;
    const int wpos0 = u.L - u.n + wr0 / G;
    const int wpos1 = u.L - u.n + max(0, min(wr0 + 31, u.rows - 1)) / G;
    const int wlo1 = (a.window > 0 && wpos1 + 1 > a.window) ? wpos1 + 1 - a.window : 0;

    if (warp == 0) tc::alloc(&tmem_base, Tg::COLS);
    tc::fence_proxy_async_smem();  // the Q tile is read by the tensor cores
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = tmem_base;
    const uint32_t tm_row = tm + (static_cast<uint32_t>(warp * 32) << 16);   // this warp's 32 lanes

    float m = -INFINITY, l = 0.f;
    // FP32 output accumulator: registers at d <= 128, TMEM columns at d = 256
    float o[D <= 128 ? D : 1];
#pragma unroll
    for (int d = 0; d < (D <= 128 ? D : 1); ++d) o[d] = 0.f;
    if constexpr (D == 256) {
        float z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tc::st32(tm_row + Tg::OACC + 32 * c, z);
        tc::wait_st();
    }
    bool fail = false;
    for (int st = 0; st < nst; ++st) {
        cp_async_wait<0>();            // this stage's copies (this thread's) have landed
        if (__syncthreads_or(fail)) {  // ... everyone's; the previous stage's tiles are free
            fail = true;
            break;
        }
        if (st + 1 < nst)
            load_stage_tc<D>(a, bt, hk, sp0 + (st + 1) * tcg::kPages,
                             min(tcg::kPages, sp1 - sp0 - (st + 1) * tcg::kPages),
                             sb + Tg::STG + ((st + 1) & 1) * Tg::SLOT);
        cp_async_commit();
        const int pgs = sp0 + st * tcg::kPages;
        const int np = min(tcg::kPages, sp1 - pgs);
        const int t0 = pgs * kBS;
        const uint8_t* stg = sm + Tg::STG + (st & 1) * Tg::SLOT;

        // ---- 1. the stage's K and V^T operand tiles
        convert_stage<D>(stg, sm + Tg::KT, sm + Tg::VT, t, t0, np, u.kmin, u.kmax);
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();

        // ---- 2. S = Q K^T
        const bool stalled = st == a.stall_stage && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
        if (t == 0 && !stalled) {
            tc::fence_after_sync();
            constexpr uint32_t id_s = tc::idesc_f16_f32(128, tcg::kKeys);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (ks & 3) * 32;
                tc::mma_f16(tm, tc::desc_k_sw128(sb + Tg::QT + (ks >> 2) * 16384 + off),
                            tc::desc_k_sw128(sb + Tg::KT + (ks >> 2) * (tcg::kKeys * 128) + off), id_s, ks > 0);
            }
            tc::commit(&bars[0]);
        }
        const bool ok_s = mbar_wait_bounded(&bars[0], st & 1, a.wait_ns);
        tc::fence_after_sync();

        // ---- 3. this row's scores -> online softmax -> its row of P
        float sv[64];
        tc::ld32(tm_row, *reinterpret_cast<float(*)[32]>(sv));
        tc::ld32(tm_row + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
        tc::wait_ld(*reinterpret_cast<float(*)[32]>(sv));
        tc::wait_ld(*reinterpret_cast<float(*)[32]>(sv + 32));
        const bool interior = np == tcg::kPages && t0 + tcg::kKeys - 1 <= wpos0 && t0 >= wlo1;
        float mx = -INFINITY;
        if (interior) {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                sv[j] *= cs;
                mx = fmaxf(mx, sv[j]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const int key = t0 + j;
                const bool valid = j < np * kBS && rv && key >= lq && key <= pq;
                sv[j] = valid ? sv[j] * cs : -INFINITY;
                mx = fmaxf(mx, sv[j]);
            }
        }
        const float mn = fmaxf(m, mx);
        const float muse = mn == -INFINITY ? 0.f : mn;
        const float alpha = fast_exp2(m - muse);
        m = mn;
        float ls = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t pw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p0 = fast_exp2(sv[8 * c + 2 * e] - muse), p1 = fast_exp2(sv[8 * c + 2 * e + 1] - muse);
                ls += p0 + p1;
                pw[e] = pack_f16x2(p0, p1);
            }
            *reinterpret_cast<uint4*>(sm + Tg::KT + t * 128 + ((c ^ (t & 7)) << 4)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
        l = l * alpha + ls;
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        if (__syncthreads_or(!ok_s)) {
            fail = true;
            break;
        }

        // ---- 4. O_tile = P V (d = 256: two halves of 128 output dimensions,
        // one after the other through the same O_tile columns)
#pragma unroll
        for (int oh = 0; oh < D / Tg::ON; ++oh) {
            if (oh > 0) {  // every row's load of the previous half is done before the MMA overwrites it
                tc::fence_before_sync();
                if (__syncthreads_or(fail)) {
                    fail = true;
                    break;
                }
            }
            if (t == 0) {
                tc::fence_after_sync();
                constexpr uint32_t id_o = tc::idesc_f16_f32(128, Tg::ON);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_f16(tm + 64, tc::desc_k_sw128(sb + Tg::KT + ks * 32),
                                tc::desc_k_sw128(sb + Tg::VT + oh * Tg::ON * 128 + ks * 32), id_o, ks > 0);
                tc::commit(&bars[1]);
            }
            // bars[1] completes D / ON times per stage
            fail = !mbar_wait_bounded(&bars[1], (st * (D / Tg::ON) + oh) & 1, a.wait_ns);
            tc::fence_after_sync();

            // ---- 5. fold this row's tile into the FP32 accumulator,
            // O = O * alpha + O_tile (IEEE FMA, FP32): the two-level accumulation
#pragma unroll
            for (int c = 0; c < Tg::ON / 32; ++c) {
                float x[32];
                tc::ld32(tm_row + 64 + 32 * c, x);
                if constexpr (D <= 128) {
                    tc::wait_ld(x);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[32 * c + j] = fmaf(o[32 * c + j], alpha, x[j]);
                } else {
                    float y[32];
                    const uint32_t acc = tm_row + Tg::OACC + oh * Tg::ON + 32 * c;
                    tc::ld32(acc, y);
                    tc::wait_ld(x);
                    tc::wait_ld(y);
#pragma unroll
                    for (int j = 0; j < 32; ++j) y[j] = fmaf(y[j], alpha, x[j]);
                    tc::st32(acc, y);
                }
            }
            if constexpr (D == 256) tc::wait_st();
        }
        // a failed wait (possibly in some threads only) ends the loop at the
        // next stage's __syncthreads_or, where every thread agrees
        tc::fence_before_sync();
    }
    cp_async_wait<0>();
    fail = __syncthreads_or(fail);
    if (fail) {
        if (t == 0) report(a.err, FP8KV_ERR_TIMEOUT);
    } else if (D == 256 || rv) {
        if constexpr (D == 256) {
            // The accumulator moves from TMEM to registers, 32 columns at a
            // time.  tcgen05.ld is warp-collective (.sync.aligned): every
            // thread loads, including those whose row is past the tile's
            // last, and only valid rows store.
            const int64_t unit = (static_cast<int64_t>(b) * a.num_kv_heads + hk) * a.tiles + tile;
            const float so = l > 0.f ? a.v_scale / l : 0.f;
            uint4* orow = reinterpret_cast<uint4*>(a.out + (static_cast<int64_t>(u.q0 + r / G) * a.num_q_heads + hk * G + r % G) * D);
            const int64_t slot = (unit * a.splits + split) * a.rows + t;
            float4* po = reinterpret_cast<float4*>(a.part_o + slot * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float x[32];
                tc::ld32(tm_row + Tg::OACC + 32 * c, x);
                tc::wait_ld(x);
                if (!rv) continue;
                if (a.splits == 1) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        orow[4 * c + i] = make_uint4(pack_bf16x2(x[8 * i] * so, x[8 * i + 1] * so),
                                                     pack_bf16x2(x[8 * i + 2] * so, x[8 * i + 3] * so),
                                                     pack_bf16x2(x[8 * i + 4] * so, x[8 * i + 5] * so),
                                                     pack_bf16x2(x[8 * i + 6] * so, x[8 * i + 7] * so));
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        po[8 * c + i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
                }
            }
            if (rv && a.splits > 1) a.part_ml[slot] = make_float2(m, l);
        } else {
        const int64_t unit = (static_cast<int64_t>(b) * a.num_kv_heads + hk) * a.tiles + tile;
        if (a.splits == 1) {
            const float so = l > 0.f ? a.v_scale / l : 0.f;
            uint4* orow = reinterpret_cast<uint4*>(a.out + (static_cast<int64_t>(u.q0 + r / G) * a.num_q_heads + hk * G + r % G) * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c)
                orow[c] = make_uint4(pack_bf16x2(o[8 * c] * so, o[8 * c + 1] * so), pack_bf16x2(o[8 * c + 2] * so, o[8 * c + 3] * so),
                                     pack_bf16x2(o[8 * c + 4] * so, o[8 * c + 5] * so), pack_bf16x2(o[8 * c + 6] * so, o[8 * c + 7] * so));
        } else {
            const int64_t slot = (unit * a.splits + split) * a.rows + t;
            float4* po = reinterpret_cast<float4*>(a.part_o + slot * D);
#pragma unroll
            for (int c = 0; c < D / 4; ++c) po[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            a.part_ml[slot] = make_float2(m, l);
        }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::dealloc(tm, Tg::COLS);
    }
}

// ---------------------------------------------------------------------------
// The warp-specialised prefill kernel (d = 64 and 128, chunks of at least two
// tiles).
//
// A CTA takes two consecutive query tiles of one (kv head, sequence), 256
// rows, and one key range, walked in stages of 128 keys (two staging
// granules of 64 keys); each stage's K and V operand tiles are built once for
// both tiles.  The roles run concurrently and hand work over through
// mbarriers (every wait bounded):
//   * warps 8-11 (converters): cp.async the fp8 pages of stage s + 1 into a
//     two-stage staging ring, then convert stage s's K into the f16 K tile
//     (once the score MMAs of stage s - 1 have read it) and its V, transposed,
//     into one of two f16 V^T tiles (once the value MMAs of stage s - 2 have);
//   * one thread of warp 12 (the MMA issuer), tile by tile in turn: once the
//     tile's P of stage s is written, O += P V (A = P read from TMEM) into the
//     tile's FP32 accumulator in TMEM, then S = Q K^T of stage s + 1 (N = 128
//     keys) into the tile's S columns.  The tensor cores run the MMAs one
//     thread issues in issue order, so S(s + 1) overwrites the columns only
//     after P V of stage s has read P from them;
//   * warps 0-3 and 4-7 (one warpgroup per tile, thread = row = TMEM lane):
//     load the row of S, online softmax in log2 units, write the row of P
//     (f16, two per column) over the S just read, in TMEM.  The running
//     maximum the row's O and l refer to moves only when the stage's maximum
//     exceeds it by more than 2^8 (so P stays below 2^8); then, before the
//     stage's P V, the warp rescales its rows of O in TMEM.  The tensor-core
//     sums of O continue across stages in FP32.
// The two tiles ping-pong: while one tile's warpgroup runs its softmax, the
// tensor cores run the other tile's P V and next S, and the converters
// prepare the next stage.
namespace ws {
constexpr int kTiles = 2;                  // query tiles of 128 rows per CTA
constexpr int kConvWarp0 = 8;              // warps 8-11 convert
constexpr int kMmaWarp = 12;               // warp 12 issues the MMAs
constexpr int kThreads = 13 * 32;
constexpr int kKeys = 128;                 // keys per stage
constexpr int kGran = kKeys / tcg::kKeys;  // staging granules (64 keys, 4 pages) per stage
constexpr int kPages = kKeys / kBS;        // pages per stage
constexpr int kStg = 2;                    // stages in the fp8 staging ring
constexpr int kConvBar = 2;                // named barrier of the converter warps
constexpr float kRescaleLog2 = 8.f;        // a row's maximum moves when exceeded by more than this
}  // namespace ws

template <int D>
struct WsGeo {
    static constexpr int NB = D / 64;
    static constexpr int QTB = NB * 128 * 128;          // one Q tile: 128 rows x d
    static constexpr int KAT = ws::kKeys * 128;         // one 128-byte atom column of the K tile (128 keys)
    static constexpr int KTB = NB * KAT;                // the K tile: 128 keys x d
    static constexpr int VAT = D * 128;                 // one atom column of the V^T tile: d rows x 64 keys
    static constexpr int VTB = ws::kGran * VAT;         // the V^T tile: d rows x 128 keys
    static constexpr int GSLOT = 2 * tcg::kKeys * D;    // one fp8 staging granule: 64 K rows, then 64 V rows
    static constexpr int QT = 0;
    static constexpr int KT = QT + ws::kTiles * QTB;
    static constexpr int VT = KT + KTB;
    static constexpr int STG = VT + 2 * VTB;
    static constexpr int SMEM = STG + ws::kStg * ws::kGran * GSLOT;   // 224 KB at d = 128, 112 KB at 64
    // TMEM per tile: S in [0, 128) (P written over its first 64 columns), the
    // FP32 output accumulator in [128, 128 + d)
    static constexpr uint32_t OC = ws::kKeys;
    static constexpr uint32_t TC = 256;
    static constexpr uint32_t COLS = ws::kTiles * TC;   // 512
    static_assert(D == 64 || D == 128, "the warp-specialised two-tile kernel covers d = 64 and 128");
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier over n threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Packed FP32 pairs (sm_100 family): d = a * b + c and d += a, lane by lane,
// one instruction for two values.
__device__ __forceinline__ void fma_f32x2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                          float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add_f32x2(float& d0, float& d1, float a0, float a1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1));
}

// A bounded mbarrier wait that also gives up as soon as another thread of the
// CTA has given up (the shared abort flag); the first to run out sets it.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            return false;
        }
    }
}

template <int D, int G>
__global__ void __launch_bounds__(ws::kThreads, 1) paged_prefill_ws_kernel(const Args a) {
    using Wg = WsGeo<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t k_full, k_empty, v_full[2], v_empty[2];
    __shared__ uint64_t s_full[ws::kTiles], p_full[ws::kTiles];
    __shared__ uint64_t done_bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_sh;
    volatile int* abort_flag = &abort_sh;
    uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        mbar_init(&k_full, 128);           // the converter threads
        mbar_init(&k_empty, 1);            // tcgen05.commit
        for (int j = 0; j < 2; ++j) {      // one per V^T tile
            mbar_init(&v_full[j], 128);
            mbar_init(&v_empty[j], 1);
        }
        for (int i = 0; i < ws::kTiles; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);    // the tile's warpgroup
        }
        mbar_init(&done_bar, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    griddep_wait();                // inputs may come from the previous grid on the stream
    griddep_launch_dependents();
    const int b = blockIdx.z, hk = blockIdx.y;
    const int pair = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
    Unit u[ws::kTiles];
    if (!make_unit<G>(a, b, 2 * pair, blockIdx.x == 0 && hk == 0 && tid == 0, u[0])) return;
    const bool has1 = make_unit<G>(a, b, 2 * pair + 1, false, u[1]);
    // the pair's keys: the first tile's window starts first, the second tile's rows end last
    const int kmin = u[0].kmin, kmax = has1 ? u[1].kmax : u[0].kmax;
    const int pg0 = kmin / kBS, np_all = kmax / kBS - pg0 + 1;
    const int sp0 = pg0 + static_cast<int>(static_cast<int64_t>(split) * np_all / a.splits);
    const int sp1 = pg0 + static_cast<int>(static_cast<int64_t>(split + 1) * np_all / a.splits);
    const int nst = (sp1 - sp0 + ws::kPages - 1) / ws::kPages;
    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;

    // ---- role set-up: the warpgroups build their Q tiles; the converters
    // start the first stages' copies
    const int ti = warp >> 2;                     // the tile of warps 0-7
    const int tt = tid & 127;                     // row within the tile
    const Unit& uu = u[ti < ws::kTiles ? ti : 0];
    const int r = uu.R0 + tt;
    const bool rv = warp < 8 && (ti == 0 || has1) && r < uu.rows;
    float cs = 0.f;
    int pq = 0, lq = 0, wpos0 = 0, wlo1 = 0;
    if (warp < 8) {
        // the bf16 row in 16-byte chunks, read twice (its largest magnitude,
        // then the copy) to keep few of them in registers
        constexpr int NC = D / 8;
        const int tok = rv ? r / G : 0, hq = hk * G + (rv ? r % G : 0);
        const uint4* qrow =
            reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(uu.q0 + tok) * a.num_q_heads + hq) * D);
        float qmax = 0.f;
#pragma unroll 4
        for (int c = 0; c < NC; ++c) {
            const uint4 qv = rv ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
            const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                qmax = fmaxf(qmax, fmaxf(fabsf(bf16_to_f32(w4[e] & 0xFFFF)), fabsf(bf16_to_f32(w4[e] >> 16))));
        }
        int shift = 0;
        if (qmax > 0.f) {
            const int e = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFF) - 127;
            shift = max(-100, min(100, 14 - e));
        }
        // a negative score scale goes into Q, so that the row's scale cs is
        // positive and the maximum of the scaled scores is cs times the raw maximum
        const float up = (a.score_scale < 0.f ? -1.f : 1.f) * __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
#pragma unroll 4
        for (int c = 0; c < NC; ++c) {
            const uint4 qv = rv ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
            const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
            uint32_t f[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                f[e] = pack_f16x2(bf16_to_f32(w4[e] & 0xFFFF) * up, bf16_to_f32(w4[e] >> 16) * up);
            *reinterpret_cast<uint4*>(sm + Wg::QT + ti * Wg::QTB + (c >> 3) * 16384 + tt * 128 +
                                      (((c & 7) ^ (tt & 7)) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
        }
        cs = fabsf(a.score_scale) * __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
        pq = uu.L - uu.n + (rv ? r / G : 0);
        lq = (a.window > 0 && pq + 1 > a.window) ? pq + 1 - a.window : 0;
        // the warp's first position and its last valid row's window start: a
        // stage of keys in [wlo1, wpos0] is attended in full by every row of the warp
        const int wr0 = uu.R0 + (warp & 3) * 32;
        wpos0 = uu.L - uu.n + wr0 / G;
        const int wpos1 = uu.L - uu.n + max(0, min(wr0 + 31, uu.rows - 1)) / G;
        wlo1 = (a.window > 0 && wpos1 + 1 > a.window) ? wpos1 + 1 - a.window : 0;
        if (!(ti == 0 || has1)) wpos0 = -1;       // no valid row: never the fast path
    }
    // the converters' copies of stage s: granule g's pages into staging granule
    // (s % kStg) * kGran + g; one commit group per stage
    auto load_stage = [&](int s, int ct) {
        if (s < nst)
            for (int g = 0; g < ws::kGran; ++g) {
                const int pg = sp0 + s * ws::kPages + g * tcg::kPages;
                const int npg = min(tcg::kPages, sp1 - pg);
                if (npg > 0)
                    load_stage_tc<D>(a, bt, hk, pg, npg, sb + Wg::STG + ((s % ws::kStg) * ws::kGran + g) * Wg::GSLOT,
                                     ct);
            }
        cp_async_commit();
    };
    if (warp >= ws::kConvWarp0 && warp < ws::kMmaWarp) load_stage(0, tid - ws::kConvWarp0 * 32);
    if (warp == 0) tc::alloc(&tmem_base, Wg::COLS);
    tc::fence_proxy_async_smem();  // the Q tiles are read by the tensor cores
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = tmem_base;

    // A pair whose second tile has no rows still runs it (its rows are
    // masked and never stored): skipping the tile's roles measured 10% slower
    // on full pairs, through the branch structure it adds.
    float m = -INFINITY, l = 0.f;
    if (warp < 8) {
        // ---------------------------------------------------------- softmax and fold of tile ti
        const uint32_t trow = tm + ti * Wg::TC + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        {
            float z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tc::st32(trow + Wg::OC + 32 * c, z);
            tc::wait_st();
        }
        for (int st = 0; st < nst; ++st) {
            // S of stage st is in; its commit also covers the P V of stage
            // st - 1, so O is complete and P's columns are free
            const bool ok = wait_or_abort(&s_full[ti], st & 1, a.wait_ns, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;   // warp-uniform: the TMEM loads below are collective
            tc::fence_after_sync();
            const int pgs = sp0 + st * ws::kPages;
            const int nk = min(ws::kPages, sp1 - pgs) * kBS;    // the stage's keys
            const int t0 = pgs * kBS;
            const bool interior = nk == ws::kKeys && t0 + ws::kKeys - 1 <= wpos0 && t0 >= wlo1;
            // the row of S in two halves of 64 keys, read twice (its maximum,
            // then P) to keep 64 values in registers; cs >= 0, so the maximum
            // of the scaled scores is cs times that of the raw ones
            auto load_half = [&](int h, float (&sv)[64]) {
                tc::ld32(trow + 64 * h, *reinterpret_cast<float(*)[32]>(sv));
                tc::ld32(trow + 64 * h + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
                tc::wait_ld(*reinterpret_cast<float(*)[32]>(sv));
                tc::wait_ld(*reinterpret_cast<float(*)[32]>(sv + 32));
            };
            auto key_ok = [&](int jj) {
                const int key = t0 + jj;
                return jj < nk && rv && key >= lq && key <= pq;
            };
            float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float sv[64];
                load_half(h, sv);
                if (interior) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) mr[j & 3] = fmaxf(mr[j & 3], sv[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) mr[j & 3] = fmaxf(mr[j & 3], key_ok(64 * h + j) ? sv[j] : -INFINITY);
                }
            }
            const float mraw = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
            const float mx = mraw == -INFINITY ? -INFINITY : mraw * cs;
            // the reference maximum moves only by more than 8 (log2 units);
            // a row that had none (m = -inf) holds O = 0 and l = 0
            const float mn = fmaxf(m, mx);
            const bool upd = mn > m + ws::kRescaleLog2;
            const bool held = upd && m != -INFINITY;
            float alpha = 1.f;
            if (upd) {
                alpha = fast_exp2(m - mn);
                l *= alpha;
                m = mn;
            }
            if (__any_sync(0xffffffffu, held)) {
                // O = O * alpha for the warp's rows (1 where the row keeps its maximum)
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float x[32];
                    tc::ld32(trow + Wg::OC + 32 * c, x);
                    tc::wait_ld(x);
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] *= alpha;
                    tc::st32(trow + Wg::OC + 32 * c, x);
                }
            }
            const float nmuse = m == -INFINITY ? 0.f : -m;
            float lp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                // P of keys [64h, 64h + 64) goes to columns [32h, 32h + 32),
                // whose S (keys [32h, 32h + 32)) has been read already
                float sv[64];
                load_half(h, sv);
                float pw[32];
                if (interior) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {   // key pairs in packed FP32 pairs
                        float x0, x1;
                        fma_f32x2(x0, x1, sv[2 * j], sv[2 * j + 1], cs, cs, nmuse, nmuse);
                        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                        if (j & 1) add_f32x2(lp[2], lp[3], p0, p1);
                        else add_f32x2(lp[0], lp[1], p0, p1);
                        pw[j] = __uint_as_float(pack_f16x2(p0, p1));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {   // masked keys weigh 0 (also when cs = 0)
                        const float p0 = key_ok(64 * h + 2 * j) ? fast_exp2(fmaf(sv[2 * j], cs, nmuse)) : 0.f;
                        const float p1 = key_ok(64 * h + 2 * j + 1) ? fast_exp2(fmaf(sv[2 * j + 1], cs, nmuse)) : 0.f;
                        lp[j & 3] += p0 + p1;
                        pw[j] = __uint_as_float(pack_f16x2(p0, p1));
                    }
                }
                tc::st32(trow + 32 * h, pw);
            }
            const float ls = (lp[0] + lp[1]) + (lp[2] + lp[3]);
            l += ls;
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(&p_full[ti]);      // P (and the rescaled O) are in TMEM
        }
    } else if (warp < ws::kMmaWarp) {
        // ---------------------------------------------------------- converters
        const int ct = tid - ws::kConvWarp0 * 32;
        for (int st = 0; st < nst; ++st) {
            load_stage(st + 1, ct);          // its staging granules were read in iteration st - 1
            cp_async_wait<1>();              // this thread's copies of stage st have landed
            const uint8_t* stg = sm + Wg::STG + (st % ws::kStg) * ws::kGran * Wg::GSLOT;
            const int pgs = sp0 + st * ws::kPages;
            // the K tile is free once the score MMAs of stage st - 1 have completed
            bool ok = st == 0 || wait_or_abort(&k_empty, (st - 1) & 1, a.wait_ns, abort_flag);
            if (named_bar_or(ws::kConvBar, 128, !ok)) break;   // every copy of stage st landed (or all give up)
#pragma unroll
            for (int g = 0; g < ws::kGran; ++g)
                if (pgs + g * tcg::kPages < sp1)   // an empty granule's keys are masked
                    convert_stage_k<D, Wg::KAT>(stg + g * Wg::GSLOT, sm + Wg::KT + g * (tcg::kKeys * 128), ct);
            tc::fence_proxy_async_smem();    // the tile is read by the tensor cores
            mbar_arrive(&k_full);
            // V^T tile st & 1 is free once the value MMAs of stage st - 2 have completed
            const int j = st & 1;
            ok = st < 2 || wait_or_abort(&v_empty[j], ((st >> 1) + 1) & 1, a.wait_ns, abort_flag);
            if (named_bar_or(ws::kConvBar, 128, !ok)) break;
#pragma unroll
            for (int g = 0; g < ws::kGran; ++g) {
                const int pg = pgs + g * tcg::kPages;
                convert_stage_v<D>(stg + g * Wg::GSLOT, sm + Wg::VT + j * Wg::VTB + g * Wg::VAT, ct, pg * kBS,
                                   min(tcg::kPages, sp1 - pg), kmin, kmax);   // zeros past the range
            }
            tc::fence_proxy_async_smem();
            mbar_arrive(&v_full[j]);
            named_bar_sync(ws::kConvBar, 128);  // the staging granules are read before they are refilled
        }
        cp_async_wait<0>();
    } else if (lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        constexpr uint32_t id_s = tc::idesc_f16_f32(128, ws::kKeys);
        constexpr uint32_t id_o = tc::idesc_f16_f32(128, D);
        const bool stall_cta = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
        // S = Q K^T of stage s for tile i (N = 128 keys), into the tile's S columns
        auto issue_s = [&](int i, int s) {
            if (s == a.stall_stage && stall_cta) return;   // test hook: this tile's S never arrives
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (ks & 3) * 32;
                tc::mma_f16(tm + i * Wg::TC, tc::desc_k_sw128(sb + Wg::QT + i * Wg::QTB + (ks >> 2) * 16384 + off),
                            tc::desc_k_sw128(sb + Wg::KT + (ks >> 2) * Wg::KAT + off), id_s, ks > 0);
            }
            tc::commit(&s_full[i]);
        };
        bool ok = nst == 0 || wait_or_abort(&k_full, 0, a.wait_ns, abort_flag);
        if (ok && nst > 0) {
            tc::fence_after_sync();
            for (int i = 0; i < ws::kTiles; ++i) issue_s(i, 0);
            tc::commit(&k_empty);            // the K tile is free when the score MMAs complete
        }
        for (int st = 0; st < nst && ok; ++st) {
            for (int i = 0; i < ws::kTiles; ++i) {
                if (!wait_or_abort(&p_full[i], st & 1, a.wait_ns, abort_flag) ||
                    (i == 0 && !wait_or_abort(&v_full[st & 1], (st >> 1) & 1, a.wait_ns, abort_flag))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                // O += P V: P (128 rows x 128 keys) from the S columns [0, 64)
#pragma unroll
                for (int ks = 0; ks < ws::kKeys / 16; ++ks)
                    tc::mma_f16_ts(tm + i * Wg::TC + Wg::OC, tm + i * Wg::TC + ks * 8,
                                   tc::desc_k_sw128(sb + Wg::VT + (st & 1) * Wg::VTB + (ks >> 2) * Wg::VAT + (ks & 3) * 32),
                                   id_o, 1);
                if (i == ws::kTiles - 1) tc::commit(&v_empty[st & 1]);   // the V^T tile is free when both tiles' P V complete
                if (st + 1 < nst) {
                    if (i == 0) {
                        if (!wait_or_abort(&k_full, (st + 1) & 1, a.wait_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                    }
                    issue_s(i, st + 1);
                    if (i == ws::kTiles - 1) tc::commit(&k_empty);
                }
            }
        }
        // every MMA this thread issued completes before TMEM is released
        tc::commit(&done_bar);
        mbar_wait_bounded(&done_bar, 0, tcg::kWaitNs);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const bool failed = *abort_flag != 0;
    if (failed) {
        if (tid == 0) report(a.err, FP8KV_ERR_TIMEOUT);
    } else if (warp < 8 && (ti == 0 || has1)) {
        // ---- the rows' outputs (or partials) from the TMEM accumulator; every
        // thread of the warp loads (tcgen05.ld is collective), valid rows store
        const uint32_t trow = tm + ti * Wg::TC + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const int tile = 2 * pair + ti;
        const int64_t unit = (static_cast<int64_t>(b) * a.num_kv_heads + hk) * a.tiles + tile;
        const float so = l > 0.f ? a.v_scale / l : 0.f;
        uint4* orow = reinterpret_cast<uint4*>(
            a.out + (static_cast<int64_t>(uu.q0 + (rv ? r / G : 0)) * a.num_q_heads + hk * G + (rv ? r % G : 0)) * D);
        const int64_t slot = (unit * a.splits + split) * a.rows + tt;
        float4* po = reinterpret_cast<float4*>(a.part_o + slot * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float x[32];
            tc::ld32(trow + Wg::OC + 32 * c, x);
            tc::wait_ld(x);
            if (!rv) continue;
            if (a.splits == 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    orow[4 * c + i] = make_uint4(pack_bf16x2(x[8 * i] * so, x[8 * i + 1] * so),
                                                 pack_bf16x2(x[8 * i + 2] * so, x[8 * i + 3] * so),
                                                 pack_bf16x2(x[8 * i + 4] * so, x[8 * i + 5] * so),
                                                 pack_bf16x2(x[8 * i + 6] * so, x[8 * i + 7] * so));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) po[8 * c + i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
            }
        }
        if (rv && a.splits > 1) a.part_ml[slot] = make_float2(m, l);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::dealloc(tm, Wg::COLS);
    }
}

// ---------------------------------------------------------------------------
// The warp-specialised one-tile prefill kernel (used at d = 256; written for
// d = 64 too): one 128-row tile per CTA.  A row's d FP32 outputs live in TMEM
// (columns [256, 512) at d = 256, [128, 192) at d = 64); S has its own
// columns [0, 64) and the P.V tile [64, 64 + min(d, 128)), computed in halves
// of 128 output dimensions at d = 256.  Roles, handing over through mbarriers (every wait
// bounded, a shared abort flag ending all of them):
//   * warps 4-7 (converters): cp.async stage s + 1 into a 2-slot staging
//     ring; convert stage s's K into the K tile once the score MMAs of stage
//     s - 1 have finished with it, and its V^T into the V^T tile once the
//     value MMAs of stage s - 1 have;
//   * one thread of warp 8 (MMA issuer): S(s) = Q K^T; once P(s) is written,
//     O_tile = P V^T for output dimensions [0, 128), and, once that half has
//     been folded, for [128, 256);
//   * warps 0-3 (thread = row): softmax of S(s) into P(s), then the fold of
//     each half into the accumulator, O = O * alpha + O_tile.
// S(s + 1) runs while the rows fold stage s; the conversions run beside both.
namespace ws1 {
constexpr int kConvWarp0 = 4;              // warps 4-7 convert
constexpr int kMmaWarp = 8;                // warp 8 issues the MMAs
constexpr int kThreads = 9 * 32;
constexpr int kConvBar = 2;                // named barrier of the converter warps
}  // namespace ws1

template <int D>
struct Ws1Geo {
    static constexpr int NB = D / 64;
    static constexpr int QTB = NB * 128 * 128;          // Q tile: 128 rows x d
    static constexpr int KTB = NB * tcg::kKeys * 128;   // K tile: 64 keys x d
    static constexpr int VTB = D * 128;                 // V^T tile: d rows x 64 keys
    static constexpr int PTB = 128 * 128;               // P tile: 128 rows x 64 keys
    static constexpr int SLOT = 2 * tcg::kKeys * D;     // one fp8 staging slot: K rows, then V rows
    static constexpr int QT = 0, KT = QT + QTB, VT = KT + KTB, PT = VT + VTB, STG = PT + PTB;
    static constexpr int SMEM = STG + 2 * SLOT;         // 208 KB at d = 256, 64 KB at 64
    static constexpr int ON = D > 128 ? 128 : D;        // output dimensions of one P.V half
    static constexpr int NH = D / ON;                   // halves: 2 at d = 256, else 1
    static constexpr uint32_t S_COL = 0, OT_COL = 64;
    static constexpr uint32_t OACC_COL = D == 256 ? 256 : 128;
    static constexpr uint32_t COLS = D == 256 ? 512 : 256;
    static constexpr int kCtasPerSm = D == 64 ? 2 : 1;  // 2 x 64 KB of shared memory and 2 x 256 TMEM columns
    static_assert(OT_COL + ON <= OACC_COL && OACC_COL + D <= COLS, "TMEM columns");
    static_assert(D == 64 || D == 256, "the one-tile warp-specialised kernel covers d = 64 and 256");
};

template <int D, int G>
__global__ void __launch_bounds__(ws1::kThreads, Ws1Geo<D>::kCtasPerSm) paged_prefill_ws1_kernel(const Args a) {
    using namespace ws1;
    using Wg = Ws1Geo<D>;
    constexpr int QT = Wg::QT, KT = Wg::KT, VT = Wg::VT, PT = Wg::PT, STG = Wg::STG, SLOT = Wg::SLOT;
    constexpr uint32_t S_COL = Wg::S_COL, OT_COL = Wg::OT_COL, OACC_COL = Wg::OACC_COL, COLS = Wg::COLS;
    constexpr int ON = Wg::ON, NH = Wg::NH;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t k_full, k_empty, v_full, v_empty, s_full, p_full, o_full[NH], o_free, done_bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_sh;
    volatile int* abort_flag = &abort_sh;
    uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        mbar_init(&k_full, 128);
        mbar_init(&v_full, 128);
        mbar_init(&k_empty, 1);
        mbar_init(&v_empty, 1);
        mbar_init(&s_full, 1);
        mbar_init(&p_full, 128);
        for (int h = 0; h < NH; ++h) mbar_init(&o_full[h], 1);
        mbar_init(&o_free, 128);
        mbar_init(&done_bar, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    griddep_wait();                // inputs may come from the previous grid on the stream
    griddep_launch_dependents();
    const int b = blockIdx.z, hk = blockIdx.y;
    const int tile = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
    Unit u;
    if (!make_unit<G>(a, b, tile, blockIdx.x == 0 && hk == 0 && tid == 0, u)) return;
    const int pg0 = u.kmin / kBS, np_all = u.kmax / kBS - pg0 + 1;
    const int sp0 = pg0 + static_cast<int>(static_cast<int64_t>(split) * np_all / a.splits);
    const int sp1 = pg0 + static_cast<int>(static_cast<int64_t>(split + 1) * np_all / a.splits);
    const int nst = (sp1 - sp0 + tcg::kPages - 1) / tcg::kPages;
    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;

    // ---- set-up: the rows build the Q tile; the converters start stage 0's copies
    const int r = u.R0 + tid;
    const bool rv = warp < 4 && r < u.rows;
    float cs = 0.f;
    int pq = 0, lq = 0, wpos0 = 0, wlo1 = 0;
    if (warp < 4) {
        // the bf16 row in 16-byte chunks, read twice (its largest magnitude,
        // then the copy) to keep few of them in registers
        constexpr int NC = D / 8;
        const int tok = rv ? r / G : 0, hq = hk * G + (rv ? r % G : 0);
        const uint4* qrow =
            reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(u.q0 + tok) * a.num_q_heads + hq) * D);
        float qmax = 0.f;
#pragma unroll 4
        for (int c = 0; c < NC; ++c) {
            const uint4 qv = rv ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
            const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                qmax = fmaxf(qmax, fmaxf(fabsf(bf16_to_f32(w4[e] & 0xFFFF)), fabsf(bf16_to_f32(w4[e] >> 16))));
        }
        int shift = 0;
        if (qmax > 0.f) {
            const int e = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFF) - 127;
            shift = max(-100, min(100, 14 - e));
        }
        // a negative score scale goes into Q, so that the row's scale cs is
        // positive and the maximum of the scaled scores is cs times the raw maximum
        const float up = (a.score_scale < 0.f ? -1.f : 1.f) * __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
#pragma unroll 4
        for (int c = 0; c < NC; ++c) {
            const uint4 qv = rv ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
            const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
            uint32_t f[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                f[e] = pack_f16x2(bf16_to_f32(w4[e] & 0xFFFF) * up, bf16_to_f32(w4[e] >> 16) * up);
            *reinterpret_cast<uint4*>(sm + QT + (c >> 3) * 16384 + tid * 128 + (((c & 7) ^ (tid & 7)) << 4)) =
                make_uint4(f[0], f[1], f[2], f[3]);
        }
        cs = fabsf(a.score_scale) * __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
        pq = u.L - u.n + (rv ? r / G : 0);
        lq = (a.window > 0 && pq + 1 > a.window) ? pq + 1 - a.window : 0;
        const int wr0 = u.R0 + warp * 32;
        wpos0 = u.L - u.n + wr0 / G;
        const int wpos1 = u.L - u.n + max(0, min(wr0 + 31, u.rows - 1)) / G;
        wlo1 = (a.window > 0 && wpos1 + 1 > a.window) ? wpos1 + 1 - a.window : 0;
    } else if (warp < kMmaWarp) {
        const int ct = tid - kConvWarp0 * 32;
        if (nst > 0)
            load_stage_tc<D>(a, bt, hk, sp0, min(tcg::kPages, sp1 - sp0), sb + STG, ct);
        cp_async_commit();
    }
    if (warp == 0) tc::alloc(&tmem_base, COLS);
    tc::fence_proxy_async_smem();  // the Q tile is read by the tensor cores
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = tmem_base;

    float m = -INFINITY, l = 0.f;
    if (warp < 4) {
        // ---------------------------------------------------------- softmax and fold
        const uint32_t trow = tm + (static_cast<uint32_t>(warp * 32) << 16);
        {
            float z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tc::st32(trow + OACC_COL + 32 * c, z);
            tc::wait_st();
        }
        uint8_t* prow = sm + PT + tid * 128;
        for (int st = 0; st < nst; ++st) {
            bool ok = wait_or_abort(&s_full, st & 1, a.wait_ns, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;   // warp-uniform: the TMEM loads below are collective
            tc::fence_after_sync();
            const int pgs = sp0 + st * tcg::kPages;
            const int np = min(tcg::kPages, sp1 - pgs);
            const int t0 = pgs * kBS;
            const bool interior = np == tcg::kPages && t0 + tcg::kKeys - 1 <= wpos0 && t0 >= wlo1;
            float sv[64];
            tc::ld32(trow + S_COL, *reinterpret_cast<float(*)[32]>(sv));
            tc::ld32(trow + S_COL + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
            tc::wait_ld(*reinterpret_cast<float(*)[32]>(sv));
            tc::wait_ld(*reinterpret_cast<float(*)[32]>(sv + 32));
            // cs >= 0: the maximum of the scaled scores is cs times the raw one
            auto key_ok = [&](int j) {
                const int key = t0 + j;
                return j < np * kBS && rv && key >= lq && key <= pq;
            };
            float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (interior) {
#pragma unroll
                for (int j = 0; j < 64; ++j) mr[j & 3] = fmaxf(mr[j & 3], sv[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) mr[j & 3] = fmaxf(mr[j & 3], key_ok(j) ? sv[j] : -INFINITY);
            }
            const float mraw = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
            const float mx = mraw == -INFINITY ? -INFINITY : mraw * cs;
            const float mn = fmaxf(m, mx);
            const float muse = mn == -INFINITY ? 0.f : mn;
            const float alpha = fast_exp2(m - muse);
            m = mn;
            float lp[4] = {0.f, 0.f, 0.f, 0.f};
            // pof(j, p0, p1): the weights of keys j and j + 1
            auto emit = [&](auto pof) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t pw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float p0, p1;
                        pof(8 * c + 2 * e, p0, p1);
                        add_f32x2(lp[2 * (e & 1)], lp[2 * (e & 1) + 1], p0, p1);
                        pw[e] = pack_f16x2(p0, p1);
                    }
                    *reinterpret_cast<uint4*>(prow + ((c ^ (tid & 7)) << 4)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                }
            };
            if (interior) {
                emit([&](int j, float& p0, float& p1) {   // key pairs in packed FP32 pairs
                    float x0, x1;
                    fma_f32x2(x0, x1, sv[j], sv[j + 1], cs, cs, -muse, -muse);
                    p0 = fast_exp2(x0);
                    p1 = fast_exp2(x1);
                });
            } else {   // masked keys weigh 0 (also when cs = 0)
                emit([&](int j, float& p0, float& p1) {
                    p0 = key_ok(j) ? fast_exp2(fmaf(sv[j], cs, -muse)) : 0.f;
                    p1 = key_ok(j + 1) ? fast_exp2(fmaf(sv[j + 1], cs, -muse)) : 0.f;
                });
            }
            l = l * alpha + ((lp[0] + lp[1]) + (lp[2] + lp[3]));
            tc::fence_proxy_async_smem();  // P is read by the tensor cores
            tc::fence_before_sync();
            mbar_arrive(&p_full);
            // O = O * alpha + O_tile (IEEE FMA, FP32), one half of the output dimensions at a time
            bool okh = true;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                ok = wait_or_abort(&o_full[h], st & 1, a.wait_ns, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {
                    okh = false;
                    break;
                }
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < ON / 32; ++c) {
                    float x[32], y[32];
                    tc::ld32(trow + OT_COL + 32 * c, x);
                    tc::ld32(trow + OACC_COL + ON * h + 32 * c, y);
                    tc::wait_ld(x);
                    tc::wait_ld(y);
#pragma unroll
                    for (int j = 0; j < 32; ++j) y[j] = fmaf(y[j], alpha, x[j]);
                    tc::st32(trow + OACC_COL + ON * h + 32 * c, y);
                }
                tc::wait_st();
                tc::fence_before_sync();
                mbar_arrive(&o_free);      // the MMA may overwrite O_tile
            }
            if (!okh) break;
        }
    } else if (warp < kMmaWarp) {
        // ---------------------------------------------------------- converters
        const int ct = tid - kConvWarp0 * 32;
        for (int st = 0; st < nst; ++st) {
            if (st + 1 < nst)
                load_stage_tc<D>(a, bt, hk, sp0 + (st + 1) * tcg::kPages,
                                 min(tcg::kPages, sp1 - sp0 - (st + 1) * tcg::kPages),
                                 sb + STG + ((st + 1) & 1) * SLOT, ct);
            cp_async_commit();
            cp_async_wait<1>();              // this thread's copies of stage st have landed
            // the K tile is free once the score MMAs of stage st - 1 have completed
            bool ok = st == 0 || wait_or_abort(&k_empty, (st - 1) & 1, a.wait_ns, abort_flag);
            if (named_bar_or(kConvBar, 128, !ok)) break;   // every copy of stage st landed (or all give up)
            const uint8_t* stg = sm + STG + (st & 1) * SLOT;
            const int pgs = sp0 + st * tcg::kPages;
            const int np = min(tcg::kPages, sp1 - pgs);
            convert_stage_k<D>(stg, sm + KT, ct);
            tc::fence_proxy_async_smem();
            mbar_arrive(&k_full);
            // the V^T tile is free once the value MMAs of stage st - 1 have completed
            ok = st == 0 || wait_or_abort(&v_empty, (st - 1) & 1, a.wait_ns, abort_flag);
            if (named_bar_or(kConvBar, 128, !ok)) break;
            convert_stage_v<D>(stg, sm + VT, ct, pgs * kBS, np, u.kmin, u.kmax);
            tc::fence_proxy_async_smem();
            mbar_arrive(&v_full);
            named_bar_sync(kConvBar, 128);   // the staging slot is read before it is refilled
        }
        cp_async_wait<0>();
    } else if (lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        constexpr uint32_t id_s = tc::idesc_f16_f32(128, tcg::kKeys);
        constexpr uint32_t id_o = tc::idesc_f16_f32(128, ON);
        const bool stall_cta = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
        for (int st = 0; st < nst; ++st) {
            if (!wait_or_abort(&k_full, st & 1, a.wait_ns, abort_flag)) break;
            tc::fence_after_sync();
            // S(st) overwrites S(st - 1), which the rows loaded before writing P(st - 1)
            if (!(st == a.stall_stage && stall_cta)) {   // test hook: this stage's S never arrives
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks & 3) * 32;
                    tc::mma_f16(tm + S_COL, tc::desc_k_sw128(sb + QT + (ks >> 2) * 16384 + off),
                                tc::desc_k_sw128(sb + KT + (ks >> 2) * (tcg::kKeys * 128) + off), id_s, ks > 0);
                }
                tc::commit(&s_full);
            }
            tc::commit(&k_empty);             // the K tile is free when the score MMAs complete
            if (!wait_or_abort(&p_full, st & 1, a.wait_ns, abort_flag)) break;
            if (!wait_or_abort(&v_full, st & 1, a.wait_ns, abort_flag)) break;
            tc::fence_after_sync();
            bool ok = true;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                // O_tile is free once the rows have folded the previous half
                const int f = NH * st + h;    // this half's fold index
                if (f > 0 && !wait_or_abort(&o_free, (f - 1) & 1, a.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_f16(tm + OT_COL, tc::desc_k_sw128(sb + PT + ks * 32),
                                tc::desc_k_sw128(sb + VT + h * ON * 128 + ks * 32), id_o, ks > 0);
                tc::commit(&o_full[h]);
            }
            if (!ok) break;
            tc::commit(&v_empty);             // the V^T tile is free when the value MMAs complete
        }
        // every MMA this thread issued completes before TMEM is released
        tc::commit(&done_bar);
        mbar_wait_bounded(&done_bar, 0, tcg::kWaitNs);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const bool failed = *abort_flag != 0;
    if (failed) {
        if (tid == 0) report(a.err, FP8KV_ERR_TIMEOUT);
    } else if (warp < 4) {
        // ---- the rows' outputs (or partials) from the TMEM accumulator; every
        // thread of the warp loads (tcgen05.ld is collective), valid rows store
        const uint32_t trow = tm + (static_cast<uint32_t>(warp * 32) << 16);
        const int64_t unit = (static_cast<int64_t>(b) * a.num_kv_heads + hk) * a.tiles + tile;
        const float so = l > 0.f ? a.v_scale / l : 0.f;
        uint4* orow = reinterpret_cast<uint4*>(
            a.out + (static_cast<int64_t>(u.q0 + (rv ? r / G : 0)) * a.num_q_heads + hk * G + (rv ? r % G : 0)) * D);
        const int64_t slot = (unit * a.splits + split) * a.rows + tid;
        float4* po = reinterpret_cast<float4*>(a.part_o + slot * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float x[32];
            tc::ld32(trow + OACC_COL + 32 * c, x);
            tc::wait_ld(x);
            if (!rv) continue;
            if (a.splits == 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    orow[4 * c + i] = make_uint4(pack_bf16x2(x[8 * i] * so, x[8 * i + 1] * so),
                                                 pack_bf16x2(x[8 * i + 2] * so, x[8 * i + 3] * so),
                                                 pack_bf16x2(x[8 * i + 4] * so, x[8 * i + 5] * so),
                                                 pack_bf16x2(x[8 * i + 6] * so, x[8 * i + 7] * so));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) po[8 * c + i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
            }
        }
        if (rv && a.splits > 1) a.part_ml[slot] = make_float2(m, l);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::dealloc(tm, COLS);
    }
}

// Combines a unit's split partials row by row in FP32: with M the largest
// row maximum, weight_s = 2^(m_s - M), out = v_scale * sum_s weight_s o_s /
// sum_s weight_s l_s, rounded to bf16.  A CTA covers 8 rows of a unit, a
// warp one row; each lane owns D/32 dimensions and keeps 8 splits' loads in
// flight.  Every split writes its partial (zeros and m = -inf when it has no
// keys for the row), so all loads are of written values.
template <int D, int G>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const Args a) {
    constexpr int PER = D / 32;   // dimensions per lane: 2, 4 or 8
    __shared__ float wsm[8][kMaxSplits];
    const int b = blockIdx.z, hk = blockIdx.y;
    const int groups = a.rows / 8;
    const int tile = blockIdx.x / groups, grp = blockIdx.x % groups;
    Unit u;
    const bool ok = make_unit<G>(a, b, tile, false, u);  // only the lengths: read before the wait
    griddep_wait();                                      // the partials are complete and visible
    if (!ok) return;
    // a CTA of this call gave up a wait: its partials are missing, and the
    // error word says so
    if (*reinterpret_cast<volatile uint32_t*>(a.err) == FP8KV_ERR_TIMEOUT) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rr = grp * 8 + warp;                       // row within the tile
    const int r = u.R0 + rr;
    if (r >= u.rows) return;                             // whole warp; no CTA-wide sync follows
    const int64_t unit = (static_cast<int64_t>(b) * a.num_kv_heads + hk) * a.tiles + tile;
    const int64_t slot0 = unit * a.splits * a.rows + rr;  // split s at slot0 + s * rows
    float mmax = -INFINITY;
    for (int sp = lane; sp < a.splits; sp += 32) mmax = fmaxf(mmax, a.part_ml[slot0 + sp * a.rows].x);
#pragma unroll
    for (int off = 16; off; off >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, off));
    float lsum = 0.f;
    for (int sp = lane; sp < a.splits; sp += 32) {
        const float2 ml = a.part_ml[slot0 + sp * a.rows];
        const float wgt = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - mmax);
        wsm[warp][sp] = wgt;
        lsum += wgt * ml.y;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    __syncwarp();
    const float so = lsum > 0.f ? a.v_scale / lsum : 0.f;
    const float* po = a.part_o + slot0 * D + lane * PER;
    const int64_t stride = static_cast<int64_t>(a.rows) * D;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    int sp = 0;
    for (; sp + 8 <= a.splits; sp += 8) {
        float v[8][PER];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int e = 0; e < PER; e += 2) {
                const float2 x = *reinterpret_cast<const float2*>(po + (sp + i) * stride + e);
                v[i][e] = x.x;
                v[i][e + 1] = x.y;
            }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float wgt = wsm[warp][sp + i];
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = fmaf(wgt, v[i][e], acc[e]);
        }
    }
    for (; sp < a.splits; ++sp) {
        const float wgt = wsm[warp][sp];
#pragma unroll
        for (int e = 0; e < PER; e += 2) {
            const float2 x = *reinterpret_cast<const float2*>(po + sp * stride + e);
            acc[e] = fmaf(wgt, x.x, acc[e]);
            acc[e + 1] = fmaf(wgt, x.y, acc[e + 1]);
        }
    }
    uint16_t* orow = a.out + (static_cast<int64_t>(u.q0 + r / G) * a.num_q_heads + hk * G + r % G) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2)
        *reinterpret_cast<uint32_t*>(orow + e) = pack_bf16x2(acc[e] * so, acc[e + 1] * so);
}

// Split plan: the tiles a sequence's chunk may need, how many CTAs share each
// unit's key range (choose_splits in prefill_plan.h) and the workspace layout.
struct Plan {
    int tiles = 0;
    int splits = 1;
    size_t ml = kHeader;   // offset of the (m, l) partials
    size_t o = kHeader;    // offset of the output partials
    size_t total = kHeader;
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Query rows per tile (one TMEM lane each).
inline int rows_per_tile(int) { return kRowsTC; }

// Query tiles of 128 rows per (sequence, kv head) for a chunk of max_q_len.
inline int tiles_of(int max_q_len, int G) {
    return static_cast<int>((static_cast<int64_t>(max_q_len) * G + kRowsTC - 1) / kRowsTC);
}

// Which kernel runs: 2, the warp-specialised one-tile kernel, at d = 256;
// 1, the warp-specialised one with two tiles per CTA, at d = 64 and 128 when
// a sequence's chunk spans at least two tiles (at d = 64 it measured 617
// against 442 TFLOP/s for the one-tile kernel at 2048-token chunks); else 0,
// paged_prefill_tc_kernel, one tile per CTA.
inline int kernel_kind(int D, int tiles) {
    if (D == 256) return 2;
    return tiles >= 2 ? 1 : 0;
}
inline int tiles_per_cta(int kind) { return kind == 1 ? ws::kTiles : 1; }

Plan make_plan(int batch, int max_q_len, int max_seq_len, int G, int Hkv, int D, int window, int sms, int per_sm) {
    Plan pl;
    const int rows = rows_per_tile(D);
    pl.tiles = tiles_of(max_q_len, G);
    const int tpc = tiles_per_cta(kernel_kind(D, pl.tiles));
    const int64_t units = static_cast<int64_t>(pl.tiles) * Hkv * batch;
    const int64_t ctas = static_cast<int64_t>((pl.tiles + tpc - 1) / tpc) * Hkv * batch;
    int64_t pages = (static_cast<int64_t>(max_seq_len) + kBS - 1) / kBS;
    if (window > 0) pages = std::min<int64_t>(pages, (static_cast<int64_t>(window) + rows * tpc) / kBS + 2);
    pl.splits = choose_splits(ctas, pages, static_cast<int64_t>(sms) * per_sm);
    if (pl.splits > 1) {
        const size_t slots = static_cast<size_t>(units) * pl.splits * rows;
        pl.ml = kHeader;
        pl.o = pl.ml + align256(slots * sizeof(float2));
        pl.total = pl.o + align256(slots * D * sizeof(float));
    }
    return pl;
}

// The prefill kernel of a kind (kernel_kind) for (D, G), its dynamic shared
// memory and its threads.
template <int D, int G>
void kernel_of(int kind, void (**fn)(const Args), size_t* smem, int* threads) {
    if constexpr (D == 64 || D == 128) {
        if (kind == 1) {
            *fn = paged_prefill_ws_kernel<D, G>;
            *smem = static_cast<size_t>(WsGeo<D>::SMEM) + 1024;
            *threads = ws::kThreads;
            return;
        }
    }
    if constexpr (D == 256) {
        if (kind == 2) {
            *fn = paged_prefill_ws1_kernel<D, G>;
            *smem = static_cast<size_t>(Ws1Geo<D>::SMEM) + 1024;
            *threads = ws1::kThreads;
            return;
        }
    }
    *fn = paged_prefill_tc_kernel<D, G>;
    *smem = static_cast<size_t>(TcGeo<D>::SMEM) + 1024;
    *threads = kThreads;
}

template <int D>
bool kernel_of_g(int G, int kind, void (**fn)(const Args), size_t* smem, int* threads) {
    switch (G) {
        case 1: kernel_of<D, 1>(kind, fn, smem, threads); return true;
        case 2: kernel_of<D, 2>(kind, fn, smem, threads); return true;
        case 4: kernel_of<D, 4>(kind, fn, smem, threads); return true;
        case 8: kernel_of<D, 8>(kind, fn, smem, threads); return true;
        case 16: kernel_of<D, 16>(kind, fn, smem, threads); return true;
        default: return false;
    }
}

// Resident CTAs per SM of the prefill kernel for (D, G, kind) on the current
// device (the occupancy calculator, with the kernel's shared-memory opt-in
// applied); 0 on failure.  Cached per device.
int resident_per_sm(int D, int G, int kind) {
    static std::atomic<int> cache[3][3][5][64] = {};
    const int di = D == 64 ? 0 : (D == 128 ? 1 : 2);
    const int gi = G == 1 ? 0 : (G == 2 ? 1 : (G == 4 ? 2 : (G == 8 ? 3 : 4)));
    const int wi = kind;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        const int c = cache[wi][di][gi][dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    void (*fn)(const Args) = nullptr;
    size_t smem = 0;
    int threads = 0;
    const bool ok = D == 64 ? kernel_of_g<64>(G, kind, &fn, &smem, &threads)
                            : (D == 128 ? kernel_of_g<128>(G, kind, &fn, &smem, &threads)
                                        : kernel_of_g<256>(G, kind, &fn, &smem, &threads));
    if (!ok) return 0;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1) return 0;
    if (dev >= 0 && dev < 64) cache[wi][di][gi][dev].store(n, std::memory_order_relaxed);
    return n;
}

template <int D, int G>
cudaError_t launch(const Args& a, int batch, cudaStream_t s) {
    const int kind = kernel_kind(D, a.tiles);
    void (*kernel)(const Args) = nullptr;
    size_t smem = 0;
    int threads = 0;
    kernel_of<D, G>(kind, &kernel, &smem, &threads);
    static std::atomic<uint64_t> done_mask[3] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit == 0 || !(done_mask[kind].load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        done_mask[kind].fetch_or(bit, std::memory_order_release);
    }
    // Both grids may start before the previous work on the stream ends; each
    // waits (griddepcontrol.wait) before touching what that work wrote.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const int tpc = tiles_per_cta(kind);
    const int ctas_x = (a.tiles + tpc - 1) / tpc;
    cfg.gridDim = dim3(static_cast<unsigned>(ctas_x * a.splits), static_cast<unsigned>(a.num_kv_heads),
                       static_cast<unsigned>(batch));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess || a.splits == 1) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(a.tiles * (a.rows / 8)), static_cast<unsigned>(a.num_kv_heads),
                       static_cast<unsigned>(batch));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, prefill_merge_kernel<D, G>, a);
}

template <int D>
cudaError_t launch_g(int G, const Args& a, int batch, cudaStream_t s) {
    switch (G) {
        case 1: return launch<D, 1>(a, batch, s);
        case 2: return launch<D, 2>(a, batch, s);
        case 4: return launch<D, 4>(a, batch, s);
        case 8: return launch<D, 8>(a, batch, s);
        case 16: return launch<D, 16>(a, batch, s);
        default: return cudaErrorInvalidValue;
    }
}

// Shape checks shared by the size query and the call.
fp8kv_status check_shape(int batch, int max_q_len, int max_seq_len, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size) {
    if (batch < 0 || batch > 65535 || num_kv_heads < 1 || num_kv_heads > 65535 || num_q_heads < 1 ||
        num_q_heads % num_kv_heads != 0 || max_seq_len < 0 || max_q_len < 0 || max_q_len > max_seq_len)
        return FP8KV_ERR_INVALID_ARG;
    const int G = num_q_heads / num_kv_heads;
    if (!(head_dim == 64 || head_dim == 128 || head_dim == 256) || block_size != kBS ||
        !(G == 1 || G == 2 || G == 4 || G == 8 || G == 16))
        return FP8KV_ERR_UNSUPPORTED;
    const int64_t tiles = (static_cast<int64_t>(max_q_len) * G + kRowsTC - 1) / kRowsTC;
    if (tiles * kMaxSplits > INT32_MAX) return FP8KV_ERR_UNSUPPORTED;
    return FP8KV_OK;
}

}  // namespace prefill
}  // namespace fp8kv

extern "C" size_t fp8kv_paged_prefill_workspace_size(int batch, int max_q_len, int max_seq_len, int num_q_heads,
                                                     int num_kv_heads, int head_dim, int block_size, int window) {
    using namespace fp8kv::prefill;
    if (check_shape(batch, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size) != FP8KV_OK)
        return 0;
    int sms = 0;
    if (fp8kv::device_sms(&sms) != 0) return 0;
    const int G = num_q_heads / num_kv_heads;
    const int per_sm = resident_per_sm(head_dim, G, kernel_kind(head_dim, tiles_of(max_q_len, G)));
    if (per_sm < 1) return 0;
    return make_plan(batch, max_q_len, max_seq_len, G, num_kv_heads, head_dim, window > 0 ? window : 0, sms, per_sm)
        .total;
}

namespace {

fp8kv_status prefill_impl(const void* q, int64_t num_q_tokens, const uint8_t* k_cache, const uint8_t* v_cache,
                          int64_t num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* seq_lens, const int32_t* q_starts, int max_q_len, int max_seq_len, int batch,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size, float k_scale,
                          float v_scale, float sm_scale, int window, void* out, void* workspace,
                          size_t workspace_bytes, void* stream, int stall_stage, uint64_t wait_ns) {
    using namespace fp8kv::prefill;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const fp8kv_status sh = check_shape(batch, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                                        block_size);
    if (sh != FP8KV_OK) return sh;
    if (num_blocks < 1 || max_blocks_per_seq < 0 || num_q_tokens < 0) return FP8KV_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !(k_scale > 0) || !std::isfinite(v_scale) || !(v_scale > 0) ||
        !std::isfinite(sm_scale))
        return FP8KV_ERR_INVALID_ARG;
    if (num_blocks >= (INT64_C(1) << 31) || num_blocks * num_kv_heads >= (INT64_C(1) << 31))
        return FP8KV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_blocks_per_seq) * block_size < max_seq_len) return FP8KV_ERR_INVALID_ARG;
    if (batch == 0 || max_q_len == 0 || num_q_tokens == 0) return FP8KV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !q_starts || !out) return FP8KV_ERR_INVALID_ARG;
    if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(out)) return FP8KV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(q_starts) & 3u))
        return FP8KV_ERR_INVALID_ARG;
    int sms = 0;
    if (fp8kv::device_sms(&sms) != 0) return FP8KV_ERR_CUDA;
    const int G = num_q_heads / num_kv_heads;
    const int per_sm = resident_per_sm(head_dim, G, kernel_kind(head_dim, tiles_of(max_q_len, G)));
    if (per_sm < 1) return FP8KV_ERR_CUDA;
    const Plan pl = make_plan(batch, max_q_len, max_seq_len, G, num_kv_heads, head_dim, window > 0 ? window : 0, sms,
                              per_sm);
    if (!workspace || workspace_bytes < pl.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FP8KV_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    Args a;
    a.q = static_cast<const uint16_t*>(q);
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.q_starts = q_starts;
    a.out = static_cast<uint16_t*>(out);
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.part_ml = reinterpret_cast<float2*>(ws + pl.ml);
    a.part_o = reinterpret_cast<float*>(ws + pl.o);
    a.num_blocks = num_blocks;
    a.num_q_tokens = num_q_tokens;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.max_seq_len = max_seq_len;
    a.max_q_len = max_q_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.tiles = pl.tiles;
    a.rows = rows_per_tile(head_dim);
    a.splits = pl.splits;
    a.window = window > 0 ? window : 0;
    a.score_scale = sm_scale * k_scale * kLog2e;
    a.v_scale = v_scale;
    a.wait_ns = wait_ns;
    a.stall_stage = stall_stage;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (head_dim) {
        case 64: e = launch_g<64>(G, a, batch, s); break;
        case 128: e = launch_g<128>(G, a, batch, s); break;
        default: e = launch_g<256>(G, a, batch, s); break;
    }
    return e == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA;
}

}  // namespace

extern "C" fp8kv_status fp8kv_paged_prefill(const void* q, int64_t num_q_tokens, const uint8_t* k_cache,
                                            const uint8_t* v_cache, int64_t num_blocks, const int32_t* block_tables,
                                            int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* q_starts,
                                            int max_q_len, int max_seq_len, int batch, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size, float k_scale,
                                            float v_scale, float sm_scale, int window, void* out, void* workspace,
                                            size_t workspace_bytes, void* stream) {
    FP8KV_TRACE("fp8kv_paged_prefill");
    return prefill_impl(q, num_q_tokens, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                        q_starts, max_q_len, max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                        k_scale, v_scale, sm_scale, window, out, workspace, workspace_bytes, stream, -1,
                        fp8kv::prefill::tcg::kWaitNs);
}

extern "C" fp8kv_status fp8kv_debug_paged_prefill_stall(
    const void* q, int64_t num_q_tokens, const uint8_t* k_cache, const uint8_t* v_cache, int64_t num_blocks,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* q_starts,
    int max_q_len, int max_seq_len, int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    float k_scale, float v_scale, float sm_scale, int window, void* out, void* workspace, size_t workspace_bytes,
    void* stream, int stall_stage, uint64_t wait_limit_ns) {
    FP8KV_TRACE("fp8kv_debug_paged_prefill_stall");
    if (stall_stage < 0 || wait_limit_ns == 0 || wait_limit_ns > fp8kv::prefill::tcg::kWaitNs)
        return FP8KV_ERR_INVALID_ARG;
    return prefill_impl(q, num_q_tokens, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                        q_starts, max_q_len, max_seq_len, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                        k_scale, v_scale, sm_scale, window, out, workspace, workspace_bytes, stream, stall_stage,
                        wait_limit_ns);
}
