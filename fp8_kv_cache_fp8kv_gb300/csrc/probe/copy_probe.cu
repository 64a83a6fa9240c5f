// Copy-pipeline probe: how fast can one GB300 stream the pages of a paged KV
// cache into shared memory, by copy mechanism, with no attention math?
//
// The decode kernel's design rests on these numbers: the pages are 2 KB (one
// kv head of 16 tokens at d = 128) in random physical order, K and V in two
// arrays, the whole step's pages (8 sequences of 18000-22000 tokens, 8 kv
// heads) split into equal contiguous ranges, one per CTA, in the decode
// kernel's unit order.  Each variant copies every page of K and of V once;
// the consumer side only waits for a stage and releases it.
//
//   tma:     TMA 4-D tensor boxes (one per page) issued by `producers` warps
//            per CTA (half for K, half for V) into an mbarrier-guarded ring of
//            12 stages of 2 pages; 4 consumer warps.  The decode kernel's first
//            design used 2 producer warps.
//   cpasync: every warp streams its own contiguous share of the CTA's range
//            with 16-byte cp.async copies into a private ring of 3 stages of 2
//            pages (the current decode kernel's pipeline); block ids are read
//            32 at a time, one window ahead.
//   ldg:     plain 16-byte loads into registers, 16 warps per SM, each warp
//            reading whole pages (a bound on what the DRAM serves).
//
// Prints one line per variant: pages, median microseconds of 20 launches, GB/s
// of K+V bytes.  Every wait on an mbarrier is bounded (0.5 s); a wait that
// runs out sets an error flag, which the program reports.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <numeric>
#include <random>
#include <vector>

#define CHECK(x)                                                                                  \
    do {                                                                                          \
        cudaError_t e_ = (x);                                                                     \
        if (e_ != cudaSuccess) {                                                                  \
            std::printf("CUDA error %s at line %d: %s\n", #x, __LINE__, cudaGetErrorString(e_)); \
            std::exit(1);                                                                         \
        }                                                                                         \
    } while (0)

namespace {

constexpr int kD = 128, kHkv = 8, kPage = 16 * kD, kPps = 2, kHalf = kPps * kPage;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool wait_bounded(uint64_t* b, uint32_t parity) {
    const uint64_t t0 = now_ns();
    while (!try_wait(b, parity))
        if (now_ns() - t0 > 500000000ull) return false;
    return true;
}

struct Pages {
    const int* ids;    // physical block of each page, in range order
    const int* heads;  // kv head of each page
    const int* start;  // [ranges + 1]
};

// --------------------------------------------------------------------------- tma
__global__ void __launch_bounds__(512) tma_probe(const __grid_constant__ CUtensorMap tk,
                                                 const __grid_constant__ CUtensorMap tv, Pages pg, int producers,
                                                 unsigned* err) {
    constexpr int S = 12, NC = 4;
    extern __shared__ uint8_t raw[];
    uint8_t* ring = raw + ((1024u - (su32(raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + S * 2 * kHalf);
    uint64_t* empty = full + 2 * S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * S; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&full[i])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&empty[i])) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int j0 = pg.start[blockIdx.x], n = pg.start[blockIdx.x + 1] - j0;
    const int nst = (n + kPps - 1) / kPps;
    if (warp >= NC) {  // producers: array (pw & 1), stages sub, sub + nsub, ...
        const int pw = warp - NC, arr = pw & 1, sub = pw >> 1, nsub = producers >> 1;
        const CUtensorMap* tm = arr ? &tv : &tk;
        int last = -1;
        bool ok = true;
        for (int st = sub; st < nst && ok; st += nsub) {
            int id = 0, h = 0;
            if (lane < kPps && st * kPps + lane < n) {
                id = pg.ids[j0 + st * kPps + lane];
                h = pg.heads[j0 + st * kPps + lane];
            }
            const int id1 = __shfl_sync(0xffffffffu, id, 1), h1 = __shfl_sync(0xffffffffu, h, 1);
            if (lane == 0) {
                const int slot = st % S, np = min(kPps, n - st * kPps);
                if (st >= S && !wait_bounded(&empty[arr * S + slot], ((st / S) & 1) ^ 1)) {
                    atomicExch(err, 1u);
                    ok = false;
                } else {
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&full[arr * S + slot])),
                                 "r"(np * kPage)
                                 : "memory");
                    for (int p = 0; p < np; ++p) {
                        const uint32_t dst = su32(ring + slot * 2 * kHalf + arr * kHalf + p * kPage);
                        asm volatile(
                            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                            " [%0], [%1, {0, 0, %2, %3}], [%4];" ::"r"(dst),
                            "l"(reinterpret_cast<uint64_t>(tm)), "r"(p ? h1 : h), "r"(p ? id1 : id),
                            "r"(su32(&full[arr * S + slot]))
                            : "memory");
                    }
                    last = st;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (lane == 0)  // no copy may land after the CTA exits
            for (int t = sub; t <= last; t += nsub)
                if (t + S > last) wait_bounded(&full[arr * S + t % S], (t / S) & 1);
        return;
    }
    for (int st = warp; st < nst; st += NC) {
        const int slot = st % S;
        for (int arr = 0; arr < 2; ++arr) {
            if (!wait_bounded(&full[arr * S + slot], (st / S) & 1)) {
                atomicExch(err, 2u);
                return;
            }
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(&empty[arr * S + slot])) : "memory");
        }
    }
}

// --------------------------------------------------------------------------- cpasync
template <int W>
__global__ void __launch_bounds__(W * 32) cpasync_probe(const uint8_t* K, const uint8_t* V, Pages pg) {
    constexpr int R = 3;
    extern __shared__ uint8_t raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring = su32(raw) + warp * R * 2 * kHalf;
    const int c0 = pg.start[blockIdx.x], cn = pg.start[blockIdx.x + 1] - c0;
    const int j0 = c0 + cn * warp / W, n = c0 + cn * (warp + 1) / W - j0;  // this warp's share
    const int nst = (n + kPps - 1) / kPps;
    int win = 0, win_h = 0, nxt = 0, nxt_h = 0, base = 0;
    if (lane < n) { win = pg.ids[j0 + lane]; win_h = pg.heads[j0 + lane]; }
    if (32 + lane < n) { nxt = pg.ids[j0 + 32 + lane]; nxt_h = pg.heads[j0 + 32 + lane]; }
    int ist = 0;
    auto issue = [&]() {
        if (ist < nst) {
            for (int p = 0; p < kPps && ist * kPps + p < n; ++p) {
                const int pgi = ist * kPps + p;
                if (pgi - base >= 32) {
                    win = nxt; win_h = nxt_h; base += 32;
                    nxt = nxt_h = 0;
                    if (base + 32 + lane < n) { nxt = pg.ids[j0 + base + 32 + lane]; nxt_h = pg.heads[j0 + base + 32 + lane]; }
                }
                const int id = __shfl_sync(0xffffffffu, win, pgi - base), h = __shfl_sync(0xffffffffu, win_h, pgi - base);
                const size_t off = (static_cast<size_t>(id) * kHkv + h) * kPage;
                const uint32_t dst = ring + (ist % R) * 2 * kHalf + p * kPage;
                for (int i = lane * 16; i < kPage; i += 512) {
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + i), "l"(K + off + i) : "memory");
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + kHalf + i), "l"(V + off + i) : "memory");
                }
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        ++ist;
    };
    issue();
    issue();
    for (int st = 0; st < nst; ++st) {
        issue();
        asm volatile("cp.async.wait_group 2;" ::: "memory");
        __syncwarp();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// --------------------------------------------------------------------------- ldg
__global__ void __launch_bounds__(256) ldg_probe(const uint8_t* K, const uint8_t* V, Pages pg, unsigned* sink) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j0 = pg.start[blockIdx.x], j1 = pg.start[blockIdx.x + 1];
    uint32_t acc = 0;
    for (int j = j0 + warp; j < j1; j += 8) {
        const size_t off = (static_cast<size_t>(pg.ids[j]) * kHkv + pg.heads[j]) * kPage;
        uint4 x[4], y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] = __ldcs(reinterpret_cast<const uint4*>(K + off) + i * 32 + lane);
            y[i] = __ldcs(reinterpret_cast<const uint4*>(V + off) + i * 32 + lane);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc ^= x[i].x ^ y[i].y ^ x[i].z ^ y[i].w;
    }
    if (acc == 0x9e3779b9u) atomicAdd(sink, 1u);  // keeps the loads
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <typename F>
float median_us(F&& launch) {
    cudaEvent_t a, b;
    CHECK(cudaEventCreate(&a));
    CHECK(cudaEventCreate(&b));
    std::vector<float> t;
    for (int r = 0; r < 23; ++r) {
        CHECK(cudaEventRecord(a));
        launch();
        CHECK(cudaEventRecord(b));
        CHECK(cudaEventSynchronize(b));
        float ms = 0;
        CHECK(cudaEventElapsedTime(&ms, a, b));
        if (r >= 3) t.push_back(ms * 1e3f);
    }
    CHECK(cudaGetLastError());
    std::sort(t.begin(), t.end());
    CHECK(cudaEventDestroy(a));
    CHECK(cudaEventDestroy(b));
    return t[t.size() / 2];
}

}  // namespace

int main() {
    int sms = 0;
    CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
    std::mt19937_64 rng(20);
    std::vector<int> blocks(8);
    int64_t nb = 0;
    for (int& b : blocks) {
        b = (18000 + static_cast<int>(rng() % 4001) + 15) / 16;
        nb += b;
    }
    std::vector<int> perm(nb);
    std::iota(perm.begin(), perm.end(), 0);
    std::shuffle(perm.begin(), perm.end(), rng);
    std::vector<int> ids, heads;  // unit order: (sequence, kv head), pages in logical order
    for (int s = 0, first = 0; s < 8; first += blocks[s], ++s)
        for (int h = 0; h < kHkv; ++h)
            for (int i = 0; i < blocks[s]; ++i) {
                ids.push_back(perm[first + i]);
                heads.push_back(h);
            }
    const int64_t P = static_cast<int64_t>(ids.size());
    const size_t bytes = static_cast<size_t>(nb) * kHkv * kPage;
    uint8_t *K, *V;
    CHECK(cudaMalloc(&K, bytes));
    CHECK(cudaMalloc(&V, bytes));
    CHECK(cudaMemset(K, 1, bytes));
    CHECK(cudaMemset(V, 2, bytes));
    int *d_ids, *d_heads, *d_start;
    unsigned* d_err;
    CHECK(cudaMalloc(&d_ids, P * sizeof(int)));
    CHECK(cudaMalloc(&d_heads, P * sizeof(int)));
    CHECK(cudaMalloc(&d_start, (2 * sms + 1) * sizeof(int)));
    CHECK(cudaMalloc(&d_err, 2 * sizeof(unsigned)));
    CHECK(cudaMemset(d_err, 0, 2 * sizeof(unsigned)));
    CHECK(cudaMemcpy(d_ids, ids.data(), P * sizeof(int), cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_heads, heads.data(), P * sizeof(int), cudaMemcpyHostToDevice));
    const int C = 2 * sms;  // two CTAs per SM, as the decode kernel
    std::vector<int> start(C + 1);
    for (int c = 0; c <= C; ++c) start[c] = static_cast<int>(static_cast<int64_t>(c) * P / C);
    CHECK(cudaMemcpy(d_start, start.data(), (C + 1) * sizeof(int), cudaMemcpyHostToDevice));
    const Pages pg{d_ids, d_heads, d_start};
    const double kv = 2.0 * P * kPage;
    std::printf("pages %lld, K+V %.1f MB, %d CTAs\n", static_cast<long long>(P), kv / 1e6, C);

    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    CHECK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
    CUtensorMap tk, tv;
    const cuuint64_t dims[4] = {kD, 16, kHkv, static_cast<cuuint64_t>(nb)};
    const cuuint64_t strides[3] = {kD, 16 * kD, 16 * kD * kHkv};
    const cuuint32_t box[4] = {kD, 16, 1, 1}, one[4] = {1, 1, 1, 1};
    for (int a = 0; a < 2; ++a)
        if (reinterpret_cast<EncodeFn>(fn)(a ? &tv : &tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, a ? V : K, dims, strides,
                                           box, one, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            std::printf("tensor map encoding failed\n");
            return 1;
        }
    const size_t tma_smem = 1024 + 12 * 2 * kHalf + 4 * 12 * sizeof(uint64_t);
    CHECK(cudaFuncSetAttribute(tma_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(tma_smem)));
    for (int prod : {2, 4, 8}) {
        const float us = median_us([&] { tma_probe<<<C, 32 * (4 + prod), tma_smem>>>(tk, tv, pg, prod, d_err); });
        std::printf("tma producers=%d: %.2f us %.1f GB/s\n", prod, us, kv / us / 1e3);
    }
    const size_t cp_smem = 4 * 3 * 2 * kHalf;
    CHECK(cudaFuncSetAttribute(cpasync_probe<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(cp_smem)));
    {
        const float us = median_us([&] { cpasync_probe<4><<<C, 128, cp_smem>>>(K, V, pg); });
        std::printf("cpasync warps=4 ring=3: %.2f us %.1f GB/s\n", us, kv / us / 1e3);
    }
    {
        const float us = median_us([&] { ldg_probe<<<C, 256>>>(K, V, pg, d_err + 1); });
        std::printf("ldg warps=16/SM: %.2f us %.1f GB/s\n", us, kv / us / 1e3);
    }
    unsigned err[2];
    CHECK(cudaMemcpy(err, d_err, sizeof(err), cudaMemcpyDeviceToHost));
    std::printf("wait errors: %u\n", err[0]);
    return err[0] != 0;
}
