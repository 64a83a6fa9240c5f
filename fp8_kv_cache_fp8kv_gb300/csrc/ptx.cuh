// Inline-PTX building blocks for the sm_103a kernels of libfp8kv: mbarriers,
// TMA tensor loads, the fp8/f16 conversions, the mixed-precision FP32 FMA of
// the CUDA-core path and the m16n8k16 tensor-core MMA.
// Every wait on an mbarrier is bounded in time; a wait that runs out reports
// failure to its caller instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace fp8kv {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most
// `limit_ns` nanoseconds.  Returns false if the wait ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- programmatic dependent launch

// Lets the grid launched after this one on the stream start early.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits until the grids this one depends on have completed and their memory
// operations are visible.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- TMA

// 4-D tiled tensor load into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const void* tmap, uint64_t* bar, int c0, int c1,
                                            int c2, int c3, uint64_t cache_policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)),
        "l"(cache_policy)
        : "memory");
}

// 16-byte asynchronous global -> shared copy (L2 only, no L1 allocation) with
// an L2 cache-policy hint.  Completion is tracked per thread by commit groups.
__device__ __forceinline__ void cp_async_16(uint32_t smem_dst, const void* src, uint64_t cache_policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_dst), "l"(src),
                 "l"(cache_policy)
                 : "memory");
}

// The same copy with the default L2 policy.
__device__ __forceinline__ void cp_async_16(uint32_t smem_dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(src) : "memory");
}

// Closes the calling thread's current group of cp.async copies.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Waits until at most N of the calling thread's most recent copy groups are
// still in flight.  Copies always complete: this wait ends by itself.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Orders this thread's earlier generic-proxy global writes before its (and,
// after a barrier, its group's) later async-proxy operations such as TMA loads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------- conversions

// Two E4M3 codes (low byte first) -> f16x2 (exact: every E4M3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two_codes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two_codes));
    return r;
}

// Both halves of a 32-bit word of codes -> two f16x2 (bytes 0,1 -> lo; 2,3 -> hi).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Both halves of a 32-bit word of E5M2 codes -> two f16x2.  An E5M2 code is
// the upper byte of the f16 with the same value (same sign, 5 exponent bits
// with bias 15, leading 2 mantissa bits), so this is a byte move.
__device__ __forceinline__ void e5m2x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("prmt.b32 %0, %1, 0, 0x1404;" : "=r"(lo) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0x3424;" : "=r"(hi) : "r"(w));
}

// fp32 pair -> E5M2 pair with round-to-nearest-even and saturation to
// +-57344; `lo` lands in bits 0-7, `hi` in bits 8-15.
__device__ __forceinline__ uint16_t f32x2_to_e5m2x2_satfinite(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// fp32 pair -> E4M3 pair with round-to-nearest-even and saturation to +-448;
// `lo` lands in bits 0-7, `hi` in bits 8-15.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2_satfinite(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- CUDA-core FP32 accumulation

// acc_lo += a.lo * b.lo, acc_hi += a.hi * b.hi for f16x2 words a, b: the
// products of two f16 values are exact in FP32 and each sum is rounded once
// to FP32 (mixed-precision fma, f16 operands, FP32 addend and result).
__device__ __forceinline__ void fma_f16x2_f32(float& acc_lo, float& acc_hi, uint32_t a, uint32_t b) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(a), "r"(b));
}

// acc_lo += a.lo * b, acc_hi += a.hi * b for an f16x2 word a and an f16 b.
__device__ __forceinline__ void fma_f16x2_f16_f32(float& acc_lo, float& acc_hi, uint32_t a, uint16_t b) {
    asm("{\n\t.reg .b16 al, ah;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, %3, %0;\n\t"
        "fma.rn.f32.f16 %1, ah, %3, %1;\n\t}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(a), "h"(b));
}

// ---------------------------------------------------------------- tensor cores

// D = A(16x16, row) * B(16x8, col) + C, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// The same with bf16 operands.
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                               const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// Transposes an 8x8 matrix of 16-bit values held in the m16n8 fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t r;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

}  // namespace fp8kv
