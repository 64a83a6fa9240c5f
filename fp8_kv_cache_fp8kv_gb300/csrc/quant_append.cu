// Quantise-on-append: bf16 K/V rows -> E4M3 codes written into cache pages
// through a slot mapping.
//
// The operation is the one gpusmith.com, "FP8 KV Cache Quantization: Capacity
// Gains and Accuracy Risk", describes in "Scales and calibration" (each K and
// V tensor is divided by a scale, then cast; one scale per tensor, or one per
// kv head for the per-attention-head granularity) with the format of
// "What FP8 KV changes" (E4M3, 1 byte per element, maximum normal 448).  The
// divide is one IEEE fp32 division; the cast is the hardware's
// round-to-nearest-even, saturating-finite conversion.
//
// The same kernel writes E5M2 codes (the other FP8 format: 2 mantissa bits,
// maximum 57,344, same page) when asked for them.
//
// HBM-bound elementwise kernel: each thread turns 16 bf16 values (32 bytes,
// two 16-byte loads) into 16 codes (one 16-byte store).  The grid is a
// multiple of the SM count and strides over all (token, head, 16-dim chunk)
// work items of K and then V.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fp8kv.h"
#include "trace.cuh"
#include "ptx.cuh"

namespace fp8kv {

template <bool E5M2>
__global__ void __launch_bounds__(256) quant_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, const int64_t* __restrict__ slot_mapping,
    int64_t num_tokens, uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, int64_t num_slots,
    int num_kv_heads, int head_dim, int block_size, float k_scale, float v_scale,
    const float* __restrict__ k_scales, const float* __restrict__ v_scales) {
    // A decode launched right after may get resident now (it waits for this
    // grid before reading anything).
    griddep_launch_dependents();
    // This grid may have started before the previous one on the stream
    // finished (programmatic launch): that grid may have produced the inputs
    // or still read the cache, so wait for it before touching either.
    griddep_wait();
    const int64_t chunks_per_row = head_dim / 16;
    const int64_t chunks_per_token = chunks_per_row * num_kv_heads;
    const int64_t per_tensor = num_tokens * chunks_per_token;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < 2 * per_tensor;
         i += stride) {
        const bool is_v = i >= per_tensor;
        const int64_t j = is_v ? i - per_tensor : i;
        const int64_t t = j / chunks_per_token;
        const int64_t rem = j - t * chunks_per_token;
        const int64_t hk = rem / chunks_per_row;
        const int64_t c = rem - hk * chunks_per_row;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0 || slot >= num_slots) continue;
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        const uint4* src = (is_v ? v_new : k_new) + 2 * j;
        const uint4 a = __ldcs(src);
        const uint4 b = __ldcs(src + 1);
        // per-tensor scale, or the kv head's own one ([Hkv] arrays)
        const float* hs = is_v ? v_scales : k_scales;
        const float s = hs ? __ldg(hs + hk) : (is_v ? v_scale : k_scale);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // two bf16 words = four consecutive elements e0..e3 (e0 in the low half)
            const uint32_t w0 = w[2 * q], w1 = w[2 * q + 1];
            const float e0 = __uint_as_float(w0 << 16), e1 = __uint_as_float(w0 & 0xFFFF0000u);
            const float e2 = __uint_as_float(w1 << 16), e3 = __uint_as_float(w1 & 0xFFFF0000u);
            uint16_t lo, hi;
            if constexpr (E5M2) {
                lo = f32x2_to_e5m2x2_satfinite(__fdiv_rn(e0, s), __fdiv_rn(e1, s));
                hi = f32x2_to_e5m2x2_satfinite(__fdiv_rn(e2, s), __fdiv_rn(e3, s));
            } else {
                lo = f32x2_to_e4m3x2_satfinite(__fdiv_rn(e0, s), __fdiv_rn(e1, s));
                hi = f32x2_to_e4m3x2_satfinite(__fdiv_rn(e2, s), __fdiv_rn(e3, s));
            }
            o[q] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        uint8_t* dst = (is_v ? v_cache : k_cache) + ((blk * num_kv_heads + hk) * block_size + off) * head_dim + c * 16;
        *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace fp8kv

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool good_scale(float s) { return std::isfinite(s) && s > 0.0f; }

}  // namespace

namespace {

fp8kv_status append_impl(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t num_tokens,
                         uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks, int block_size, int num_kv_heads,
                         int head_dim, float k_scale, float v_scale, const float* k_scales, const float* v_scales,
                         void* stream, bool e5m2 = false) {
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || num_kv_heads < 1) return FP8KV_ERR_INVALID_ARG;
    if (!good_scale(k_scale) || !good_scale(v_scale)) return FP8KV_ERR_INVALID_ARG;
    if ((k_scales == nullptr) != (v_scales == nullptr)) return FP8KV_ERR_INVALID_ARG;
    if (k_scales && ((reinterpret_cast<uintptr_t>(k_scales) & 3u) || (reinterpret_cast<uintptr_t>(v_scales) & 3u)))
        return FP8KV_ERR_INVALID_ARG;
    if (head_dim % 16 != 0 || head_dim < 16 || head_dim > 1024) return FP8KV_ERR_UNSUPPORTED;
    if (!k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache)) return FP8KV_ERR_INVALID_ARG;
    if (num_tokens == 0) return FP8KV_OK;
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)) return FP8KV_ERR_INVALID_ARG;
    const int64_t kLimit = INT64_C(1) << 60;
    if (num_blocks > kLimit / (static_cast<int64_t>(block_size) * num_kv_heads * head_dim)) return FP8KV_ERR_INVALID_ARG;
    if (num_tokens > kLimit / (static_cast<int64_t>(num_kv_heads) * head_dim)) return FP8KV_ERR_INVALID_ARG;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8KV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FP8KV_ERR_CUDA;
    const int64_t items = 2 * num_tokens * num_kv_heads * (head_dim / 16);
    const int threads = 256;
    int64_t blocks = (items + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    // May get resident while the previous grid on the stream finishes; the
    // kernel waits for it (griddepcontrol.wait) before touching memory.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(
        &cfg, e5m2 ? fp8kv::quant_append_kernel<true> : fp8kv::quant_append_kernel<false>,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, num_tokens, k_cache,
        v_cache, num_blocks * block_size, num_kv_heads, head_dim, block_size, k_scale, v_scale, k_scales, v_scales);
    return err == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA;
}

}  // namespace

extern "C" fp8kv_status fp8kv_quant_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                           int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                           int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                                           float k_scale, float v_scale, void* stream) {
    FP8KV_TRACE("fp8kv_quant_append");
    return append_impl(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, block_size, num_kv_heads,
                       head_dim, k_scale, v_scale, nullptr, nullptr, stream);
}

extern "C" fp8kv_status fp8kv_quant_append_per_head(const void* k_new, const void* v_new,
                                                    const int64_t* slot_mapping, int64_t num_tokens,
                                                    uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                                                    int block_size, int num_kv_heads, int head_dim,
                                                    const float* k_scales, const float* v_scales, void* stream) {
    FP8KV_TRACE("fp8kv_quant_append_per_head");
    if (num_tokens > 0 && (!k_scales || !v_scales)) return FP8KV_ERR_INVALID_ARG;
    return append_impl(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, block_size, num_kv_heads,
                       head_dim, 1.0f, 1.0f, k_scales, v_scales, stream);
}

extern "C" fp8kv_status fp8kv_quant_append_e5m2(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                                int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                                int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                                                float k_scale, float v_scale, void* stream) {
    FP8KV_TRACE("fp8kv_quant_append_e5m2");
    return append_impl(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, block_size, num_kv_heads,
                       head_dim, k_scale, v_scale, nullptr, nullptr, stream, true);
}
