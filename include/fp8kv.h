/*
 * libfp8kv -- fp8 (E4M3) paged KV cache: quantise-on-append, single-query
 * (decode) grouped-query attention and chunked-prefill attention over the
 * cache, for NVIDIA GB300 (sm_103a).
 *
 * Sources the operations follow (the FP8 KV-cache web pages):
 *   [G] gpusmith.com, "FP8 KV Cache Quantization: Capacity Gains and Accuracy
 *       Risk": "What FP8 KV changes" (E4M3, 1 byte/element, max normal 448),
 *       "Scales and calibration" (divide by a per-tensor scale, then cast),
 *       "Attention backend interactions" (the kernel must read fp8 directly,
 *       dequantisation fused), "Why the KV cache sets long-context capacity"
 *       (paged, block-granular cache).
 *   [P] particula.tech, "KV Cache Quantization: What FP8 and q8_0 Cost in
 *       Accuracy", opening section (partial results accumulate in real FP32
 *       registers).
 *   [V] phantomic12 summary of the vLLM FP8 KV-cache blog: "ACCURACY AT LONG
 *       CONTEXT" (the P.V contraction runs over the context, >= 100K tokens),
 *       "DECODE COST" (sliding windows of 128 and 512).
 *   [A] phantomic12 record flops/ctx-fp8-kv-cache-long-context-accuracy:
 *       "Arithmetic intensity" (decode attention streams the cache at about
 *       2g flop per fp8 byte: memory-bound).
 *
 * Conventions for every entry point:
 *   - All pointers except `stream` are DEVICE pointers owned by the caller.
 *     The library allocates nothing and keeps no state between calls (the one
 *     exception is the fixed scratch array of fp8kv_paged_decode_noalloc).
 *     The entry points are safe to call from several host threads.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  Nothing is synchronised.
 *   - Invalid arguments return an error status and launch nothing.  A failed
 *     launch returns FP8KV_ERR_CUDA.  Faults during execution surface at the
 *     caller's next synchronisation, as for any CUDA kernel.
 *   - bf16 means IEEE bfloat16 stored as 2-byte little-endian values.
 */
#ifndef FP8KV_H_
#define FP8KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8KV_OK = 0,
    FP8KV_ERR_INVALID_ARG = 1, /* null pointer, bad size, non-finite/<=0 scale, misalignment */
    FP8KV_ERR_UNSUPPORTED = 2, /* shape outside the supported set (see below)                */
    FP8KV_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the required size         */
    FP8KV_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed                 */
    FP8KV_ERR_TIMEOUT = 5      /* a kernel gave up a bounded wait (read via fp8kv_read_error) */
} fp8kv_status;

/* Static, human-readable name of a status code. */
const char* fp8kv_status_string(fp8kv_status status);

/*
 * Quantise-on-append [G "Scales and calibration"; G "What FP8 KV changes"].
 *
 * For every token t < num_tokens, kv head h and dim i:
 *     code = E4M3( fp32(k_new[t][h][i]) / k_scale )     (same for V)
 * with one IEEE fp32 division followed by one round-to-nearest-even,
 * saturating-finite conversion (|x| >= 448 -> +-448, NaN -> NaN).  The code
 * is written at slot s = slot_mapping[t] = block * block_size + offset:
 *     k_cache[block][h][offset][i] = code.
 *
 *   k_new, v_new   bf16 [num_tokens][num_kv_heads][head_dim], contiguous,
 *                  16-byte aligned
 *   slot_mapping   int64 [num_tokens]; a negative slot skips the token (padding);
 *                  a slot >= num_blocks * block_size is out of range and is
 *                  skipped too (nothing is written for it)
 *   k_cache,       uint8 E4M3 [num_blocks][num_kv_heads][block_size][head_dim]
 *   v_cache        (one page = one (block, head) pair = block_size*head_dim
 *                  contiguous bytes), 16-byte aligned
 *   k_scale,       per-tensor scales, finite and > 0
 *   v_scale
 * Supported: head_dim % 16 == 0 and 16 <= head_dim <= 1024; block_size >= 1.
 * num_tokens == 0 is a no-op.
 */
fp8kv_status fp8kv_quant_append(const void* k_new, const void* v_new,
                                const int64_t* slot_mapping, int64_t num_tokens,
                                uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                                int block_size, int num_kv_heads, int head_dim,
                                float k_scale, float v_scale, void* stream);

/*
 * Workspace bytes fp8kv_paged_decode needs for this problem on the CURRENT
 * device (the split-context plan depends on its SM count).  Returns 0 if the
 * arguments are invalid or no device is available.
 */
size_t fp8kv_paged_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                         int head_dim, int max_seq_len, int block_size,
                                         int window);

/*
 * Zero-fills a workspace (asynchronously on `stream`).  A workspace must be
 * zero-filled once before its first fp8kv_paged_decode call; every call that
 * completes leaves it ready for the next one (its per-unit split counters
 * back at zero).  After a call that failed with
 * FP8KV_ERR_TIMEOUT the workspace must be zero-filled again.  Calls that share one workspace must be ordered (same
 * stream or explicit dependencies).
 */
fp8kv_status fp8kv_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Reads (and clears) the workspace's error word: 0 = no error, otherwise an
 * fp8kv_status (FP8KV_ERR_TIMEOUT, or FP8KV_ERR_INVALID_ARG for an
 * out-of-range block id met on the device).  Synchronises `stream`.
 */
fp8kv_status fp8kv_read_error(void* workspace, uint32_t* code, void* stream);

/*
 * Paged fp8 decode attention [G "Attention backend interactions";
 * V "ACCURACY AT LONG CONTEXT"; P opening section].
 *
 * For batch b, query head h (kv head hk = h / g, g = num_q_heads/num_kv_heads),
 * with L = seq_lens[b] (the current token included) and the attended keys
 * t in [lo, L), lo = (window > 0 && L > window) ? L - window : 0:
 *     k^_t = decode(k_cache[page(t)][hk][t % bs][:]) * k_scale
 *     v^_t = decode(v_cache[page(t)][hk][t % bs][:]) * v_scale
 *     s_t  = sm_scale * sum_i q[b][h][i] * k^_t[i]
 *     out[b][h][:] = sum_t exp(s_t - max s) v^_t / sum_t exp(s_t - max s)
 * page(t) = block_tables[b][t / block_size].  Scores, the softmax and P.V are
 * accumulated in FP32; split-context partial results are merged in FP32; the
 * result is rounded to bf16 (RNE).  L == 0 writes zeros.
 *
 *   q              bf16 [batch][num_q_heads][head_dim], contiguous, 16-B aligned
 *   k_cache,       uint8 E4M3 [num_blocks][num_kv_heads][block_size][head_dim],
 *   v_cache        16-byte aligned (the layout fp8kv_quant_append writes)
 *   block_tables   int32 [batch][max_blocks_per_seq]; entries past a sequence's
 *                  last page are never read; an entry outside [0, num_blocks)
 *                  is replaced by block 0 and reported via fp8kv_read_error
 *   seq_lens       int32 [batch] on the device; each must satisfy
 *                  0 <= seq_lens[b] <= min(max_seq_len, max_blocks_per_seq*block_size)
 *   max_seq_len    host-side upper bound of seq_lens (sizes the split plan)
 *   sm_scale       softmax scale (usually 1/sqrt(head_dim)); finite
 *   window         <= 0: full attention; > 0: attend the last `window` keys
 *   out            bf16 [batch][num_q_heads][head_dim], 16-byte aligned
 *   workspace      >= fp8kv_paged_decode_workspace_size(...) bytes, 256-B
 *                  aligned, zero-filled before first use (fp8kv_workspace_init)
 * Supported: head_dim in {64, 128, 256}; block_size == 16;
 *            g in {1, 2, 4, 8, 16}; num_blocks * num_kv_heads < 2^31.  At g = 16
 *            each kv head runs as two units of 8 query heads, each reading the
 *            head's pages (the kernels put a unit's heads on the MMA's n side).
 */
fp8kv_status fp8kv_paged_decode(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                int64_t num_blocks, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* seq_lens,
                                int max_seq_len, int batch, int num_q_heads, int num_kv_heads,
                                int head_dim, int block_size, float k_scale, float v_scale,
                                float sm_scale, int window, void* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Per-attention-head scales [G "Scales and calibration": per-tensor or
 * per-attention-head k/v scales, [num_kv_heads] each].
 *
 * The same operations as fp8kv_quant_append, fp8kv_paged_decode and
 * fp8kv_decode_step, with one K scale and one V scale per kv head instead of
 * one per tensor: elements of kv head h are divided by k_scales[h]
 * (v_scales[h]) before the cast, and its codes stand for
 * decode(code) * scale[h] in the attention.
 *
 *   k_scales, v_scales  DEVICE fp32 [num_kv_heads], 4-byte aligned, finite and
 *                       > 0 (not checked on the device: other values give
 *                       unspecified codes and outputs); read by the kernels
 *                       after they wait for the previous work on the stream.
 *   all other arguments, the workspace and the errors as the per-tensor calls.
 * With every k_scales[h] == k_scale and v_scales[h] == v_scale the results
 * are bit-identical to the per-tensor calls.
 */
fp8kv_status fp8kv_quant_append_per_head(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                         int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                         int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                                         const float* k_scales, const float* v_scales, void* stream);

fp8kv_status fp8kv_paged_decode_per_head(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                         int64_t num_blocks, const int32_t* block_tables,
                                         int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                         int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, const float* k_scales, const float* v_scales,
                                         float sm_scale, int window, void* out, void* workspace,
                                         size_t workspace_bytes, void* stream);

fp8kv_status fp8kv_decode_step_per_head(const void* q, const void* k_new, const void* v_new,
                                        uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                                        const int32_t* block_tables, int max_blocks_per_seq,
                                        const int32_t* seq_lens, int max_seq_len, int batch,
                                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                        const float* k_scales, const float* v_scales, float sm_scale,
                                        int window, void* out, void* workspace, size_t workspace_bytes,
                                        void* stream);

/*
 * The E5M2 cache [G "What FP8 KV changes": the other FP8 format, 2 mantissa
 * bits and a maximum of 57,344; E4M3 is the default].
 *
 * The same operations as fp8kv_quant_append, fp8kv_paged_decode and
 * fp8kv_decode_step with E5M2 codes (S.EEEEE.MM, exponent bias 15,
 * subnormals m * 2^-16): code = E5M2(fp32(x) / scale) with one IEEE fp32
 * division and one round-to-nearest-even, saturating-finite conversion
 * (|x| >= 57344 and infinities -> +-57344, NaN -> NaN).  A code stands for
 * its exact value times the scale; E5M2 values are exact in f16, so the
 * decode runs the same tensor-core path.  Arguments, layout, workspace and
 * errors as the E4M3 calls.
 */
fp8kv_status fp8kv_quant_append_e5m2(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                     int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                     int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                                     float k_scale, float v_scale, void* stream);

fp8kv_status fp8kv_paged_decode_e5m2(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                     int64_t num_blocks, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                     int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, float k_scale, float v_scale, float sm_scale,
                                     int window, void* out, void* workspace, size_t workspace_bytes,
                                     void* stream);

fp8kv_status fp8kv_decode_step_e5m2(const void* q, const void* k_new, const void* v_new,
                                    uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* seq_lens, int max_seq_len, int batch,
                                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                    float k_scale, float v_scale, float sm_scale, int window, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Which units perform the two contractions of the decode attention. */
typedef enum {
    FP8KV_ENGINE_DEFAULT = 0,      /* the library's choice for the shape (the faster one measured) */
    FP8KV_ENGINE_TENSOR_CORES = 1, /* m16n8k16 f16 MMA per stage tile, folded into FP32 registers */
    FP8KV_ENGINE_CUDA_CORES = 2    /* FP32 fma chains of exact f16 products on the CUDA cores     */
} fp8kv_engine;

/*
 * fp8kv_paged_decode with the contraction engine chosen by the caller
 * [P opening section (FP32 accumulation); A "Arithmetic intensity" (at M = g
 * the contractions are small next to the bytes streamed, so either unit may
 * keep up; the default is the one measured faster)].
 *
 * Same operation, arguments, workspace and errors as fp8kv_paged_decode; the
 * engines differ only in rounding order (both accumulate in FP32 and meet the
 * same tolerance).  An engine value outside fp8kv_engine is
 * FP8KV_ERR_INVALID_ARG.
 */
fp8kv_status fp8kv_paged_decode_engine(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                       int64_t num_blocks, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* seq_lens,
                                       int max_seq_len, int batch, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, float k_scale, float v_scale,
                                       float sm_scale, int window, void* out, void* workspace,
                                       size_t workspace_bytes, void* stream, int engine);

/*
 * The bf16 twin of fp8kv_paged_decode: the same attention over a paged cache
 * that stores bf16 K and V instead of E4M3 codes -- the baseline the fp8 cache
 * is compared against [G "What FP8 KV changes" (1 byte per element against
 * bf16's 2); V "DECODE COST" (cost per cached token, fp8 against bf16)].
 *
 *   k_cache, v_cache  bf16 [num_blocks][num_kv_heads][block_size][head_dim],
 *                     16-byte aligned (no scales: the values are the cache)
 *   all other arguments, the workspace and the errors as fp8kv_paged_decode.
 *
 * Scores and P.V run on the tensor cores with bf16 operands (P rounded to
 * bf16) and FP32 accumulation, each stage's tile added into FP32 registers.
 * Supported: head_dim in {64, 128, 256}; block_size == 16; g in {1, 2, 4, 8, 16}.
 */
fp8kv_status fp8kv_paged_decode_bf16(const void* q, const void* k_cache, const void* v_cache,
                                     int64_t num_blocks, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* seq_lens,
                                     int max_seq_len, int batch, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, float sm_scale, int window,
                                     void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * One decode step: append, then attend [G "Scales and calibration";
 * G "Attention backend interactions"; V "ACCURACY AT LONG CONTEXT"].
 *
 * Equivalent to fp8kv_quant_append of each sequence's newest row followed by
 * fp8kv_paged_decode, in one launch: for every b with
 * L = seq_lens[b] > 0 the row k_new[b] (v_new[b]) is quantised exactly as
 * fp8kv_quant_append does and written at token L-1 of the sequence, i.e. at
 * page block_tables[b][(L-1)/block_size], offset (L-1) % block_size; then the
 * attention of fp8kv_paged_decode runs over the cache including that token.
 *
 *   k_new, v_new   bf16 [batch][num_kv_heads][head_dim], 16-byte aligned
 *   all other arguments as for fp8kv_paged_decode (k_cache / v_cache are
 *   written).  Sequences of length 0 append nothing; a page whose block id is
 *   out of range is not written (the error word reports it).
 */
fp8kv_status fp8kv_decode_step(const void* q, const void* k_new, const void* v_new, uint8_t* k_cache,
                               uint8_t* v_cache, int64_t num_blocks, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                               int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               float k_scale, float v_scale, float sm_scale, int window, void* out,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * fp8kv_decode_step for a caller whose per-step inputs and result live in
 * host memory (an engine that computes q and the new K/V rows on the host, or
 * a test harness).  No counterpart on the pages: it only moves the step's
 * inputs and output across the host link around the step above.
 *
 * On `stream`, in order: one copy of in_bytes bytes from h_in to d_in, the
 * decode step, and the step's output (batch*num_q_heads*head_dim bf16) into
 * h_out.  When the device can address h_out (page-locked host memory under
 * unified addressing, e.g. cudaHostAlloc or a registered buffer) the step's
 * kernels store the output there directly, across the host link, and `out`
 * is not written; otherwise the output goes to `out` and one copy moves it
 * to h_out.  It returns once the work is enqueued; h_out is valid after the
 * caller synchronises the stream.
 *
 *   h_in    host buffer (page-locked for an asynchronous copy) holding the
 *           step's inputs exactly as they must appear at d_in
 *   d_in    device buffer of in_bytes bytes; q, k_new, v_new and seq_lens are
 *           device pointers, usually into d_in (the caller chooses the layout)
 *   h_out   host buffer for the output (page-locked for an asynchronous copy)
 *   all other arguments as for fp8kv_decode_step.
 * Errors: those of fp8kv_decode_step (checked before anything is enqueued);
 * null h_in, d_in or h_out with in_bytes > 0 is FP8KV_ERR_INVALID_ARG; a
 * failed copy is FP8KV_ERR_CUDA.
 */
fp8kv_status fp8kv_decode_step_host(const void* h_in, void* d_in, size_t in_bytes, void* h_out,
                                    const void* q, const void* k_new, const void* v_new, uint8_t* k_cache,
                                    uint8_t* v_cache, int64_t num_blocks, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                    int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, float k_scale, float v_scale, float sm_scale, int window,
                                    void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free paged decode.  This entry point has no counterpart on the
 * pages: it exists for callers that cannot allocate device memory when they
 * decode -- e.g. a serving engine that reserved nearly all HBM for its own
 * paged KV pool, host code under a no-allocation rule, or a binding without a
 * CUDA allocator -- and so cannot provide the workspace fp8kv_paged_decode
 * takes.  It computes exactly what fp8kv_paged_decode computes, with the same
 * arguments minus the workspace.
 *
 * Scratch: a fixed 8 MiB array compiled into the library (every device that
 * loads the library keeps it until the process exits).  The call allocates
 * nothing and calls no allocating routine; it zeroes the array's header
 * (the error word) and its per-unit split counters (one cudaMemsetAsync on
 * `stream`), and then runs the decode.  The split partials need no clearing:
 * every call writes the ones it reads.
 *   - A problem whose split-merge scratch would exceed 8 MiB is rejected with
 *     FP8KV_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress); make that first call before
 *     any stream capture.  The address is kept for the life of the process:
 *     after a device reset (cudaDeviceReset) the array moves, so do not call
 *     this entry point on a device that was reset.
 *   - All calls share the one array: calls that overlap on the GPU (different
 *     streams without ordering, or different host threads) race and corrupt
 *     each other's results.  Order them.
 *   - Device-side errors (an out-of-range block id) are not reported by this
 *     variant; use fp8kv_paged_decode with a workspace to read them.
 */
fp8kv_status fp8kv_paged_decode_noalloc(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                        int64_t num_blocks, const int32_t* block_tables,
                                        int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                        int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                        int block_size, float k_scale, float v_scale, float sm_scale,
                                        int window, void* out, void* stream);

/*
 * Chunked-prefill attention over the paged E4M3 cache [G "Attention backend
 * interactions" (the prefill pass reads the same fp8 cache as decode);
 * V "ACCURACY AT LONG CONTEXT" (P.V over the context in FP32)].
 *
 * Sequence b holds L = seq_lens[b] tokens in the cache, its n = q_len[b] =
 * q_starts[b+1] - q_starts[b] newest ones included (append them first with
 * fp8kv_quant_append).  Query row i < n of the sequence sits at position
 * p = L - n + i and attends the keys t in [lo(p), p], lo(p) = (window > 0 &&
 * p + 1 > window) ? p + 1 - window : 0 -- causal, optionally within a
 * sliding window; row by row this is fp8kv_paged_decode of a sequence of
 * length p + 1:
 *     s_t = sm_scale * sum_i q[r][h][i] * decode(k code of t)[i] * k_scale
 *     out[r][h][:] = sum_t exp(s_t - max s) decode(v code of t) * v_scale
 *                    / sum_t exp(s_t - max s)
 * with r = q_starts[b] + i.  Scores, the softmax and P.V accumulate in FP32
 * (key-range partials, when the call splits a long range over several CTAs,
 * are merged in FP32); the result is rounded to bf16 (RNE).
 *
 *   q              bf16 [num_q_tokens][num_q_heads][head_dim], the query rows of
 *                  all sequences packed in order, 16-byte aligned
 *   num_q_tokens   rows of q and out (q_starts[batch])
 *   k_cache,       uint8 E4M3 caches, layout as fp8kv_paged_decode
 *   v_cache
 *   block_tables   int32 [batch][max_blocks_per_seq]; only the pages a query
 *                  attends are read
 *   seq_lens       int32 [batch] on the device, 0 <= seq_lens[b] <= max_seq_len
 *   q_starts       int32 [batch + 1] on the device, non-decreasing, q_starts[0] = 0,
 *                  q_starts[b+1] - q_starts[b] <= min(seq_lens[b], max_q_len)
 *   max_q_len      host-side upper bound of the q_len (sizes the grid)
 *   window         <= 0: causal over the whole prefix; > 0: the last `window` keys
 *   out            bf16 [num_q_tokens][num_q_heads][head_dim], 16-byte aligned
 *   workspace      >= fp8kv_paged_prefill_workspace_size(...) bytes, 256-byte
 *                  aligned, zero-filled before first use (fp8kv_workspace_init);
 *                  its first word is the error word fp8kv_read_error reads: an
 *                  out-of-range block id (block 0 is read instead), or a
 *                  seq_lens / q_starts entry outside the bounds above (the
 *                  sequence is clamped, or skipped if its rows would fall
 *                  outside q / out).  Calls that share a workspace must be
 *                  ordered.  Missing or too small: FP8KV_ERR_WORKSPACE.
 * Supported: head_dim in {64, 128, 256}; block_size == 16; g in {1, 2, 4, 8, 16};
 *            num_blocks * num_kv_heads < 2^31.  batch == 0, max_q_len == 0 or
 *            num_q_tokens == 0 is a no-op.
 */
/*
 * Workspace bytes fp8kv_paged_prefill needs for this problem on the CURRENT
 * device: the key-range split plan depends on its SM count and on how many
 * prefill CTAs it holds at once.  At least 256 (the error word); larger
 * when the call splits key ranges.  Returns 0 if the arguments are invalid
 * or no device is available.
 */
size_t fp8kv_paged_prefill_workspace_size(int batch, int max_q_len, int max_seq_len, int num_q_heads,
                                          int num_kv_heads, int head_dim, int block_size, int window);

fp8kv_status fp8kv_paged_prefill(const void* q, int64_t num_q_tokens, const uint8_t* k_cache,
                                 const uint8_t* v_cache, int64_t num_blocks, const int32_t* block_tables,
                                 int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* q_starts,
                                 int max_q_len, int max_seq_len, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size, float k_scale,
                                 float v_scale, float sm_scale, int window, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Failure-path test hooks.  No counterpart on the pages: the pages' failure
 * mode is silent (a wrong answer, no error), and these make the library's
 * answer to a stall observable.  A kernel wait that runs out writes
 * FP8KV_ERR_TIMEOUT into the workspace error word, waits (with the normal
 * limit) for the copies it has in flight, frees what it holds and returns.
 * Later calls on that workspace skip their work until it is zero-filled again
 * (fp8kv_workspace_init).  Nothing faults and nothing hangs: every wait is
 * bounded.
 *
 * fp8kv_debug_paged_decode_stall: fp8kv_paged_decode_engine with
 * FP8KV_ENGINE_CUDA_CORES (the engine whose copies run through barriers),
 * except that the K producer of CTA 0 never issues stage `stall_stage` and
 * every ring wait gives up after wait_limit_ns nanoseconds.
 *
 * fp8kv_debug_paged_prefill_stall: fp8kv_paged_prefill, except that CTA
 * (0, 0, 0) never issues the score MMAs of stage `stall_stage` and the MMA
 * waits give up after wait_limit_ns nanoseconds.
 *
 * Both: stall_stage >= 0 and 0 < wait_limit_ns <= 500,000,000, else
 * FP8KV_ERR_INVALID_ARG; all other arguments and errors as the wrapped call.
 */
fp8kv_status fp8kv_debug_paged_decode_stall(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                            int64_t num_blocks, const int32_t* block_tables,
                                            int max_blocks_per_seq, const int32_t* seq_lens, int max_seq_len,
                                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, float k_scale, float v_scale, float sm_scale,
                                            int window, void* out, void* workspace, size_t workspace_bytes,
                                            void* stream, int stall_stage, uint64_t wait_limit_ns);

fp8kv_status fp8kv_debug_paged_prefill_stall(const void* q, int64_t num_q_tokens, const uint8_t* k_cache,
                                             const uint8_t* v_cache, int64_t num_blocks,
                                             const int32_t* block_tables, int max_blocks_per_seq,
                                             const int32_t* seq_lens, const int32_t* q_starts, int max_q_len,
                                             int max_seq_len, int batch, int num_q_heads, int num_kv_heads,
                                             int head_dim, int block_size, float k_scale, float v_scale,
                                             float sm_scale, int window, void* out, void* workspace,
                                             size_t workspace_bytes, void* stream, int stall_stage,
                                             uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* FP8KV_H_ */
