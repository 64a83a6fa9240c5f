// Static split of one launch's attended pages over its CTAs.
//
// The pages of every (sequence, kv head) unit are laid end to end (P pages in
// all) and cut into C contiguous ranges of equal size (+-1 page), one per CTA:
// CTA c takes [c*P/C, (c+1)*P/C).  Equal ranges measured fastest on GB300;
// ranges weighted towards either half of the grid (the first and the second
// resident CTA of each SM) were slower.  Plain host/device arithmetic: the same
// functions run in the kernel and in the host-side checks.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define FP8KV_HD __host__ __device__ __forceinline__
#else
#define FP8KV_HD inline
#endif

namespace fp8kv {

struct Partition {
    int64_t P;  // pages
    int C;      // CTAs with work (1 <= C <= P)
};

FP8KV_HD Partition make_partition(int64_t P, int C) { return Partition{P, C}; }

// First page of CTA c's range; range_start(q, C) == P.
FP8KV_HD int64_t range_start(const Partition& q, int c) { return static_cast<int64_t>(c) * q.P / q.C; }

// The CTA whose range holds page p (0 <= p < P): the largest c with
// c * P / C <= p, i.e. c * P < (p + 1) * C.
FP8KV_HD int cta_of(const Partition& q, int64_t p) { return static_cast<int>(((p + 1) * q.C - 1) / q.P); }

}  // namespace fp8kv

#undef FP8KV_HD
