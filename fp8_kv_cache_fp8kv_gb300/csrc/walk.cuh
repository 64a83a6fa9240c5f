// How one CTA of the decode kernel walks its range of the flattened page list,
// and how its warps share that walk.
//
// The attended pages of every (sequence, kv head) unit are laid end to end:
// unit u = b*Hkv + hk holds pages [Hkv*pre[b] + hk*n_b, ... + n_b), where
// pre[] is the exclusive prefix of the per-sequence page counts n_b.  A CTA's
// range [s, e) overlaps one or more units; each overlap is a "segment".
// Every segment is cut into NW equal contiguous shares, one per warp of the
// CTA; the last warp's share ends with the segment's last page.  A warp reads
// the block ids of its shares in windows of up to 32 consecutive pages that
// never straddle a segment.
//
// Plain host/device integer arithmetic: the kernel and the host-side checks
// run the same functions.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define FP8KV_HD __host__ __device__ __forceinline__
#else
#define FP8KV_HD inline
#endif

namespace fp8kv {

struct Walker {
    int b, hk, n;   // sequence, kv head, pages per unit of this sequence
    int64_t base;   // global index of the unit's first page
    int64_t g;      // global index of the segment's first page
};

// The segment holding global page s (0 <= s < Hkv*pre[B]).
FP8KV_HD void walk_start(Walker& w, const int32_t* pre, int B, int Hkv, int64_t s) {
    int lo = 0, hi = B - 1;  // largest b with Hkv*pre[b] <= s (it has pages, since s < total)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(Hkv) * pre[mid] <= s) lo = mid; else hi = mid - 1;
    }
    w.b = lo;
    w.n = pre[lo + 1] - pre[lo];
    const int64_t off = s - static_cast<int64_t>(Hkv) * pre[lo];
    w.hk = static_cast<int>(off / w.n);
    w.base = static_cast<int64_t>(Hkv) * pre[lo] + static_cast<int64_t>(w.hk) * w.n;
    w.g = s;
}

// The next unit's segment (only called while the range continues past this unit).
FP8KV_HD void walk_next(Walker& w, const int32_t* pre, int Hkv) {
    if (++w.hk == Hkv) {
        w.hk = 0;
        do { ++w.b; } while (pre[w.b + 1] == pre[w.b]);
        w.n = pre[w.b + 1] - pre[w.b];
    }
    w.base = static_cast<int64_t>(Hkv) * pre[w.b] + static_cast<int64_t>(w.hk) * w.n;
    w.g = w.base;
}

// Pages of segment x of a range that ends at e.
FP8KV_HD int seg_pages(const Walker& x, int64_t e) {
    const int64_t end = x.base + x.n < e ? x.base + x.n : e;
    return static_cast<int>(end - x.g);
}

// Whether segment x ends where its unit ends (it holds the unit's last page).
FP8KV_HD bool seg_reaches_unit_end(const Walker& x, int64_t e) { return x.base + x.n <= e; }

// Whether the range continues past segment x.
FP8KV_HD bool seg_is_last(const Walker& x, int64_t e) { return x.base + x.n >= e; }

// Warp `warp` of `nw`: its share [q0, q1) of segment x (segment-relative pages).
FP8KV_HD void warp_share(const Walker& x, int64_t e, int warp, int nw, int& q0, int& q1) {
    const int64_t np = seg_pages(x, e);
    q0 = static_cast<int>(np * warp / nw);
    q1 = static_cast<int>(np * (warp + 1) / nw);
}

// A window of a warp's pages: [start, start + n) of segment w, n <= 32; the
// warp's share of that segment ends at hi.
struct WinPos {
    Walker w;
    int start, n, hi;
    bool valid;
};

FP8KV_HD WinPos make_win(const Walker& w, int start, int hi) {
    WinPos y;
    y.w = w;
    y.start = start;
    y.hi = hi;
    y.n = hi - start < 32 ? hi - start : 32;
    y.valid = true;
    return y;
}

// The first segment at or after x (x itself when `include_x`) in which the
// warp's share is not empty, as its first window; invalid if there is none.
FP8KV_HD WinPos first_window_from(Walker x, bool include_x, const int32_t* pre, int Hkv, int64_t e, int warp,
                                  int nw) {
    WinPos y;
    y.valid = false;
    y.w = x;
    y.start = y.n = y.hi = 0;
    if (!include_x) {
        if (seg_is_last(x, e)) return y;
        walk_next(x, pre, Hkv);
    }
    while (true) {
        int q0, q1;
        warp_share(x, e, warp, nw, q0, q1);
        if (q1 > q0) return make_win(x, q0, q1);
        if (seg_is_last(x, e)) return y;
        walk_next(x, pre, Hkv);
    }
}

// The window after x: the next 32 pages of the same share, else the first
// window of the next segment with a non-empty share.
FP8KV_HD WinPos next_window(const WinPos& x, const int32_t* pre, int Hkv, int64_t e, int warp, int nw) {
    if (!x.valid) return x;
    if (x.start + x.n < x.hi) return make_win(x.w, x.start + x.n, x.hi);
    return first_window_from(x.w, false, pre, Hkv, e, warp, nw);
}

// Whether window x holds its unit's last page (segment-relative page hi - 1).
FP8KV_HD bool window_holds_unit_end(const WinPos& x, int64_t e) {
    return x.valid && x.start + x.n == seg_pages(x.w, e) && seg_reaches_unit_end(x.w, e);
}

}  // namespace fp8kv

#undef FP8KV_HD
