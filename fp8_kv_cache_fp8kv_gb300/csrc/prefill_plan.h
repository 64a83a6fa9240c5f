// Key-range split plan of the chunked prefill (host code, plain C++).
//
// A prefill unit is (tile of query rows, kv head, sequence).  When the units
// do not fill one wave of resident CTAs, each unit's key pages are split
// over several CTAs whose FP32 partials a merge kernel combines.  The split
// count minimises
//     waves(units * splits) * (pages per split + kSplitCtaPages)
//         + (splits > 1 ? kMergePages : 0)
// where kSplitCtaPages stands for a CTA's fixed cost (query tile, first load
// latency, partial write) and kMergePages for the merge kernel, both in units
// of one page's work; each split covers at least kMinSplitPages pages, and
// there are at most kMaxSplits.
#pragma once

#include <cstdint>

namespace fp8kv {
namespace prefill {

constexpr int kMaxSplits = 64;
constexpr int kMinSplitPages = 8;       // a split covers at least 128 keys
constexpr int64_t kSplitCtaPages = 8;
constexpr int64_t kMergePages = 4;

// units: CTAs without splitting; pages: the most key pages a unit attends;
// slots: CTAs resident at once on the device (SMs x CTAs per SM).
inline int choose_splits(int64_t units, int64_t pages, int64_t slots) {
    if (units <= 0 || slots <= 0 || units >= slots) return 1;
    auto cost = [&](int64_t sp) {
        const int64_t waves = (units * sp + slots - 1) / slots;
        return waves * ((pages + sp - 1) / sp + kSplitCtaPages) + (sp > 1 ? kMergePages : 0);
    };
    int best = 1;
    int64_t best_cost = cost(1);
    for (int sp = 2; sp <= kMaxSplits && static_cast<int64_t>(sp) * kMinSplitPages <= pages; ++sp) {
        const int64_t c = cost(sp);
        if (c < best_cost) {
            best = sp;
            best_cost = c;
        }
    }
    return best;
}

}  // namespace prefill
}  // namespace fp8kv
