// NVTX ranges around the library's entry points, so that a profiler
// (Nsight Systems, or ncu with --nvtx) shows each call and the kernels it
// launched under the call's name.  NVTX v3 is header-only: with no tool
// attached a range costs a few nanoseconds and loads nothing.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace fp8kv {

struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace fp8kv

// Opens a range named after the enclosing entry point for the rest of its scope.
#define FP8KV_TRACE(name) ::fp8kv::TraceRange fp8kv_trace_range_(name)
