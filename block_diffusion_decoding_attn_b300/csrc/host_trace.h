// NVTX ranges around the C ABI's compute entry points, so that a profiler's
// timeline (Nsight Systems, or ncu with --nvtx) shows which call enqueued
// which kernels. The NVTX v3 headers are header-only: with no tool attached a
// range costs one call through a function pointer that does nothing. Host
// code only.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace tt {

struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace tt
