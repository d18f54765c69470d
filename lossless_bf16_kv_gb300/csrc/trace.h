// trace.h -- NVTX ranges around the library's public calls, so that a
// profiler timeline (Nsight Systems, ncu's NVTX filters) shows which codec
// call enqueued which kernels.  NVTX 3 is header-only: with no tool attached a
// range costs a function-pointer check.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace splitzip {

class TraceRange {
public:
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace splitzip
