// trace.h -- NVTX ranges around the library's entry points.
//
// Every call that enqueues device work opens a named range for its duration
// on the host, so a timeline tool (Nsight Systems, ncu's NVTX filters) shows
// which library call launched which kernels.  NVTX v3 is header-only: with no
// tool attached the push and pop are a check of a null function pointer.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace pkv_trace {
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};
}  // namespace pkv_trace

#define PKV_NVTX_RANGE(name) pkv_trace::Range pkv_nvtx_range_(name)
