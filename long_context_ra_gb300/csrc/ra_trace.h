// Named ranges around every entry point for timeline profilers (NVTX v3,
// header-only).  With no profiler attached a range costs a pointer check; a
// tool that records NVTX (Nsight Systems, Nsight Compute's range filters)
// shows each call of the library as a range named after the entry point.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace ra {

struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace ra

#define RA_TRACE(name) ::ra::TraceRange ra_trace_range_(name)
