// Internal side of the launch tracing (la_trace_enable / la_trace_collect).
#pragma once

#include <cuda_runtime.h>

namespace la {

// Records a start event on construction and a stop event on destruction on
// `s`, when tracing is enabled and the event pool has room; otherwise no-op.
class TraceScope {
public:
    TraceScope(const char* name, cudaStream_t s);
    ~TraceScope();
    TraceScope(const TraceScope&) = delete;
    TraceScope& operator=(const TraceScope&) = delete;

private:
    cudaStream_t stream_;
    int slot_;
};

}  // namespace la
