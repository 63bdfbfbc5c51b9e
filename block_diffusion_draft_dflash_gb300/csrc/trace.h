// Optional launch tracing: CUDA events around each kernel launch of the library, on the
// launch stream, summed per kernel class.  Off unless dflash_trace_enable(1) was called;
// not used while a stream is being captured into a graph.
#pragma once
#include <cuda_runtime.h>

namespace df {
bool trace_on();
void trace_begin(const char* tag, cudaStream_t st);
void trace_end(cudaStream_t st);

struct TraceScope {
  cudaStream_t st;
  bool on;
  TraceScope(const char* tag, cudaStream_t s) : st(s), on(trace_on()) {
    if (on) trace_begin(tag, st);
  }
  ~TraceScope() {
    if (on) trace_end(st);
  }
};
}  // namespace df

#define DF_TRACE(tag, st) ::df::TraceScope _df_trace_scope_(tag, st)
