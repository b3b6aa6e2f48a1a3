// Optional per-kernel timing: when enabled, every launch site records a
// start/stop cudaEvent pair on the launching stream; moe_trace_read()
// accumulates the elapsed times per kernel kind.
#pragma once
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

void trace_begin(int kind, cudaStream_t s);
void trace_end(int kind, cudaStream_t s);

struct TraceScope {
  int kind;
  cudaStream_t s;
  TraceScope(int k, cudaStream_t st) : kind(k), s(st) { trace_begin(kind, s); }
  ~TraceScope() { trace_end(kind, s); }
};

}  // namespace moe
