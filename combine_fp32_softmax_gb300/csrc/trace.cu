// Per-kernel timing with CUDA events (see trace.h).  Host-only bookkeeping;
// events are recycled through a pool.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "trace.h"

namespace moe {
namespace {

struct Pending {
  int kind;
  cudaEvent_t start, stop;
};

std::mutex g_mu;
bool g_on = false;
std::vector<cudaEvent_t> g_pool;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_open[MOE_K_COUNT];  // start events awaiting their stop
double g_ms[MOE_K_COUNT] = {0};
int g_count[MOE_K_COUNT] = {0};

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void settle_locked() {
  for (const Pending& p : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.stop) == cudaSuccess && cudaEventElapsedTime(&ms, p.start, p.stop) == cudaSuccess) {
      g_ms[p.kind] += ms;
      g_count[p.kind] += 1;
    }
    g_pool.push_back(p.start);
    g_pool.push_back(p.stop);
  }
  g_pending.clear();
}

const char* kNames[MOE_K_COUNT] = {"route",     "hist",          "scan",      "scatter",   "gather",
                                   "gemm1_swiglu", "gemm2_scale", "combine",   "combine_bwd", "gemm_dh",
                                   "dw_reduce", "route_bwd",     "gemm_dx",   "dispatch_bwd", "gemm_dw13",
                                   "gemm_dw2",  "megakernel", "megakernel_bwd", "route_tables", "bwd_gemms"};

}  // namespace

void trace_begin(int kind, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || kind < 0 || kind >= MOE_K_COUNT) return;
  cudaEvent_t e = take_event();
  cudaEventRecord(e, s);
  g_open[kind].push_back(e);
}

void trace_end(int kind, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (kind < 0 || kind >= MOE_K_COUNT || g_open[kind].empty()) return;
  cudaEvent_t start = g_open[kind].back();
  g_open[kind].pop_back();
  cudaEvent_t stop = take_event();
  cudaEventRecord(stop, s);
  g_pending.push_back({kind, start, stop});
}

}  // namespace moe

extern "C" {

int moe_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(moe::g_mu);
  moe::g_on = on != 0;
  return MOE_OK;
}

int moe_trace_reset(void) {
  std::lock_guard<std::mutex> lk(moe::g_mu);
  moe::settle_locked();
  for (int k = 0; k < MOE_K_COUNT; ++k) {
    moe::g_ms[k] = 0;
    moe::g_count[k] = 0;
  }
  return MOE_OK;
}

int moe_trace_read(int kind, double* total_ms, int* launches) {
  if (kind < 0 || kind >= MOE_K_COUNT || !total_ms || !launches) return MOE_ERR_ARG;
  std::lock_guard<std::mutex> lk(moe::g_mu);
  moe::settle_locked();
  *total_ms = moe::g_ms[kind];
  *launches = moe::g_count[kind];
  return MOE_OK;
}

const char* moe_trace_kind_name(int kind) {
  return (kind >= 0 && kind < MOE_K_COUNT) ? moe::kNames[kind] : "";
}

}  // extern "C"
