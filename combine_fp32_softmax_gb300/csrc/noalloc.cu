// moe_dispatch for callers that cannot hand the library a workspace.
//
// moe_dispatch keeps its scratch (the per-block expert histogram, the
// scanned block bases and the device error word) in the caller's workspace.
// Some callers have no way to provide one: a framework operator registered
// with a zero-byte workspace, or code whose device memory was planned up
// front by a host framework so that nothing may call cudaMalloc (or an
// allocating library routine) while it runs.  moe_dispatch_noalloc gives
// those callers the same token mapping and gather with the scratch in a
// fixed-size array compiled into the library's device image.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

// Scratch capacity: the error word (64 ints) plus two [E][ceil(T/32)]
// int32 tables; 2^20 ints = 4 MiB, enough for E * ceil(T/32) <= 524,256
// (e.g. 64 experts and 262,144 tokens, or 256 experts and 65,536 tokens).
// Every GPU that loads the library holds this array until the process exits.
constexpr long long kScratchInts = 1ll << 20;
constexpr long long kErrInts = 64;
static __device__ __align__(256) int g_dispatch_scratch[kScratchInts];

// Device address of g_dispatch_scratch per device, looked up on the first
// call made with that device current (host code cannot use the symbol's name
// as a device pointer: on the host it names a stand-in, not device memory).
// The set-up runs under a lock, once per device; later calls only load the
// published address.  The address belongs to the CUDA context current at
// set-up: after a device reset the process must restart before calling this
// entry point again on that device.
constexpr int kMaxDevices = 64;
std::atomic<int*> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mu;

// First call on the current device: loads the modules of this file and of
// the dispatch kernels (under lazy module loading that is when the scratch
// array is placed in device memory), then looks up the array's address.
int* scratch_on_current_device(int dev) {
  int* addr = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (addr) return addr;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  addr = g_scratch_addr[dev].load(std::memory_order_relaxed);
  if (addr) return addr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return nullptr;
  if (moe::preload_dispatch_kernels() != cudaSuccess) return nullptr;
  (void)moe::num_sms();
  addr = static_cast<int*>(p);
  g_scratch_addr[dev].store(addr, std::memory_order_release);
  return addr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_dispatch_noalloc(const moe_cfg* cfg, const int32_t* topk_idx, const uint16_t* x, int32_t* counts,
                                    int32_t* offsets, int32_t* dest, int32_t* row_token, int32_t* row_slot,
                                    uint16_t* Xp, void* stream) {
  using namespace moe;
  if (!cfg || !topk_idx || !counts || !offsets || !dest || !row_token || !row_slot) return MOE_ERR_ARG;
  const moe_cfg& c = *cfg;
  if (c.T < 1 || c.E < 1 || c.E > 256 || c.k < 1 || c.k > c.E || c.k > 8 || c.d_model < 64 || c.d_model % 64)
    return MOE_ERR_SHAPE;
  if (static_cast<long long>(c.T) * c.k >= (1ll << 31) - 256) return MOE_ERR_SHAPE;
  for (const void* p : {static_cast<const void*>(topk_idx), static_cast<const void*>(counts),
                        static_cast<const void*>(offsets), static_cast<const void*>(dest),
                        static_cast<const void*>(row_token), static_cast<const void*>(row_slot),
                        static_cast<const void*>(x), static_cast<const void*>(Xp)})
    if (p && !aligned16(p)) return MOE_ERR_ALIGN;
  const int nb = ceil_div(c.T, kRouteTokensPerBlock);
  const long long table = static_cast<long long>(c.E) * nb;
  if (kErrInts + 2 * table > kScratchInts) return MOE_ERR_SHAPE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  int* err = scratch_on_current_device(dev);
  if (!err) return MOE_ERR_CUDA;
  int32_t* hist = err + kErrInts;
  int32_t* base = hist + table;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // hist and base are fully overwritten by their kernels; only the error
  // word must start at zero.
  if (cudaMemsetAsync(err, 0, sizeof(int) * kErrInts, s) != cudaSuccess) return MOE_ERR_CUDA;
  const int R = c.T * c.k;
  if (launch_hist(topk_idx, c.T, c.E, c.k, hist, nb, err, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_scan(hist, c.E, nb, R, base, counts, offsets, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_scatter(topk_idx, base, c.T, c.E, c.k, nb, dest, row_token, row_slot, err, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (x && Xp && launch_gather_rows_bf16(x, row_token, c.T, R, c.d_model, Xp, MOE_K_GATHER, err, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
