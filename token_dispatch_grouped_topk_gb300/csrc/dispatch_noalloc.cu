// moe_dispatch_noalloc: dispatch for callers that cannot allocate device
// memory.  Some callers have no way to obtain a workspace: code that runs
// while a CUDA graph is being captured (cudaMalloc is not allowed there),
// runtimes that forbid device allocation after start-up or give this library
// no allocator, and latency-critical loops that cannot pay for cudaMalloc's
// implicit device synchronisation.  This entry point needs no workspace
// argument: its scratch (the per-block route histograms) lives in a
// file-scope device array of fixed size that every GPU loading this library
// holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"

namespace {

// 1 MiB of scratch: room for E * ceil(T / (8 * (32 / K))) int32 block counts.
constexpr size_t kNoAllocScratchBytes = size_t{1} << 20;
static __device__ __align__(256) unsigned char g_dispatch_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current and cached.
moe_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_dispatch_noalloc(const void* x, const int64_t* topk_idx, const float* topk_w, int T,
                                int H, int K, int E, int R, void* recv, int32_t* counts,
                                int32_t* src_map, int32_t* dev_status, moe_stream_t stream) {
  const size_t need = moe_dispatch_workspace_size(T, K, E);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;  // larger than the built-in scratch
  void* scratch = nullptr;
  if (moe_status st = scratch_for_current_device(&scratch); st != MOE_OK) return st;
  return moe_dispatch(x, topk_idx, topk_w, T, H, K, E, R, recv, counts, src_map, dev_status,
                      scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
