// moe_dispatch_noalloc: dispatch for callers that cannot allocate device
// memory.  Some callers have no way to obtain a workspace: serving runtimes
// that reserve all device memory at start-up and forbid allocation afterwards,
// hosts (plain C programs, other language runtimes) that link this library
// without handing it an allocator, and latency-critical loops that cannot pay
// for cudaMalloc's implicit device synchronisation.  This entry point needs no
// workspace argument: its scratch (the per-block route histograms) lives in a
// file-scope device array of fixed size that every GPU loading this library
// holds until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"

namespace {

// 1 MiB of scratch: room for E * ceil(T / (8 * (32 / K))) int32 block counts.
constexpr size_t kNoAllocScratchBytes = size_t{1} << 20;
static __device__ __align__(256) unsigned char g_dispatch_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Per device: the context the address was looked up in, and the address.
CUcontext g_scratch_ctx[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (no link-time
// dependency on the driver library); nullptr if it cannot be resolved.
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// Device address of the scratch array in the current device's current
// context.  In host code the array's name is only a host-side stand-in, so the
// address is looked up with that device current and cached per device; the
// cache is keyed by the context as well, because after cudaDeviceReset the
// module is loaded again into a new context, possibly at another address.
moe_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (get_ctx == nullptr || get_ctx(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  if (ctx == nullptr) {
    // No context current yet: cudaSetDevice initialises the device's primary
    // context (the one the launches below use) and makes it current.
    if (cudaSetDevice(dev) != cudaSuccess || get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
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
