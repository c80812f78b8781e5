// Self-test of the device-side failure path: the two bounded waits the
// pipelined kernels use -- an mbarrier wait, and the acquire wait on a global
// completion counter that gates the down tiles of the one-launch GEMM form --
// each run on something that nothing will complete.  Both give up after their
// time limit; the kernel reports MOE_DEV_TIMEOUT in dev_status[0], which of
// the two waits gave up as bits of dev_status[1] (1: mbarrier, 2: counter),
// and returns normally, so the context stays usable.
#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// A counter nothing increments.
__device__ int g_selftest_counter = 0;

__global__ void bounded_wait_selftest_kernel(int32_t* dev_status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // one arrival expected; none will come
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag)) {
    atomicOr(dev_status, kDevTimeout);
    atomicOr(dev_status + 1, 1);
  }
  if (threadIdx.x == 32 && !wait_count(&g_selftest_counter, 1, &abort_flag)) {
    atomicOr(dev_status, kDevTimeout);
    atomicOr(dev_status + 1, 2);
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_bounded_wait(int32_t* dev_status, moe_stream_t stream) {
  if (dev_status == nullptr) return MOE_ERR_INVALID_ARG;
  moe::bounded_wait_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev_status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
