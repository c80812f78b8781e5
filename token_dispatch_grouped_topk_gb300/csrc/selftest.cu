// Self-test of the device-side failure path: the bounded mbarrier wait every
// pipelined kernel here uses, run on a barrier that nothing will complete.
// The wait gives up after its time limit, the kernel reports MOE_DEV_TIMEOUT
// in the status word and returns normally, so the context stays usable.
#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

__global__ void bounded_wait_selftest_kernel(int32_t* dev_status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // one arrival expected; none will come
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag)) atomicOr(dev_status, kDevTimeout);
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_bounded_wait(int32_t* dev_status, moe_stream_t stream) {
  if (dev_status == nullptr) return MOE_ERR_INVALID_ARG;
  moe::bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev_status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
