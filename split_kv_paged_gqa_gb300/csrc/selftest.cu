// selftest.cu - the decode kernels' bounded-wait failure path, run out on
// purpose (sm_103a).
//
// Every mbarrier wait in the decode kernels gives up after a time limit,
// records FD_DEVSTAT_WAIT_TIMEOUT in the plan's status word and returns
// false, so a pipeline that never delivers ends its kernel instead of hanging
// the GPU. A healthy decode call never reaches that branch; this kernel does.
// It waits, with the same routine (mbar_wait_warp), on a fresh barrier that
// nothing ever arrives on, under a short caller-given limit.
#include <cuda_runtime.h>

#include "fd.h"
#include "plan.h"
#include "ptx.cuh"

namespace {

__global__ void fd_wait_selftest_kernel(unsigned *status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    fd::mbar_init(&bar, 1);
    fd::fence_mbar_init();
  }
  __syncthreads();
  // phase 0 of the barrier never completes: the wait runs out after limit_ns
  fd::mbar_wait_warp(&bar, 0, status, limit_ns);
}

}  // namespace

extern "C" fd_status fd_selftest_wait_timeout(fd_plan *plan, unsigned limit_us, fd_stream_t stream) {
  using fd::fail;
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  if (plan->device < 0 || !plan->status) return fail(FD_ERR_WORKSPACE, "host-only plan has no status word");
  if (limit_us < 1 || limit_us > fd::kWaitLimitNs / 1000)
    return fail(FD_ERR_INVALID_ARG, "limit %u us outside [1, %llu]", limit_us, fd::kWaitLimitNs / 1000);
  fd::DeviceGuard guard(plan->device);
  fd_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      plan->status, static_cast<unsigned long long>(limit_us) * 1000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "wait self-test launch failed: %s", cudaGetErrorString(e));
  return FD_OK;
}
