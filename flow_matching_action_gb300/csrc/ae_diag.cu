// ae_selftest_wait_timeout: exercises the device-side failure path of the
// library's bounded waits without faulting or hanging the GPU.
//
// Every mbarrier wait of the tensor-core kernels gives up after a cycle budget,
// records kDevTimeout in the context's host-mapped status word and returns.
// This entry point runs that same wait (tc::mbar_wait) in a one-warp kernel on
// an mbarrier that nothing ever completes, with a budget the caller chooses, so
// a test can check that the wait gives up, the status becomes sticky and the
// host reports AE_ERR_DEVICE.  No copy, MMA or TMEM allocation is in flight
// while the wait runs, so giving up leaves nothing behind.
#include "ae_internal.h"
#include "ae_tc.cuh"

namespace ae {
namespace {

__global__ void __launch_bounds__(32) k_wait_selftest(long long budget, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);  // one arrival completes the phase; none ever comes
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, &abort_flag, status, budget);
}

}  // namespace
}  // namespace ae

extern "C" ae_status ae_selftest_wait_timeout(ae_ctx* c, int64_t budget_cycles) {
  if (c == nullptr || budget_cycles < 0) return AE_ERR_INVALID_ARG;
  ae::k_wait_selftest<<<1, 32, 0, c->stream>>>((long long)budget_cycles, c->status_dev);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    c->last_msg = std::string("self-test wait kernel: ") + cudaGetErrorString(e);
    return AE_ERR_CUDA;
  }
  return AE_OK;
}
