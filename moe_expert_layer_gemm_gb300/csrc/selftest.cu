// Self-test of the failure path every pipelined kernel relies on: a bounded mbarrier wait that
// runs out.  One block initialises an mbarrier that nothing ever arrives on and waits for its
// first phase through the same bounded wait the GEMMs use (with a short limit); the wait gives
// up, raises the block's abort flag, records DEVERR_WAIT_TIMEOUT in the device error word and
// the kernel returns normally, so the context stays usable.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns, int* err,
                                                          int* observed) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    const bool ok = ptx::mbar_wait(&bar, 0u, &abort_flag, err, limit_ns);
    *observed = (ok ? 1 : 0) | (abort_flag ? 2 : 0);
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_selftest_wait_timeout(int32_t* observed, void* stream) {
  if (!observed) {
    set_error("moe_selftest_wait_timeout: observed is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // 50 ms: long enough to be a real wait, short enough for a test
  return launch("selftest_wait_timeout", wait_timeout_kernel, dim3(1), dim3(32), 0, st,
                static_cast<uint64_t>(50000000ull), device_error_word(), observed);
}
