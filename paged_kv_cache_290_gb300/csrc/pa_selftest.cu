// Test hook: drive the bounded mbarrier wait to its limit (see include/pa_selftest.h).
#include <cuda_runtime.h>

#include <string>

#include "pa.h"
#include "pa_common.cuh"
#include "pa_kernels.h"
#include "pa_selftest.h"

namespace {

constexpr uint64_t kSelftestMaxNs = 100000000ull;  // 100 ms

// One warp: lane 0 waits on an mbarrier with one expected arrival that never comes.  The wait
// gives up after limit_ns and sets the timeout bit; nothing else is in flight.
__global__ void __launch_bounds__(32) wait_without_arrival_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    pa::mbar_init(pa::smem_addr(&bar), 1);
    pa::mbar_init_fence();
    pa::mbar_wait(pa::smem_addr(&bar), 0, err, limit_ns);
  }
  __syncwarp();
}

}  // namespace

extern "C" int pa_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns < PA_WAIT_LIMIT_MIN_NS || limit_ns > kSelftestMaxNs)
    return pa::set_last_error(PA_ERR_INVALID_ARG, "self-test wait limit must be in [" +
                                                      std::to_string(PA_WAIT_LIMIT_MIN_NS) +
                                                      ", 100000000] ns");
  unsigned* err = nullptr;
  cudaError_t e = pa::error_word(stream, &err);
  if (e != cudaSuccess)
    return pa::set_last_error(PA_ERR_CUDA, std::string("error word: ") + cudaGetErrorString(e));
  wait_without_arrival_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, limit_ns);
  if ((e = cudaGetLastError()) != cudaSuccess)
    return pa::set_last_error(PA_ERR_CUDA, std::string("self-test launch: ") +
                                               cudaGetErrorString(e));
  pa::set_last_error(PA_OK, "");
  return PA_OK;
}
