// selftest.cu -- the bounded-wait self-test exported by the library.
//
// A kernel waits on an mbarrier that nothing completes, with the same
// bounded wait the GEMM pipeline uses, and must come back with
// TWELL_ERR_DEVICE_TIMEOUT in the status word: the failure path is exercised
// without faulting or hanging the GPU.
#include "common.cuh"
#include "internal.h"

namespace tw {

namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nobody arrives on `bar`: the wait must give up after limit_ns
    if (!mbar_wait(&bar, 0, nullptr, limit_ns)) set_status(status, TWELL_ERR_DEVICE_TIMEOUT);
  }
}

}  // namespace

}  // namespace tw

using namespace tw;

extern "C" twell_status twell_selftest_wait_timeout(int32_t limit_us, void* stream) {
  if (limit_us <= 0 || limit_us > 10000000) return TWELL_ERR_INVALID_ARG;
  int* status = device_status_ptr();
  if (!status) return TWELL_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  wait_timeout_kernel<<<1, 32, 0, s>>>((uint64_t)limit_us * 1000ull, status);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
