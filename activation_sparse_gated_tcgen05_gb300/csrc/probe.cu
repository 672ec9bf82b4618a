// probe.cu -- self-checks and measurement helpers exported by the library.
//
//   * a bounded-wait self-test: a kernel waits on an mbarrier that nothing
//     completes, with the same bounded wait the GEMM pipeline uses, and must
//     come back with TWELL_ERR_DEVICE_TIMEOUT in the status word (the failure
//     path is exercised without faulting or hanging the GPU);
//   * a row-gather probe: warps read whole rows of a table at given row ids
//     with 16-byte loads (the access pattern of the sparse kernels), giving
//     the achievable gather bandwidth for a table resident in L2 or not.
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

// Each warp gathers rows_per_warp rows (ids from idx) of row_vecs 16-byte
// vectors and folds them into one word so the loads are not dead.
__global__ void __launch_bounds__(256) gather_probe_kernel(const uint4* __restrict__ table,
                                                           int row_vecs,
                                                           const int* __restrict__ idx, long long n,
                                                           uint32_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const long long warp = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long warps = (long long)gridDim.x * 8;
  uint32_t acc = 0;
  for (long long i = warp; i < n; i += warps) {
    const uint4* row = table + (long long)idx[i] * row_vecs;
#pragma unroll 4
    for (int v = lane; v < row_vecs; v += 32) {
      const uint4 w = ldg_v4(row + v);
      acc ^= w.x ^ w.y ^ w.z ^ w.w;
    }
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if (lane == 0) out[warp] = acc;
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

extern "C" twell_status twell_probe_gather(const void* table, int64_t table_rows, int32_t row_bytes,
                                           const int32_t* idx, int64_t n_idx, uint32_t* out,
                                           int32_t blocks, void* stream) {
  if (!table || !idx || !out || table_rows <= 0 || n_idx < 0 || blocks <= 0) return TWELL_ERR_INVALID_ARG;
  if (row_bytes <= 0 || row_bytes % 16 != 0) return TWELL_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(table) & 15u) != 0) return TWELL_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  {
    ProfScope prof("gather_probe", s);
    gather_probe_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(table),
                                               row_bytes / 16, idx, (long long)n_idx, out);
  }
  count_launch();
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
