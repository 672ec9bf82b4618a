// gather_probe.cu -- row-gather bandwidth probe, a measurement helper built
// into its own library (libtwell_probe.so) for the benchmark; it is not part
// of the FFN library or its C ABI.
//
// Warps read whole rows of a table at given row ids with 16-byte loads, the
// access pattern of the sparse gather kernels, which gives the achievable
// gather bandwidth for a table resident in L2 or not.
#include <stdint.h>

#include "common.cuh"

namespace {

// Each warp gathers rows (ids from idx, ids outside [0, table_rows) are
// skipped) of row_vecs 16-byte vectors and folds them into one word so the
// loads are not dead.  out holds one word per warp of the grid.
__global__ void __launch_bounds__(256)
    gather_probe_kernel(const uint4* __restrict__ table, long long table_rows, int row_vecs,
                        const int* __restrict__ idx, long long n, uint32_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const long long warp = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long warps = (long long)gridDim.x * 8;
  uint32_t acc = 0;
  for (long long i = warp; i < n; i += warps) {
    const int r = idx[i];
    if (r < 0 || r >= table_rows) continue;  // warp-uniform: one id per warp
    const uint4* row = table + (long long)r * row_vecs;
#pragma unroll 4
    for (int v = lane; v < row_vecs; v += 32) {
      const uint4 w = tw::ldg_v4(row + v);
      acc ^= w.x ^ w.y ^ w.z ^ w.w;
    }
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if (lane == 0) out[warp] = acc;
}

}  // namespace

// Status codes follow twell.h: 0 ok, 1 invalid argument, 2 unsupported,
// 3 misaligned, 5 CUDA error.
//   table      device, table_rows rows of row_bytes bytes (16-byte aligned)
//   idx        device int32 [n_idx] row ids
//   out        device uint32 [out_words], at least blocks * 8 words
extern "C" int32_t twell_probe_gather(const void* table, int64_t table_rows, int32_t row_bytes,
                                      const int32_t* idx, int64_t n_idx, uint32_t* out,
                                      int64_t out_words, int32_t blocks, void* stream) {
  if (!table || !idx || !out || table_rows <= 0 || n_idx < 0 || blocks <= 0) return 1;
  if (out_words < (int64_t)blocks * 8) return 1;
  if (row_bytes <= 0 || row_bytes % 16 != 0) return 2;
  if ((reinterpret_cast<uintptr_t>(table) & 15u) != 0) return 3;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  gather_probe_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(table),
                                             (long long)table_rows, row_bytes / 16, idx,
                                             (long long)n_idx, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}
