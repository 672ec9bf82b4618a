// pack.cu -- TwELL pack from a dense pre-activation, hybrid ELL / dense routing,
// and the row gather that feeds routed rows to the dense tensor-core path.
//
// Format (page 2 "Sakana AI and NVIDIA introduce TwELL with CUDA kernels ...",
// section "¿Qué hace distinto a TwELL frente a ELL clásico?"): the columns of
// the gate activation are cut into tiles of width T_n; each (row, tile) keeps
// its live values and their in-tile columns locally, plus a count.
#include "common.cuh"
#include "internal.h"

namespace tw {

namespace {

constexpr int kWarpsPerBlock = 8;

template <int E, bool F32>
__device__ __forceinline__ void load_elems(const void* a, long long off, uint32_t (&g)[E]) {
  if (F32) {
    const float* p = reinterpret_cast<const float*>(a) + off;
    if (E == 4) {
      const float4 v = *reinterpret_cast<const float4*>(p);
      g[0] = relu_bf16_bits(v.x);
      g[1] = relu_bf16_bits(v.y);
      g[2] = relu_bf16_bits(v.z);
      g[3] = relu_bf16_bits(v.w);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(p);
      g[0] = relu_bf16_bits(v.x);
      g[1] = relu_bf16_bits(v.y);
    }
  } else {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(a) + off;
    if (E == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      g[0] = relu_bf16_bits(bf16_bits_to_float(v.x & 0xFFFFu));
      g[1] = relu_bf16_bits(bf16_bits_to_float(v.x >> 16));
      g[2] = relu_bf16_bits(bf16_bits_to_float(v.y & 0xFFFFu));
      g[3] = relu_bf16_bits(bf16_bits_to_float(v.y >> 16));
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
      g[0] = relu_bf16_bits(bf16_bits_to_float(v & 0xFFFFu));
      g[1] = relu_bf16_bits(bf16_bits_to_float(v >> 16));
    }
  }
}

// One warp per row.  Lane l holds columns [l*E, l*E+E) of each tile; a warp
// prefix sum over per-lane live counts gives every live entry its slot, so
// slots follow ascending column order.
template <int E, bool F32>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    pack_dense_kernel(const void* a, int M, int f, int T, int cap, uint16_t* val, uint8_t* idx,
                      uint8_t* cnt, int* row_nnz) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * kWarpsPerBlock;
  const int tile_n = 32 * E;
  for (int m = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); m < M; m += warps) {
    int nnz = 0;
    for (int t = 0; t < T; ++t) {
      uint32_t g[E];
      load_elems<E, F32>(a, (long long)m * f + (long long)t * tile_n + lane * E, g);
      int c = 0;
#pragma unroll
      for (int e = 0; e < E; ++e) c += (g[e] & 0x7FFFu) ? 1 : 0;
      const int incl = warp_incl_scan(c);
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      int pos = incl - c;
      const long long slot0 = ((long long)m * T + t) * cap;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (g[e] & 0x7FFFu) {
          if (pos < cap) {
            val[slot0 + pos] = (uint16_t)g[e];
            idx[slot0 + pos] = (uint8_t)(lane * E + e);
          }
          ++pos;
        }
      }
      if (lane == 0) cnt[(long long)m * T + t] = (uint8_t)total;
      nnz += total;
    }
    if (lane == 0) row_nnz[m] = nnz;
  }
}

// Per-row routing decision and ELL compaction, one warp per row.  Lane l
// owns tiles l, l+32, ...; a prefix sum over tile counts places each tile's
// entries, which keeps global columns ascending.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_rows_kernel(const uint16_t* val, const uint8_t* idx, const uint8_t* cnt,
                      const int* row_nnz, int M, int T, int tile_n, int cap, int W,
                      uint16_t* ell_val, uint16_t* ell_col, int* ell_nnz, int* flags) {
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (m >= M) return;
  const uint8_t* crow = cnt + (long long)m * T;
  bool over = false;
  for (int t = lane; t < T; t += 32) over |= crow[t] > cap;
  over = __any_sync(0xffffffffu, over);
  const bool routed = over || row_nnz[m] > W;
  if (lane == 0) flags[m] = routed ? 1 : 0;
  if (routed) {
    if (lane == 0) ell_nnz[m] = 0;
    return;
  }
  int base = 0;
  for (int t0 = 0; t0 < T; t0 += 32) {
    const int t = t0 + lane;
    const int c = t < T ? crow[t] : 0;
    const int incl = warp_incl_scan(c);
    const int excl = incl - c;
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    // the group's entries are spread over the lanes: entry e belongs to the
    // tile whose inclusive count first exceeds e (binary search over lanes)
    for (int e = lane; e - lane < total; e += 32) {
      int lo = 0;
#pragma unroll
      for (int step = 16; step >= 1; step >>= 1) {
        const int v = __shfl_sync(0xffffffffu, incl, lo + step - 1);
        if (v <= e) lo += step;
      }
      const int ex = __shfl_sync(0xffffffffu, excl, lo);
      if (e < total) {
        const int tt = t0 + lo;
        const long long src = ((long long)m * T + tt) * cap + (e - ex);
        const long long dst = (long long)m * W + base + e;
        int il = idx[src];
        TW_CHECK_INDEX(il, il < tile_n);
        ell_val[dst] = val[src];
        ell_col[dst] = (uint16_t)(tt * tile_n + il);
      }
    }
    base += total;
  }
  if (lane == 0) ell_nnz[m] = base;
}

// Stable list of routed rows: one block scans the flags in order.  More
// routed rows than the caller's capacity dense_cap records TWELL_ERR_CAPACITY.
constexpr int kListThreads = 1024;
constexpr int kListItems = 16;

__global__ void __launch_bounds__(kListThreads)
    route_list_kernel(const int* flags, int M, int* dense_rows, int* n_dense, int dense_cap,
                      int* status) {
  __shared__ int warp_tot[kListThreads / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < M; base += kListThreads * kListItems) {
    const int r0 = base + tid * kListItems;
    // flags may alias dense_rows (in-place compaction): read them all first;
    // every write below lands at an index <= the flag it replaces, and the
    // block barrier separates this iteration's reads from its writes.
    unsigned bits = 0;
#pragma unroll
    for (int i = 0; i < kListItems; ++i)
      if (r0 + i < M && flags[r0 + i]) bits |= 1u << i;
    const int c = __popc(bits);
    const int incl = warp_incl_scan(c);
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = warp_tot[lane];
      const int vi = warp_incl_scan(v);
      warp_tot[lane] = vi - v;
    }
    __syncthreads();
    int pos = carry + warp_tot[warp] + incl - c;
#pragma unroll
    for (int i = 0; i < kListItems; ++i)
      if (bits & (1u << i)) dense_rows[pos++] = r0 + i;
    __syncthreads();
    if (tid == kListThreads - 1) carry = pos;
    __syncthreads();
  }
  if (tid == 0) {
    *n_dense = carry;
    if (carry > dense_cap) set_status(status, TWELL_ERR_CAPACITY);
  }
}

// dst[i] = src[rows[i]] for i < n (n on the device); rows [n, roundup(n, 128))
// of dst are zeroed so tensor-core tiles over dst see zeros, not stale bytes.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    gather_rows_kernel(const uint16_t* src, int M, int d, const int* rows, const int* n_rows,
                       uint16_t* dst, int dst_rows) {
  const int n = min(*n_rows, dst_rows);
  const int limit = min(dst_rows, ((n + 127) / 128) * 128);
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * kWarpsPerBlock;
  const int vecs = d / 8;
  for (int i = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); i < limit; i += warps) {
    uint4* o = reinterpret_cast<uint4*>(dst + (long long)i * d);
    if (i < n) {
      const int r = rows[i];
      const uint4* s = reinterpret_cast<const uint4*>(src + (long long)r * d);
      if (r >= 0 && r < M)
        for (int v = lane; v < vecs; v += 32) o[v] = s[v];
    } else {
      for (int v = lane; v < vecs; v += 32) o[v] = make_uint4(0, 0, 0, 0);
    }
  }
}

// Sum the split-K partials of the routed rows in fixed order (split 0, 1, ...)
// and scatter the bf16 result to out[rows[r]] -- deterministic, no atomics.
__global__ void __launch_bounds__(256)
    splitk_scatter_kernel(const float* __restrict__ part, int buf_rows, int row_cap, int num_kb,
                          int s_max, const int* __restrict__ n_rows, const int* __restrict__ rows,
                          int M, int N, uint16_t* __restrict__ out) {
  const int n = min(*n_rows, row_cap);
  if (n <= 0) return;
  const int rows_eff = ((n + 127) / 128) * 128;
  int splits, kps;
  splitk_plan(rows_eff, buf_rows, num_kb, s_max, splits, kps);
  const int vecs = N / 8;
  const long long total = (long long)n * vecs;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / vecs), c = (int)(i % vecs) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int sp = 0; sp < splits; ++sp) {
      const float4* src =
          reinterpret_cast<const float4*>(part + ((long long)sp * rows_eff + r) * N + c);
      const float4 a = src[0], b = src[1];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    const int dst = rows[r];
    if (dst < 0 || dst >= M) continue;
    *reinterpret_cast<uint4*>(out + (long long)dst * N + c) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

int blocks_for(long long warps_needed) {
  long long b = (warps_needed + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const long long cap = (long long)num_sms() * 16;
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_splitk_scatter(const float* part, int buf_rows, int row_cap, int num_kb,
                                  int s_max, const int* n_rows, const int* rows, int M, int N,
                                  void* out, cudaStream_t s) {
  {
    ProfScope prof("splitk_scatter", s);
    splitk_scatter_kernel<<<num_sms() * 2, 256, 0, s>>>(part, buf_rows, row_cap, num_kb, s_max,
                                                        n_rows, rows, M, N,
                                                        reinterpret_cast<uint16_t*>(out));
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_pack_dense(const void* a, int a_f32, int M, int f, int tile_n, int cap,
                              const twell_tiles& out, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const int T = f / tile_n;
  const int grid = blocks_for(M);
  auto* val = reinterpret_cast<uint16_t*>(out.val);
  if (tile_n == 128) {
    if (a_f32)
      {
        ProfScope prof("pack_dense", s);
        pack_dense_kernel<4, true><<<grid, kWarpsPerBlock * 32, 0, s>>>(a, M, f, T, cap, val, out.idx,
                                                                        out.cnt, out.row_nnz);
      }
    else
      {
        ProfScope prof("pack_dense", s);
        pack_dense_kernel<4, false><<<grid, kWarpsPerBlock * 32, 0, s>>>(a, M, f, T, cap, val,
                                                                         out.idx, out.cnt,
                                                                         out.row_nnz);
      }
  } else {
    if (a_f32)
      {
        ProfScope prof("pack_dense", s);
        pack_dense_kernel<2, true><<<grid, kWarpsPerBlock * 32, 0, s>>>(a, M, f, T, cap, val, out.idx,
                                                                        out.cnt, out.row_nnz);
      }
    else
      {
        ProfScope prof("pack_dense", s);
        pack_dense_kernel<2, false><<<grid, kWarpsPerBlock * 32, 0, s>>>(a, M, f, T, cap, val,
                                                                         out.idx, out.cnt,
                                                                         out.row_nnz);
      }
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_route(const twell_tiles& in, int M, int f, int tile_n, int cap,
                         const twell_hybrid& out, int* flags, int dense_cap, cudaStream_t s) {
  if (M == 0) return cudaMemsetAsync(out.n_dense, 0, sizeof(int), s);
  {
    const cudaError_t ce = checked_setup();
    if (ce != cudaSuccess) return ce;
  }
  const int T = f / tile_n;
  const int grid = (M + kWarpsPerBlock - 1) / kWarpsPerBlock;
  {
    ProfScope prof("route_rows", s);
    route_rows_kernel<<<grid, kWarpsPerBlock * 32, 0, s>>>(
        reinterpret_cast<const uint16_t*>(in.val), in.idx, in.cnt, in.row_nnz, M, T, tile_n, cap,
        out.ell_width, reinterpret_cast<uint16_t*>(out.ell_val), out.ell_col, out.ell_nnz, flags);
  }
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    ProfScope prof("route_list", s);
    route_list_kernel<<<1, kListThreads, 0, s>>>(flags, M, out.dense_rows, out.n_dense, dense_cap,
                                                 device_status_ptr());
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* src, int M, int d, const int* rows, const int* n_rows,
                               void* dst, int dst_rows, cudaStream_t s) {
  if (dst_rows == 0) return cudaSuccess;
  {
    ProfScope prof("gather_rows", s);
    // two blocks per SM: the rows are strided over the grid, and with no row
    // routed (the count is on the device) every block only reads the count
    const int grid = min(blocks_for(dst_rows), 2 * num_sms());
    gather_rows_kernel<<<grid, kWarpsPerBlock * 32, 0, s>>>(
        reinterpret_cast<const uint16_t*>(src), M, d, rows, n_rows, reinterpret_cast<uint16_t*>(dst),
        dst_rows);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace tw
