// sparse_fwd.cu -- fused sparse up + down projection over packed activations.
//
// Page 2 "Sakana AI and NVIDIA introduce TwELL with CUDA kernels ...", section
// "¿Qué hace distinto a TwELL frente a ELL clásico?": one kernel reads the
// packed gate activations and performs the up and down projections together;
// the intermediate never reaches global memory.
//
// A team of TEAM warps owns one token row m; the d_model axis is split across
// the team in 256-element (512-byte) slabs, VPL slabs per warp, so every
// weight-row read is a run of coalesced 16-byte loads.  For each live entry
// (j, g) of the row:
//   u = x_m . Wu[:, j]          (x_m held in registers as packed bf16, WuT[j]
//                                gathered; bf16 x bf16 -> fp32 FMA)
//   h = g * u                   (fp32, kept in registers)
//   y_m += h * Wd[j, :]         (fp32-pair accumulators in registers)
// and y_m is written once as bf16.  Entries are processed B at a time, 2*B
// weight rows in flight per warp.  Loads are never predicated: slots past
// the row's last entry read neuron 0 with gate 0 (their h is exactly 0), and
// lanes past d_model read the row's first slab against a zero x, so the load
// sequence has no zero-fill selects.  Up to d_model = 1024 a single warp owns
// the row (no cross-warp reduction); wider rows split it over a team whose
// partial dot products meet in shared memory behind a named barrier.  Wide
// ELL rows (the training path) instead take two gathers, up and down, that
// meet no barrier per batch (ell_gather.cuh); TwELL rows of any width take
// this kernel.
#include <cooperative_groups.h>

#include "common.cuh"
#include "ell_gather.cuh"
#include "internal.h"

namespace tw {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kPassFirst = 1, kPassLast = 2;

template <int TEAM>
__device__ __forceinline__ int slab_elem(int lane, int wt, int v) {
  return 8 * (lane + 32 * (wt + TEAM * v));
}

// Row state of one warp: its share of x_m (packed bf16), of the fp32
// accumulator y_m (pairs), and the in-row offsets of its VPL slabs (clamped
// to the first slab past d_model).
template <int VPL>
struct RowCtx {
  uint4 xv[VPL];
  uint64_t acc[VPL][4];
  int eoff[VPL];
};

// Process `count` (<= 32) entries whose (column, gate) sit in lanes 0..count-1.
template <int TEAM, int VPL, int B, int ROWS>
__device__ __forceinline__ void process_entries(RowCtx<VPL>& c, int jl, float gl, int count,
                                                const uint16_t* __restrict__ wuT,
                                                const uint16_t* __restrict__ wd, int d, int lane,
                                                int wt, int team, float (*red)[ROWS][TEAM][B],
                                                int& buf) {
  static_assert(32 % B == 0, "a batch never reaches past lane 31");
  for (int i = 0; i < count; i += B) {
    // lanes >= count hold (0, 0): a valid row with a zero gate
    int j[B];
    float g[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      j[b] = __shfl_sync(kFull, jl, (i + b) & 31);
      g[b] = __shfl_sync(kFull, gl, (i + b) & 31);
    }
    uint4 wu[B][VPL], wdv[B][VPL];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const uint16_t* pu = wuT + (long long)j[b] * d;
      const uint16_t* pd = wd + (long long)j[b] * d;
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        wu[b][v] = ldg_v4(pu + c.eoff[v]);
        wdv[b][v] = ldg_v4(pd + c.eoff[v]);
      }
    }
    float p[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int v = 0; v < VPL; ++v) dot8_bf16(c.xv[v], wu[b][v], a0, a1);
      p[b] = a0 + a1;
    }
    if constexpr (B == 2) {
      warp_sum2(p[0], p[B - 1]);
    } else {
#pragma unroll
      for (int b = 0; b < B; ++b) p[b] = warp_sum(p[b]);
    }
    if constexpr (TEAM > 1) {
      if (lane == 0)
#pragma unroll
        for (int b = 0; b < B; ++b) red[buf][team][wt][b] = p[b];
      named_barrier(1 + team, 32 * TEAM);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < TEAM; ++w) sum += red[buf][team][w][b];
        p[b] = sum;
      }
      buf ^= 1;
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const uint64_t h2 = f2_splat(g[b] * p[b]);
#pragma unroll
      for (int v = 0; v < VPL; ++v) axpy8_f2(h2, wdv[b][v], c.acc[v]);
    }
  }
}

template <int TEAM, int VPL, int B, bool ELL>
__global__ void __launch_bounds__(256, VPL > 2 ? 2 : 3)
    sparse_fwd_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wuT,
                      const uint16_t* __restrict__ wd, int M, int d,
                      const uint16_t* __restrict__ val, const uint8_t* __restrict__ idx,
                      const uint8_t* __restrict__ cnt, int T, int tile_n, int cap,
                      const uint16_t* __restrict__ ell_val, const uint16_t* __restrict__ ell_col,
                      const int* __restrict__ ell_nnz, int W, uint16_t* __restrict__ y,
                      float* __restrict__ part, int j_lo, int j_hi, int pass, int* status) {
  constexpr int ROWS = 8 / TEAM;
  __shared__ float red[2][ROWS][TEAM][B];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / TEAM, wt = warp % TEAM;
  const int m = blockIdx.x * ROWS + team;
  if (m >= M) return;

  const bool first = pass & kPassFirst, last = pass & kPassLast;
  // x, y and the y carry stream through once per pass: evict-first, so the
  // gathered weight rows keep L2
  const uint64_t pol = l2_evict_first_policy();
  RowCtx<VPL> c;
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = slab_elem<TEAM>(lane, wt, v);
    c.eoff[v] = e < d ? e : 0;
    c.xv[v] = e < d ? ldg_v4_hint(x + (long long)m * d + e, pol) : make_uint4(0, 0, 0, 0);
    if (first || e >= d) {
#pragma unroll
      for (int k = 0; k < 4; ++k) c.acc[v][k] = 0;
    } else {  // running sum of the earlier neuron chunks
      const float* pp = part + (long long)m * d + e;
      const uint4 q0 = ldg_v4_hint(pp, pol), q1 = ldg_v4_hint(pp + 4, pol);
      c.acc[v][0] = f2_make(q0.x, q0.y);
      c.acc[v][1] = f2_make(q0.z, q0.w);
      c.acc[v][2] = f2_make(q1.x, q1.y);
      c.acc[v][3] = f2_make(q1.z, q1.w);
    }
  }
  int buf = 0;

  if (ELL) {
    int n = ell_nnz[m];
    TW_CHECK_INDEX(n, n >= 0 && n <= W);
    // a row's columns ascend: the chunk [j_lo, j_hi) is the slice [a, b)
    int a = 0, b = n;
    if (!(first && last)) {
      a = b = 0;
      for (int s0 = 0; s0 < n; s0 += 32) {
        const int jc = s0 + lane < n ? (int)ell_col[(long long)m * W + s0 + lane] : 0x7fffffff;
        a += __popc(__ballot_sync(kFull, jc < j_lo));
        b += __popc(__ballot_sync(kFull, jc < j_hi));
      }
    }
    for (int e0 = a; e0 < b; e0 += 32) {
      const int count = min(32, b - e0);
      int jl = 0;
      float gl = 0.f;
      if (lane < count) {
        const long long s = (long long)m * W + e0 + lane;
        jl = ell_col[s];
        TW_CHECK_INDEX(jl, jl < T * tile_n);
        gl = bf16_bits_to_float(ell_val[s]);
      }
      process_entries<TEAM, VPL, B, ROWS>(c, jl, gl, count, wuT, wd, d, lane, wt, team, red,
                                          buf);
    }
  } else {
    for (int t0 = 0; t0 < T; t0 += 32) {
      const int t = t0 + lane;
      const int craw = t < T ? cnt[(long long)m * T + t] : 0;
      if (craw > cap && wt == 0) set_status(status, TWELL_ERR_CAPACITY);
      const int ct = min(craw, cap);
      const int incl = warp_incl_scan(ct);
      const int excl = incl - ct;
      const int total = __shfl_sync(kFull, incl, 31);
      for (int e0 = 0; e0 < total; e0 += 32) {
        const int e = e0 + lane;
        int lo = 0;  // owner lane: number of lanes whose inclusive count is <= e
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
          const int v = __shfl_sync(kFull, incl, lo + step - 1);
          if (v <= e) lo += step;
        }
        const int ex = __shfl_sync(kFull, excl, lo);
        int jl = 0;
        float gl = 0.f;
        if (e < total) {
          const int tt = t0 + lo;
          const long long sl = ((long long)m * T + tt) * cap + (e - ex);
          int il = idx[sl];
          TW_CHECK_INDEX(il, il < tile_n);
          jl = tt * tile_n + il;
          gl = bf16_bits_to_float(val[sl]);
        }
        process_entries<TEAM, VPL, B, ROWS>(c, jl, gl, min(32, total - e0), wuT, wd, d, lane,
                                            wt, team, red, buf);
      }
    }
  }

#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = slab_elem<TEAM>(lane, wt, v);
    if (e >= d) continue;
    if (last) {
      st_v4_hint(y + (long long)m * d + e, f2x4_to_bf8(c.acc[v]), pol);
    } else {
      float* pp = part + (long long)m * d + e;
      st_v4_hint(pp, make_uint4((uint32_t)c.acc[v][0], (uint32_t)(c.acc[v][0] >> 32),
                                (uint32_t)c.acc[v][1], (uint32_t)(c.acc[v][1] >> 32)), pol);
      st_v4_hint(pp + 4, make_uint4((uint32_t)c.acc[v][2], (uint32_t)(c.acc[v][2] >> 32),
                                    (uint32_t)c.acc[v][3], (uint32_t)(c.acc[v][3] >> 32)), pol);
    }
  }
}

// Small batches (TwELL rows): too few rows to fill the GPU one team per row,
// so each row's tiles are split over the CL blocks of a thread-block cluster.
// Block `rank` accumulates the entries of tiles [T rank / CL, T (rank+1) / CL)
// in registers and stages its partial y_m in shared memory; after a cluster
// barrier, block `rank` sums columns [rank d / CL, (rank+1) d / CL) of every
// row over the cluster's blocks in rank order (distributed shared memory)
// and writes y.  Deterministic; no global scratch.
template <int TEAM, int VPL, int B>
__global__ void __launch_bounds__(256, VPL > 2 ? 2 : 3)
    sparse_fwd_cluster_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wuT,
                              const uint16_t* __restrict__ wd, int M, int d,
                              const uint16_t* __restrict__ val, const uint8_t* __restrict__ idx,
                              const uint8_t* __restrict__ cnt, int T, int tile_n, int cap,
                              uint16_t* __restrict__ y, int* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  constexpr int ROWS = 8 / TEAM;
  extern __shared__ __align__(16) float part[];  // [ROWS][d] partial y of this block
  __shared__ float red[2][ROWS][TEAM][B];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / TEAM, wt = warp % TEAM;
  const int m0 = (int)(blockIdx.x / CL) * ROWS;  // the cluster's first row
  const int m = m0 + team;
  const bool row_ok = m < M;  // no early exit: every block reaches the cluster barriers

  RowCtx<VPL> c;
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = slab_elem<TEAM>(lane, wt, v);
    c.eoff[v] = e < d ? e : 0;
    c.xv[v] = (e < d && row_ok) ? ldg_v4(x + (long long)m * d + e) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < 4; ++k) c.acc[v][k] = 0;
  }
  int buf = 0;
  if (row_ok) {
    const int t_lo = (int)((long long)T * rank / CL), t_hi = (int)((long long)T * (rank + 1) / CL);
    for (int t0 = t_lo; t0 < t_hi; t0 += 32) {
      const int t = t0 + lane;
      const int craw = t < t_hi ? cnt[(long long)m * T + t] : 0;
      if (craw > cap && wt == 0) set_status(status, TWELL_ERR_CAPACITY);
      const int ct = min(craw, cap);
      const int incl = warp_incl_scan(ct);
      const int excl = incl - ct;
      const int total = __shfl_sync(kFull, incl, 31);
      for (int e0 = 0; e0 < total; e0 += 32) {
        const int e = e0 + lane;
        int lo = 0;
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
          const int v = __shfl_sync(kFull, incl, lo + step - 1);
          if (v <= e) lo += step;
        }
        const int ex = __shfl_sync(kFull, excl, lo);
        int jl = 0;
        float gl = 0.f;
        if (e < total) {
          const int tt = t0 + lo;
          const long long sl = ((long long)m * T + tt) * cap + (e - ex);
          int il = idx[sl];
          TW_CHECK_INDEX(il, il < tile_n);
          jl = tt * tile_n + il;
          gl = bf16_bits_to_float(val[sl]);
        }
        process_entries<TEAM, VPL, B, ROWS>(c, jl, gl, min(32, total - e0), wuT, wd, d, lane,
                                            wt, team, red, buf);
      }
    }
  }
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = slab_elem<TEAM>(lane, wt, v);
    if (e < d) {
      float4* pp = reinterpret_cast<float4*>(part + team * d + e);
      pp[0] = make_float4(f2_lo(c.acc[v][0]), f2_hi(c.acc[v][0]), f2_lo(c.acc[v][1]),
                          f2_hi(c.acc[v][1]));
      pp[1] = make_float4(f2_lo(c.acc[v][2]), f2_hi(c.acc[v][2]), f2_lo(c.acc[v][3]),
                          f2_hi(c.acc[v][3]));
    }
  }
  cluster.sync();
  // columns [rank * cols, (rank + 1) * cols) of the cluster's rows, 8 per thread
  const int cols = d / CL;
  for (int i = threadIdx.x * 8; i < ROWS * cols; i += 256 * 8) {
    const int r = i / cols, col = rank * cols + (i - r * cols);
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < CL; ++q) {
      const float4* src = reinterpret_cast<const float4*>(
          cluster.map_shared_rank(part + r * d + col, (unsigned)q));
      const float4 a = src[0], b = src[1];
      s[0] += a.x; s[1] += a.y; s[2] += a.z; s[3] += a.w;
      s[4] += b.x; s[5] += b.y; s[6] += b.z; s[7] += b.w;
    }
    if (m0 + r < M)
      *reinterpret_cast<uint4*>(y + (long long)(m0 + r) * d + col) =
          make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                     pack_bf16x2(s[6], s[7]));
  }
  cluster.sync();  // no block leaves while another still reads its shared memory
}

template <int TEAM, int VPL>
cudaError_t launch_cluster(const void* x, const void* wuT, const void* wd, int M, int d,
                           const twell_tiles* tiles, int T, int tile_n, int cap, int CL, void* y,
                           cudaStream_t s) {
  constexpr int ROWS = 8 / TEAM;
  const int groups = (M + ROWS - 1) / ROWS;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(groups * CL));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = (size_t)ROWS * d * sizeof(float);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  {
    ProfScope prof("sparse_fwd", s);
    e = cudaLaunchKernelEx(&cfg, sparse_fwd_cluster_kernel<TEAM, VPL, 2>,
                           reinterpret_cast<const uint16_t*>(x),
                           reinterpret_cast<const uint16_t*>(wuT),
                           reinterpret_cast<const uint16_t*>(wd), M, d,
                           reinterpret_cast<const uint16_t*>(tiles->val), tiles->idx, tiles->cnt, T,
                           tile_n, cap, reinterpret_cast<uint16_t*>(y), device_status_ptr());
  }
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int TEAM, int VPL, bool ELL>
cudaError_t launch_team(const void* x, const void* wuT, const void* wd, int M, int d, int f,
                        const twell_tiles* tiles, int T, int tile_n, int cap,
                        const twell_hybrid* route, void* y, float* part, int chunks,
                        cudaStream_t s) {
  constexpr int ROWS = 8 / TEAM;
  const int grid = (M + ROWS - 1) / ROWS;
  for (int c = 0; c < chunks; ++c) {
    const int j_lo = (int)((long long)f * c / chunks), j_hi = (int)((long long)f * (c + 1) / chunks);
    const int pass = (c == 0 ? kPassFirst : 0) | (c == chunks - 1 ? kPassLast : 0);
    {
      ProfScope prof("sparse_fwd", s);
      sparse_fwd_kernel<TEAM, VPL, 2, ELL><<<grid, 256, 0, s>>>(
          reinterpret_cast<const uint16_t*>(x), reinterpret_cast<const uint16_t*>(wuT),
          reinterpret_cast<const uint16_t*>(wd), M, d,
          tiles ? reinterpret_cast<const uint16_t*>(tiles->val) : nullptr,
          tiles ? tiles->idx : nullptr, tiles ? tiles->cnt : nullptr, T, tile_n, cap,
          route ? reinterpret_cast<const uint16_t*>(route->ell_val) : nullptr,
          route ? route->ell_col : nullptr, route ? route->ell_nnz : nullptr,
          route ? route->ell_width : 0, reinterpret_cast<uint16_t*>(y), part, j_lo, j_hi, pass,
          device_status_ptr());
    }
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Wide rows: the fused gather split into an up gather (h = g x.Wu per entry)
// and a down gather (y = sum h Wd), each over one weight matrix in its own
// L2-sized neuron passes (ell_gather.cuh), over ELL rows (training) or TwELL
// tiles (inference, when the caller gives a workspace for h).  TEAM and VPL
// are the fused kernel's, so y is bit-identical to it.
template <int TEAM, int VPL, class Src, class Chunk>
cudaError_t launch_split(const void* x, const void* wuT, const void* wd, int M, int d, Src src,
                         int chunks, Chunk set_chunk, void* y, float* part, float* hbuf,
                         cudaStream_t s) {
  constexpr int ROWS = 8 / TEAM;
  EllDotArgs up{};
  up.vec = reinterpret_cast<const uint16_t*>(x);
  up.rows = reinterpret_cast<const uint16_t*>(wuT);
  up.M = M;
  up.d = d;
  up.out = hbuf;
  for (int c = 0; c < chunks; ++c) {
    Src sc = set_chunk(src, c, true);
    {
      ProfScope prof("sparse_fwd_up", s);
      // two-slab warps take four entries per batch, four-slab warps two
      // (measured on the 2B- and 8B-class shapes)
      if constexpr (VPL <= 2)
        ell_dot_kernel<TEAM, VPL, 4, 2, kDotH><<<(M + ROWS - 1) / ROWS, 256, 0, s>>>(up, sc);
      else
        ell_dot_kernel<TEAM, VPL, 2, 3, kDotH><<<(M + ROWS - 1) / ROWS, 256, 0, s>>>(up, sc);
    }
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  constexpr int DV = 2;  // down: two slabs per warp, two entries per batch
  EllAxpyArgs down{};
  down.rows0 = reinterpret_cast<const uint16_t*>(wd);
  down.M = M;
  down.d = d;
  down.coef = hbuf;
  down.part = part;
  down.out = reinterpret_cast<uint16_t*>(y);
  const int wpr = (d + 256 * DV - 1) / (256 * DV);
  const long long blocks = ((long long)M * wpr + 7) / 8;
  for (int c = 0; c < chunks; ++c) {
    Src sc = set_chunk(src, c, false);
    down.pass = (c == 0 ? kEllPassFirst : 0) | (c == chunks - 1 ? kEllPassLast : 0);
    {
      ProfScope prof("sparse_fwd_down", s);
      ell_axpy_kernel<DV, 2, 4><<<(unsigned)blocks, 256, 0, s>>>(down, sc);
    }
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ELL rows up to d_model = 1024 take the fused kernel, wider ones the split
// up and down gathers (the fused kernel when twell_set_split_gathers(0));
// TwELL rows take the fused kernel, split over clusters for small batches,
// or the split gathers when wide and given a workspace for h.
template <int TEAM, int VPL, bool ELL>
cudaError_t launch_shape(const void* x, const void* wuT, const void* wd, int M, int d, int f,
                         const twell_tiles* tiles, int T, int tile_n, int cap,
                         const twell_hybrid* route, void* y, float* part, float* hbuf, int chunks,
                         int cl, cudaStream_t s) {
  if constexpr (ELL && TEAM > 1) {
    if (!split_gathers())
      return launch_team<TEAM, VPL, true>(x, wuT, wd, M, d, f, nullptr, T, tile_n, cap, route, y,
                                          part, chunks, s);
    if (!hbuf) return cudaErrorInvalidValue;
    EllSrc src{reinterpret_cast<const uint16_t*>(route->ell_val), route->ell_col, route->ell_nnz,
               route->ell_width, 0, f, 1, f};
    const int n = part ? l2_chunks(2.0 * (double)f * d, 0.75, 0.5) : 1;
    auto chunk = [f, n](EllSrc c, int i, bool) {
      c.j_lo = (int)((long long)f * i / n);
      c.j_hi = (int)((long long)f * (i + 1) / n);
      c.whole = n == 1;
      return c;
    };
    return launch_split<TEAM, VPL>(x, wuT, wd, M, d, src, n, chunk, y, part, hbuf, s);
  } else if constexpr (ELL) {
    return launch_team<TEAM, VPL, true>(x, wuT, wd, M, d, f, nullptr, T, tile_n, cap, route, y,
                                        part, chunks, s);
  } else {
    if (cl > 1) return launch_cluster<TEAM, VPL>(x, wuT, wd, M, d, tiles, T, tile_n, cap, cl, y, s);
    if constexpr (TEAM > 1) {
      if (hbuf && split_gathers()) {  // wide TwELL rows with a workspace for h: the split gathers
        TwellSrc src{reinterpret_cast<const uint16_t*>(tiles->val), tiles->idx, tiles->cnt, T,
                     tile_n, cap, 0, T, nullptr};
        const int n = part ? l2_chunks(2.0 * (double)f * d, 0.75, 0.5) : 1;
        int* status = device_status_ptr();
        auto chunk = [T, n, status](TwellSrc c, int i, bool up) {
          c.t_lo = (int)((long long)T * i / n);
          c.t_hi = (int)((long long)T * (i + 1) / n);
          c.status = up ? status : nullptr;  // the up gather flags overfull tiles once
          return c;
        };
        return launch_split<TEAM, VPL>(x, wuT, wd, M, d, src, n, chunk, y, part, hbuf, s);
      }
    }
    return launch_team<TEAM, VPL, false>(x, wuT, wd, M, d, f, tiles, T, tile_n, cap, nullptr, y,
                                         nullptr, 1, s);
  }
}

template <bool ELL>
cudaError_t launch_fmt(const void* x, const void* wuT, const void* wd, int M, int d, int f,
                       const twell_tiles* tiles, int T, int tile_n, int cap,
                       const twell_hybrid* route, void* y, float* part, float* hbuf, int chunks,
                       cudaStream_t s) {
#define TW_FWD(TEAM, VPL)                                                                       \
  launch_shape<TEAM, VPL, ELL>(x, wuT, wd, M, d, f, tiles, T, tile_n, cap, route, y, part, hbuf, \
                               chunks, cl, s)
  // TwELL rows too few to give every SM two blocks: split each row over a
  // cluster of up to 8 blocks, widening while the grid stays within four
  // blocks per SM (a row's slices then stay short even for the heaviest rows)
  int cl = 1;
  if (!ELL) {
    const int team = d <= 1024 ? 1 : d <= 4096 ? 4 : 8;
    const int groups = (M + 8 / team - 1) / (8 / team);
    if (groups < 2 * num_sms())
      while (cl < 8 && groups * cl * 2 <= 4 * num_sms() && 2 * cl <= T &&
             d % (64 * 2 * cl) == 0)
        cl *= 2;
  }
  if (d <= 512) return TW_FWD(1, 2);
  if (d <= 1024) return TW_FWD(1, 4);
  if (d <= 2048) return TW_FWD(4, 2);
  if (d <= 4096) return TW_FWD(4, 4);
  return TW_FWD(8, 4);
#undef TW_FWD
}

}  // namespace

cudaError_t launch_sparse_fwd(const void* x, const void* wuT, const void* wd, int M, int d, int f,
                              const twell_tiles* tiles, int tile_n, int cap,
                              const twell_hybrid* route, void* y, float* part, float* hbuf,
                              cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  cudaError_t ce = checked_setup();
  if (ce != cudaSuccess) return ce;
  const int T = f / tile_n;
  if (route) {
    // Wu^T and Wd rows: split the neuron axis into L2-sized passes once they
    // exceed 3/4 of L2 (partial sums in `part`, same accumulation order; on
    // the 2B-class shape, 67 MB of weights, two passes were slower than one)
    const int chunks = part ? l2_chunks(2.0 * 2.0 * (double)f * d, 0.75, 0.5) : 1;
    return launch_fmt<true>(x, wuT, wd, M, d, f, nullptr, T, tile_n, cap, route, y, part, hbuf,
                            chunks, s);
  }
  return launch_fmt<false>(x, wuT, wd, M, d, f, tiles, T, tile_n, cap, nullptr, y, part, hbuf, 1,
                           s);
}

}  // namespace tw
