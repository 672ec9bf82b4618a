// sparse_bwd.cu -- backward of the sparse gated FFN over the ELL rows.
//
// Training path of page 2 "Sakana AI and NVIDIA introduce TwELL with CUDA
// kernels ...", section "¿Qué hace distinto a TwELL frente a ELL clásico?"
// (hybrid ELL rows), with the L1 term of section "Receta de entrenamiento".
// For a live entry (m, j) with stored gate g > 0:
//   dh = dY_m . Wd[j, :],  u = x_m . Wu[:, j],  h = g u
//   du = dh g,  da = dh u + lambda        (ReLU' = 1 on live entries)
//   dX_m += du Wu[:, j]^T + da Wg[:, j]^T
//   dWd[j] += h dY_m,  dWu^T[j] += du x_m,  dWg^T[j] += da x_m
// Dead entries contribute exactly zero, so visiting live entries only is the
// exact gradient.
//
// Three phases, all deterministic (no floating-point atomics):
//   1. csc_*: a column-major (neuron-major) index of the live entries, rows
//      ascending inside every neuron.  Per 32-row block and neuron a bitmask
//      of the rows that use the neuron gives every entry its rank without any
//      ordering race: rank = prefix over groups of 32 blocks + prefix over the
//      blocks of its group + popcount of lower bits.
//   2. bwd_rows: one team of warps per row computes dh, u, du, da, h per entry
//      (stored at the entry's neuron-major position) and dX_m.  Rows wider
//      than 1024 take two gathers instead (dh; then u with du, da, h and dX),
//      which meet one barrier per 32 entries (ell_gather.cuh).
// Gathered rows are loaded without predicates: a batch slot past the last
// entry reads neuron (or row) 0 with zero coefficients, and lanes past
// d_model read the first slab against zero x / dY, so no zero-fill selects
// sit between the loads and the arithmetic.
//   3. bwd_neurons: one team per neuron sums its entries in ascending row
//      order into dWd[j], dWu^T[j], dWg^T[j] (fp32, written once).
#include "common.cuh"
#include "ell_gather.cuh"
#include "internal.h"

namespace tw {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 8;
constexpr int kPassFirst = 1, kPassLast = 2;

// ---------------------------------------------------------------- CSC index
__global__ void __launch_bounds__(kWarps * 32)
    csc_mark_kernel(const uint16_t* __restrict__ ell_col, const int* __restrict__ ell_nnz, int M,
                    int W, int f, unsigned* __restrict__ mask) {
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (m >= M) return;
  int n = ell_nnz[m];
  TW_CHECK_INDEX(n, n >= 0 && n <= W);
  unsigned* mrow = mask + (long long)(m >> 5) * f;
  const unsigned bit = 1u << (m & 31);
  for (int s = lane; s < n; s += 32) {
    int j = ell_col[(long long)m * W + s];
    TW_CHECK_INDEX(j, j < f);
    atomicOr(mrow + j, bit);
  }
}

// Column scan of the row masks.  CTA c handles neurons [32 c, 32 c + 32)
// over every row block, 32 blocks at a time (warp w: block 32 g + w; lane:
// neuron), with a running count per neuron:
//   off[b][j] = live rows of neuron j in the blocks before b
//   tot[j]    = live rows of neuron j
// The CTA that finishes last (a ticket on the zeroed counter `done`) forms
// csc_ptr[0..f] = exclusive prefix of tot.
__global__ void __launch_bounds__(1024)
    csc_scan_kernel(const unsigned* __restrict__ mask, int NB, int f, int* __restrict__ off,
                    int* __restrict__ tot, unsigned* __restrict__ done, int* __restrict__ csc_ptr) {
  __shared__ int c[32][33];
  __shared__ int carry[32];
  __shared__ int warp_tot[32];
  __shared__ int chunk_carry;
  __shared__ bool last;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int j = blockIdx.x * 32 + lane;
  const int NG = (NB + 31) / 32;
  if (tid < 32) carry[tid] = 0;
  for (int g0 = 0; g0 < NG; g0 += 8) {
    // eight groups' mask words in flight before the first is scanned
    int v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int b = (g0 + k) * 32 + w;
      v[k] = (j < f && b < NB) ? __popc(mask[(long long)b * f + j]) : 0;  // coalesced over j
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (g0 + k >= NG) break;  // uniform over the CTA
      __syncthreads();          // the previous group's reads of c (and carry's init) are done
      c[w][lane] = v[k];
      __syncthreads();
      {  // warp w scans neuron 32 c + w over the group's blocks (lane)
        const int x = c[lane][w];
        const int incl = warp_incl_scan(x);
        c[lane][w] = carry[w] + incl - x;
        __syncwarp();
        if (lane == 31) carry[w] += incl;
      }
      __syncthreads();
      const int b = (g0 + k) * 32 + w;
      if (j < f && b < NB) off[(long long)b * f + j] = c[w][lane];
    }
  }
  __syncthreads();
  if (tid < 32 && blockIdx.x * 32 + tid < f) tot[blockIdx.x * 32 + tid] = carry[tid];
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid == 0) chunk_carry = 0;
  __syncthreads();
  for (int base = 0; base < f; base += 1024) {
    const int jj = base + tid;
    const int t = jj < f ? __ldcg(tot + jj) : 0;  // other CTAs' totals: from L2
    const int incl = warp_incl_scan(t);
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int x = warp_tot[lane];
      warp_tot[lane] = warp_incl_scan(x) - x;
    }
    __syncthreads();
    const int ex = chunk_carry + warp_tot[w] + incl - t;
    if (jj < f) csc_ptr[jj] = ex;
    __syncthreads();
    if (tid == 1023) chunk_carry = ex + t;
    __syncthreads();
  }
  if (tid == 0) csc_ptr[f] = chunk_carry;
}

__global__ void __launch_bounds__(kWarps * 32)
    csc_place_kernel(const uint16_t* __restrict__ ell_col, const int* __restrict__ ell_nnz, int M,
                     int W, int f, const unsigned* __restrict__ mask, const int* __restrict__ off,
                     const int* __restrict__ csc_ptr, int* __restrict__ csc_row,
                     int* __restrict__ slot_pos) {
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (m >= M) return;
  int n = ell_nnz[m];
  TW_CHECK_INDEX(n, n >= 0 && n <= W);
  const long long blk = (long long)(m >> 5) * f;
  const unsigned below = (1u << (m & 31)) - 1u;
  for (int s = lane; s < n; s += 32) {
    int j = ell_col[(long long)m * W + s];
    TW_CHECK_INDEX(j, j < f);
    const int pos = csc_ptr[j] + off[blk + j] + __popc(mask[blk + j] & below);
    csc_row[pos] = m;
    slot_pos[(long long)m * W + s] = pos;
  }
}

// ---------------------------------------------------------------- row phase
template <int TEAM>
__device__ __forceinline__ int slab(int lane, int wt, int v) {
  return 8 * (lane + 32 * (wt + TEAM * v));
}

// One team of TEAM warps per ELL row; fp32-pair arithmetic as in the forward.
template <int TEAM, int VPL, int B, int MINB>
__global__ void __launch_bounds__(256, MINB)
    bwd_rows_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ dy,
                    const uint16_t* __restrict__ wgT, const uint16_t* __restrict__ wuT,
                    const uint16_t* __restrict__ wd, int M, int d,
                    const uint16_t* __restrict__ ell_val, const uint16_t* __restrict__ ell_col,
                    const int* __restrict__ ell_nnz, int W, const int* __restrict__ slot_pos,
                    float lambda, float4* __restrict__ csc_vals, uint16_t* __restrict__ dx,
                    float* __restrict__ part, int j_lo, int j_hi, int pass) {
  static_assert(32 % B == 0, "a batch never reaches past lane 31");
  constexpr int ROWS = 8 / TEAM;
  __shared__ float red[2][ROWS][TEAM][2 * B];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / TEAM, wt = warp % TEAM;
  const int m = blockIdx.x * ROWS + team;
  if (m >= M) return;

  const bool first = pass & kPassFirst, last = pass & kPassLast;
  // x, dY and the dX carry stream through once per pass: evict-first, so the
  // pass's weight rows keep L2
  const uint64_t pol = l2_evict_first_policy();
  uint4 xp[VPL], dyp[VPL];  // x_m, dY_m slabs, packed bf16
  uint64_t acc[VPL][4];
  int eoff[VPL];  // slab offsets, lanes past d_model read the first slab
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = slab<TEAM>(lane, wt, v);
    const bool ok = e < d;
    eoff[v] = ok ? e : 0;
    xp[v] = ok ? ldg_v4_hint(x + (long long)m * d + e, pol) : make_uint4(0, 0, 0, 0);
    dyp[v] = ok ? ldg_v4_hint(dy + (long long)m * d + e, pol) : make_uint4(0, 0, 0, 0);
    if (first || !ok) {
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[v][k] = 0;
    } else {  // dX_m of the earlier neuron chunks
      const float* pp = part + (long long)m * d + e;
      const uint4 q0 = ldg_v4_hint(pp, pol), q1 = ldg_v4_hint(pp + 4, pol);
      acc[v][0] = f2_make(q0.x, q0.y);
      acc[v][1] = f2_make(q0.z, q0.w);
      acc[v][2] = f2_make(q1.x, q1.y);
      acc[v][3] = f2_make(q1.z, q1.w);
    }
  }
  int buf = 0;
  int n = ell_nnz[m];
  TW_CHECK_INDEX(n, n >= 0 && n <= W);
  // a row's columns ascend: the neuron chunk [j_lo, j_hi) is the slice [a, b)
  int a = 0, bnd = n;
  if (!(first && last)) {
    a = bnd = 0;
    for (int s0 = 0; s0 < n; s0 += 32) {
      const int jc = s0 + lane < n ? (int)ell_col[(long long)m * W + s0 + lane] : 0x7fffffff;
      a += __popc(__ballot_sync(kFull, jc < j_lo));
      bnd += __popc(__ballot_sync(kFull, jc < j_hi));
    }
  }
  for (int e0 = a; e0 < bnd; e0 += 32) {
    const int count = min(32, bnd - e0);
    int jl = 0, pl = 0;  // slots past the row's end: neuron 0, gate 0
    float gl = 0.f;
    if (lane < count) {
      const long long s = (long long)m * W + e0 + lane;
      jl = ell_col[s];
      TW_CHECK_INDEX(jl, jl >= j_lo && jl < j_hi);  // the pass's neuron chunk
      gl = bf16_bits_to_float(ell_val[s]);
      pl = slot_pos[s];
      TW_CHECK_INDEX(pl, pl >= 0 && (long long)pl < (long long)M * W);
    }
    for (int i = 0; i < count; i += B) {
      int j[B], pos[B];
      float g[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int src = (i + b) & 31;
        j[b] = __shfl_sync(kFull, jl, src);
        pos[b] = __shfl_sync(kFull, pl, src);
        g[b] = __shfl_sync(kFull, gl, src);
      }
      // unpredicated loads: a slot past the end reads neuron 0's rows
      uint4 wdv[B][VPL], wuv[B][VPL], wgv[B][VPL];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const long long row = (long long)j[b] * d;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          wdv[b][v] = ldg_v4(wd + row + eoff[v]);
          wuv[b][v] = ldg_v4(wuT + row + eoff[v]);
          wgv[b][v] = ldg_v4(wgT + row + eoff[v]);
        }
      }
      float dh[B], u[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float a0 = 0.f, a1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          dot8_bf16(dyp[v], wdv[b][v], a0, a1);
          dot8_bf16(xp[v], wuv[b][v], c0, c1);
        }
        dh[b] = a0 + a1;
        u[b] = c0 + c1;
      }
      if constexpr (B == 1) {
        warp_sum2(dh[0], u[0]);
      } else if constexpr (B == 2) {
        warp_sum4(dh[0], u[0], dh[B - 1], u[B - 1]);
      } else {
#pragma unroll
        for (int b = 0; b < B; ++b) {
          dh[b] = warp_sum(dh[b]);
          u[b] = warp_sum(u[b]);
        }
      }
      if constexpr (TEAM > 1) {
        if (lane == 0)
#pragma unroll
          for (int b = 0; b < B; ++b) {
            red[buf][team][wt][2 * b] = dh[b];
            red[buf][team][wt][2 * b + 1] = u[b];
          }
        named_barrier(1 + team, 32 * TEAM);
#pragma unroll
        for (int b = 0; b < B; ++b) {
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int w = 0; w < TEAM; ++w) {
            s0 += red[buf][team][w][2 * b];
            s1 += red[buf][team][w][2 * b + 1];
          }
          dh[b] = s0;
          u[b] = s1;
        }
        buf ^= 1;
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        // a slot past the end has g = 0 (du = 0) and must add no da either
        const bool live = i + b < count;
        const float du = dh[b] * g[b];
        const float da = live ? fmaf(dh[b], u[b], lambda) : 0.f;
        if (live && wt == 0 && lane == 0) csc_vals[pos[b]] = make_float4(du, da, g[b] * u[b], 0.f);
        const uint64_t du2 = f2_splat(du), da2 = f2_splat(da);
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          axpy8_f2(du2, wuv[b][v], acc[v]);
          axpy8_f2(da2, wgv[b][v], acc[v]);
        }
      }
    }
  }
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = slab<TEAM>(lane, wt, v);
    if (e >= d) continue;
    if (last) {
      *reinterpret_cast<uint4*>(dx + (long long)m * d + e) = f2x4_to_bf8(acc[v]);
    } else {
      float* pp = part + (long long)m * d + e;
      st_v4_hint(pp, make_uint4((uint32_t)acc[v][0], (uint32_t)(acc[v][0] >> 32),
                                (uint32_t)acc[v][1], (uint32_t)(acc[v][1] >> 32)), pol);
      st_v4_hint(pp + 4, make_uint4((uint32_t)acc[v][2], (uint32_t)(acc[v][2] >> 32),
                                    (uint32_t)acc[v][3], (uint32_t)(acc[v][3] >> 32)), pol);
    }
  }
}

// ---------------------------------------------------------------- neuron phase
// One team per neuron; each warp owns VPL slabs of the column window
// [c0, c1) of d_model and needs no cross-warp communication, so narrow slabs
// (VPL = 1) buy occupancy and more gathered rows in flight per SM.  PARTS
// selects the outputs: kNeuD gathers dY rows for dWd, kNeuX gathers x rows
// for dWu^T and dWg^T, and kNeuD | kNeuX does both in one pass.  Each output
// element sums its entries in ascending row order either way, and a column
// window owns its output columns outright, so windows need no carry.
constexpr int kNeuD = 1, kNeuX = 2;

template <int TEAM, int VPL, int B, int MINB, int PARTS>
__global__ void __launch_bounds__(256, MINB)
    bwd_neurons_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ dy, int M,
                       int d, int f, int c0, int c1, const int* __restrict__ csc_ptr,
                       const int* __restrict__ csc_row,
                       const float4* __restrict__ csc_vals, float* __restrict__ dwgT,
                       float* __restrict__ dwuT, float* __restrict__ dwd) {
  constexpr bool DO_D = PARTS & kNeuD, DO_X = PARTS & kNeuX;
  constexpr int ROWS = 8 / TEAM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / TEAM, wt = warp % TEAM;
  const int j = blockIdx.x * ROWS + team;
  if (j >= f) return;
  uint64_t ad[DO_D ? VPL : 1][4], au[DO_X ? VPL : 1][4], ag[DO_X ? VPL : 1][4];
#pragma unroll
  for (int v = 0; v < VPL; ++v)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (DO_D) ad[v][k] = 0;
      if constexpr (DO_X) au[v][k] = ag[v][k] = 0;
    }

  int eoff[VPL];  // slab offsets, lanes past the window read its first slab
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = c0 + slab<TEAM>(lane, wt, v);
    eoff[v] = e < c1 ? e : c0;
  }
  const int p0 = csc_ptr[j], p1 = csc_ptr[j + 1];
  for (int e0 = p0; e0 < p1; e0 += 32) {
    const int count = min(32, p1 - e0);
    int ml = 0;  // slots past the neuron's end: row 0 with zero coefficients
    float4 vl = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < count) {
      ml = csc_row[e0 + lane];
      TW_CHECK_INDEX(ml, ml >= 0 && ml < M);
      vl = csc_vals[e0 + lane];
    }
    for (int i = 0; i < count; i += B) {
      int m[B];
      float du[B], da[B], h[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        // with B not dividing 32 the last batch reaches past lane 31: those
        // slots take row 0 with zero coefficients, like slots past the end
        const bool in = 32 % B == 0 || i + b < 32;
        const int src = (i + b) & 31;
        m[b] = __shfl_sync(kFull, ml, src);
        if constexpr (DO_X) {
          du[b] = __shfl_sync(kFull, vl.x, src);
          da[b] = __shfl_sync(kFull, vl.y, src);
        }
        if constexpr (DO_D) h[b] = __shfl_sync(kFull, vl.z, src);
        if (!in) {
          m[b] = 0;
          du[b] = da[b] = h[b] = 0.f;
        }
      }
      uint4 xv[DO_X ? B : 1][VPL], dyv[DO_D ? B : 1][VPL];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const long long row = (long long)m[b] * d;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          if constexpr (DO_X) xv[b][v] = ldg_v4(x + row + eoff[v]);
          if constexpr (DO_D) dyv[b][v] = ldg_v4(dy + row + eoff[v]);
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          if constexpr (DO_D) axpy8_f2(f2_splat(h[b]), dyv[b][v], ad[v]);
          if constexpr (DO_X) {
            const uint64_t du2 = f2_splat(du[b]), da2 = f2_splat(da[b]);
            uint64_t xf[4];
            bf8_to_f2(xv[b][v], xf);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              au[v][k] = f2_fma(du2, xf[k], au[v][k]);
              ag[v][k] = f2_fma(da2, xf[k], ag[v][k]);
            }
          }
        }
      }
    }
  }
  // dW rows are written once: evict-first so they do not displace x / dY
  const uint64_t pol = l2_evict_first_policy();
  const long long row = (long long)j * d;
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = c0 + slab<TEAM>(lane, wt, v);
    if (e < c1) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if constexpr (DO_D) {
          const uint64_t d0 = ad[v][2 * q], d1 = ad[v][2 * q + 1];
          st_v4_hint(dwd + row + e + 4 * q,
                     make_uint4((uint32_t)d0, (uint32_t)(d0 >> 32), (uint32_t)d1, (uint32_t)(d1 >> 32)), pol);
        }
        if constexpr (DO_X) {
          const uint64_t u0 = au[v][2 * q], u1 = au[v][2 * q + 1];
          const uint64_t g0 = ag[v][2 * q], g1 = ag[v][2 * q + 1];
          st_v4_hint(dwuT + row + e + 4 * q,
                     make_uint4((uint32_t)u0, (uint32_t)(u0 >> 32), (uint32_t)u1, (uint32_t)(u1 >> 32)), pol);
          st_v4_hint(dwgT + row + e + 4 * q,
                     make_uint4((uint32_t)g0, (uint32_t)(g0 >> 32), (uint32_t)g1, (uint32_t)(g1 >> 32)), pol);
        }
      }
    }
  }
}

template <int TEAM, int VPL, int B, int MINB>
cudaError_t rows_team(const void* x, const void* dy, const void* wgT, const void* wuT,
                      const void* wd, int M, int d, int f, const twell_hybrid& r,
                      const int* slot_pos, float lambda, float4* csc_vals, void* dx, float* part,
                      int chunks, cudaStream_t s) {
  constexpr int ROWS = 8 / TEAM;
  for (int c = 0; c < chunks; ++c) {
    const int j_lo = (int)((long long)f * c / chunks), j_hi = (int)((long long)f * (c + 1) / chunks);
    const int pass = (c == 0 ? kPassFirst : 0) | (c == chunks - 1 ? kPassLast : 0);
    {
      ProfScope prof("bwd_rows", s);
      bwd_rows_kernel<TEAM, VPL, B, MINB><<<(M + ROWS - 1) / ROWS, 256, 0, s>>>(
          reinterpret_cast<const uint16_t*>(x), reinterpret_cast<const uint16_t*>(dy),
          reinterpret_cast<const uint16_t*>(wgT), reinterpret_cast<const uint16_t*>(wuT),
          reinterpret_cast<const uint16_t*>(wd), M, d,
          reinterpret_cast<const uint16_t*>(r.ell_val), r.ell_col, r.ell_nnz, r.ell_width,
          slot_pos, lambda, csc_vals, reinterpret_cast<uint16_t*>(dx), part, j_lo, j_hi, pass);
    }
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// One launch per column window: windows of d / windows columns (a multiple
// of 8, so every slab stays 16-byte aligned), the team covering one window.
template <int TEAM, int VPL, int B, int MINB, int PARTS>
cudaError_t neurons_team(const void* x, const void* dy, int M, int d, int f, const int* csc_ptr,
                         const int* csc_row, const float4* csc_vals, float* dwgT, float* dwuT,
                         float* dwd, cudaStream_t s, int windows = 1) {
  constexpr int ROWS = 8 / TEAM;
  const int width = d / windows;
  if (width % 8 != 0 || width > TEAM * 32 * 8 * VPL) return cudaErrorInvalidValue;
  for (int w = 0; w < windows; ++w) {
    {
      ProfScope prof(PARTS == kNeuD ? "bwd_neurons_dy" : PARTS == kNeuX ? "bwd_neurons_x" : "bwd_neurons", s);
      bwd_neurons_kernel<TEAM, VPL, B, MINB, PARTS><<<(f + ROWS - 1) / ROWS, 256, 0, s>>>(
          reinterpret_cast<const uint16_t*>(x), reinterpret_cast<const uint16_t*>(dy), M, d, f,
          w * width, (w + 1) * width, csc_ptr, csc_row, csc_vals, dwgT, dwuT, dwd);
    }
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

// blk_counts holds the scan's finish counter (32 ints), the row masks and
// the block offsets ([ceil(M/32)][f] ints each) and the neuron totals (f).
cudaError_t launch_csc_build(const twell_hybrid& r, int M, int f, int* blk_counts, int* csc_ptr,
                             int* csc_row, int* slot_pos, cudaStream_t s) {
  const int NB = (M + 31) / 32;
  unsigned* done = reinterpret_cast<unsigned*>(blk_counts);
  unsigned* mask = done + 32;
  {
    const cudaError_t ce = checked_setup();
    if (ce != cudaSuccess) return ce;
  }
  int* off = blk_counts + 32 + (long long)NB * f;
  int* tot = off + (long long)NB * f;
  // the counter and the masks start at zero
  cudaError_t e = cudaMemsetAsync(done, 0, sizeof(unsigned) * (32 + (size_t)NB * f), s);
  if (e != cudaSuccess) return e;
  if (M == 0) return cudaMemsetAsync(csc_ptr, 0, sizeof(int) * ((size_t)f + 1), s);
  {
    ProfScope prof("csc_mark", s);
    csc_mark_kernel<<<(M + kWarps - 1) / kWarps, kWarps * 32, 0, s>>>(r.ell_col, r.ell_nnz, M,
                                                                      r.ell_width, f, mask);
  }
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    ProfScope prof("csc_scan", s);
    csc_scan_kernel<<<(f + 31) / 32, 1024, 0, s>>>(mask, NB, f, off, tot, done, csc_ptr);
  }
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    ProfScope prof("csc_place", s);
    csc_place_kernel<<<(M + kWarps - 1) / kWarps, kWarps * 32, 0, s>>>(
        r.ell_col, r.ell_nnz, M, r.ell_width, f, mask, off, csc_ptr, csc_row, slot_pos);
  }
  count_launch();
  return cudaGetLastError();
}

namespace {

// Wide ELL rows: the fused row phase split into two gathers (ell_gather.cuh)
//   dh = dY_m . Wd[j]                                   over Wd
//   u = x_m . Wu[:, j]; du, da, h per entry;
//   dX_m = sum du Wu[:, j]^T + da Wg[:, j]^T             over Wu^T and Wg^T
// each in its own L2-sized neuron passes.  Per entry the arithmetic is the
// fused kernel's; dX sums each group of 32 entries' du Wu^T terms before its
// da Wg^T terms (see ell_grad_dx_kernel).
template <int TEAM, int VPL>
cudaError_t split_rows(const void* x, const void* dy, const void* wgT, const void* wuT,
                       const void* wd, int M, int d, int f, const twell_hybrid& r,
                       const int* slot_pos, float lambda, float4* csc_vals, void* dx, float* part,
                       float* dhbuf, cudaStream_t s) {
  constexpr int ROWS = 8 / TEAM;
  const unsigned grid = (unsigned)((M + ROWS - 1) / ROWS);
  EllDotArgs p{};
  p.M = M;
  p.d = d;
  p.out = dhbuf;
  p.vec = reinterpret_cast<const uint16_t*>(dy);
  p.rows = reinterpret_cast<const uint16_t*>(wd);
  EllSrc src{reinterpret_cast<const uint16_t*>(r.ell_val), r.ell_col, r.ell_nnz, r.ell_width, 0,
             f, 1, f};
  const int dot_chunks = part ? l2_chunks(2.0 * (double)f * d, 0.75, 0.5) : 1;
  for (int c = 0; c < dot_chunks; ++c) {
    src.j_lo = (int)((long long)f * c / dot_chunks);
    src.j_hi = (int)((long long)f * (c + 1) / dot_chunks);
    src.whole = dot_chunks == 1;
    {
      ProfScope prof("bwd_dh", s);
      // two-slab warps take four entries per batch, four-slab warps two
      if constexpr (VPL <= 2)
        ell_dot_kernel<TEAM, VPL, 4, 2, kDotDh><<<grid, 256, 0, s>>>(p, src);
      else
        ell_dot_kernel<TEAM, VPL, 2, 3, kDotDh><<<grid, 256, 0, s>>>(p, src);
    }
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  EllGradDxArgs g{};
  g.x = reinterpret_cast<const uint16_t*>(x);
  g.wuT = reinterpret_cast<const uint16_t*>(wuT);
  g.wgT = reinterpret_cast<const uint16_t*>(wgT);
  g.M = M;
  g.d = d;
  g.dh = dhbuf;
  g.slot_pos = slot_pos;
  g.lambda = lambda;
  g.csc_vals = csc_vals;
  g.part = part;
  g.dx = reinterpret_cast<uint16_t*>(dx);
  // the gradient + dX gather runs eight warps per row (half the dot
  // gathers' slabs per warp, four entries per batch, four blocks per SM):
  // on the 2B- and 8B-class shapes 19 % / 20 % faster than the dot
  // gathers' team shape (two entries, two blocks), and 14 % / 14 % faster
  // than separate gradient and dX gathers
  constexpr int GT = 8, GV = (TEAM * VPL + 7) / 8;
  const int gd_chunks = part ? l2_chunks(4.0 * (double)f * d, 0.75, 0.5) : 1;
  for (int c = 0; c < gd_chunks; ++c) {
    src.j_lo = (int)((long long)f * c / gd_chunks);
    src.j_hi = (int)((long long)f * (c + 1) / gd_chunks);
    src.whole = gd_chunks == 1;
    g.pass = (c == 0 ? kEllPassFirst : 0) | (c == gd_chunks - 1 ? kEllPassLast : 0);
    {
      ProfScope prof("bwd_grad_dx", s);
      if constexpr (GV <= 2)
        ell_grad_dx_kernel<GT, GV, 4, 4><<<(unsigned)M, 256, 0, s>>>(g, src);
      else
        ell_grad_dx_kernel<GT, GV, 2, 2><<<(unsigned)M, 256, 0, s>>>(g, src);
    }
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_sparse_bwd_rows(const void* x, const void* dy, const void* wgT, const void* wuT,
                                   const void* wd, int M, int d, int f, const twell_hybrid& route,
                                   const int* slot_pos, float lambda, float4* csc_vals, void* dx,
                                   float* part, float* dhbuf, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  {
    const cudaError_t ce = checked_setup();
    if (ce != cudaSuccess) return ce;
  }
  if (d > 1024 && split_gathers()) {  // wide rows: the split gathers, the forward's team shapes
    if (!dhbuf) return cudaErrorInvalidValue;
#define TW_SPLIT(T, V)                                                                          \
  split_rows<T, V>(x, dy, wgT, wuT, wd, M, d, f, route, slot_pos, lambda, csc_vals, dx, part,  \
                   dhbuf, s)
    if (d <= 2048) return TW_SPLIT(4, 2);
    if (d <= 4096) return TW_SPLIT(4, 4);
    return TW_SPLIT(8, 4);
#undef TW_SPLIT
  }
  // Wd, Wu^T and Wg^T rows: L2-sized neuron passes once they exceed half of
  // L2 (x, dY and dX stream through L2 beside them), chunks of at most 0.65
  // of L2 (measured with this kernel on 101 MB and 352 MB of weights: two
  // passes beat one by 7 %, four beat six and eight), dX_m carried in `part`
  // (fp32) with the accumulation order unchanged
  const int chunks = part ? l2_chunks(3.0 * 2.0 * (double)f * d, 0.5, 0.65) : 1;
#define TW_ROWS(T, V, B, MINB)                                                                 \
  rows_team<T, V, B, MINB>(x, dy, wgT, wuT, wd, M, d, f, route, slot_pos, lambda, csc_vals, dx, \
                           part, chunks, s)
  // wider rows here only with the split gathers switched off; team shapes as
  // measured on the 2B- and 8B-class shapes (one entry per batch from d = 2048)
  if (d <= 512) return TW_ROWS(1, 2, 2, 2);
  if (d <= 1024) return TW_ROWS(1, 4, 1, 2);
  if (d <= 2048) return TW_ROWS(4, 2, 1, 3);
  if (d <= 4096) return TW_ROWS(4, 4, 1, 2);
  return TW_ROWS(8, 4, 2, 1);
#undef TW_ROWS
}

cudaError_t launch_sparse_bwd_neurons(const void* x, const void* dy, int M, int d, int f,
                                      const int* csc_ptr, const int* csc_row,
                                      const float4* csc_vals, float* dwgT, float* dwuT, float* dwd,
                                      cudaStream_t s) {
  if (f == 0) return cudaSuccess;
  {
    const cudaError_t ce = checked_setup();
    if (ce != cudaSuccess) return ce;
  }
#define TW_NEU(T, V, B, MINB, P) \
  neurons_team<T, V, B, MINB, P>(x, dy, M, d, f, csc_ptr, csc_row, csc_vals, dwgT, dwuT, dwd, s)
#define TW_NEU_W(T, V, B, MINB, P, NW) \
  neurons_team<T, V, B, MINB, P>(x, dy, M, d, f, csc_ptr, csc_row, csc_vals, dwgT, dwuT, dwd, s, \
                                 NW)
  // Once x and dY together outgrow L2 the phase runs twice, over dY rows
  // (dWd) and over x rows (dWu^T, dWg^T): each pass gathers from a table half
  // the size, so more of its rows hit in L2.  A pass whose table (x or dY,
  // 2 M d bytes) still outgrows half of L2 runs in column windows, each
  // gathering a column slice of the rows (d / 2 columns: a table half the
  // size again) and writing its own columns of dW, so no partial sums are
  // carried between launches.
  if (4.0 * (double)M * d > 0.75 * l2_bytes()) {
    cudaError_t e;
    const int windows = (2.0 * (double)M * d > 0.5 * l2_bytes() && d % 16 == 0) ? 2 : 1;
    if (d <= 1024) {
      if ((e = TW_NEU(4, 1, 4, 4, kNeuD)) != cudaSuccess) return e;
      return TW_NEU(4, 1, 4, 4, kNeuX);
    }
    if (d <= 2048) {
      if ((e = TW_NEU(8, 1, 4, 4, kNeuD)) != cudaSuccess) return e;
      return TW_NEU(8, 1, 4, 3, kNeuX);
    }
    if (d <= 4096 && windows == 2) {  // 2048-column windows: the 2048-wide shapes
      if ((e = TW_NEU_W(8, 1, 4, 4, kNeuD, 2)) != cudaSuccess) return e;
      return TW_NEU_W(8, 1, 4, 3, kNeuX, 2);
    }
    if (d <= 4096) {  // four blocks per SM: 14 % faster on the 8B-class shape than three
      if ((e = TW_NEU(8, 2, 4, 4, kNeuD)) != cudaSuccess) return e;
      return TW_NEU(8, 2, 4, 4, kNeuX);
    }
    if ((e = TW_NEU(8, 4, 2, 2, kNeuD)) != cudaSuccess) return e;
    return TW_NEU(8, 4, 2, 2, kNeuX);
  }
  // one 256-element slab per warp (short accumulators, 3-4 blocks per SM)
  // while a block's 8 warps cover d_model; at d = 4096 batches of three rows
  // (6 % faster than two on the 8B-class shape)
  constexpr int kBoth = kNeuD | kNeuX;
  if (d <= 256) return TW_NEU(1, 1, 2, 4, kBoth);
  if (d <= 512) return TW_NEU(2, 1, 2, 4, kBoth);
  if (d <= 1024) return TW_NEU(4, 1, 2, 4, kBoth);
  if (d <= 2048) return TW_NEU(8, 1, 4, 3, kBoth);
  if (d <= 4096) return TW_NEU(8, 2, 3, 2, kBoth);
  return TW_NEU(8, 4, 2, 1, kBoth);
#undef TW_NEU
#undef TW_NEU_W
}

}  // namespace tw
