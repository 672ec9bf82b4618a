// ell_gather.cuh -- the two gathers that ELL rows wider than 1024 are split
// into, shared by the forward and the backward row phase.
//
// Page 2 "Sakana AI and NVIDIA introduce TwELL with CUDA kernels ...",
// section "¿Qué hace distinto a TwELL frente a ELL clásico?", fuses the up
// and down projections into one gather.  For wide rows that kernel needs a
// team of warps per row whose partial dot products meet at a barrier for
// every batch of entries, and it gathers two or three weight rows per entry,
// so on large shapes its table outgrows L2 and it runs in several neuron
// passes.  Split in two:
//
//   ell_dot_kernel   per ELL entry e = (m, j): the dot product of a row
//                    vector v_m (x_m or dY_m) with a gathered weight row
//                    R[j] (Wu^T[j] or Wd[j]).  The team forms each dot
//                    exactly as the fused kernels do (same slabs, same warp
//                    and cross-warp summation order) but meets at its named
//                    barrier once per 32 entries: lane i keeps the warp's
//                    partial of entry i and the team sums 32 partials at once.
//                    The epilogue runs per entry on lane i:
//                      kDotH     h = g u                  (forward, u = x.Wu)
//                      kDotDh    dh                       (backward, dY.Wd)
//   ell_axpy_kernel  out_m = sum_e c_e R[j_e]: independent warps, each
//                    owning VPL slabs of one row, accumulate the per-entry
//                    coefficients in entry order -- y = sum h Wd in the
//                    forward.
//   ell_grad_dx_kernel  the backward's u, du, da, h per entry and dX in one
//                    gather over Wu^T and Wg^T (see below).
//
// The forward's per-entry arithmetic and y's accumulation order are those of
// the fused kernels, so y is bit-identical to them; the backward's gradient
// + dX gather sums the same terms in another grouping.  Each kernel gathers one or two weight
// matrices (a smaller table than the fused kernel's, so fewer L2-sized
// passes), and none waits at a barrier per batch.  Entries come from an entry source: the ELL rows of the training
// path (EllSrc) or the TwELL tiles of the inference path (TwellSrc); the
// per-entry buffers hold a row's entries contiguously, in order.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace tw {
namespace {

constexpr int kDotH = 0, kDotDh = 1;
constexpr int kEllPassFirst = 1, kEllPassLast = 2;

// Element offset of slab v of warp wt in a team of TEAM warps: slabs of 256
// elements (32 lanes x 8) dealt round-robin over the team.
template <int TEAM>
__device__ __forceinline__ int team_slab(int lane, int wt, int v) {
  return 8 * (lane + 32 * (wt + TEAM * v));
}

// [a, b): the entries of row m whose columns lie in [j_lo, j_hi).  A row's
// columns ascend, so the chunk is one contiguous slice.
__device__ __forceinline__ void ell_slice(const uint16_t* __restrict__ ell_col, long long row_off,
                                          int n, int j_lo, int j_hi, bool whole, int lane, int& a,
                                          int& b) {
  a = 0;
  b = n;
  if (whole) return;
  a = b = 0;
  for (int s0 = 0; s0 < n; s0 += 32) {
    const int jc = s0 + lane < n ? (int)ell_col[row_off + s0 + lane] : 0x7fffffff;
    a += __popc(__ballot_sync(0xffffffffu, jc < j_lo));
    b += __popc(__ballot_sync(0xffffffffu, jc < j_hi));
  }
}

// Entry sources.  for_groups(m, lane, f) visits row m's live entries in
// ascending column order, 32 at a time: f(count, j, slot, e) with lane
// i < count holding entry i's column j, its slot (the index of its value in
// the source's bf16 value array) and e, its index in the per-entry buffers
// (row m's entries at consecutive e); lanes >= count hold j = 0.
struct EllSrc {
  const uint16_t* val;  // [M][W] bf16 gate values
  const uint16_t* col;  // [M][W] columns, ascending in a row
  const int* nnz;       // [M]
  int W;
  int j_lo, j_hi, whole;  // neuron chunk [j_lo, j_hi); whole: every entry
  int f;                  // d_ff (columns are below it)
  template <class F>
  __device__ __forceinline__ void for_groups(int m, int lane, F&& fn) const {
    const long long row_off = (long long)m * W;
    int n = nnz[m];
    TW_CHECK_INDEX(n, n >= 0 && n <= W);
    int a, b;
    ell_slice(col, row_off, n, j_lo, j_hi, whole, lane, a, b);
    for (int e0 = a; e0 < b; e0 += 32) {
      const int count = min(32, b - e0);
      const long long s = row_off + e0 + lane;
      int j = lane < count ? (int)col[s] : 0;
      TW_CHECK_INDEX(j, j < f);
      fn(count, j, s, s);
    }
  }
};

struct TwellSrc {
  const uint16_t* val;  // [M][T][C] bf16 gate values
  const uint8_t* idx;   // [M][T][C] column inside the tile
  const uint8_t* cnt;   // [M][T] live count (only the first C are stored)
  int T, tile_n, cap;
  int t_lo, t_hi;       // tile chunk: neurons [t_lo tile_n, t_hi tile_n)
  int* status;          // non-null: a tile with cnt > C sets TWELL_ERR_CAPACITY
  template <class F>
  __device__ __forceinline__ void for_groups(int m, int lane, F&& f) const {
    // a row's entries at [m T C, m T C + row_nnz): its tiles' stored entries
    // in order, whatever tile chunk a pass covers (entries of earlier tiles
    // counted first)
    long long e_row = (long long)m * T * cap;
    for (int t0 = 0; t0 < t_lo; t0 += 32) {
      const int t = t0 + lane;
      const int c = t < t_lo ? min((int)cnt[(long long)m * T + t], cap) : 0;
      e_row += __reduce_add_sync(0xffffffffu, c);
    }
    for (int t0 = t_lo; t0 < t_hi; t0 += 32) {
      const int t = t0 + lane;
      const int craw = t < t_hi ? cnt[(long long)m * T + t] : 0;
      if (status && craw > cap) set_status(status, TWELL_ERR_CAPACITY);
      const int ct = min(craw, cap);
      const int incl = warp_incl_scan(ct);
      const int excl = incl - ct;
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      for (int e0 = 0; e0 < total; e0 += 32) {
        const int e = e0 + lane;
        int lo = 0;  // owner lane: number of lanes whose inclusive count is <= e
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
          const int v = __shfl_sync(0xffffffffu, incl, lo + step - 1);
          if (v <= e) lo += step;
        }
        const int ex = __shfl_sync(0xffffffffu, excl, lo);
        int jl = 0;
        long long sl = 0;
        if (e < total) {
          const int tt = t0 + lo;
          sl = ((long long)m * T + tt) * cap + (e - ex);
          int il = idx[sl];
          TW_CHECK_INDEX(il, il < tile_n);
          jl = tt * tile_n + il;
        }
        f(min(32, total - e0), jl, sl, e_row + e);
      }
      e_row += total;
    }
  }
};

struct EllDotArgs {
  const uint16_t* vec;   // [M][d] row vectors (x or dY)
  const uint16_t* rows;  // [f][d] gathered weight rows (Wu^T or Wd)
  int M, d;
  float* out;            // kDotH: h, kDotDh: dh  (per entry, the source's buffer index)
};

template <int TEAM, int VPL, int B, int MINB, int MODE, class Src>
__global__ void __launch_bounds__(256, MINB) ell_dot_kernel(const EllDotArgs p, const Src src) {
  static_assert(B % 2 == 0 && 32 % B == 0, "entries are summed over the warp in pairs");
  constexpr int ROWS = 8 / TEAM;
  __shared__ float red[2][ROWS][TEAM][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / TEAM, wt = warp % TEAM;
  const int m = blockIdx.x * ROWS + team;
  if (m >= p.M) return;
  const int d = p.d;

  const uint64_t pol = l2_evict_first_policy();  // the row vectors stream through
  uint4 vv[VPL];
  int eoff[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = team_slab<TEAM>(lane, wt, v);
    eoff[v] = e < d ? e : 0;
    vv[v] = e < d ? ldg_v4_hint(p.vec + (long long)m * d + e, pol) : make_uint4(0, 0, 0, 0);
  }
  int buf = 0;
  src.for_groups(m, lane, [&](int count, int jl, long long s, long long he) {
    float mine = 0.f;  // the warp's partial dot product of entry lane
    for (int i = 0; i < count; i += B) {
      int j[B];
#pragma unroll
      for (int b = 0; b < B; ++b) j[b] = __shfl_sync(0xffffffffu, jl, (i + b) & 31);
      uint4 r[B][VPL];
#pragma unroll
      for (int b = 0; b < B; ++b)
#pragma unroll
        for (int v = 0; v < VPL; ++v) r[b][v] = ldg_v4(p.rows + (long long)j[b] * d + eoff[v]);
      float q[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) dot8_bf16(vv[v], r[b][v], a0, a1);
        q[b] = a0 + a1;
      }
#pragma unroll
      for (int b = 0; b < B; b += 2) warp_sum2(q[b], q[b + 1]);
#pragma unroll
      for (int b = 0; b < B; ++b)
        if (lane == i + b) mine = q[b];
    }
    float dot = mine;
    if constexpr (TEAM > 1) {
      red[buf][team][wt][lane] = mine;
      named_barrier(1 + team, 32 * TEAM);
      dot = 0.f;
#pragma unroll
      for (int w = 0; w < TEAM; ++w) dot += red[buf][team][w][lane];
      buf ^= 1;
    }
    if (wt != 0 || lane >= count) return;
    if constexpr (MODE == kDotDh) {
      p.out[he] = dot;
    } else {  // kDotH
      p.out[he] = bf16_bits_to_float(src.val[s]) * dot;
    }
  });
}

struct EllAxpyArgs {
  const uint16_t* rows0;  // [f][d] weight rows scaled by the per-entry coefficient
  int M, d;
  const float* coef;      // per entry (the source's buffer index)
  int pass;               // kEllPassFirst: start from 0, kEllPassLast: store out
  float* part;            // [M][d] fp32 carry between neuron passes
  uint16_t* out;          // [M][d] bf16 result
};

template <int VPL, int B, int MINB, class Src>
__global__ void __launch_bounds__(256, MINB) ell_axpy_kernel(const EllAxpyArgs p, const Src src) {
  static_assert(32 % B == 0, "a batch never reaches past lane 31");
  const int lane = threadIdx.x & 31;
  const int d = p.d;
  const int wpr = (d + 256 * VPL - 1) / (256 * VPL);  // warps per row
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int m = (int)(gw / wpr), sg = (int)(gw % wpr);
  if (m >= p.M) return;

  const bool first = p.pass & kEllPassFirst, last = p.pass & kEllPassLast;
  const uint64_t pol = l2_evict_first_policy();  // the result and its carry stream through
  uint64_t acc[VPL][4];
  int eoff[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = 8 * lane + 256 * (sg * VPL + v);
    eoff[v] = e < d ? e : 0;
    if (first || e >= d) {
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[v][k] = 0;
    } else {
      const float* pp = p.part + (long long)m * d + e;
      const uint4 q0 = ldg_v4_hint(pp, pol), q1 = ldg_v4_hint(pp + 4, pol);
      acc[v][0] = f2_make(q0.x, q0.y);
      acc[v][1] = f2_make(q0.z, q0.w);
      acc[v][2] = f2_make(q1.x, q1.y);
      acc[v][3] = f2_make(q1.z, q1.w);
    }
  }
  src.for_groups(m, lane, [&](int count, int jl, long long, long long he) {
    // slots past the group: neuron 0 with a zero coefficient
    const float c0 = lane < count ? p.coef[he] : 0.f;
    for (int i = 0; i < count; i += B) {
      int j[B];
      float k0[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        j[b] = __shfl_sync(0xffffffffu, jl, (i + b) & 31);
        k0[b] = __shfl_sync(0xffffffffu, c0, (i + b) & 31);
      }
      uint4 r0[B][VPL];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const long long row = (long long)j[b] * d;
#pragma unroll
        for (int v = 0; v < VPL; ++v) r0[b][v] = ldg_v4(p.rows0 + row + eoff[v]);
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const uint64_t s0 = f2_splat(k0[b]);
#pragma unroll
        for (int v = 0; v < VPL; ++v) axpy8_f2(s0, r0[b][v], acc[v]);
      }
    }
  });
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = 8 * lane + 256 * (sg * VPL + v);
    if (e >= d) continue;
    if (last) {
      st_v4_hint(p.out + (long long)m * d + e, f2x4_to_bf8(acc[v]), pol);
    } else {
      float* pp = p.part + (long long)m * d + e;
      st_v4_hint(pp, make_uint4((uint32_t)acc[v][0], (uint32_t)(acc[v][0] >> 32),
                                (uint32_t)acc[v][1], (uint32_t)(acc[v][1] >> 32)), pol);
      st_v4_hint(pp + 4, make_uint4((uint32_t)acc[v][2], (uint32_t)(acc[v][2] >> 32),
                                    (uint32_t)acc[v][3], (uint32_t)(acc[v][3] >> 32)), pol);
    }
  }
}

// The gradient gather and the dX gather of the backward rows in one pass
// over Wu^T and Wg^T.  Per ELL entry e = (m, j), with dh from the dh gather:
//   u = x_m . Wu[:, j],  du = dh g,  da = dh u + lambda,  h = g u
//   dX_m += du Wu[:, j]^T + da Wg[:, j]^T
// du is known before u, so the Wu^T row the dot product reads also feeds
// dX straight away; da needs the whole dot product, which the team forms
// once per group of 32 entries, after which the group's Wg^T rows are read.
// Each entry reads Wu^T[j] and Wg^T[j] once (4 d bytes instead of the 6 d
// of a gradient gather plus a dX gather).  Per dX element the sum runs
// group by group: the group's du Wu^T terms in entry order, then its
// da Wg^T terms.  The team and slab layout are ell_dot_kernel's (the team
// size is the caller's choice, so u is summed over that many warps).
struct EllGradDxArgs {
  const uint16_t* x;     // [M][d] bf16
  const uint16_t* wuT;   // [f][d] bf16
  const uint16_t* wgT;   // [f][d] bf16
  int M, d;
  const float* dh;       // dh per entry (the source's buffer index)
  const int* slot_pos;   // neuron-major position of each slot
  float lambda;          // L1 coefficient
  float4* csc_vals;      // (du, da, h, 0) at the neuron-major position
  int pass;              // kEllPassFirst: start from 0, kEllPassLast: store dx
  float* part;           // [M][d] fp32 dX carry between neuron passes
  uint16_t* dx;          // [M][d] bf16 result
};

template <int TEAM, int VPL, int B, int MINB>
__global__ void __launch_bounds__(256, MINB)
    ell_grad_dx_kernel(const EllGradDxArgs p, const EllSrc src) {
  static_assert(B % 2 == 0 && 32 % B == 0, "entries are summed over the warp in pairs");
  constexpr int ROWS = 8 / TEAM;
  __shared__ float red[2][ROWS][TEAM][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / TEAM, wt = warp % TEAM;
  const int m = blockIdx.x * ROWS + team;
  if (m >= p.M) return;
  const int d = p.d;
  const bool first = p.pass & kEllPassFirst, last = p.pass & kEllPassLast;

  const uint64_t pol = l2_evict_first_policy();  // x and the dX carry stream through
  uint4 xv[VPL];
  int eoff[VPL];
  uint64_t acc[VPL][4];
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = team_slab<TEAM>(lane, wt, v);
    eoff[v] = e < d ? e : 0;
    xv[v] = e < d ? ldg_v4_hint(p.x + (long long)m * d + e, pol) : make_uint4(0, 0, 0, 0);
    if (first || e >= d) {
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[v][k] = 0;
    } else {  // dX_m of the earlier neuron chunks
      const float* pp = p.part + (long long)m * d + e;
      const uint4 q0 = ldg_v4_hint(pp, pol), q1 = ldg_v4_hint(pp + 4, pol);
      acc[v][0] = f2_make(q0.x, q0.y);
      acc[v][1] = f2_make(q0.z, q0.w);
      acc[v][2] = f2_make(q1.x, q1.y);
      acc[v][3] = f2_make(q1.z, q1.w);
    }
  }
  int buf = 0;
  src.for_groups(m, lane, [&](int count, int jl, long long s, long long he) {
    // entry `lane` of the group; slots past it: neuron 0 with zero coefficients
    const bool live = lane < count;
    const float dhl = live ? p.dh[he] : 0.f;
    const float gl = live ? bf16_bits_to_float(src.val[s]) : 0.f;
    const float dul = dhl * gl;
    float mine = 0.f;  // the warp's partial dot product of entry lane
    // Wu^T rows: dot products with x_m, and du Wu[:, j]^T into dX_m
    for (int i = 0; i < count; i += B) {
      int j[B];
      float du[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        j[b] = __shfl_sync(0xffffffffu, jl, (i + b) & 31);
        du[b] = __shfl_sync(0xffffffffu, dul, (i + b) & 31);
      }
      uint4 r[B][VPL];
#pragma unroll
      for (int b = 0; b < B; ++b)
#pragma unroll
        for (int v = 0; v < VPL; ++v) r[b][v] = ldg_v4(p.wuT + (long long)j[b] * d + eoff[v]);
      float q[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) dot8_bf16(xv[v], r[b][v], a0, a1);
        q[b] = a0 + a1;
        const uint64_t s2 = f2_splat(du[b]);
#pragma unroll
        for (int v = 0; v < VPL; ++v) axpy8_f2(s2, r[b][v], acc[v]);
      }
#pragma unroll
      for (int b = 0; b < B; b += 2) warp_sum2(q[b], q[b + 1]);
#pragma unroll
      for (int b = 0; b < B; ++b)
        if (lane == i + b) mine = q[b];
    }
    float u = mine;
    if constexpr (TEAM > 1) {
      red[buf][team][wt][lane] = mine;
      named_barrier(1 + team, 32 * TEAM);
      u = 0.f;
#pragma unroll
      for (int w = 0; w < TEAM; ++w) u += red[buf][team][w][lane];
      buf ^= 1;
    }
    const float dal = live ? fmaf(dhl, u, p.lambda) : 0.f;  // ReLU'(a) = 1 on a live entry
    if (wt == 0 && live) {
      long long pos = p.slot_pos[s];
      TW_CHECK_INDEX(pos, pos >= 0 && pos < (long long)p.M * src.W);
      p.csc_vals[pos] = make_float4(dul, dal, gl * u, 0.f);
    }
    // Wg^T rows: da Wg[:, j]^T into dX_m
    for (int i = 0; i < count; i += B) {
      int j[B];
      float da[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        j[b] = __shfl_sync(0xffffffffu, jl, (i + b) & 31);
        da[b] = __shfl_sync(0xffffffffu, dal, (i + b) & 31);
      }
      uint4 r[B][VPL];
#pragma unroll
      for (int b = 0; b < B; ++b)
#pragma unroll
        for (int v = 0; v < VPL; ++v) r[b][v] = ldg_v4(p.wgT + (long long)j[b] * d + eoff[v]);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const uint64_t s2 = f2_splat(da[b]);
#pragma unroll
        for (int v = 0; v < VPL; ++v) axpy8_f2(s2, r[b][v], acc[v]);
      }
    }
  });
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = team_slab<TEAM>(lane, wt, v);
    if (e >= d) continue;
    if (last) {
      st_v4_hint(p.dx + (long long)m * d + e, f2x4_to_bf8(acc[v]), pol);
    } else {
      float* pp = p.part + (long long)m * d + e;
      st_v4_hint(pp, make_uint4((uint32_t)acc[v][0], (uint32_t)(acc[v][0] >> 32),
                                (uint32_t)acc[v][1], (uint32_t)(acc[v][1] >> 32)), pol);
      st_v4_hint(pp + 4, make_uint4((uint32_t)acc[v][2], (uint32_t)(acc[v][2] >> 32),
                                    (uint32_t)acc[v][3], (uint32_t)(acc[v][3] >> 32)), pol);
    }
  }
}

}  // namespace
}  // namespace tw
