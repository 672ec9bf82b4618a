// gemm_tc.cuh -- persistent tcgen05 GEMM engine for sm_103a with fused epilogues.
//
// One CTA per SM.  Warp roles (384 threads):
//   warp 0      TMA producer: fills a STAGES-deep ring of A / B tiles in shared
//               memory (128-byte swizzle), one elected lane
//   warp 1      MMA issuer: tcgen05.mma 128 x 256 x 16 (bf16 in, fp32 in TMEM),
//               one elected lane; commits free smem stages and finished tiles
//   warp 2      TMEM owner: allocates / frees 512 columns (two accumulators)
//   warps 4..11 epilogue: warp w reads TMEM lane quarter w % 4 (the quarter a
//               warp may touch) and column half (w - 4) / 4, so each thread
//               owns one accumulator row and half of its 256 columns
// Two 256-column accumulators let the epilogue of tile i overlap the
// mainloop of tile i+1.  Tiles are visited in a grouped raster so CTAs that
// run together share A rows and B columns in L2.  The CTA-pair form of the
// same kernel (PAIR, see "kernel" below) runs 2-CTA clusters on 256 x 256
// tiles with tcgen05.mma.cta_group::2.
//
// Operands: A (M x K) and B (N x K), each K-major ([rows][K], K contiguous) or
// MN-major ([K][rows]).  Epilogues:
//   EPI_STORE     C = acc (bf16 or fp32, optional += into fp32, optional row map)
//   EPI_PACK      ReLU + TwELL pack of the gate activation (no dense write)
//   EPI_GATED     B = [Wg tile ; Wu tile]: h = bf16(ReLU(a)) * u, optional g, u
//   EPI_BWD_GATE  acc = dh: du = dh * g, da = (dh * u + lambda) * 1[g > 0]
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace tw {

// ---- CTA-pair forms (cta_group::2).  A kernel uses either these or the
// single-CTA forms of common.cuh for alloc / dealloc / relinquish / mma /
// commit, never both.  The pair is the two CTAs of a 2-CTA cluster: rank 0 issues the
// MMAs, which read A and B from both CTAs' shared memory (same offsets) and
// write each CTA's own accumulator rows into that CTA's TMEM.

// Collective over the pair: one warp of each CTA executes it.
TW_DEV void tmem_alloc_pair(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(holder)),
               "r"(ncols)
               : "memory");
}
TW_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
TW_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Arrive once on the barrier at this shared-memory offset in every CTA of
// `cta_mask` when the pair MMAs issued so far are done.
TW_DEV void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// D[tmem] (+)= A * B^T over the pair: M = 256 (128 rows from each CTA), N
// columns of B (the first N/2 rows of B from rank 0, the rest from rank 1).
TW_DEV void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
TW_DEV uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

// TMA load into this CTA's shared memory whose completion is counted on a
// barrier of either CTA of the pair (a shared::cluster address).
TW_DEV void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                             int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

// Arrive on a barrier given by its shared::cluster address.
TW_DEV void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

TW_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
TW_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

enum EpiKind { EPI_STORE = 0, EPI_PACK = 1, EPI_GATED = 2, EPI_BWD_GATE = 3, EPI_BWD_GATE_RT = 4 };

constexpr int kBM = 128;
constexpr int kBN = 256;  // MMA N (for EPI_GATED: 128 gate + 128 up columns)
constexpr int kBK = 64;   // one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kGemmThreads = 384;
constexpr int kEpiThreads = 256;  // warps 4..11
constexpr int kGroupM = 16;
constexpr uint32_t kTmemCols = 512;
constexpr int kStageBytes = 4096;  // per epilogue warp: 32 rows x 128 B output staging
constexpr int kGemmSmem =
    kStages * (kABytes + kBBytes) + 8 * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;

// Gate activations.  ReLU is the sparse path's gate; SiLU serves only the
// dense comparator (the unmodified gated FFN) and only on the TMA-store path,
// where the saved "g" holds bf16(a) so the backward can recompute SiLU.
constexpr int kActRelu = 0, kActSilu = 1;

struct GemmParams {
  int M, N, K;          // M: rows (buffer capacity), N: output columns, K: reduction
  const int* m_dev;     // optional device row count: rows used = min(M, *m_dev)
  const int* k_dev;     // optional device K: K used = min(K, *k_dev)
  int n_tiles;          // tiles along N
  int k_split;          // K segment length in k-blocks: segment s reads B (s even) or B2 (s odd)
  int a_seg_off;        // MN-major A only: if > 0, the K range is run twice, the second time
                        // with A's M coordinate shifted by a_seg_off (B rows repeat): C += A0^T B + A1^T B
  int pad_rows;         // store every row of a visited tile that is < M (zero padding)
  int tma_out;          // outputs go through shared memory and TMA stores (tensor maps O0..O2)
  int act;              // gate activation of EPI_GATED / EPI_BWD_GATE: kActRelu or kActSilu
  int cluster_k;        // EPI_PACK only: > 1 = split K over the blocks of a cluster (see kernel)
  int split_k_max;      // > 1: split K (plan from splitk_plan); split s stores its fp32 partial
                        // at rows [s * rows_eff, (s + 1) * rows_eff) of the output map
  int split_rows;       // rows of that output map (0: M)
  int* status;
  // EPI_STORE
  void* c;
  long long ldc;
  int c_f32;
  int accumulate;
  const int* row_map;   // destination row of output row r (scatter), or null
  // EPI_PACK
  uint16_t* val;
  uint8_t* idx;
  uint8_t* cnt;
  int* row_nnz;
  int T, cap, tile_n;
  // EPI_GATED (outputs [M][N], leading dimension ldh)
  uint16_t* h;
  uint16_t* g_out;
  uint16_t* u_out;
  long long ldh;        // leading dimension of h
  long long h_lo_off;   // if > 0: h is stored as bf16 hi at [r][j] plus bf16 lo at [r][j + h_lo_off]
  long long ldgu;       // leading dimension of g / u (written by EPI_GATED, read by EPI_BWD_GATE)
  float* u_f32;         // EPI_GATED: u kept in fp32 instead of u_out (bf16)
  const float* u_f32_in;  // EPI_BWD_GATE: read u from here (fp32) instead of u_in
  // EPI_BWD_GATE: g, u in [M][ldh]; du -> dd[r][j], da -> dd[r][dd_seg + j]; with
  // dd_split the bf16 residuals follow: du lo at 2*dd_seg, da lo at 3*dd_seg
  const uint16_t* g_in;
  const uint16_t* u_in;
  uint16_t* dd;
  long long ld_dd;
  long long dd_seg;
  int dd_split;
  float lambda;
};

__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int& mb, int& nb) {
  const int per_group = kGroupM * n_tiles;
  const int g = tile / per_group;
  const int first = g * kGroupM;
  const int gm = min(kGroupM, m_tiles - first);
  const int r = tile - g * per_group;
  mb = first + r % gm;
  nb = r / gm;
}

// unit -> (tile index, K split): split-major for split-K partials written to
// global memory; with cluster split-K the splits of one tile are the blocks
// of one cluster, so they are adjacent in the grid
__device__ __forceinline__ void unit_coords(int unit, int tiles, int cluster_k, int& tile,
                                            int& ks) {
  if (cluster_k > 1) {
    tile = unit / cluster_k;
    ks = unit - tile * cluster_k;
  } else {
    ks = unit / tiles;
    tile = unit - ks * tiles;
  }
}

// ------------------------------------------------------------------ epilogues
// Output staging: each epilogue warp owns a 4 KB shared-memory buffer; lane r
// writes row r of a 32-row box (128-byte swizzle for 128-byte rows, 64-byte
// swizzle for 64-byte rows, matching the tensor maps, so the 16-byte writes
// of a warp hit distinct banks) and lane 0 sends the box with a TMA store.
struct Stager {
  uint8_t* buf;
  int lane;
  int n;          // stores issued so far
  bool whole;     // the last buffer handed out was the whole 4 KB
  // 128-byte rows: the whole buffer; waits until no store still reads it
  __device__ __forceinline__ uint8_t* full() {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    whole = true;
    return buf;
  }
  // 64-byte rows: the two 2 KB halves in turn, one store may stay in flight
  // (none if that store read the whole buffer)
  __device__ __forceinline__ uint8_t* half() {
    if (lane == 0) {
      if (whole)
        bulk_wait_read<0>();
      else
        bulk_wait_read<1>();
    }
    __syncwarp();
    whole = false;
    return buf + ((n & 1) << 11);
  }
  __device__ __forceinline__ void put128(uint8_t* b, int c, const uint4& v) const {
    *reinterpret_cast<uint4*>(b + lane * 128 + ((c ^ (lane & 7)) << 4)) = v;
  }
  __device__ __forceinline__ void put64(uint8_t* b, int c, const uint4& v) const {
    *reinterpret_cast<uint4*>(b + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = v;
  }
  __device__ __forceinline__ void send(const CUtensorMap* map, const uint8_t* b, int col, int row,
                                       bool reduce_add = false) {
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
      if (reduce_add)
        tma_reduce_add_2d(map, b, col, row);
      else
        tma_store_2d(map, b, col, row);
      bulk_commit();
    }
    ++n;
  }
  __device__ __forceinline__ void drain() {
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
};

struct OutMaps {
  const CUtensorMap* o0;
  const CUtensorMap* o1;
  const CUtensorMap* o2;
};

template <int EPI>
struct Epilogue;

template <>
struct Epilogue<EPI_STORE> {
  static __device__ __forceinline__ void run(const GemmParams& p, uint32_t tacc, int row,
                                             bool row_ok, int n0, int N, int half, Stager& st,
                                             const OutMaps& om, int row0) {
    if (p.tma_out) {
      // C through TMA: bf16 in 64-column boxes, fp32 in 32-column boxes (+= via reduce-add)
#pragma unroll 1
      for (int c0 = half * (kBN / 2); c0 < (half + 1) * (kBN / 2); c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tacc + c0, r);
        tmem_wait_ld();
        // box wholly outside C (warp-uniform); split-K partials fill split_rows rows
        if (n0 + c0 >= N || row0 >= (p.split_rows > 0 ? p.split_rows : p.M)) continue;
        if (p.c_f32) {
          uint8_t* b = st.full();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            st.put128(b, v, make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]));
          st.send(om.o0, b, n0 + c0, row0, p.accumulate != 0);
        } else {
          uint8_t* b = st.half();
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st.put64(b, v,
                     make_uint4(pack_bf16x2(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]))));
          st.send(om.o0, b, n0 + c0, row0);
        }
      }
      return;
    }
    const int dst_row = (row_ok && p.row_map) ? p.row_map[row] : row;
#pragma unroll 1
    for (int c0 = half * (kBN / 2); c0 < (half + 1) * (kBN / 2); c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tacc + c0, r);
      tmem_wait_ld();
      if (!row_ok) continue;
      const int col = n0 + c0;
      if (p.c_f32) {
        float* dst = reinterpret_cast<float*>(p.c) + (long long)dst_row * p.ldc + col;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          if (col + 4 * v + 4 <= N) {
            float4 o = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                   __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            float4* q = reinterpret_cast<float4*>(dst + 4 * v);
            if (p.accumulate) {
              float4 old = *q;
              o.x += old.x;
              o.y += old.y;
              o.z += old.z;
              o.w += old.w;
            }
            *q = o;
          }
        }
      } else {
        uint16_t* dst = reinterpret_cast<uint16_t*>(p.c) + (long long)dst_row * p.ldc + col;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (col + 8 * v + 8 <= N) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
            o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
            o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
            o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
            *reinterpret_cast<uint4*>(dst + 8 * v) = o;
          }
        }
      }
    }
  }
};

// Select r[i] for a runtime i in [0, 32) without indexing registers
// dynamically (which would spill r to local memory): a 5-level select tree.
__device__ __forceinline__ uint32_t select32(const uint32_t (&r)[32], int i) {
  uint32_t a[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) a[k] = (i & 16) ? r[k + 16] : r[k];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = (i & 8) ? a[k + 8] : a[k];
#pragma unroll
  for (int k = 0; k < 4; ++k) a[k] = (i & 4) ? a[k + 4] : a[k];
#pragma unroll
  for (int k = 0; k < 2; ++k) a[k] = (i & 2) ? a[k + 2] : a[k];
  return (i & 1) ? a[1] : a[0];
}

// ReLU + TwELL pack.  The accumulator holds 256 gate columns = 256 / T_n
// TwELL tiles; this thread owns one row and one column half, scans its
// columns in ascending order and writes the live ones to its (row, tile)
// slots.  bf16(ReLU(a)) > 0 exactly when a > 2^-134 (the largest fp32 that
// rounds to bf16 zero is 2^-134, a tie to even; NaN compares false), so one
// compare per column builds the live mask and values are only extracted for
// the (rare) live columns.
template <>
struct Epilogue<EPI_PACK> {
  // With cluster split-K the leader block adds `part`, the sum of the other
  // blocks' partial accumulators staged [column][row] in its shared memory.
  static __device__ __forceinline__ void add_partial(const float* part, int r_local, int col,
                                                     uint32_t (&r)[32]) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      r[i] = __float_as_uint(__uint_as_float(r[i]) + part[(col + i) * kBM + r_local]);
  }
  static __device__ __forceinline__ void run(const GemmParams& p, uint32_t tacc, int row,
                                             bool row_ok, int n0, int /*N*/, int half, Stager&,
                                             const OutMaps&, int, float* part = nullptr,
                                             int r_local = 0) {
    const float kLiveMin = __uint_as_float(0x00008000u);  // 2^-134
    const int tiles_here = (kBN / 2) / p.tile_n;
    const int chunks_per_tile = p.tile_n / 32;
    const int col0 = half * (kBN / 2);
    int nnz = 0;
#pragma unroll 1
    for (int tt = 0; tt < tiles_here; ++tt) {
      const int t = (n0 + col0) / p.tile_n + tt;
      const bool tile_ok = row_ok && t < p.T;
      const long long slot0 = ((long long)row * p.T + t) * p.cap;
      int c = 0;
#pragma unroll 1
      for (int ch = 0; ch < chunks_per_tile; ++ch) {
        uint32_t r[32];
        tmem_ld32(tacc + col0 + tt * p.tile_n + ch * 32, r);
        tmem_wait_ld();
        if (!tile_ok) continue;
        if (part) add_partial(part, r_local, col0 + tt * p.tile_n + ch * 32, r);
        uint32_t mask = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) mask |= (__uint_as_float(r[i]) > kLiveMin ? 1u : 0u) << i;
        while (mask) {
          const int i = __ffs(mask) - 1;
          mask &= mask - 1;
          if (c < p.cap) {
            p.val[slot0 + c] = (uint16_t)relu_bf16_bits(__uint_as_float(select32(r, i)));
            p.idx[slot0 + c] = (uint8_t)(ch * 32 + i);
          }
          ++c;
        }
      }
      if (tile_ok) {
        p.cnt[(long long)row * p.T + t] = (uint8_t)c;
        nnz += c;
      }
    }
    if (row_ok && nnz) atomicAdd(p.row_nnz + row, nnz);
  }
};

// Dense gated activation: accumulator columns [0,128) = a (gate), [128,256) =
// u (up) of the same 128 neurons.  h = bf16(ReLU(a)) * u, stored bf16.
template <>
struct Epilogue<EPI_GATED> {
  static __device__ __forceinline__ void run(const GemmParams& p, uint32_t tacc, int row,
                                             bool row_ok, int n0, int N, int half, Stager& st,
                                             const OutMaps& om, int row0) {
    // here n0 is the neuron offset (tile index * 128); this thread takes 64 neurons
#pragma unroll 1
    for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 32) {
      uint32_t ra[32], ru[32];
      tmem_ld32(tacc + c0, ra);
      tmem_ld32(tacc + 128 + c0, ru);
      tmem_wait_ld();
      {  // h (its lo half, g, u) through shared memory and TMA stores, 32 neurons a box
        if (n0 + c0 >= N || row0 >= p.M) continue;
        uint32_t hw[16], gw[16], uw[16];
        if (p.act == kActSilu) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float a0 = __uint_as_float(ra[2 * q]), a1 = __uint_as_float(ra[2 * q + 1]);
            const float u0 = __uint_as_float(ru[2 * q]), u1 = __uint_as_float(ru[2 * q + 1]);
            const float s0 = a0 / (1.0f + __expf(-a0)), s1 = a1 / (1.0f + __expf(-a1));
            hw[q] = pack_bf16x2(s0 * u0, s1 * u1);
            gw[q] = pack_bf16x2(a0, a1);  // pre-activation, for the backward
            uw[q] = pack_bf16x2(u0, u1);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const uint32_t g0 = relu_bf16_bits(__uint_as_float(ra[2 * q]));
            const uint32_t g1 = relu_bf16_bits(__uint_as_float(ra[2 * q + 1]));
            const float u0 = __uint_as_float(ru[2 * q]), u1 = __uint_as_float(ru[2 * q + 1]);
            hw[q] = pack_bf16x2(bf16_bits_to_float(g0) * u0, bf16_bits_to_float(g1) * u1);
            gw[q] = g0 | (g1 << 16);
            uw[q] = pack_bf16x2(u0, u1);
          }
        }
        uint8_t* b = st.half();
#pragma unroll
        for (int v = 0; v < 4; ++v)
          st.put64(b, v, make_uint4(hw[4 * v], hw[4 * v + 1], hw[4 * v + 2], hw[4 * v + 3]));
        st.send(om.o0, b, n0 + c0, row0);
        if (p.h_lo_off) {  // h - bf16(h) in the same map, h_lo_off columns on
          uint32_t lw[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float2 hr = unpack_bf16x2(hw[q]);
            float h0, h1;
            if (p.act == kActSilu) {
              const float a0 = __uint_as_float(ra[2 * q]), a1 = __uint_as_float(ra[2 * q + 1]);
              h0 = a0 / (1.0f + __expf(-a0)) * __uint_as_float(ru[2 * q]);
              h1 = a1 / (1.0f + __expf(-a1)) * __uint_as_float(ru[2 * q + 1]);
            } else {
              h0 = bf16_bits_to_float(relu_bf16_bits(__uint_as_float(ra[2 * q]))) *
                   __uint_as_float(ru[2 * q]);
              h1 = bf16_bits_to_float(relu_bf16_bits(__uint_as_float(ra[2 * q + 1]))) *
                   __uint_as_float(ru[2 * q + 1]);
            }
            lw[q] = pack_bf16x2(h0 - hr.x, h1 - hr.y);
          }
          b = st.half();
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st.put64(b, v, make_uint4(lw[4 * v], lw[4 * v + 1], lw[4 * v + 2], lw[4 * v + 3]));
          st.send(om.o0, b, n0 + c0 + (int)p.h_lo_off, row0);
        }
        if (p.g_out) {
          b = st.half();
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st.put64(b, v, make_uint4(gw[4 * v], gw[4 * v + 1], gw[4 * v + 2], gw[4 * v + 3]));
          st.send(om.o1, b, n0 + c0, row0);
        }
        if (p.u_f32) {  // u kept in fp32: 32 columns are a 128-byte row
          b = st.full();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            st.put128(b, v, make_uint4(ru[4 * v], ru[4 * v + 1], ru[4 * v + 2], ru[4 * v + 3]));
          st.send(om.o2, b, n0 + c0, row0);
        } else if (p.u_out) {
          b = st.half();
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st.put64(b, v, make_uint4(uw[4 * v], uw[4 * v + 1], uw[4 * v + 2], uw[4 * v + 3]));
          st.send(om.o2, b, n0 + c0, row0);
        }
      }
    }
  }
};

// acc = dh = dY Wd^T for 256 neurons.  du = dh * g, da = (dh * u + lambda) if
// g > 0 else 0 (SiLU: see below); both stored bf16 into dd = [du | da].
TW_DEV void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

template <>
struct Epilogue<EPI_BWD_GATE> {
  // Issued before the tile's accumulator is ready: pulls this thread's g and
  // u (its row, its 128 columns: two 128-byte lines each) into L2, so the
  // epilogue's loads do not wait on DRAM.
  static __device__ __forceinline__ void prefetch(const GemmParams& p, int row, int n0, int half,
                                                  int N) {
    const int c = n0 + half * (kBN / 2);
    if (row >= p.M || c >= N) return;
    const long long gu = (long long)row * p.ldgu + c;
    prefetch_l2(p.g_in + gu);
    prefetch_l2(p.g_in + gu + 64);
    prefetch_l2(p.u_in + gu);
    prefetch_l2(p.u_in + gu + 64);
  }
  static __device__ __forceinline__ void run(const GemmParams& p, uint32_t tacc, int row,
                                             bool row_ok, int n0, int N, int half, Stager& st,
                                             const OutMaps& om, int row0) {
    const long long seg = p.dd_seg;
#pragma unroll 1
    for (int c0 = half * (kBN / 2); c0 < (half + 1) * (kBN / 2); c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tacc + c0, r);
      tmem_wait_ld();
      {  // du, da through shared memory and TMA stores, 32 columns a box
        if (n0 + c0 >= N || row0 >= p.M) continue;
        uint32_t duw[16], daw[16];
        const bool in = row < p.M;
        const long long gu = (long long)row * p.ldgu + n0 + c0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 g8 = in ? *reinterpret_cast<const uint4*>(p.g_in + gu + 8 * v)
                              : make_uint4(0, 0, 0, 0);
          const uint4 u8 = in ? *reinterpret_cast<const uint4*>(p.u_in + gu + 8 * v)
                              : make_uint4(0, 0, 0, 0);
          const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w};
          const uint32_t uw[4] = {u8.x, u8.y, u8.z, u8.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 g = unpack_bf16x2(gw[q]);
            const float2 u = unpack_bf16x2(uw[q]);
            const float dh0 = __uint_as_float(r[8 * v + 2 * q]);
            const float dh1 = __uint_as_float(r[8 * v + 2 * q + 1]);
            if (p.act == kActSilu) {  // g holds a: du = dh silu(a), da = dh u silu'(a)
              const float sg0 = 1.0f / (1.0f + __expf(-g.x)), sg1 = 1.0f / (1.0f + __expf(-g.y));
              duw[4 * v + q] = pack_bf16x2(dh0 * (g.x * sg0), dh1 * (g.y * sg1));
              daw[4 * v + q] = pack_bf16x2(dh0 * u.x * (sg0 * (1.0f + g.x * (1.0f - sg0))),
                                           dh1 * u.y * (sg1 * (1.0f + g.y * (1.0f - sg1))));
            } else {
              duw[4 * v + q] = pack_bf16x2(dh0 * g.x, dh1 * g.y);
              daw[4 * v + q] = pack_bf16x2(g.x > 0.f ? fmaf(dh0, u.x, p.lambda) : 0.f,
                                           g.y > 0.f ? fmaf(dh1, u.y, p.lambda) : 0.f);
            }
          }
        }
        uint8_t* b = st.half();
#pragma unroll
        for (int v = 0; v < 4; ++v)
          st.put64(b, v, make_uint4(duw[4 * v], duw[4 * v + 1], duw[4 * v + 2], duw[4 * v + 3]));
        st.send(om.o0, b, n0 + c0, row0);
        b = st.half();
#pragma unroll
        for (int v = 0; v < 4; ++v)
          st.put64(b, v, make_uint4(daw[4 * v], daw[4 * v + 1], daw[4 * v + 2], daw[4 * v + 3]));
        st.send(om.o0, b, n0 + c0 + (int)seg, row0);
      }
    }
  }
};


// Routed rows' variant (its own instantiation, so the dense comparator's
// epilogue stays lean): g bf16, u fp32, and dd = [du | da | du lo | da lo].
template <>
struct Epilogue<EPI_BWD_GATE_RT> {
  // as for EPI_BWD_GATE; u is fp32 here (four lines)
  static __device__ __forceinline__ void prefetch(const GemmParams& p, int row, int n0, int half,
                                                  int N) {
    const int c = n0 + half * (kBN / 2);
    if (row >= p.M || c >= N) return;
    const long long gu = (long long)row * p.ldgu + c;
    prefetch_l2(p.g_in + gu);
    prefetch_l2(p.g_in + gu + 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) prefetch_l2(p.u_f32_in + gu + 32 * i);
  }
  // du, da from dh and the saved g, u (ReLU: da = dh u + lambda on live
  // entries; SiLU: g holds a, du = dh silu(a), da = dh u silu'(a))
  static __device__ __forceinline__ void grads(const GemmParams& p, float dh, float g, float u,
                                               float& du, float& da) {
    if (p.act == kActSilu) {
      const float sg = 1.0f / (1.0f + __expf(-g));
      du = dh * (g * sg);
      da = dh * u * (sg * (1.0f + g * (1.0f - sg)));
    } else {
      du = dh * g;
      da = g > 0.f ? fmaf(dh, u, p.lambda) : 0.f;
    }
  }
  static __device__ __forceinline__ void send16(Stager& st, const CUtensorMap* m,
                                                const uint32_t (&w)[16], int col, int row0) {
    uint8_t* b = st.half();
#pragma unroll
    for (int v = 0; v < 4; ++v) st.put64(b, v, make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]));
    st.send(m, b, col, row0);
  }
  static __device__ __forceinline__ void run(const GemmParams& p, uint32_t tacc, int row,
                                             bool /*row_ok*/, int n0, int N, int half, Stager& st,
                                             const OutMaps& om, int row0) {
    const int seg = (int)p.dd_seg;
    const bool in = row < p.M;
#pragma unroll 1
    for (int c0 = half * (kBN / 2); c0 < (half + 1) * (kBN / 2); c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tacc + c0, r);
      tmem_wait_ld();
      // du, da through shared memory and TMA stores, 32 columns a box
      if (n0 + c0 >= N || row0 >= p.M) continue;
      const long long gu = (long long)row * p.ldgu + n0 + c0;
      uint32_t duw[16], daw[16];
      {  // routed rows: u fp32, du and da also as bf16 residuals [du lo | da lo]
        uint32_t dul[16], dal[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 g8 = in ? *reinterpret_cast<const uint4*>(p.g_in + gu + 8 * v)
                              : make_uint4(0, 0, 0, 0);
          const float4 u0 = in ? *reinterpret_cast<const float4*>(p.u_f32_in + gu + 8 * v)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 u1 = in ? *reinterpret_cast<const float4*>(p.u_f32_in + gu + 8 * v + 4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w};
          const float uf[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 g = unpack_bf16x2(gw[q]);
            float du0, du1, da0, da1;
            grads(p, __uint_as_float(r[8 * v + 2 * q]), g.x, uf[2 * q], du0, da0);
            grads(p, __uint_as_float(r[8 * v + 2 * q + 1]), g.y, uf[2 * q + 1], du1, da1);
            duw[4 * v + q] = pack_bf16x2(du0, du1);
            daw[4 * v + q] = pack_bf16x2(da0, da1);
            const float2 duh = unpack_bf16x2(duw[4 * v + q]);
            const float2 dah = unpack_bf16x2(daw[4 * v + q]);
            dul[4 * v + q] = pack_bf16x2(du0 - duh.x, du1 - duh.y);
            dal[4 * v + q] = pack_bf16x2(da0 - dah.x, da1 - dah.y);
          }
        }
        send16(st, om.o0, duw, n0 + c0, row0);
        send16(st, om.o0, daw, n0 + c0 + seg, row0);
        send16(st, om.o0, dul, n0 + c0 + 2 * seg, row0);
        send16(st, om.o0, dal, n0 + c0 + 3 * seg, row0);
      }
    }
  }
};

// ------------------------------------------------------------------ kernel
// PAIR = true: the CTA-pair form.  The kernel runs as 2-CTA clusters; a pair
// owns 256 x 256 output tiles, rank r of the pair loads A rows [128 r, 128 r
// + 128) of the tile and B rows (output columns) [128 r, 128 r + 128) into
// its own ring, and rank 0's MMA warp issues 256 x 256 x 16 MMAs that read
// both rings and leave each rank's 128 accumulator rows in that rank's TMEM.
// Per SM this halves the B bytes staged and read per MMA, which is what
// bounds the single-CTA 128 x 256 tile.  A stage holds 32 KB per CTA (16 KB
// A + 16 KB B), so the same shared memory gives a 6-deep ring.  Not used
// with split-K or cluster split-K.
constexpr int kPairStages = 6;
static_assert(kPairStages * (kABytes + kBBytes / 2) <= kStages * (kABytes + kBBytes),
              "the pair ring fits the single-CTA ring's shared memory");

template <bool A_MN, bool B_MN, int EPI, bool PAIR = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmO0,
                const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2,
                const GemmParams p) {
  constexpr int STAGES = PAIR ? kPairStages : kStages;
  constexpr int B_BYTES = PAIR ? kBBytes / 2 : kBBytes;  // B bytes per stage in this CTA
  constexpr int TILE_M = PAIR ? 2 * kBM : kBM;           // output rows per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * kABytes;
  uint8_t* sOut = sB + STAGES * B_BYTES;  // 8 x 4 KB epilogue staging buffers
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + 8 * kStageBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // a pair (PAIR) or a CTA walks the units group, group + n_groups, ...
  const int rank = PAIR ? (int)cluster_rank() : 0;
  const int group = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_groups = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  int M_eff = p.M;
  if (p.m_dev) M_eff = min(M_eff, *p.m_dev);
  int K_eff = p.K;
  if (p.k_dev) K_eff = min(K_eff, *p.k_dev);
  const int m_tiles = (M_eff + TILE_M - 1) / TILE_M;
  const int kb_pass = (K_eff + kBK - 1) / kBK;
  const int num_kb = (A_MN && p.a_seg_off > 0) ? 2 * kb_pass : kb_pass;
  const int tiles = m_tiles * p.n_tiles;
  int splits = 1, kps = num_kb;
  const int cluster_k = (!PAIR && EPI == EPI_PACK && p.cluster_k > 1) ? p.cluster_k : 1;
  if (cluster_k > 1) {
    splits = cluster_k;
    kps = (num_kb + cluster_k - 1) / cluster_k;
  } else if (!PAIR && p.split_k_max > 1 && num_kb > 0 && M_eff > 0) {
    splitk_plan(m_tiles * kBM, p.split_rows > 0 ? p.split_rows : p.M, num_kb, p.split_k_max,
                splits, kps);
  }
  const int total = (num_kb > 0 && M_eff > 0) ? tiles * splits : 0;
  // nothing to do (e.g. no routed rows): leave before touching TMEM or
  // barriers (uniform over a pair: both ranks have the same group)
  if (total == 0 || group >= total) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      // PAIR: one arrival per epilogue warp of both ranks, on rank 0's barrier
      mbar_init(&tempty[a], PAIR ? 2 * (kEpiThreads / 32) : kEpiThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_holder, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && total > 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmB2);
      // PAIR: both ranks' loads complete on rank 0's full barriers
      const uint32_t full0 = PAIR ? cluster_addr(&full[0], 0) : 0u;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int unit = group; unit < total && ok; unit += n_groups) {
        int mb, nb, tile, ks;
        unit_coords(unit, tiles, cluster_k, tile, ks);
        tile_coords(tile, m_tiles, p.n_tiles, mb, nb);
        const int kb1 = min(num_kb, (ks + 1) * kps);
        for (int kb = ks * kps; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = sA + stage * kABytes;
          uint8_t* b_dst = sB + stage * B_BYTES;
          if constexpr (PAIR) {
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * (kABytes + B_BYTES));
            const uint32_t fb = full0 + 8u * (uint32_t)stage;
            const int m0 = mb * TILE_M + rank * kBM;  // this rank's A rows
            if (!A_MN) {
              tma_load_2d_pair(a_dst, &tmA, fb, kb * kBK, m0);
            } else {
              const bool second = kb >= kb_pass;
              const int ka = (second ? kb - kb_pass : kb) * kBK;
              const int ma = m0 + (second ? p.a_seg_off : 0);
              tma_load_2d_pair(a_dst, &tmA, fb, ma, ka);
              tma_load_2d_pair(a_dst + 8192, &tmA, fb, ma + 64, ka);
            }
            if (EPI == EPI_GATED) {
              // rank 0 holds the tile's 128 gate rows, rank 1 its 128 up rows
              tma_load_2d_pair(b_dst, rank ? &tmB2 : &tmB, fb, kb * kBK, nb * 128);
            } else {
              const int kbb = (A_MN && kb >= kb_pass) ? kb - kb_pass : kb;  // B rows repeat
              const int seg = kbb / p.k_split;
              const CUtensorMap* mp = (seg & 1) ? &tmB2 : &tmB;
              const int kk = kbb - seg * p.k_split;
              const int n0 = nb * kBN + rank * (kBN / 2);  // this rank's B rows
              if (!B_MN) {
                tma_load_2d_pair(b_dst, mp, fb, kk * kBK, n0);
              } else {
                tma_load_2d_pair(b_dst, mp, fb, n0, kk * kBK);
                tma_load_2d_pair(b_dst + 8192, mp, fb, n0 + 64, kk * kBK);
              }
            }
          } else {
            mbar_arrive_expect_tx(&full[stage], kABytes + kBBytes);
            if (!A_MN) {
              tma_load_2d(a_dst, &tmA, &full[stage], kb * kBK, mb * kBM);
            } else {
              const bool second = kb >= kb_pass;
              const int ka = (second ? kb - kb_pass : kb) * kBK;
              const int ma = mb * kBM + (second ? p.a_seg_off : 0);
              tma_load_2d(a_dst, &tmA, &full[stage], ma, ka);
              tma_load_2d(a_dst + 8192, &tmA, &full[stage], ma + 64, ka);
            }
            if (EPI == EPI_GATED) {
              tma_load_2d(b_dst, &tmB, &full[stage], kb * kBK, nb * 128);
              tma_load_2d(b_dst + 16384, &tmB2, &full[stage], kb * kBK, nb * 128);
            } else {
              const int kbb = (A_MN && kb >= kb_pass) ? kb - kb_pass : kb;  // B rows repeat
              const int seg = kbb / p.k_split;
              const CUtensorMap* mp = (seg & 1) ? &tmB2 : &tmB;
              const int kk = kbb - seg * p.k_split;
              if (!B_MN) {
                tma_load_2d(b_dst, mp, &full[stage], kk * kBK, nb * kBN);
              } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  tma_load_2d(b_dst + i * 8192, mp, &full[stage], nb * kBN + 64 * i, kk * kBK);
              }
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if constexpr (PAIR) {
        // rank 0's MMA warp signals this CTA's empty barriers from the other
        // SM: wait for the release of the last STAGES fills, so no arrival
        // is still on its way when the CTA leaves
        for (int i = 0; i < STAGES && ok; ++i) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) ok = false;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        set_status(p.status, TWELL_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && total > 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16(TILE_M, kBN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int unit = group; unit < total && ok; unit += n_groups, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        int tile, ks;
        unit_coords(unit, tiles, cluster_k, tile, ks);
        const int kb0 = ks * kps, kb1 = min(num_kb, (ks + 1) * kps);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kABytes);
          const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = A_MN ? sdesc_sw128(a0 + k * 2048, 8192, 1024)
                                     : sdesc_sw128(a0 + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b0 + k * 2048, 8192, 1024)
                                     : sdesc_sw128(b0 + k * 32, 16, 1024);
            if constexpr (PAIR)
              tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
            else
              tc_mma_bf16(d_tmem, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          }
          if constexpr (PAIR)
            tc_commit_pair(&empty[stage], 0x3);
          else
            tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) {
          if constexpr (PAIR)
            tc_commit_pair(&tfull[acc], 0x3);
          else
            tc_commit(&tfull[acc]);
        }
      }
      if (!ok) {
        set_status(p.status, TWELL_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int r_local = quarter * 32 + lane;
    Stager st{sOut + (warp - 4) * kStageBytes, lane, 0, false};
    const OutMaps om{&tmO0, &tmO1, &tmO2};
    const uint32_t tempty0 = PAIR ? cluster_addr(&tempty[0], 0) : 0u;
    int it = 0;
    for (int unit = group; unit < total; unit += n_groups, ++it) {
      int mb, nb, tile, ks;
      unit_coords(unit, tiles, cluster_k, tile, ks);
      tile_coords(tile, m_tiles, p.n_tiles, mb, nb);
      const int row_off = cluster_k > 1 ? 0 : ks * m_tiles * kBM;  // split-K partial rows
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      const int m_row0 = mb * TILE_M + rank * kBM;  // this CTA's first output row of the tile
      const int row = m_row0 + r_local;
      const int n0 = (EPI == EPI_GATED) ? nb * 128 : nb * kBN;
      if constexpr (EPI == EPI_BWD_GATE || EPI == EPI_BWD_GATE_RT)
        Epilogue<EPI>::prefetch(p, row, n0, half, p.N);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
        set_status(p.status, TWELL_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const bool row_ok = p.pad_rows ? (row < p.M) : (row < M_eff);
      const uint32_t tacc = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
      if (cluster_k > 1) {
        // one unit per block: split 0 packs after the cluster barrier below;
        // the other splits stage their accumulator [column][row] in the
        // operand buffers, idle now that every MMA of the tile has completed
        if (ks > 0) {
          float* part = reinterpret_cast<float*>(sA);
#pragma unroll 1
          for (int c0 = half * (kBN / 2); c0 < (half + 1) * (kBN / 2); c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tacc + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) part[(c0 + i) * kBM + r_local] = __uint_as_float(r[i]);
          }
        }
        continue;
      }
      Epilogue<EPI>::run(p, tacc, row, row_ok, n0, p.N, half, st, om,
                         row_off + m_row0 + quarter * 32);
      tc_fence_before();
      if constexpr (PAIR) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
      } else {
        mbar_arrive(&tempty[acc]);
      }
    }
    st.drain();  // staged stores finish reading shared memory before the CTA exits
  }

  if constexpr (EPI == EPI_PACK) {
    if (cluster_k > 1) {
      // every thread of every block of the cluster passes both barriers (all
      // waits above are bounded, so a block that gave up still arrives)
      namespace cg = cooperative_groups;
      cg::cluster_group cluster = cg::this_cluster();
      cluster.sync();  // partials staged
      int mb = 0, nb = 0, tile = 0, ks = 1;
      if (total > 0) {
        unit_coords(blockIdx.x, tiles, cluster_k, tile, ks);
        tile_coords(tile, m_tiles, p.n_tiles, mb, nb);
      }
      if (ks == 0 && !*abort_flag) {  // uniform over the leader block
        // the whole block sums the other splits' partials of the tile's valid
        // rows into its own shared memory, rank order, every remote value of
        // an element requested before any is added
        float* rsum = reinterpret_cast<float*>(sA);
        const float* src[7];
#pragma unroll
        for (int q = 1; q < 8; ++q)
          src[q - 1] = q < cluster_k ? cluster.map_shared_rank(rsum, (unsigned)q) : rsum;
        const int vrows = min(kBM, M_eff - mb * kBM);
        const int n_el = vrows * kBN;
        // four elements per pass: their remote values are all in flight together
        for (int e0 = threadIdx.x; e0 < n_el; e0 += 4 * kGemmThreads) {
          int o[4];
          float v[4][7];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = min(e0 + k * kGemmThreads, n_el - 1);
            const int col = e / vrows;
            o[k] = col * kBM + (e - col * vrows);
#pragma unroll
            for (int q = 1; q < 8; ++q) v[k][q - 1] = q < cluster_k ? src[q - 1][o[k]] : 0.f;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < 7; ++q) acc += v[k][q];
            if (e0 + k * kGemmThreads < n_el) rsum[o[k]] = acc;
          }
        }
        __syncthreads();
        if (warp >= 4) {
          const int quarter = warp & 3;
          const int half = (warp - 4) >> 2;
          const int r_local = quarter * 32 + lane;
          const int row = mb * kBM + r_local;
          const uint32_t tacc = tmem_base + ((uint32_t)(quarter * 32) << 16);
          Stager st{sOut + (warp - 4) * kStageBytes, lane, 0, false};
          const OutMaps om{&tmO0, &tmO1, &tmO2};
          Epilogue<EPI>::run(p, tacc, row, row < M_eff, nb * kBN, p.N, half, st, om, 0, rsum,
                             r_local);
        }
      }
      cluster.sync();  // no block leaves while the leader still reads its partial
    }
  }

  __syncthreads();
  if constexpr (PAIR) {
    // neither rank leaves (or frees TMEM) while the other may still signal
    // its barriers or have its shared memory read by the pair's MMAs
    cluster_sync_all();
    if (warp == 2) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, kTmemCols);
    }
  } else {
    if (warp == 2) {
      tc_fence_after();
      tmem_dealloc(tmem_base, kTmemCols);
    }
  }
}

}  // namespace tw
