// gate_smallm.cu -- gate GEMM with the TwELL pack for small batches (M <= 64).
//
// Page 2 "Sakana AI and NVIDIA introduce TwELL with CUDA kernels ...",
// section "¿Qué hace distinto a TwELL frente a ELL clásico?": the gate
// activation is packed per T_n-wide tile inside the gate matmul's epilogue.
// Section "¿Cuál es el problema que TwELL resuelve?" names the regime this
// kernel serves: earlier activation-sparse kernels only covered one token at
// a time, where the gate matmul is a matrix-vector product bound by reading
// Wg from HBM.
//
// With a handful of tokens the usual orientation (tokens on the MMA's
// 128-row M dimension) pads M to 128 and spreads Wg over few, wide tiles.
// Here the operands are swapped: a tile is 128 neurons (rows of Wg^T, the
// MMA's M) by NP tokens (x padded to 16, 32 or 64 rows, the MMA's N), one
// block per tile and SM, streaming its slice of Wg through a TMA ring of
// about 200 KB (measured on the 8B-class shape: ~45 GB/s per SM with eight
// 16 KB stages; an L2 prefetch of the whole slice ahead of the ring made the
// first data arrive later and the kernel slower).  Where the tiles are
// fewer than the SMs, K is split over the blocks of a thread-block cluster.
// The accumulator holds one neuron per TMEM lane and one token per column,
// and the pack works across lanes: per token, each warp ballots which of its
// 32 neurons are live; a lane per token then combines the four warps' counts
// into the TwELL count and walks its warp's live neurons in ascending order
// to their slots.  The blocks of a cluster sum their partial accumulators
// through distributed shared memory in rank order (deterministic; no global
// scratch).
//
// Warp roles (192 threads): warps 0-3 epilogue (warp w owns TMEM lanes
// 32w..32w+31, the only lanes it may read), warp 4 TMA producer, warp 5
// TMEM allocator and MMA issuer.  Every mbarrier wait is bounded.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace tw {

namespace {

constexpr int kSmThreads = 192;
constexpr int kSmBM = 128;  // neurons per tile (MMA M)
constexpr int kSmBK = 64;   // one 128-byte swizzle row of bf16
constexpr int kSmABytes = kSmBM * kSmBK * 2;

template <int NP>
struct SmCfg {
  static constexpr int kBPS = 1;  // k-blocks (TMA boxes of A and of B) per ring stage
  static constexpr int kBBytes = kBPS * NP * kSmBK * 2;
  static constexpr int kABytes = kBPS * kSmABytes;
  static constexpr int kStages = (200 * 1024) / (kABytes + kBBytes);
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = NP <= 32 ? 32 : 64;
  // stage buffers (1024-byte aligned: up to 1008 bytes of slack), barriers,
  // and the per-token warp counts of the pack (one block per SM)
  static constexpr int kSmem = kStages * kStageBytes + 1008 + 256 + NP * 4 * 4;
  static_assert(NP * kSmBM * 4 <= kStages * kStageBytes, "partials fit in the stage buffers");
  static_assert(kSmem <= 227 * 1024, "one block's shared memory");
};

struct SmallGateParams {
  int M, num_kb, kps;  // tokens, k-blocks of d_model, k-blocks per cluster rank
  int T, tile_n, cap;  // TwELL tiles per row, tile width, slots per tile
  uint16_t* val;
  uint8_t* idx;
  uint8_t* cnt;
  int* row_nnz;
  int* status;
};

template <int NP>
__global__ void __launch_bounds__(kSmThreads, 1)
    gate_pack_smallm_kernel(const __grid_constant__ CUtensorMap tmW,
                            const __grid_constant__ CUtensorMap tmX, const SmallGateParams p) {
  using C = SmCfg<NP>;
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                            // stages x 128 neuron rows of Wg^T
  uint8_t* sB = smem + C::kStages * C::kABytes;  // stages x NP token rows of x
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::kStages * C::kBBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // per token: live neurons of each epilogue warp
  int (*s_cnt)[4] = reinterpret_cast<int (*)[4]>(reinterpret_cast<uint8_t*>(full) + 256);

  const int KS = (int)cluster.num_blocks();
  const int ks = (int)cluster.block_rank();
  const int nt = (int)blockIdx.x / KS;  // neuron tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb0 = ks * p.kps, kb1 = min(p.num_kb, kb0 + p.kps);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; kb += C::kBPS) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const int nb = min(C::kBPS, kb1 - kb);
        mbar_arrive_expect_tx(&full[stage], (uint32_t)nb * (kSmABytes + NP * kSmBK * 2));
        for (int b = 0; b < nb; ++b) {
          tma_load_2d(sA + stage * C::kABytes + b * kSmABytes, &tmW, &full[stage],
                      (kb + b) * kSmBK, nt * kSmBM);
          tma_load_2d(sB + stage * C::kBBytes + b * NP * kSmBK * 2, &tmX, &full[stage],
                      (kb + b) * kSmBK, 0);
        }
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        set_status(p.status, TWELL_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kSmBM, NP, false, false);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; kb += C::kBPS) {
        if (!mbar_wait(&full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nb = min(C::kBPS, kb1 - kb);
        for (int b = 0; b < nb; ++b) {
          const uint32_t a0 = smem_u32(sA + stage * C::kABytes + b * kSmABytes);
          const uint32_t b0 = smem_u32(sB + stage * C::kBBytes + b * NP * kSmBK * 2);
#pragma unroll
          for (int k = 0; k < kSmBK / 16; ++k)
            tc_mma_bf16(tmem, sdesc_sw128(a0 + k * 32, 16, 1024),
                        sdesc_sw128(b0 + k * 32, 16, 1024), idesc,
                        (kb + b != kb0 || k != 0) ? 1u : 0u);
        }
        tc_commit(&empty[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        tc_commit(tfull);
      } else {
        set_status(p.status, TWELL_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- epilogue
  // The accumulator stays in TMEM; each thread (neuron 32 warp + lane of the
  // tile) reads it 32 tokens at a time.
  constexpr int kChunks = (NP + 31) / 32;
  float* part = reinterpret_cast<float*>(smem);  // [NP][128] partial of a rank > 0
  const int nrow = warp * 32 + lane;
  const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
  if (warp < 4) {
    if (!mbar_wait(tfull, 0, abort_flag)) {
      set_status(p.status, TWELL_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      // every MMA of this block has completed (tfull), so its operand buffers
      // are free: ranks > 0 stage their partial there, [token][neuron]
      if (ks > 0) {
#pragma unroll
        for (int h = 0; h < kChunks; ++h) {
          uint32_t r[32];
          tmem_ld32(taddr + 32 * h, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * h + i < NP) part[(32 * h + i) * kSmBM + nrow] = __uint_as_float(r[i]);
        }
      }
    }
  }
  // every thread of every block of the cluster passes both barriers (all
  // waits above are bounded, so a block that gave up still arrives)
  cluster.sync();
  if (ks == 0 && warp < 4 && !*abort_flag) {
    // ReLU + TwELL pack across the tile's neurons.  bf16(ReLU(a)) > 0 exactly
    // when a > 2^-134 (the largest fp32 that rounds to bf16 zero).
    const float kLiveMin = __uint_as_float(0x00008000u);
    const int per_tile = p.tile_n / 32;     // warps per TwELL tile: 4 or 2
    const int t = nt * (kSmBM / p.tile_n) + warp / per_tile;
    const int w0 = warp - warp % per_tile;  // first warp of this TwELL tile
    // this block's operand buffers are free (its MMAs completed): the
    // chunk's values [token][neuron]
    float* sv = reinterpret_cast<float*>(smem);
    uint32_t mk = 0;
#pragma unroll 1
    for (int h = 0; h < kChunks; ++h) {
      if (32 * h >= p.M) break;  // block-uniform
      uint32_t r[32];
      tmem_ld32(taddr + 32 * h, r);
      tmem_wait_ld();
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      // partials of ranks 1, 2, ... added in rank order
      for (int q = 1; q < KS; ++q) {
        const float* rp = cluster.map_shared_rank(part, (unsigned)q);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (32 * h + i < NP) v[i] += rp[(32 * h + i) * kSmBM + nrow];
      }
      mk = 0;
      // pass 1 (unrolled over the chunk's tokens): lane i keeps this warp's
      // live mask of token 32 h + i; the values go to shared memory
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int m = 32 * h + i;
        sv[i * kSmBM + nrow] = v[i];
        if (m < NP && m < p.M) {  // warp-uniform
          const uint32_t b = __ballot_sync(0xffffffffu, v[i] > kLiveMin);
          if (lane == i) {
            mk = b;
            s_cnt[m][warp] = __popc(b);
          }
        }
      }
      named_barrier(1, 128);
      // pass 2, a lane per token: the TwELL count of the token's tile from
      // the warps' counts, then this warp's live neurons, ascending, to
      // their slots after those of the warps before it
      {
        const int m = 32 * h + lane;
        if (m < NP && m < p.M) {
          int pre = 0, total = 0;
          for (int w = w0; w < w0 + per_tile; ++w) {
            const int c = s_cnt[m][w];
            pre += w < warp ? c : 0;
            total += c;
          }
          const long long slot0 = ((long long)m * p.T + t) * p.cap;
          int slot = pre;
          for (uint32_t bits = mk; bits && slot < p.cap; bits &= bits - 1u, ++slot) {
            const int n = __ffs(bits) - 1;  // neuron 32 warp + n of the 128-neuron tile
            p.val[slot0 + slot] = (uint16_t)relu_bf16_bits(sv[lane * kSmBM + warp * 32 + n]);
            p.idx[slot0 + slot] = (uint8_t)((warp * 32 + n) % p.tile_n);
          }
          if (warp == w0) {
            p.cnt[(long long)m * p.T + t] = (uint8_t)total;
            if (total) atomicAdd(p.row_nnz + m, total);
          }
        }
      }
      named_barrier(1, 128);  // sv is rewritten by the next chunk
    }
  }
  if (warp < 4) tc_fence_before();
  cluster.sync();  // no block leaves while rank 0 still reads its partial
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NP>
cudaError_t launch_np(const CUtensorMap& tw_map, const CUtensorMap& tx_map,
                      const SmallGateParams& p, int n_tiles, int ks, cudaStream_t s) {
  using C = SmCfg<NP>;
  auto kern = gate_pack_smallm_kernel<NP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_tiles * ks));
  cfg.blockDim = dim3(kSmThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    ProfScope prof("gemm_gate_pack", s);
    e = cudaLaunchKernelEx(&cfg, kern, tw_map, tx_map, p);
  }
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool gate_pack_smallm_fits(int M, int d, int f, int tile_n) {
  return M >= 1 && M <= kSmallGateMaxM && d % kSmBK == 0 && f % kSmBM == 0 &&
         (tile_n == 64 || tile_n == 128);
}

cudaError_t launch_gate_pack_smallm(const void* x, const void* wgT, int M, int d, int f,
                                    int tile_n, int cap, const twell_tiles& out, cudaStream_t s) {
  if (!gate_pack_smallm_fits(M, d, f, tile_n)) return cudaErrorInvalidValue;
  const int NP = M <= 16 ? 16 : M <= 32 ? 32 : 64;
  const int n_tiles = f / kSmBM;
  const int num_kb = d / kSmBK;
  // K split over a cluster: the largest power of two (at most 8) dividing
  // the k-blocks that keeps every rank at four k-blocks or more and the grid
  // within one block per SM (all resident at once)
  int ks = 1;
  for (int next = 2; next <= 8; next *= 2) {
    if (num_kb % next != 0 || num_kb / next < 4 || (long long)n_tiles * next > num_sms())
      break;
    ks = next;
  }
  CUtensorMap tw_map, tx_map;
  if (!make_tma_map_bf16(&tw_map, Mat{wgT, f, d, d}, kSmBK, kSmBM)) return cudaErrorInvalidValue;
  if (!make_tma_map_bf16(&tx_map, Mat{x, M, d, d}, kSmBK, (uint32_t)NP))
    return cudaErrorInvalidValue;
  SmallGateParams p{};
  p.M = M;
  p.num_kb = num_kb;
  p.kps = num_kb / ks;
  p.T = f / tile_n;
  p.tile_n = tile_n;
  p.cap = cap;
  p.val = reinterpret_cast<uint16_t*>(out.val);
  p.idx = out.idx;
  p.cnt = out.cnt;
  p.row_nnz = out.row_nnz;
  p.status = device_status_ptr();
  if (NP == 16) return launch_np<16>(tw_map, tx_map, p, n_tiles, ks, s);
  if (NP == 32) return launch_np<32>(tw_map, tx_map, p, n_tiles, ks, s);
  return launch_np<64>(tw_map, tx_map, p, n_tiles, ks, s);
}

}  // namespace tw
