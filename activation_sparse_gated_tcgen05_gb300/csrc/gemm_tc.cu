// gemm_tc.cu -- host side of the tcgen05 GEMM engine: TMA tensor maps and
// persistent launches of the instantiated kernels.
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_tc.cuh"
#include "internal.h"

namespace tw {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [outer][inner] matrix with leading
// dimension ld (elements), 128-byte swizzled boxes of box_inner x box_outer.
bool make_map(CUtensorMap* m, const Mat& a, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn || !a.ptr || a.rows <= 0 || a.cols <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)a.cols, (cuuint64_t)a.rows};
  cuuint64_t strides[1] = {(cuuint64_t)a.ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output map for TMA stores: box_cols x 32 rows, swizzle matching the row
// bytes of the staging buffer (128-byte or 64-byte rows).
bool make_out_map(CUtensorMap* m, const OutMat& o) {
  auto fn = encode_fn();
  if (!fn || !o.ptr || o.rows <= 0 || o.cols <= 0) return false;
  const int esz = o.f32 ? 4 : 2;
  const int row_bytes = o.box_cols * esz;
  if (row_bytes != 128 && row_bytes != 64) return false;
  cuuint64_t dims[2] = {(cuuint64_t)o.cols, (cuuint64_t)o.rows};
  cuuint64_t strides[1] = {(cuuint64_t)o.ld * esz};
  cuuint32_t box[2] = {(cuuint32_t)o.box_cols, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, o.f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(o.ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool make_tma_map_bf16(CUtensorMap* m, const Mat& a, uint32_t box_inner, uint32_t box_outer) {
  return make_map(m, a, box_inner, box_outer);
}

namespace {

// Clusters of the CTA-pair kernel that fit on the device at once (0: none,
// or the query failed), cached per device.
template <bool A_MN, bool B_MN, int EPI>
int pair_clusters() {
  constexpr int kDevices = 64;
  static int cache[kDevices] = {0};  // 0 = not asked yet, -1 = unavailable
  const int dev = current_device();
  if (dev < 0 || dev >= kDevices) return 0;
  if (cache[dev] == 0) {
    auto kern = gemm_kernel<A_MN, B_MN, EPI, true>;
    int n = 0;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kGemmSmem);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (unsigned)(num_sms() / 2));
      cfg.blockDim = dim3(kGemmThreads);
      cfg.dynamicSmemBytes = kGemmSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    }
    if (e != cudaSuccess) {
      n = 0;
      cudaGetLastError();  // the failed query's error is not left for the caller
    }
    cache[dev] = n > 0 ? n : -1;
  }
  return cache[dev] > 0 ? cache[dev] : 0;
}

template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_t(const char* name, const Mat& A, const Mat& B, const Mat* B2,
                     const GemmParams& p, cudaStream_t s, const OutMat* outs, int n_outs) {
  // CTA pairs (256 x 256 tiles) unless the GEMM splits K (split-K partials
  // and cluster split-K keep single CTAs) or the pairs would need more waves
  // of tiles than single CTAs (a pair tile takes about as long as a single
  // CTA's 128 x 256 tile)
  int clusters = 0;
  long long pair_tiles = 0;
  if (pair_gemm() && p.split_k_max <= 1 && !(EPI == EPI_PACK && p.cluster_k > 1) && p.M > 0 &&
      p.n_tiles > 0) {
    pair_tiles = (long long)((p.M + 2 * kBM - 1) / (2 * kBM)) * p.n_tiles;
    const long long single_tiles = (long long)((p.M + kBM - 1) / kBM) * p.n_tiles;
    const int sms = num_sms();
    clusters = pair_clusters<A_MN, B_MN, EPI>();
    if (clusters > 0 && sms > 0 &&
        (pair_tiles + clusters - 1) / clusters > (single_tiles + sms - 1) / sms)
      clusters = 0;
  }
  const bool pair = clusters > 0;
  CUtensorMap ta, tb, tb2;
  // A: K-major [M][K] -> box {64 (K), 128 rows}; MN-major [K][M] -> box {64 (M), 64 (K)}
  if (!make_map(&ta, A, 64, A_MN ? 64 : kBM)) return cudaErrorInvalidValue;
  // B: K-major -> box {64 (K), rows of B a CTA stages}: 128 for the gated
  // GEMM (one of [Wg ; Wu]) and for a pair (half of the tile's 256), else 256
  const uint32_t b_rows = (EPI == EPI_GATED || pair) ? 128 : kBN;
  if (!make_map(&tb, B, 64, B_MN ? 64 : b_rows)) return cudaErrorInvalidValue;
  if (B2) {
    if (!make_map(&tb2, *B2, 64, B_MN ? 64 : b_rows)) return cudaErrorInvalidValue;
  } else {
    tb2 = tb;
  }
  CUtensorMap to[3];
  for (int i = 0; i < 3; ++i) {
    if (i < n_outs) {
      if (!make_out_map(&to[i], outs[i])) return cudaErrorInvalidValue;
    } else {
      to[i] = ta;  // unused
    }
  }
  if (pair) {
    // one 2-CTA cluster per pair, at most one pair per resident cluster slot
    auto kern = gemm_kernel<A_MN, B_MN, EPI, true>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    const long long n_pairs = pair_tiles < clusters ? pair_tiles : clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * n_pairs));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kGemmSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t le;
    {
      ProfScope prof(name, s);
      le = cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2, to[0], to[1], to[2], p);
    }
    count_launch();
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
  }
  auto kern = gemm_kernel<A_MN, B_MN, EPI, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  const long long m_tiles = (p.M + kBM - 1) / kBM;
  const long long tiles = m_tiles * p.n_tiles;
  if (tiles <= 0) return cudaSuccess;
  if (EPI == EPI_PACK && p.cluster_k > 1) {
    // cluster split-K: one (tile, K split) per block, the splits of a tile in
    // one cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * p.cluster_k));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kGemmSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cluster_k;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t le;
    {
      ProfScope prof(name, s);
      le = cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2, to[0], to[1], to[2], p);
    }
    count_launch();
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
  }
  // split-K GEMMs run up to split_k_max units per output tile (the plan
  // depends on the device-side row count); blocks past the work exit at once
  const long long units = tiles * (p.split_k_max > 1 ? p.split_k_max : 1);
  const int grid = (int)(units < num_sms() ? units : num_sms());
  {
    ProfScope prof(name, s);
    kern<<<grid, kGemmThreads, kGemmSmem, s>>>(ta, tb, tb2, to[0], to[1], to[2], p);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_launch(GemmKind kind, const Mat& A, const Mat& B, const Mat* B2,
                        const GemmParams& p, cudaStream_t s, const OutMat* outs, int n_outs) {
  switch (kind) {
#define TW_CASE(K, AM, BM, E, NAME) \
  case K: return launch_t<AM, BM, E>(NAME, A, B, B2, p, s, outs, n_outs);
    TW_CASE(GK_STORE_KK, false, false, EPI_STORE, "gemm_store_kk")
    TW_CASE(GK_STORE_MK, true, false, EPI_STORE, "gemm_store_mk")
    TW_CASE(GK_STORE_KM, false, true, EPI_STORE, "gemm_store_km")
    TW_CASE(GK_STORE_MM, true, true, EPI_STORE, "gemm_store_mm")
    TW_CASE(GK_PACK, false, false, EPI_PACK, "gemm_gate_pack")
    TW_CASE(GK_GATED, false, false, EPI_GATED, "gemm_gated")
    TW_CASE(GK_BWD_GATE, false, false, EPI_BWD_GATE, "gemm_dgate")
    TW_CASE(GK_BWD_GATE_RT, false, false, EPI_BWD_GATE_RT, "gemm_dgate")
#undef TW_CASE
  }
  return cudaErrorInvalidValue;
}

}  // namespace tw
