// internal.h -- host-side interfaces between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "twell.h"

namespace tw {

struct GemmParams;

// A bf16 row-major matrix view: rows x cols elements, leading dimension ld.
struct Mat {
  const void* ptr;
  long long rows, cols, ld;
};

// An output the epilogue writes through TMA: rows x cols elements (bf16 or
// fp32), leading dimension ld, boxes of box_cols x 32 rows.
struct OutMat {
  const void* ptr;
  long long rows, cols, ld;
  int f32;
  int box_cols;
};

// Which epilogue / operand majorness a GEMM launch uses.
enum GemmKind {
  GK_STORE_KK = 0,   // A K-major, B K-major, store
  GK_STORE_MK = 1,   // A MN-major, B K-major, store
  GK_STORE_KM = 2,   // A K-major, B MN-major, store
  GK_STORE_MM = 3,   // A MN-major, B MN-major, store
  GK_PACK = 4,       // gate GEMM with the TwELL pack epilogue
  GK_GATED = 5,      // [Wg ; Wu] GEMM with the ReLU * up epilogue
  GK_BWD_GATE = 6,   // dh GEMM with the du / da epilogue
  GK_BWD_GATE_RT = 7,  // the same for routed rows (fp32 u in, bf16 hi + lo out)
};

int num_sms();
// L2 size of the current device in bytes (0 if unknown).
double l2_bytes();
// Rows wider than 1024 take the split gathers (true, the default) or the
// fused kernels (twell_set_split_gathers).
bool split_gathers();
// Large GEMMs run as CTA pairs with 256 x 256 tiles (true, the default) or
// as single CTAs with 128 x 256 tiles (twell_set_pair_gemm).
bool pair_gemm();
int current_device();
// Passes over the neuron axis for a gather whose weight rows total
// `gathered_bytes`: 1 while they fit in the fraction `fit` of L2, else
// enough chunks of at most the fraction `chunk` of L2 each.
int l2_chunks(double gathered_bytes, double fit, double chunk);
void count_launch(int n = 1);  // kernels launched by the library (process-wide)

// Brackets one kernel launch: an NVTX range named after the kernel family
// (seen by Nsight tools; a no-op without one) and, while profiling is on for
// `name` (or "*"), CUDA events recorded on the launch's stream.
struct ProfScope {
  ProfScope(const char* name, cudaStream_t s);
  ~ProfScope();
  int slot;
  cudaStream_t stream;
};
int* device_status_ptr();  // per-device status word (device address)

// NVTX range over one entry point (named after it) for Nsight timelines.
struct NvtxRange {
  explicit NvtxRange(const char* name);
  ~NvtxRange();
};

// Launch the persistent GEMM.  A is the M-side operand, B (and B2 for a
// second K range or the up half of EPI_GATED) the N-side one, each given in
// its storage layout.  Returns a CUDA error or cudaSuccess; an invalid
// tensor-map encode returns cudaErrorInvalidValue.
cudaError_t gemm_launch(GemmKind kind, const Mat& A, const Mat& B, const Mat* B2,
                        const GemmParams& p, cudaStream_t stream, const OutMat* outs = nullptr,
                        int n_outs = 0);
// 2-D tensor map over a bf16 matrix, 128-byte swizzled boxes of
// box_inner (contiguous) x box_outer elements.
bool make_tma_map_bf16(CUtensorMap* m, const Mat& a, uint32_t box_inner, uint32_t box_outer);

// Gate GEMM + TwELL pack for small batches (gate_smallm.cu): neurons on the
// MMA's M dimension, up to kSmallGateMaxM tokens on its N dimension.
constexpr int kSmallGateMaxM = 64;
bool gate_pack_smallm_fits(int M, int d, int f, int tile_n);
cudaError_t launch_gate_pack_smallm(const void* x, const void* wgT, int M, int d, int f,
                                    int tile_n, int cap, const twell_tiles& out, cudaStream_t s);

// Non-tensor-core kernels (pack.cu, sparse_fwd.cu, sparse_bwd.cu).
cudaError_t launch_pack_dense(const void* a, int a_f32, int M, int f, int tile_n, int cap,
                              const twell_tiles& out, cudaStream_t s);
// dense_cap: routed rows the workspace holds; more routed rows than that
// record TWELL_ERR_CAPACITY in the device status word.
cudaError_t launch_route(const twell_tiles& in, int M, int f, int tile_n, int cap,
                         const twell_hybrid& out, int* scan_flags, int dense_cap, cudaStream_t s);
// part holds buf_rows rows of split-K partials of at most row_cap routed rows
cudaError_t launch_splitk_scatter(const float* part, int buf_rows, int row_cap, int num_kb,
                                  int s_max, const int* n_rows, const int* rows, int M, int N,
                                  void* out, cudaStream_t s);
cudaError_t launch_gather_rows(const void* src, int M, int d, const int* rows, const int* n_rows,
                               void* dst, int dst_rows, cudaStream_t s);
// `part` ([M][d] fp32) carries y between the passes of an ELL gather split
// into L2-sized neuron chunks; it may be null when one pass suffices.
// `hbuf` ([M][ell_width] fp32) holds the per-entry h of the split up / down
// gathers used for ELL rows wider than 1024; null keeps the fused gather.
cudaError_t launch_sparse_fwd(const void* x, const void* wuT, const void* wd, int M, int d, int f,
                              const twell_tiles* tiles, int tile_n, int cap,
                              const twell_hybrid* route, void* y, float* part, float* hbuf,
                              cudaStream_t s);
cudaError_t launch_csc_build(const twell_hybrid& route, int M, int f, int* blk_counts,
                             int* csc_ptr, int* csc_row, int* slot_pos, cudaStream_t s);
// `part` ([M][d] fp32) carries dX between L2-sized neuron passes (may be null).
// `dhbuf` ([M][ell_width] fp32) holds the per-entry dh of the split row phase
// used for rows wider than 1024; null keeps the fused kernel.
cudaError_t launch_sparse_bwd_rows(const void* x, const void* dy, const void* wgT, const void* wuT,
                                   const void* wd, int M, int d, int f, const twell_hybrid& route,
                                   const int* slot_pos, float lambda, float4* csc_vals, void* dx,
                                   float* part, float* dhbuf, cudaStream_t s);
cudaError_t launch_sparse_bwd_neurons(const void* x, const void* dy, int M, int d, int f,
                                      const int* csc_ptr, const int* csc_row,
                                      const float4* csc_vals, float* dwgT, float* dwuT, float* dwd,
                                      cudaStream_t s);

}  // namespace tw
