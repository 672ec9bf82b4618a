// api.cu -- the library's C ABI: argument checks, workspace layout and the
// launch sequence of every entry point declared in twell.h.
#include <atomic>
#include <cstring>
#include <map>
#include <cmath>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "gemm_tc.cuh"
#include "internal.h"

namespace tw {

__device__ int g_device_status;

namespace {
constexpr int kMaxDevices = 64;
}  // namespace

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

namespace {
std::atomic<unsigned long long> g_launches{0};
}

void count_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

// ---------------------------------------------------------------- profiling
namespace {
struct ProfRecord {
  std::string name;
  cudaEvent_t start, stop;
};
struct ProfEntry {
  std::string name;
  int launches;
  double total_ms;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::string g_prof_filter;
std::vector<ProfRecord> g_prof_records;
std::vector<ProfEntry> g_prof_report;
}  // namespace

NvtxRange::NvtxRange(const char* name) { nvtxRangePushA(name); }
NvtxRange::~NvtxRange() { nvtxRangePop(); }

ProfScope::ProfScope(const char* name, cudaStream_t s) : slot(-1), stream(s) {
  nvtxRangePushA(name);
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof_filter != "*" && g_prof_filter != name) return;
  ProfRecord r{name, nullptr, nullptr};
  if (cudaEventCreate(&r.start) != cudaSuccess) return;
  if (cudaEventCreate(&r.stop) != cudaSuccess) {
    cudaEventDestroy(r.start);
    return;
  }
  cudaEventRecord(r.start, s);
  slot = (int)g_prof_records.size();
  g_prof_records.push_back(r);
}

ProfScope::~ProfScope() {
  nvtxRangePop();
  if (slot < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  cudaEventRecord(g_prof_records[slot].stop, stream);
}

int num_sms() {
  static int cache[kMaxDevices] = {0};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// Process-wide choice of the wide-row gathers (see twell_set_split_gathers).
std::atomic<int> g_split_gathers{1};
bool split_gathers() { return g_split_gathers.load(std::memory_order_relaxed) != 0; }

// Process-wide choice of the GEMM tile form (see twell_set_pair_gemm).
std::atomic<int> g_pair_gemm{1};
bool pair_gemm() { return g_pair_gemm.load(std::memory_order_relaxed) != 0; }

double l2_bytes() {
  static int cache[kMaxDevices] = {0};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 0.0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0) return 0.0;
    cache[dev] = n;
  }
  return (double)cache[dev];
}

int l2_chunks(double gathered_bytes, double fit, double chunk) {
  const double l2 = l2_bytes();
  if (l2 <= 0.0 || gathered_bytes <= fit * l2) return 1;
  return (int)std::ceil(gathered_bytes / (chunk * l2));
}

int* device_status_ptr() {
  static int* cache[kMaxDevices] = {nullptr};
  static std::mutex mu;
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cache[dev] = reinterpret_cast<int*>(p);
  }
  return cache[dev];
}

}  // namespace tw

using namespace tw;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every pointer given must be non-null and 16-byte aligned.
twell_status check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps) {
    if (!p) return TWELL_ERR_INVALID_ARG;
    if (!aligned16(p)) return TWELL_ERR_ALIGNMENT;
  }
  return TWELL_OK;
}

twell_status check_shape(const twell_shape* s, bool packed) {
  if (!s) return TWELL_ERR_INVALID_ARG;
  if (s->M < 0 || s->d_model <= 0 || s->d_ff <= 0) return TWELL_ERR_INVALID_ARG;
  if (s->d_model % 64 != 0 || s->d_model > 8192) return TWELL_ERR_UNSUPPORTED;
  if (s->d_ff % 128 != 0 || s->d_ff > 65535) return TWELL_ERR_UNSUPPORTED;
  if (packed) {
    if (s->tile_n != 64 && s->tile_n != 128) return TWELL_ERR_UNSUPPORTED;
    if (s->tile_cap < 1 || s->tile_cap > s->tile_n) return TWELL_ERR_UNSUPPORTED;
  }
  return TWELL_OK;
}

twell_status check_tiles(const twell_tiles* t) {
  if (!t) return TWELL_ERR_INVALID_ARG;
  return check_ptrs({t->val, t->idx, t->cnt, t->row_nnz});
}

twell_status check_route(const twell_hybrid* r) {
  if (!r) return TWELL_ERR_INVALID_ARG;
  if (r->ell_width < 0 || r->dense_cap < 0) return TWELL_ERR_INVALID_ARG;
  twell_status st = check_ptrs({r->ell_nnz, r->dense_rows, r->n_dense});
  if (st != TWELL_OK) return st;
  if (r->ell_width > 0) return check_ptrs({r->ell_val, r->ell_col});
  return TWELL_OK;
}

inline twell_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA; }

inline long long round_up(long long v, long long a) { return (v + a - 1) / a * a; }

// Bump allocator over the caller's workspace (256-byte aligned slices).
struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(reinterpret_cast<uint8_t*>(b)) {}
  template <class T>
  T* take(size_t count) {
    off = (size_t)round_up((long long)off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

// Workspace of the sparse path.  Routed-row buffers hold the route's
// capacity (dense_cap, at most M) in whole 128-row tiles (Mr rows).  The
// dense backup keeps its intermediates h, du, da as bf16 hi + lo pairs, so
// routed rows are as accurate as the fp32 gather path:
//   hr  [Mr][2f] = [h hi | h lo]
//   part [Mp][d] fp32 (Mp = M in whole tiles): the running y / dX of
//        L2-sized passes, then the split-K partials of the routed rows' y
//        and dX GEMMs
//   ur  [Mr][f]  fp32 u
//   ddr [Mr][4f] = [du hi | da hi | du lo | da lo]
struct SparseWs {
  uint16_t *xr, *hr;                    // forward fallback
  float* part;
  float* hbuf;                          // per-ELL-entry h of the split forward
  uint16_t *dyr, *gr, *ddr;             // backward fallback
  float* ur;
  int *mask_off, *csc_ptr, *csc_row, *slot_pos;
  float4* csc_vals;
  long long Mr;                         // routed-row buffer rows (capacity in whole tiles)
  long long Mp;                         // rows of part
  size_t bytes;
};

SparseWs carve_sparse(void* ws, const twell_shape& s, int W, int dense_cap, int training) {
  const long long Mp = round_up(s.M, 128);
  const long long Mr = round_up(dense_cap < s.M ? dense_cap : s.M, 128);
  const long long d = s.d_model, f = s.d_ff;
  Carve c(ws);
  SparseWs w{};
  w.Mr = Mr;
  w.Mp = Mp;
  w.xr = c.take<uint16_t>(Mr * d);
  w.hr = c.take<uint16_t>(Mr * 2 * f);
  w.part = c.take<float>(Mp * d);
  const long long E = (long long)s.M * W;
  w.hbuf = c.take<float>(E > 0 ? E : 1);
  if (training) {
    const long long NB = (s.M + 31) / 32;
    w.dyr = c.take<uint16_t>(Mr * d);
    w.gr = c.take<uint16_t>(Mr * f);
    w.ur = c.take<float>(Mr * f);
    w.ddr = c.take<uint16_t>(Mr * 4 * f);
    w.mask_off = c.take<int>(32 + 2 * NB * f + f);  // counter, masks, offsets, totals
    w.csc_ptr = c.take<int>(f + 1);
    w.csc_row = c.take<int>(E > 0 ? E : 1);
    w.slot_pos = c.take<int>(E > 0 ? E : 1);
    w.csc_vals = c.take<float4>(E > 0 ? E : 1);
  }
  w.bytes = c.off + 256;
  return w;
}

// Optional workspace of the TwELL (inference) forward for rows wider than
// 1024, where it runs as two gathers:
//   hbuf [M][T * C] fp32: h of each row's live entries, in order
//   part [M][d] fp32: y carried between L2-sized neuron passes
struct TilesWs {
  float *hbuf, *part;
  size_t bytes;
};

TilesWs carve_tiles(void* ws, const twell_shape& s) {
  TilesWs w{};
  if (s.d_model <= 1024) return w;
  Carve c(ws);
  w.hbuf = c.take<float>((long long)s.M * (s.d_ff / s.tile_n) * s.tile_cap);
  w.part = c.take<float>((long long)s.M * s.d_model);
  w.bytes = c.off + 256;
  return w;
}

struct DenseWs {
  uint16_t *h, *g, *u, *dd;
  size_t bytes;
};

DenseWs carve_dense(void* ws, const twell_shape& s, int training) {
  const long long M = s.M, f = s.d_ff;
  Carve c(ws);
  DenseWs w{};
  w.h = c.take<uint16_t>(M * f);
  if (training) {
    w.g = c.take<uint16_t>(M * f);
    w.u = c.take<uint16_t>(M * f);
    w.dd = c.take<uint16_t>(M * 2 * f);
  }
  w.bytes = c.off + 256;
  return w;
}

GemmParams base_params(int M, int N, int K, int n_tile_width) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.n_tiles = (N + n_tile_width - 1) / n_tile_width;
  p.k_split = 1 << 30;
  p.status = device_status_ptr();
  return p;
}

Mat mat(const void* p, long long rows, long long cols, long long ld) { return Mat{p, rows, cols, ld}; }

// Dense gated FFN on rows [0, m_dev or M) of x_rows (a [rows][d] buffer):
// h = bf16(ReLU(x Wg)) * (x Wu) stored bf16 (split: as hi | lo halves of a
// [rows][2f] buffer), optional g / u copies ([rows][f]).
cudaError_t gated_gemm(const void* x_rows, long long rows, const twell_shape& s, const void* wgT,
                       const void* wuT, const int* m_dev, uint16_t* h, bool split, uint16_t* g,
                       uint16_t* u, float* u32, int pad_rows, cudaStream_t st,
                       int act = kActRelu) {
  GemmParams p = base_params((int)rows, s.d_ff, s.d_model, 128);
  p.act = act;
  p.m_dev = m_dev;
  p.h = h;
  p.ldh = split ? 2LL * s.d_ff : s.d_ff;
  p.h_lo_off = split ? s.d_ff : 0;
  p.g_out = g;
  p.u_out = u;
  p.u_f32 = u32;
  p.ldgu = s.d_ff;
  p.pad_rows = pad_rows;
  const Mat A = mat(x_rows, rows, s.d_model, s.d_model);
  const Mat B = mat(wgT, s.d_ff, s.d_model, s.d_model);
  const Mat B2 = mat(wuT, s.d_ff, s.d_model, s.d_model);
  // h (with its lo half h_lo_off columns on), g and u through TMA stores
  p.tma_out = 1;
  const long long hcols = split ? 2LL * s.d_ff : s.d_ff;
  OutMat outs[3];
  outs[0] = OutMat{h, rows, hcols, p.ldh, 0, 32};
  outs[1] = OutMat{g ? g : h, rows, s.d_ff, s.d_ff, 0, 32};
  outs[2] = OutMat{u ? u : h, rows, s.d_ff, s.d_ff, 0, 32};
  if (u32) outs[2] = OutMat{u32, rows, s.d_ff, s.d_ff, 1, 32};
  return gemm_launch(GK_GATED, A, B, &B2, p, st, outs, 3);
}

// Routed rows: out[row_map[r]] = A[r] B with the K range split across CTAs
// (the few routed rows give too few output tiles to fill the GPU); each split
// stores an fp32 partial in `part` (part_rows rows) and a reduction kernel
// sums them in fixed order and scatters the bf16 rows.
constexpr int kSplitKMax = 8;
cudaError_t routed_gemm(const Mat& A, const Mat& B, const Mat* B2, long long rows, int K,
                        const twell_shape& s, int k_split, const int* m_dev, const int* row_map,
                        float* part, long long part_rows, void* out, cudaStream_t st) {
  GemmParams p = base_params((int)rows, s.d_model, K, kBN);
  p.m_dev = m_dev;
  p.k_split = k_split;
  p.c_f32 = 1;
  p.tma_out = 1;
  p.split_k_max = kSplitKMax;
  p.split_rows = (int)part_rows;
  const OutMat o{part, part_rows, s.d_model, s.d_model, 1, 32};
  cudaError_t e = gemm_launch(GK_STORE_KM, A, B, B2, p, st, &o, 1);
  if (e != cudaSuccess) return e;
  return launch_splitk_scatter(part, (int)part_rows, (int)rows, (K + kBK - 1) / kBK, kSplitKMax,
                               m_dev, row_map, s.M, s.d_model, out, st);
}

// out[row_map ? row_map[r] : r] = h[r] Wd (bf16); with split, h = hi + lo and
// the GEMM runs over K = 2f against [Wd ; Wd].
cudaError_t down_gemm(const uint16_t* h, long long rows, const twell_shape& s, const void* wd,
                      bool split, const int* m_dev, const int* row_map, void* out,
                      cudaStream_t st, float* part = nullptr, long long part_rows = 0) {
  const long long K = split ? 2LL * s.d_ff : s.d_ff;
  GemmParams p = base_params((int)rows, s.d_model, (int)K, kBN);
  p.m_dev = m_dev;
  p.row_map = row_map;
  p.c = out;
  p.ldc = s.d_model;
  p.k_split = s.d_ff / kBK;
  const Mat A = mat(h, rows, K, K);
  const Mat B = mat(wd, s.d_ff, s.d_model, s.d_model);  // [K = f][N = d], MN-major
  if (row_map && part)
    return routed_gemm(A, B, &B, rows, (int)K, s, s.d_ff / kBK, m_dev, row_map, part, part_rows,
                       out, st);
  if (!row_map && !m_dev) {
    p.tma_out = 1;
    const OutMat o{out, rows, s.d_model, s.d_model, 0, 32};
    return gemm_launch(GK_STORE_KM, A, B, &B, p, st, &o, 1);
  }
  return gemm_launch(GK_STORE_KM, A, B, &B, p, st);
}

// dd = [du | da] (split: [du | da | du lo | da lo]) from dh = dy Wd^T and g, u.
cudaError_t dgate_gemm(const void* dy_rows, long long rows, const twell_shape& s, const void* wd,
                       const int* m_dev, const uint16_t* g, const uint16_t* u, const float* u32,
                       uint16_t* dd, bool split, float lambda, int pad_rows, cudaStream_t st,
                       int act = kActRelu) {
  GemmParams p = base_params((int)rows, s.d_ff, s.d_model, kBN);
  p.act = act;
  p.m_dev = m_dev;
  p.g_in = g;
  p.u_in = u;
  p.u_f32_in = u32;
  p.ldgu = s.d_ff;
  p.dd = dd;
  p.ld_dd = (split ? 4LL : 2LL) * s.d_ff;
  p.dd_seg = s.d_ff;
  p.dd_split = split ? 1 : 0;
  p.lambda = lambda;
  p.pad_rows = pad_rows;
  const Mat A = mat(dy_rows, rows, s.d_model, s.d_model);
  const Mat B = mat(wd, s.d_ff, s.d_model, s.d_model);  // [N = f][K = d], K-major
  // du, da (and their lo halves) through TMA stores into dd [rows][2f or 4f]
  p.tma_out = 1;
  const OutMat o{dd, rows, p.ld_dd, p.ld_dd, 0, 32};
  return gemm_launch(split ? GK_BWD_GATE_RT : GK_BWD_GATE, A, B, nullptr, p, st, &o, 1);
}

// out[row_map ? row_map[r] : r] = du Wu^T + da Wg^T  (bf16): the GEMM runs over
// K = 2f (or 4f with the lo halves) against [WuT ; WgT (; WuT ; WgT)].
cudaError_t dx_gemm(const uint16_t* dd, long long rows, const twell_shape& s, const void* wgT,
                    const void* wuT, bool split, const int* m_dev, const int* row_map, void* out,
                    cudaStream_t st, float* part = nullptr, long long part_rows = 0) {
  const long long K = (split ? 4LL : 2LL) * s.d_ff;
  GemmParams p = base_params((int)rows, s.d_model, (int)K, kBN);
  p.m_dev = m_dev;
  p.row_map = row_map;
  p.c = out;
  p.ldc = s.d_model;
  p.k_split = s.d_ff / kBK;
  const Mat A = mat(dd, rows, K, K);
  const Mat B = mat(wuT, s.d_ff, s.d_model, s.d_model);   // [K][N], MN-major
  const Mat B2 = mat(wgT, s.d_ff, s.d_model, s.d_model);
  if (row_map && part)
    return routed_gemm(A, B, &B2, rows, (int)K, s, s.d_ff / kBK, m_dev, row_map, part, part_rows,
                       out, st);
  if (!row_map && !m_dev) {
    p.tma_out = 1;
    const OutMat o{out, rows, s.d_model, s.d_model, 0, 32};
    return gemm_launch(GK_STORE_KM, A, B, &B2, p, st, &o, 1);
  }
  return gemm_launch(GK_STORE_KM, A, B, &B2, p, st);
}

// C[f][d] (+)= A^T B with A = [K][f] (leading dim lda) and B = [K][d], K from k_dev or K.
// With lo_off > 0, A is a hi + lo pair (lo at column offset lo_off of the same
// rows) and C (+)= (A_hi + A_lo)^T B in one launch.
cudaError_t dw_gemm(const uint16_t* a, long long lda, const void* b, long long K,
                    const twell_shape& s, const int* k_dev, float* c, int accumulate,
                    cudaStream_t st, long long lo_off = 0) {
  GemmParams p = base_params(s.d_ff, s.d_model, (int)K, kBN);
  p.k_dev = k_dev;
  p.c = c;
  p.ldc = s.d_model;
  p.c_f32 = 1;
  p.accumulate = accumulate;
  p.a_seg_off = (int)lo_off;
  const Mat A = mat(a, K, lo_off > 0 ? lo_off + s.d_ff : s.d_ff, lda);
  const Mat B = mat(b, K, s.d_model, s.d_model);
  p.tma_out = 1;  // fp32 boxes: TMA store, or TMA reduce-add when accumulating
  const OutMat o{c, s.d_ff, s.d_model, s.d_model, 1, 32};
  return gemm_launch(GK_STORE_MM, A, B, nullptr, p, st, &o, 1);
}

}  // namespace

// ============================================================== entry points
extern "C" {

const char* twell_status_string(int32_t status) {
  switch (status) {
    case TWELL_OK: return "ok";
    case TWELL_ERR_INVALID_ARG: return "invalid argument";
    case TWELL_ERR_UNSUPPORTED: return "unsupported shape";
    case TWELL_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case TWELL_ERR_CAPACITY: return "packed tile overflow without a route";
    case TWELL_ERR_CUDA: return "CUDA error";
    case TWELL_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case TWELL_ERR_WORKSPACE: return "workspace missing or too small";
    case TWELL_ERR_INDEX: return "index out of range (checked build)";
  }
  return "unknown status";
}

int32_t twell_num_sms(void) { return num_sms(); }

uint64_t twell_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

twell_status twell_profile_begin(const char* kernel) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (auto& r : g_prof_records) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_prof_records.clear();
  g_prof_filter = kernel ? kernel : "";
  g_prof_on.store(!g_prof_filter.empty());
  return TWELL_OK;
}

int32_t twell_profile_end(void) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on.store(false);
  std::map<std::string, ProfEntry> agg;
  int bad = 0;
  for (auto& r : g_prof_records) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      ++bad;
    ProfEntry& e = agg[r.name];
    e.name = r.name;
    e.launches += 1;
    e.total_ms += ms;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_prof_records.clear();
  g_prof_report.clear();
  for (auto& kv : agg) g_prof_report.push_back(kv.second);
  return bad ? -1 : (int32_t)g_prof_report.size();
}

twell_status twell_profile_entry(int32_t i, const char** name, int32_t* launches,
                                 double* total_ms) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (i < 0 || i >= (int32_t)g_prof_report.size() || !name || !launches || !total_ms)
    return TWELL_ERR_INVALID_ARG;
  *name = g_prof_report[i].name.c_str();
  *launches = g_prof_report[i].launches;
  *total_ms = g_prof_report[i].total_ms;
  return TWELL_OK;
}

twell_status twell_get_device_status(void* stream, int32_t* out) {
  if (!out) return TWELL_ERR_INVALID_ARG;
  int* p = device_status_ptr();
  if (!p) return TWELL_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return TWELL_ERR_CUDA;
  *out = v;
  return TWELL_OK;
}

twell_status twell_pack(const void* x, const void* wgT, const twell_shape* shape,
                        const twell_tiles* out, void* stream) {
  NvtxRange nvtx("twell_pack");
  twell_status st = check_shape(shape, true);
  if (st != TWELL_OK) return st;
  if ((st = check_ptrs({x, wgT})) != TWELL_OK) return st;
  if ((st = check_tiles(out)) != TWELL_OK) return st;
  const twell_shape& s = *shape;
  if (s.M == 0) return TWELL_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(out->row_nnz, 0, sizeof(int32_t) * (size_t)s.M, cs);
  if (e != cudaSuccess) return TWELL_ERR_CUDA;
  // a handful of tokens: neurons on the MMA's M dimension (gate_smallm.cu)
  if (gate_pack_smallm_fits(s.M, s.d_model, s.d_ff, s.tile_n))
    return cuda_status(launch_gate_pack_smallm(x, wgT, s.M, s.d_model, s.d_ff, s.tile_n,
                                               s.tile_cap, *out, cs));
  GemmParams p = base_params(s.M, s.d_ff, s.d_model, kBN);
  p.val = reinterpret_cast<uint16_t*>(out->val);
  p.idx = out->idx;
  p.cnt = out->cnt;
  p.row_nnz = out->row_nnz;
  p.T = s.d_ff / s.tile_n;
  p.cap = s.tile_cap;
  p.tile_n = s.tile_n;
  // Small batches give fewer output tiles than half the SMs: split K over the
  // blocks of a cluster (up to 8, within one wave, each split at least 8 K
  // blocks so streaming Wg still outweighs summing the partials), so more SMs
  // stream Wg; the leader block sums the partials in rank order.
  const long long tiles = (long long)((s.M + kBM - 1) / kBM) * p.n_tiles;
  const int num_kb = (s.d_model + kBK - 1) / kBK;
  for (int next = 2; next <= 8; next *= 2) {
    if (tiles * next > num_sms() || next * 8 > num_kb) break;
    p.cluster_k = next;
  }
  const Mat A = mat(x, s.M, s.d_model, s.d_model);
  const Mat B = mat(wgT, s.d_ff, s.d_model, s.d_model);
  return cuda_status(gemm_launch(GK_PACK, A, B, nullptr, p, cs));
}

twell_status twell_pack_dense(const void* a, int32_t a_dtype, const twell_shape* shape,
                              const twell_tiles* out, void* stream) {
  NvtxRange nvtx("twell_pack_dense");
  twell_status st = check_shape(shape, true);
  if (st != TWELL_OK) return st;
  if (a_dtype != 0 && a_dtype != 1) return TWELL_ERR_INVALID_ARG;
  if ((st = check_ptrs({a})) != TWELL_OK) return st;
  if ((st = check_tiles(out)) != TWELL_OK) return st;
  const twell_shape& s = *shape;
  return cuda_status(launch_pack_dense(a, a_dtype, s.M, s.d_ff, s.tile_n, s.tile_cap, *out,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

twell_status hybrid_route(const twell_tiles* in, const twell_shape* shape, const twell_hybrid* out,
                          void* stream) {
  NvtxRange nvtx("hybrid_route");
  twell_status st = check_shape(shape, true);
  if (st != TWELL_OK) return st;
  if ((st = check_tiles(in)) != TWELL_OK) return st;
  if ((st = check_route(out)) != TWELL_OK) return st;
  const twell_shape& s = *shape;
  // the routing flags live in dense_rows until the stable list overwrites them
  return cuda_status(launch_route(*in, s.M, s.d_ff, s.tile_n, s.tile_cap, *out, out->dense_rows,
                                  out->dense_cap < s.M ? out->dense_cap : s.M,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

size_t twell_workspace_bytes_capped(const twell_shape* shape, int32_t ell_width,
                                    int32_t dense_cap, int32_t training) {
  if (check_shape(shape, true) != TWELL_OK || ell_width < 0 || dense_cap < 0) return 0;
  return carve_sparse(nullptr, *shape, ell_width, dense_cap, training ? 1 : 0).bytes;
}

size_t twell_workspace_bytes(const twell_shape* shape, int32_t ell_width, int32_t training) {
  if (check_shape(shape, true) != TWELL_OK) return 0;
  return twell_workspace_bytes_capped(shape, ell_width, shape->M, training);
}

int32_t twell_set_split_gathers(int32_t enable) {
  return g_split_gathers.exchange(enable ? 1 : 0) ? 1 : 0;
}

int32_t twell_set_pair_gemm(int32_t enable) {
  return g_pair_gemm.exchange(enable ? 1 : 0) ? 1 : 0;
}

size_t twell_tiles_workspace_bytes(const twell_shape* shape) {
  if (check_shape(shape, true) != TWELL_OK) return 0;
  return carve_tiles(nullptr, *shape).bytes;
}

twell_status twell_ffn_fwd(const void* x, const void* wgT, const void* wuT, const void* wd,
                           const twell_shape* shape, const twell_tiles* tiles,
                           const twell_hybrid* route, void* y, void* ws, size_t ws_bytes,
                           void* stream) {
  NvtxRange nvtx("twell_ffn_fwd");
  twell_status st = check_shape(shape, true);
  if (st != TWELL_OK) return st;
  if ((tiles == nullptr) == (route == nullptr)) return TWELL_ERR_INVALID_ARG;
  if ((st = check_ptrs({x, wuT, wd, y})) != TWELL_OK) return st;
  const twell_shape& s = *shape;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (tiles) {
    if ((st = check_tiles(tiles)) != TWELL_OK) return st;
    TilesWs w{};
    if (ws && s.d_model > 1024) {  // wide rows: the split gathers, h in the workspace
      if (ws_bytes < carve_tiles(nullptr, s).bytes) return TWELL_ERR_WORKSPACE;
      if (!aligned16(ws)) return TWELL_ERR_ALIGNMENT;
      w = carve_tiles(ws, s);
    }
    if (s.M == 0) return TWELL_OK;
    return cuda_status(launch_sparse_fwd(x, wuT, wd, s.M, s.d_model, s.d_ff, tiles, s.tile_n,
                                         s.tile_cap, nullptr, y, w.part, w.hbuf, cs));
  }
  if ((st = check_route(route)) != TWELL_OK) return st;
  if ((st = check_ptrs({wgT})) != TWELL_OK) return st;
  const SparseWs need = carve_sparse(nullptr, s, route->ell_width, route->dense_cap, 0);
  if (!ws || ws_bytes < need.bytes) return TWELL_ERR_WORKSPACE;
  if (!aligned16(ws)) return TWELL_ERR_ALIGNMENT;
  if (s.M == 0) return TWELL_OK;
  const SparseWs w = carve_sparse(ws, s, route->ell_width, route->dense_cap, 0);
  const long long Mr = w.Mr;
  // w.part carries y between L2-sized passes; the routed rows' split-K GEMM
  // reuses it afterwards on the same stream
  cudaError_t e = launch_sparse_fwd(x, wuT, wd, s.M, s.d_model, s.d_ff, nullptr, s.tile_n,
                                    s.tile_cap, route, y, w.part, w.hbuf, cs);
  if (Mr == 0) return cuda_status(e);  // no routed-row capacity: nothing else to run
  if (e == cudaSuccess)
    e = launch_gather_rows(x, s.M, s.d_model, route->dense_rows, route->n_dense, w.xr, (int)Mr, cs);
  if (e == cudaSuccess)
    e = gated_gemm(w.xr, Mr, s, wgT, wuT, route->n_dense, w.hr, true, nullptr, nullptr,
                   nullptr, 0, cs);
  if (e == cudaSuccess)
    e = down_gemm(w.hr, Mr, s, wd, true, route->n_dense, route->dense_rows, y, cs, w.part, w.Mp);
  return cuda_status(e);
}

twell_status twell_ffn_bwd(const void* x, const void* wgT, const void* wuT, const void* wd,
                           const void* dy, const twell_shape* shape, const twell_hybrid* route,
                           float l1_coeff, void* dx, float* dwgT, float* dwuT, float* dwd,
                           void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("twell_ffn_bwd");
  twell_status st = check_shape(shape, true);
  if (st != TWELL_OK) return st;
  if ((st = check_ptrs({x, wgT, wuT, wd, dy, dx, dwgT, dwuT, dwd})) != TWELL_OK) return st;
  if ((st = check_route(route)) != TWELL_OK) return st;
  const twell_shape& s = *shape;
  const SparseWs need = carve_sparse(nullptr, s, route->ell_width, route->dense_cap, 1);
  if (!ws || ws_bytes < need.bytes) return TWELL_ERR_WORKSPACE;
  if (!aligned16(ws)) return TWELL_ERR_ALIGNMENT;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const SparseWs w = carve_sparse(ws, s, route->ell_width, route->dense_cap, 1);
  const long long Mr = w.Mr;
  const long long f = s.d_ff;
  cudaError_t e = launch_csc_build(*route, s.M, s.d_ff, w.mask_off, w.csc_ptr, w.csc_row,
                                   w.slot_pos, cs);
  if (e == cudaSuccess)
    e = launch_sparse_bwd_rows(x, dy, wgT, wuT, wd, s.M, s.d_model, s.d_ff, *route, w.slot_pos,
                               l1_coeff, w.csc_vals, dx, w.part, w.hbuf, cs);
  if (e == cudaSuccess)
    e = launch_sparse_bwd_neurons(x, dy, s.M, s.d_model, s.d_ff, w.csc_ptr, w.csc_row, w.csc_vals,
                                  dwgT, dwuT, dwd, cs);
  if (s.M == 0 || Mr == 0) return cuda_status(e);
  // routed rows: dense tensor-core backward, accumulated into the same dW
  const int* nd = route->n_dense;
  if (e == cudaSuccess)
    e = launch_gather_rows(x, s.M, s.d_model, route->dense_rows, nd, w.xr, (int)Mr, cs);
  if (e == cudaSuccess)
    e = launch_gather_rows(dy, s.M, s.d_model, route->dense_rows, nd, w.dyr, (int)Mr, cs);
  if (e == cudaSuccess)
    e = gated_gemm(w.xr, Mr, s, wgT, wuT, nd, w.hr, true, w.gr, nullptr, w.ur, 1, cs);
  if (e == cudaSuccess)
    e = dgate_gemm(w.dyr, Mr, s, wd, nd, w.gr, nullptr, w.ur, w.ddr, true, l1_coeff, 1, cs);
  if (e == cudaSuccess)
    e = dx_gemm(w.ddr, Mr, s, wgT, wuT, true, nd, route->dense_rows, dx, cs, w.part, w.Mp);
  // dW += (hi + lo)^T B, both halves in one launch per weight
  if (e == cudaSuccess) e = dw_gemm(w.hr, 2 * f, w.dyr, Mr, s, nd, dwd, 1, cs, f);
  if (e == cudaSuccess) e = dw_gemm(w.ddr, 4 * f, w.xr, Mr, s, nd, dwuT, 1, cs, 2 * f);
  if (e == cudaSuccess) e = dw_gemm(w.ddr + f, 4 * f, w.xr, Mr, s, nd, dwgT, 1, cs, 2 * f);
  return cuda_status(e);
}

size_t twell_dense_workspace_bytes(const twell_shape* shape, int32_t training) {
  if (check_shape(shape, false) != TWELL_OK) return 0;
  return carve_dense(nullptr, *shape, training ? 1 : 0).bytes;
}

twell_status twell_dense_ffn_fwd_act(const void* x, const void* wgT, const void* wuT,
                                     const void* wd, const twell_shape* shape,
                                     int32_t activation, void* y, int32_t training, void* ws,
                                     size_t ws_bytes, void* stream) {
  NvtxRange nvtx("twell_dense_ffn_fwd_act");
  twell_status st = check_shape(shape, false);
  if (st != TWELL_OK) return st;
  if (activation != TWELL_ACT_RELU && activation != TWELL_ACT_SILU) return TWELL_ERR_INVALID_ARG;
  if ((st = check_ptrs({x, wgT, wuT, wd, y})) != TWELL_OK) return st;
  const twell_shape& s = *shape;
  if (!ws || ws_bytes < carve_dense(nullptr, s, training ? 1 : 0).bytes) return TWELL_ERR_WORKSPACE;
  if (!aligned16(ws)) return TWELL_ERR_ALIGNMENT;
  if (s.M == 0) return TWELL_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const DenseWs w = carve_dense(ws, s, training ? 1 : 0);
  cudaError_t e = gated_gemm(x, s.M, s, wgT, wuT, nullptr, w.h, false, training ? w.g : nullptr,
                             training ? w.u : nullptr, nullptr, 0, cs,
                             activation == TWELL_ACT_SILU ? kActSilu : kActRelu);
  if (e == cudaSuccess) e = down_gemm(w.h, s.M, s, wd, false, nullptr, nullptr, y, cs);
  return cuda_status(e);
}

twell_status twell_dense_ffn_fwd(const void* x, const void* wgT, const void* wuT, const void* wd,
                                 const twell_shape* shape, void* y, int32_t training, void* ws,
                                 size_t ws_bytes, void* stream) {
  return twell_dense_ffn_fwd_act(x, wgT, wuT, wd, shape, TWELL_ACT_RELU, y, training, ws,
                                 ws_bytes, stream);
}

twell_status twell_dense_ffn_bwd_act(const void* x, const void* wgT, const void* wuT,
                                     const void* wd, const void* dy, const twell_shape* shape,
                                     int32_t activation, float l1_coeff, void* dx, float* dwgT,
                                     float* dwuT, float* dwd, void* ws, size_t ws_bytes,
                                     void* stream) {
  NvtxRange nvtx("twell_dense_ffn_bwd_act");
  twell_status st = check_shape(shape, false);
  if (st != TWELL_OK) return st;
  if (activation != TWELL_ACT_RELU && activation != TWELL_ACT_SILU) return TWELL_ERR_INVALID_ARG;
  if (activation == TWELL_ACT_SILU && l1_coeff != 0.0f) return TWELL_ERR_INVALID_ARG;
  if ((st = check_ptrs({x, wgT, wuT, wd, dy, dx, dwgT, dwuT, dwd})) != TWELL_OK) return st;
  const twell_shape& s = *shape;
  if (!ws || ws_bytes < carve_dense(nullptr, s, 1).bytes) return TWELL_ERR_WORKSPACE;
  if (!aligned16(ws)) return TWELL_ERR_ALIGNMENT;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const long long f = s.d_ff;
  if (s.M == 0) {
    cudaError_t e = cudaMemsetAsync(dwgT, 0, sizeof(float) * f * s.d_model, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dwuT, 0, sizeof(float) * f * s.d_model, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dwd, 0, sizeof(float) * f * s.d_model, cs);
    return cuda_status(e);
  }
  const DenseWs w = carve_dense(ws, s, 1);
  cudaError_t e = dgate_gemm(dy, s.M, s, wd, nullptr, w.g, w.u, nullptr, w.dd, false, l1_coeff, 0,
                             cs, activation == TWELL_ACT_SILU ? kActSilu : kActRelu);
  if (e == cudaSuccess) e = dx_gemm(w.dd, s.M, s, wgT, wuT, false, nullptr, nullptr, dx, cs);
  if (e == cudaSuccess) e = dw_gemm(w.h, f, dy, s.M, s, nullptr, dwd, 0, cs);
  if (e == cudaSuccess) e = dw_gemm(w.dd, 2 * f, x, s.M, s, nullptr, dwuT, 0, cs);
  if (e == cudaSuccess) e = dw_gemm(w.dd + f, 2 * f, x, s.M, s, nullptr, dwgT, 0, cs);
  return cuda_status(e);
}

twell_status twell_dense_ffn_bwd(const void* x, const void* wgT, const void* wuT, const void* wd,
                                 const void* dy, const twell_shape* shape, float l1_coeff,
                                 void* dx, float* dwgT, float* dwuT, float* dwd, void* ws,
                                 size_t ws_bytes, void* stream) {
  return twell_dense_ffn_bwd_act(x, wgT, wuT, wd, dy, shape, TWELL_ACT_RELU, l1_coeff, dx, dwgT,
                                 dwuT, dwd, ws, ws_bytes, stream);
}

twell_status twell_gemm_bf16(const void* A, const void* B, void* C, int32_t M, int32_t N,
                             int32_t K, int32_t a_mn_major, int32_t b_mn_major, int32_t c_dtype,
                             int32_t accumulate, void* stream) {
  NvtxRange nvtx("twell_gemm_bf16");
  if (M < 0 || N <= 0 || K <= 0) return TWELL_ERR_INVALID_ARG;
  if (c_dtype != 0 && c_dtype != 1) return TWELL_ERR_INVALID_ARG;
  if (accumulate && c_dtype != 1) return TWELL_ERR_INVALID_ARG;
  twell_status st = check_ptrs({A, B, C});
  if (st != TWELL_OK) return st;
  if (K % 8 != 0 || N % 8 != 0) return TWELL_ERR_UNSUPPORTED;
  if (a_mn_major && M % 8 != 0) return TWELL_ERR_UNSUPPORTED;
  if (M == 0) return TWELL_OK;
  GemmParams p = base_params(M, N, K, kBN);
  p.c = C;
  p.ldc = N;
  p.c_f32 = c_dtype;
  p.accumulate = accumulate;
  const Mat a = a_mn_major ? mat(A, K, M, M) : mat(A, M, K, K);
  const Mat b = b_mn_major ? mat(B, K, N, N) : mat(B, N, K, K);
  const GemmKind kind = a_mn_major ? (b_mn_major ? GK_STORE_MM : GK_STORE_MK)
                                   : (b_mn_major ? GK_STORE_KM : GK_STORE_KK);
  p.tma_out = 1;
  const OutMat o{C, M, N, N, c_dtype, 32};
  return cuda_status(
      gemm_launch(kind, a, b, nullptr, p, reinterpret_cast<cudaStream_t>(stream), &o, 1));
}

}  // extern "C"

// ============================================== allocation-free hybrid forward
// Some callers cannot allocate device memory at the point where they run the
// FFN: code inside a CUDA graph capture or another framework's scheduler
// where cudaMalloc would break the capture or synchronise the device, plugins
// hosted by a runtime that owns every allocation, and deployments that fix
// their memory footprint up front.  twell_ffn_fwd_noalloc serves them by
// taking the routed-row scratch of the hybrid forward from a fixed array in
// the library's own device image instead of a caller workspace.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array for the current device.  Host code
// sees g_noalloc_scratch only as a host-side stand-in, so the address must
// come from cudaGetSymbolAddress, once per device, with that device current.
void* noalloc_scratch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" twell_status twell_ffn_fwd_noalloc(const void* x, const void* wgT, const void* wuT,
                                              const void* wd, const twell_shape* shape,
                                              const twell_hybrid* route, void* y, void* stream) {
  twell_status st = check_shape(shape, true);
  if (st != TWELL_OK) return st;
  if ((st = check_ptrs({x, wgT, wuT, wd, y})) != TWELL_OK) return st;
  if ((st = check_route(route)) != TWELL_OK) return st;
  const size_t need = carve_sparse(nullptr, *shape, route->ell_width, route->dense_cap, 0).bytes;
  if (need > kNoAllocScratchBytes) return TWELL_ERR_WORKSPACE;
  void* ws = noalloc_scratch();
  if (!ws) return TWELL_ERR_CUDA;
  return twell_ffn_fwd(x, wgT, wuT, wd, shape, nullptr, route, y, ws, kNoAllocScratchBytes, stream);
}
