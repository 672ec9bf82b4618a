// twell_oracle.cpp -- CPU oracle for the activation-sparse gated FFN (TwELL).
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
// statement of what the GPU path computes.  Only the test-suite, the smoke
// check and the CPU-baseline leg of the benchmark may load it; the library
// under activation_sparse_gated_tcgen05_gb300/ never does, and the two share
// no code, header, table or helper.
//
// Every floating-point quantity is computed in IEEE double (fp64), one
// output element at a time, with the loops in the order of the definitions.
// Inputs arrive already decoded to double (bf16 -> double is exact).
//
// Sources (three web pages on TwELL; page 2 is the technical one):
//   [P2-problem]  page 2 "Sakana AI and NVIDIA introduce TwELL with CUDA
//                 kernels ...", section "¿Cuál es el problema que TwELL
//                 resuelve?" -- gated feed-forward block; ReLU makes ~99.5 %
//                 of hidden activations exactly zero; classic ELLPACK needs a
//                 separate dense->sparse conversion kernel.
//   [P2-twell]    same page, section "¿Qué hace distinto a TwELL frente a ELL
//                 clásico?" -- activation columns are cut into tiles of the
//                 matmul's tile width T_n and nonzeros are packed locally
//                 inside each tile; inference reads the packed activations
//                 and does the up and down projections together; training
//                 routes rows with too many nonzeros to a dense backup.
//   [P2-recipe]   same page, section "Receta de entrenamiento" -- the gate
//                 activation is ReLU (not SiLU) and an L1 term with
//                 coefficient 2e-5 is added on the hidden activations.
//
// Readings where the pages are silent (each is listed in the design notes):
//   * "hidden activation" under L1 = the gate output g = ReLU(x Wg); the
//     penalty is unnormalised, lambda * sum(g), so d(loss)/dg = lambda.
//   * g is stored as bf16 (round to nearest even) in the packed format; a
//     column is live iff that stored value is > 0; ReLU'(0) = 0; NaN -> dead.
//   * inside a tile, live columns are kept in ascending column order; cnt
//     holds the true count; only the first C are stored.
//   * hybrid routing: a row goes to the dense backup iff some tile holds
//     more than C live columns or the row holds more than W in total; the
//     dense-row list is ascending; ELL rows keep global columns ascending.
//   * the backward pass is the chain rule of the forward definition.
//
// Weight layout (host arrays, row-major):
//   wgT[j][k] = Wg[k][j], wuT[j][k] = Wu[k][j]   (shape d_ff x d_model)
//   wd[j][k]  = Wd[j][k]                          (shape d_ff x d_model)
// so the forward is  a = x Wg,  g = ReLU(a),  u = x Wu,  h = g * u,  y = h Wd.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

int g_threads = 1;

// Run fn(lo, hi) over [0, n) split into g_threads contiguous chunks.  Each
// output element is still produced by exactly one thread with the same loop
// order, so the result does not depend on the thread count.
template <class F>
void parallel_for(int64_t n, F fn) {
  int nt = g_threads < 1 ? 1 : g_threads;
  if (nt == 1 || n < 2) {
    fn((int64_t)0, n);
    return;
  }
  if ((int64_t)nt > n) nt = (int)n;
  std::vector<std::thread> pool;
  int64_t step = (n + nt - 1) / nt;
  for (int i = 0; i < nt; ++i) {
    int64_t lo = i * step, hi = lo + step < n ? lo + step : n;
    if (lo >= hi) break;
    pool.emplace_back([=] { fn(lo, hi); });
  }
  for (auto& t : pool) t.join();
}

// bf16 <-> double.  bf16 is the top half of an IEEE binary32.
double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Round a double straight to the nearest bf16 value, ties to even.  bf16 has
// 8 significant bits and binary32's exponent range: normal numbers from
// 2^-126, subnormal spacing 2^-133, largest finite (2 - 2^-7) * 2^127.
uint16_t double_to_bf16(double v) {
  if (std::isnan(v)) return 0x7FC0;
  uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  if (a == 0.0) return sign;
  double q;  // spacing of bf16 values around a
  if (a >= std::ldexp(1.0, -126)) {
    int e;
    std::frexp(a, &e);          // a = m * 2^e with m in [0.5, 1)
    q = std::ldexp(1.0, e - 8);  // 8 significant bits
  } else {
    q = std::ldexp(1.0, -133);
  }
  double r = std::nearbyint(a / q) * q;  // default mode: ties to even
  if (r >= std::ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);  // inf
  float rf = (float)r;  // exact: r has at most 8 significant bits
  uint32_t u;
  std::memcpy(&u, &rf, 4);
  return (uint16_t)(sign | (u >> 16));
}

// The gate value the packed format stores for pre-activation a:
// ReLU, then bf16.  Returns the bf16 bits; live iff the result is > 0.
uint16_t gate_bf16(double a) { return double_to_bf16(a > 0.0 ? a : 0.0); }

double dot(const double* a, const double* b, int64_t n) {
  double s = 0.0;
  for (int64_t k = 0; k < n; ++k) s += a[k] * b[k];
  return s;
}

}  // namespace

extern "C" {

void orc_set_threads(int n) { g_threads = n < 1 ? 1 : n; }
int orc_get_threads(void) { return g_threads; }

// ---- bf16 helpers exposed for the pins -------------------------------------
void orc_double_to_bf16(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(v[i]);
}

// ---- gate pre-activation  a = x Wg   [P2-problem] --------------------------
// x [M][d], wgT [f][d]  ->  a [M][f]
void orc_gate_preact(const double* x, const double* wgT, int64_t M, int64_t d,
                     int64_t f, double* a) {
  parallel_for(M, [&](int64_t lo, int64_t hi) {
    for (int64_t m = lo; m < hi; ++m)
      for (int64_t j = 0; j < f; ++j) a[m * f + j] = dot(x + m * d, wgT + j * d, d);
  });
}

// ---- TwELL pack  [P2-twell] -------------------------------------------------
// a [M][f] (any precision, given as double).  Columns are cut into T = f/Tn
// tiles of width Tn.  For each (row m, tile t): cnt[m][t] = number of live
// columns (bf16(ReLU(a)) > 0); the first min(cnt, C) live columns in
// ascending order go to slots 0.. of val[m][t][.] (bf16 bits) and
// idx[m][t][.] (column inside the tile).  row_nnz[m] = sum over t of cnt.
// Slots at or past min(cnt, C) are left untouched.
void orc_twell_pack(const double* a, int64_t M, int64_t f, int Tn, int C,
                    uint16_t* val, uint8_t* idx, uint8_t* cnt, int32_t* row_nnz) {
  int64_t T = f / Tn;
  for (int64_t m = 0; m < M; ++m) {
    int32_t nnz = 0;
    for (int64_t t = 0; t < T; ++t) {
      int c = 0;
      for (int l = 0; l < Tn; ++l) {
        uint16_t g = gate_bf16(a[m * f + t * Tn + l]);
        bool live = (g & 0x8000) == 0 && (g & 0x7FFF) != 0;
        if (!live) continue;
        if (c < C) {
          val[(m * T + t) * C + c] = g;
          idx[(m * T + t) * C + c] = (uint8_t)l;
        }
        ++c;
      }
      cnt[m * T + t] = (uint8_t)c;
      nnz += c;
    }
    row_nnz[m] = nnz;
  }
}

// Inverse of the pack for tiles that did not overflow: g [M][f] as double.
void orc_twell_unpack(const uint16_t* val, const uint8_t* idx, const uint8_t* cnt,
                      int64_t M, int64_t f, int Tn, int C, double* g) {
  int64_t T = f / Tn;
  for (int64_t i = 0; i < M * f; ++i) g[i] = 0.0;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t t = 0; t < T; ++t) {
      int n = cnt[m * T + t] < C ? cnt[m * T + t] : C;
      for (int s = 0; s < n; ++s)
        g[m * f + t * Tn + idx[(m * T + t) * C + s]] = bf16_to_double(val[(m * T + t) * C + s]);
    }
}

// ---- hybrid ELL / dense-backup routing  [P2-twell] -------------------------
// A row is routed to the dense backup iff any of its tiles overflowed
// (cnt > C) or row_nnz > W.  Routed rows get ell_nnz = 0 and are listed in
// ascending order in dense_rows[0 .. *n_dense).  Every other row copies its
// live entries, tile by tile and slot by slot, into ell_val[m][0..]
// (bf16 bits) and ell_col[m][0..] (global column t*Tn + idx).
void orc_hybrid_route(const uint16_t* val, const uint8_t* idx, const uint8_t* cnt,
                      const int32_t* row_nnz, int64_t M, int64_t f, int Tn, int C,
                      int32_t W, uint16_t* ell_val, uint16_t* ell_col, int32_t* ell_nnz,
                      int32_t* dense_rows, int32_t* n_dense) {
  int64_t T = f / Tn;
  int32_t nd = 0;
  for (int64_t m = 0; m < M; ++m) {
    bool overflow = false;
    for (int64_t t = 0; t < T; ++t)
      if (cnt[m * T + t] > C) overflow = true;
    if (overflow || row_nnz[m] > W) {
      dense_rows[nd++] = (int32_t)m;
      ell_nnz[m] = 0;
      continue;
    }
    int32_t s = 0;
    for (int64_t t = 0; t < T; ++t)
      for (int c = 0; c < cnt[m * T + t]; ++c) {
        ell_val[m * W + s] = val[(m * T + t) * C + c];
        ell_col[m * W + s] = (uint16_t)(t * Tn + idx[(m * T + t) * C + c]);
        ++s;
      }
    ell_nnz[m] = s;
  }
  *n_dense = nd;
}

// ---- dense gated FFN forward  [P2-problem], [P2-recipe] ---------------------
// y[r][.] for the rows listed in rows[0..nrows):
//   a_j = x_m . Wg[:,j];  g_j = ReLU(a_j) (then bf16 if round_g);
//   u_j = x_m . Wu[:,j];  h_j = g_j u_j;  y_m = sum_j h_j Wd[j,:]
void orc_ffn_fwd_dense(const double* x, const double* wgT, const double* wuT,
                       const double* wd, int64_t d, int64_t f, int round_g,
                       const int64_t* rows, int64_t nrows, double* y) {
  parallel_for(nrows, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      const double* xm = x + rows[r] * d;
      double* yr = y + r * d;
      for (int64_t k = 0; k < d; ++k) yr[k] = 0.0;
      for (int64_t j = 0; j < f; ++j) {
        double a = dot(xm, wgT + j * d, d);
        double g = a > 0.0 ? a : 0.0;
        if (round_g) g = bf16_to_double(double_to_bf16(g));
        double u = dot(xm, wuT + j * d, d);
        double h = g * u;
        for (int64_t k = 0; k < d; ++k) yr[k] += h * wd[j * d + k];
      }
    }
  });
}

// ---- sparse forward from the packed format  [P2-twell] ----------------------
// Same y, visiting only the stored live entries of each row.  With a hybrid
// route the caller passes ELL rows (ell_* != NULL); otherwise TwELL tiles.
void orc_ffn_fwd_twell(const double* x, const double* wuT, const double* wd, int64_t d,
                       int64_t f, int Tn, int C, const uint16_t* val, const uint8_t* idx,
                       const uint8_t* cnt, const int64_t* rows, int64_t nrows, double* y) {
  int64_t T = f / Tn;
  parallel_for(nrows, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      int64_t m = rows[r];
      const double* xm = x + m * d;
      double* yr = y + r * d;
      for (int64_t k = 0; k < d; ++k) yr[k] = 0.0;
      for (int64_t t = 0; t < T; ++t) {
        int n = cnt[m * T + t] < C ? cnt[m * T + t] : C;
        for (int s = 0; s < n; ++s) {
          int64_t j = t * Tn + idx[(m * T + t) * C + s];
          double g = bf16_to_double(val[(m * T + t) * C + s]);
          double u = dot(xm, wuT + j * d, d);
          double h = g * u;
          for (int64_t k = 0; k < d; ++k) yr[k] += h * wd[j * d + k];
        }
      }
    }
  });
}

void orc_ffn_fwd_ell(const double* x, const double* wuT, const double* wd, int64_t d,
                     int32_t W, const uint16_t* ell_val, const uint16_t* ell_col,
                     const int32_t* ell_nnz, const int64_t* rows, int64_t nrows, double* y) {
  parallel_for(nrows, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      int64_t m = rows[r];
      const double* xm = x + m * d;
      double* yr = y + r * d;
      for (int64_t k = 0; k < d; ++k) yr[k] = 0.0;
      for (int32_t s = 0; s < ell_nnz[m]; ++s) {
        int64_t j = ell_col[m * W + s];
        double g = bf16_to_double(ell_val[m * W + s]);
        double u = dot(xm, wuT + j * d, d);
        double h = g * u;
        for (int64_t k = 0; k < d; ++k) yr[k] += h * wd[j * d + k];
      }
    }
  });
}

// ---- dense backward, whole batch  [P2-recipe] + chain rule -----------------
// Loss = sum(y * dy) + lambda * sum(g).  With g (bf16-rounded if round_g) and
// the live mask 1[g > 0]:
//   dh = dy Wd^T          dWd = h^T dy
//   du = dh * g           dWu = x^T du      (stored transposed: dwuT = du^T x)
//   da = (dh * u + lambda) * 1[g > 0]
//                         dWg = x^T da      (dwgT = da^T x)
//   dx = du Wu^T + da Wg^T
// l1_out = lambda * sum(g).  Small shapes only: it holds [M][f] arrays.
void orc_ffn_bwd_dense(const double* x, const double* wgT, const double* wuT,
                       const double* wd, const double* dy, int64_t M, int64_t d,
                       int64_t f, double lambda, int round_g, double* dx, double* dwgT,
                       double* dwuT, double* dwd, double* l1_out) {
  std::vector<double> g(M * f), u(M * f), h(M * f), du(M * f), da(M * f);
  parallel_for(M, [&](int64_t lo, int64_t hi) {
    for (int64_t m = lo; m < hi; ++m)
      for (int64_t j = 0; j < f; ++j) {
        double a = dot(x + m * d, wgT + j * d, d);
        double gj = a > 0.0 ? a : 0.0;
        if (round_g) gj = bf16_to_double(double_to_bf16(gj));
        double uj = dot(x + m * d, wuT + j * d, d);
        double dh = dot(dy + m * d, wd + j * d, d);
        g[m * f + j] = gj;
        u[m * f + j] = uj;
        h[m * f + j] = gj * uj;
        du[m * f + j] = dh * gj;
        da[m * f + j] = gj > 0.0 ? dh * uj + lambda : 0.0;
      }
  });
  double l1 = 0.0;
  for (int64_t i = 0; i < M * f; ++i) l1 += g[i];
  *l1_out = lambda * l1;
  parallel_for(f, [&](int64_t lo, int64_t hi) {
    for (int64_t j = lo; j < hi; ++j)
      for (int64_t k = 0; k < d; ++k) {
        double sd = 0.0, su = 0.0, sg = 0.0;
        for (int64_t m = 0; m < M; ++m) {
          sd += h[m * f + j] * dy[m * d + k];
          su += du[m * f + j] * x[m * d + k];
          sg += da[m * f + j] * x[m * d + k];
        }
        dwd[j * d + k] = sd;
        dwuT[j * d + k] = su;
        dwgT[j * d + k] = sg;
      }
  });
  parallel_for(M, [&](int64_t lo, int64_t hi) {
    for (int64_t m = lo; m < hi; ++m)
      for (int64_t k = 0; k < d; ++k) {
        double s = 0.0;
        for (int64_t j = 0; j < f; ++j)
          s += du[m * f + j] * wuT[j * d + k] + da[m * f + j] * wgT[j * d + k];
        dx[m * d + k] = s;
      }
  });
}

// dx for the listed rows only (same definitions; each row is independent).
void orc_ffn_bwd_dx_rows(const double* x, const double* wgT, const double* wuT,
                         const double* wd, const double* dy, int64_t d, int64_t f,
                         double lambda, int round_g, const int64_t* rows, int64_t nrows,
                         double* dx) {
  parallel_for(nrows, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      int64_t m = rows[r];
      double* out = dx + r * d;
      for (int64_t k = 0; k < d; ++k) out[k] = 0.0;
      for (int64_t j = 0; j < f; ++j) {
        double a = dot(x + m * d, wgT + j * d, d);
        double g = a > 0.0 ? a : 0.0;
        if (round_g) g = bf16_to_double(double_to_bf16(g));
        if (!(g > 0.0)) continue;  // du = da = 0 for a dead column
        double u = dot(x + m * d, wuT + j * d, d);
        double dh = dot(dy + m * d, wd + j * d, d);
        double du = dh * g, da = dh * u + lambda;
        for (int64_t k = 0; k < d; ++k) out[k] += du * wuT[j * d + k] + da * wgT[j * d + k];
      }
    }
  });
}

// dWg^T, dWu^T, dWd rows for the listed neurons only (sums over all M rows).
void orc_ffn_bwd_dw_neurons(const double* x, const double* wgT, const double* wuT,
                            const double* wd, const double* dy, int64_t M, int64_t d,
                            double lambda, int round_g, const int64_t* neurons,
                            int64_t nneur, double* dwgT, double* dwuT, double* dwd) {
  parallel_for(nneur, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      int64_t j = neurons[r];
      double *og = dwgT + r * d, *ou = dwuT + r * d, *od = dwd + r * d;
      for (int64_t k = 0; k < d; ++k) og[k] = ou[k] = od[k] = 0.0;
      for (int64_t m = 0; m < M; ++m) {
        double a = dot(x + m * d, wgT + j * d, d);
        double g = a > 0.0 ? a : 0.0;
        if (round_g) g = bf16_to_double(double_to_bf16(g));
        if (!(g > 0.0)) continue;  // dead: h = du = da = 0
        double u = dot(x + m * d, wuT + j * d, d);
        double dh = dot(dy + m * d, wd + j * d, d);
        double h = g * u, du = dh * g, da = dh * u + lambda;
        for (int64_t k = 0; k < d; ++k) {
          od[k] += h * dy[m * d + k];
          ou[k] += du * x[m * d + k];
          og[k] += da * x[m * d + k];
        }
      }
    }
  });
}

// ---- sparse backward over the hybrid format  [P2-twell] --------------------
// ELL rows visit only their stored live entries (g from ell_val); routed rows
// use the dense definitions above with g = bf16(ReLU(a)).  Outputs the whole
// dx [M][d] and dW [f][d] arrays; small shapes only.
void orc_ffn_bwd_hybrid(const double* x, const double* wgT, const double* wuT,
                        const double* wd, const double* dy, int64_t M, int64_t d, int64_t f,
                        int32_t W, const uint16_t* ell_val, const uint16_t* ell_col,
                        const int32_t* ell_nnz, const int32_t* dense_rows, int32_t n_dense,
                        double lambda, double* dx, double* dwgT, double* dwuT, double* dwd) {
  for (int64_t i = 0; i < M * d; ++i) dx[i] = 0.0;
  for (int64_t i = 0; i < f * d; ++i) dwgT[i] = dwuT[i] = dwd[i] = 0.0;
  std::vector<char> routed(M, 0);
  for (int32_t i = 0; i < n_dense; ++i) routed[dense_rows[i]] = 1;
  for (int64_t m = 0; m < M; ++m) {
    const double *xm = x + m * d, *dym = dy + m * d;
    double* dxm = dx + m * d;
    if (!routed[m]) {
      for (int32_t s = 0; s < ell_nnz[m]; ++s) {
        int64_t j = ell_col[m * W + s];
        double g = bf16_to_double(ell_val[m * W + s]);
        double dh = dot(dym, wd + j * d, d);
        double u = dot(xm, wuT + j * d, d);
        double du = dh * g, da = dh * u + lambda, h = g * u;
        for (int64_t k = 0; k < d; ++k) {
          dxm[k] += du * wuT[j * d + k] + da * wgT[j * d + k];
          dwd[j * d + k] += h * dym[k];
          dwuT[j * d + k] += du * xm[k];
          dwgT[j * d + k] += da * xm[k];
        }
      }
    } else {
      for (int64_t j = 0; j < f; ++j) {
        double a = dot(xm, wgT + j * d, d);
        double g = bf16_to_double(gate_bf16(a));
        if (!(g > 0.0)) continue;
        double dh = dot(dym, wd + j * d, d);
        double u = dot(xm, wuT + j * d, d);
        double du = dh * g, da = dh * u + lambda, h = g * u;
        for (int64_t k = 0; k < d; ++k) {
          dxm[k] += du * wuT[j * d + k] + da * wgT[j * d + k];
          dwd[j * d + k] += h * dym[k];
          dwuT[j * d + k] += du * xm[k];
          dwgT[j * d + k] += da * xm[k];
        }
      }
    }
  }
}

// ---- SiLU-gated dense FFN (comparator only)  [P2-recipe] ----------------------
// The unmodified gated FFN the recipe starts from: the gate activation is SiLU
// instead of ReLU, and there is no L1 term.
//   s_j = silu(a_j) = a_j * sigmoid(a_j),  h_j = s_j u_j,  y_m = sum_j h_j Wd[j,:]
// Backward, by the chain rule:
//   dh = dY Wd^T,  du = dh s,  da = dh u silu'(a),
//   silu'(a) = sigmoid(a) (1 + a (1 - sigmoid(a))),
//   dWd = h^T dY, dWu = x^T du, dWg = x^T da, dx = du Wu^T + da Wg^T.
static double sigmoid(double a) { return 1.0 / (1.0 + std::exp(-a)); }

void orc_ffn_fwd_dense_silu(const double* x, const double* wgT, const double* wuT,
                            const double* wd, int64_t d, int64_t f, const int64_t* rows,
                            int64_t nrows, double* y) {
  parallel_for(nrows, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      const double* xm = x + rows[r] * d;
      double* yr = y + r * d;
      for (int64_t k = 0; k < d; ++k) yr[k] = 0.0;
      for (int64_t j = 0; j < f; ++j) {
        double a = dot(xm, wgT + j * d, d);
        double s = a * sigmoid(a);
        double u = dot(xm, wuT + j * d, d);
        double h = s * u;
        for (int64_t k = 0; k < d; ++k) yr[k] += h * wd[j * d + k];
      }
    }
  });
}

// Whole-batch SiLU backward (small shapes: it holds [M][f] arrays).
void orc_ffn_bwd_dense_silu(const double* x, const double* wgT, const double* wuT,
                            const double* wd, const double* dy, int64_t M, int64_t d,
                            int64_t f, double* dx, double* dwgT, double* dwuT, double* dwd) {
  std::vector<double> h(M * f), du(M * f), da(M * f);
  parallel_for(M, [&](int64_t lo, int64_t hi) {
    for (int64_t m = lo; m < hi; ++m)
      for (int64_t j = 0; j < f; ++j) {
        double a = dot(x + m * d, wgT + j * d, d);
        double sg = sigmoid(a);
        double s = a * sg;
        double ds = sg * (1.0 + a * (1.0 - sg));
        double uj = dot(x + m * d, wuT + j * d, d);
        double dh = dot(dy + m * d, wd + j * d, d);
        h[m * f + j] = s * uj;
        du[m * f + j] = dh * s;
        da[m * f + j] = dh * uj * ds;
      }
  });
  parallel_for(f, [&](int64_t lo, int64_t hi) {
    for (int64_t j = lo; j < hi; ++j)
      for (int64_t k = 0; k < d; ++k) {
        double sd = 0.0, su = 0.0, sg = 0.0;
        for (int64_t m = 0; m < M; ++m) {
          sd += h[m * f + j] * dy[m * d + k];
          su += du[m * f + j] * x[m * d + k];
          sg += da[m * f + j] * x[m * d + k];
        }
        dwd[j * d + k] = sd;
        dwuT[j * d + k] = su;
        dwgT[j * d + k] = sg;
      }
  });
  parallel_for(M, [&](int64_t lo, int64_t hi) {
    for (int64_t m = lo; m < hi; ++m)
      for (int64_t k = 0; k < d; ++k) {
        double s = 0.0;
        for (int64_t j = 0; j < f; ++j)
          s += du[m * f + j] * wuT[j * d + k] + da[m * f + j] * wgT[j * d + k];
        dx[m * d + k] = s;
      }
  });
}

}  // extern "C"
