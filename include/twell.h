/*
 * twell.h -- C ABI of the GB300 (sm_103a) activation-sparse gated FFN library.
 *
 * The method (three web pages on TwELL; page 2, "Sakana AI and NVIDIA
 * introduce TwELL with CUDA kernels ...", is the technical one):
 *   - "¿Cuál es el problema que TwELL resuelve?": the gated feed-forward block
 *     y = (ReLU(x Wg) * (x Wu)) Wd of a Transformer++, whose ReLU gate output
 *     is ~99.5 % exact zeros; classic ELLPACK needs a separate dense->sparse
 *     conversion kernel whose cost cancels the saving.
 *   - "¿Qué hace distinto a TwELL frente a ELL clásico?": the sparse format is
 *     built inside the gate matmul's epilogue, with no extra launch and no
 *     extra global write; columns are cut into tiles of the matmul's tile
 *     width T_n and nonzeros are packed locally per tile (TwELL).  Inference
 *     runs up and down projections in one fused kernel that never writes the
 *     intermediate to global memory.  Training routes rows with too many
 *     nonzeros to a dense backup, the rest to a compact ELL matrix.
 *   - "Receta de entrenamiento": ReLU replaces SiLU as the gate activation and
 *     an L1 term (coefficient 2e-5) is added on the hidden activations.
 *
 * Conventions for every entry point
 *   - All pointers named as tensors are DEVICE pointers the caller allocated;
 *     the library allocates no device memory and keeps no per-call state.
 *     Structs (twell_shape, twell_tiles, twell_hybrid) are HOST structs passed
 *     by pointer; the pointers inside them are device pointers.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work
 *     is asynchronous on it; no entry point synchronises the host.
 *   - Layouts (row-major, bf16 = IEEE bfloat16 bits):
 *       x, dy, y, dx       bf16 [M][d_model]
 *       wgT, wuT           bf16 [d_ff][d_model]  (= Wg^T, Wu^T; nn.Linear layout)
 *       wd                 bf16 [d_ff][d_model]  (= Wd, the down projection)
 *       dwgT, dwuT, dwd    fp32 [d_ff][d_model]  (same layouts as the weights)
 *     so every neuron's three weight vectors are contiguous d_model-long rows.
 *   - Argument checks happen before any launch; a failed check returns a
 *     non-zero status and launches nothing.  Nothing aborts or throws across
 *     the ABI.  A CUDA launch error maps to TWELL_ERR_CUDA.
 *   - Errors found on the device (a tile overflow with no route, a pipeline
 *     wait that timed out) are recorded in a per-device status word that
 *     twell_get_device_status() reads and clears.
 *   - Supported shapes: d_model % 64 == 0 and >= 64; d_ff % tile_n == 0;
 *     d_ff <= 65535; tile_n in {64, 128}; 1 <= tile_cap <= tile_n; M >= 0
 *     (M == 0 is a no-op); every pointer 16-byte aligned.
 */
#ifndef TWELL_H
#define TWELL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum twell_status {
  TWELL_OK = 0,
  TWELL_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad enum */
  TWELL_ERR_UNSUPPORTED = 2,    /* shape outside the supported set above */
  TWELL_ERR_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned */
  TWELL_ERR_CAPACITY = 4,       /* a packed tile overflowed with no route */
  TWELL_ERR_CUDA = 5,           /* a CUDA call or launch failed */
  TWELL_ERR_DEVICE_TIMEOUT = 6, /* a device-side pipeline wait gave up */
  TWELL_ERR_WORKSPACE = 7,      /* workspace missing or smaller than required */
  TWELL_ERR_INDEX = 8           /* checked build only: an index read from memory
                                   (column, row, entry position) was out of range */
} twell_status;

/* Problem shape.  tile_n = T_n, the TwELL tile width (columns of the gate
 * activation per tile); tile_cap = C, the number of stored slots per tile. */
typedef struct twell_shape {
  int32_t M, d_model, d_ff, tile_n, tile_cap;
} twell_shape;

/* TwELL tiles (device).  T = d_ff / tile_n tiles per row.
 *   val      bf16 [M][T][C]  gate values g = bf16(ReLU(a)) of the live columns
 *   idx      u8   [M][T][C]  column of each value inside its tile (0..T_n-1)
 *   cnt      u8   [M][T]     true number of live columns in the tile (may be > C;
 *                            then only the first C, in ascending column, are stored)
 *   row_nnz  i32  [M]        live columns in the row (sum of cnt)
 * Slots at or past min(cnt, C) hold unspecified bytes. */
typedef struct twell_tiles {
  void* val;
  uint8_t* idx;
  uint8_t* cnt;
  int32_t* row_nnz;
} twell_tiles;

/* Hybrid ELL / dense-backup routing (device arrays, one host field).
 *   ell_val    bf16 [M][ell_width]  live gate values, ascending global column
 *   ell_col    u16  [M][ell_width]  global column (neuron) of each value
 *   ell_nnz    i32  [M]             entries used in the row; 0 for routed rows
 *   dense_rows i32  [M]             routed rows, ascending, first *n_dense valid
 *   n_dense    i32  [1]             number of routed rows (stays on the device)
 *   dense_cap  host int: how many routed rows the caller's workspace holds
 *              (0 <= dense_cap; values above M count as M).  The routed rows'
 *              buffers of the workspace, and so its size, scale with it.
 *              hybrid_route records TWELL_ERR_CAPACITY in the device status
 *              word when it routes more rows than dense_cap; the forward and
 *              backward then compute only the first dense_cap routed rows and
 *              leave the others' y / dx rows and dW terms out.  The count is
 *              on the device, so a caller that can read it may route with
 *              dense_cap = M, read *n_dense and size the workspace for exactly
 *              that many rows (setting dense_cap to it). */
typedef struct twell_hybrid {
  void* ell_val;
  uint16_t* ell_col;
  int32_t* ell_nnz;
  int32_t ell_width;
  int32_t* dense_rows;
  int32_t* n_dense;
  int32_t dense_cap;
} twell_hybrid;

/* Gate projection with the TwELL pack fused into its epilogue.
 * Source: page 2, "¿Qué hace distinto a TwELL frente a ELL clásico?" (format
 * built in the matmul epilogue; per-T_n-tile local packing) and "Receta de
 * entrenamiento" (ReLU gate).
 * Computes a = x Wg (bf16 in, fp32 accumulate on tcgen05 tensor cores), then
 * for every (row, tile) g = bf16(ReLU(a)), keeps the live (g > 0) columns in
 * ascending order and writes `out` (all four arrays).  No dense activation is
 * written to global memory.  Batches of at most 64 rows run with the
 * operands swapped (128 neurons on the MMA's M dimension, the rows padded
 * to 16, 32 or 64 on its N dimension) and pack across TMEM lanes; the
 * format is the same, the fp32 sums run in another order.
 *   x    bf16 [M][d_model], wgT bf16 [d_ff][d_model]. */
twell_status twell_pack(const void* x, const void* wgT, const twell_shape* shape,
                        const twell_tiles* out, void* stream);

/* Pack an already-dense pre-activation a [M][d_ff] into TwELL -- the separate
 * conversion step of classic ELL (page 2, "¿Cuál es el problema que TwELL
 * resuelve?").  Same output contract as twell_pack.
 *   a_dtype: 0 = a is bf16, 1 = a is fp32. */
twell_status twell_pack_dense(const void* a, int32_t a_dtype, const twell_shape* shape,
                              const twell_tiles* out, void* stream);

/* Hybrid routing of packed rows (training).  Source: page 2, "¿Qué hace
 * distinto a TwELL frente a ELL clásico?" (rows with too many nonzeros go to
 * a dense backup, the rest to a compact ELL matrix).
 * A row is routed iff some tile has cnt > tile_cap or row_nnz > ell_width.
 * Routed rows are listed ascending in dense_rows and get ell_nnz = 0; the other
 * rows are compacted into ELL, ascending global column.  ell_width >= 0.
 * The count n_dense stays on the device. */
twell_status hybrid_route(const twell_tiles* in, const twell_shape* shape,
                          const twell_hybrid* out, void* stream);

/* Bytes of workspace twell_ffn_fwd (training = 0) or twell_ffn_fwd +
 * twell_ffn_bwd (training = 1) need for this shape, ELL width and routed-row
 * capacity (the route's dense_cap; values above M count as M).  The routed
 * rows' buffers hold dense_cap rows in whole 128-row tiles; the rest grows
 * with M * ell_width (per-entry values of the backward) and M * d_model (the
 * fp32 running y / dX of L2-sized passes, and the routed rows' split-K
 * partials).  Returns 0 for an invalid shape or a negative width or capacity. */
size_t twell_workspace_bytes_capped(const twell_shape* shape, int32_t ell_width,
                                    int32_t dense_cap, int32_t training);

/* twell_workspace_bytes_capped with dense_cap = M (room for every row routed). */
size_t twell_workspace_bytes(const twell_shape* shape, int32_t ell_width, int32_t training);

/* Bytes of the optional workspace of twell_ffn_fwd with `tiles` (inference).
 * For d_model > 1024 a workspace this large (h of each row's live entries,
 * fp32, room for d_ff / tile_n * tile_cap per row, and the fp32 running y
 * between L2-sized neuron passes, [M][d_model]) lets the forward run as two
 * gathers, up then down, that meet no barrier per batch; the result is the
 * same bit for bit.
 * Returns 0 for d_model <= 1024, where no workspace is used, and for an
 * invalid shape. */
size_t twell_tiles_workspace_bytes(const twell_shape* shape);

/* Choice of the gathers for rows wider than 1024, process-wide; returns the
 * previous setting.  enable = 1 (the default): the forward runs as an up
 * gather (h = g (x . Wu[:, j]) per live entry, 4 bytes each in the
 * workspace) and a down gather (y = sum h Wd[j, :]), and the backward row
 * phase as a dh gather (over Wd) and a gradient + dX gather (over Wu^T and
 * Wg^T, each read once per entry); none meets a barrier per batch and each
 * takes one or two weight matrices per L2-sized pass.  enable = 0: the fused
 * kernels of page 2, section "¿Qué hace distinto a TwELL frente a ELL
 * clásico?" (one gather per row, h kept in registers and never written to
 * global memory).  Both give the same bytes in y; the backward sums the
 * same fp32 terms in another grouping (u over another set of warps, dX per
 * group of 32 entries), so dX and dW may differ in their last bits.  Not
 * synchronised with work in flight: change it between calls. */
int32_t twell_set_split_gathers(int32_t enable);

/* Choice of the tensor-core GEMM form, process-wide; returns the previous
 * setting.  enable = 1 (the default): GEMMs without a K split run as 2-CTA
 * clusters (tcgen05 cta_group::2) on 256 x 256 output tiles, each CTA
 * staging half of the tile's A rows and half of its B rows, unless that
 * would take more waves of tiles than the single-CTA form.  enable = 0:
 * every GEMM runs one CTA per 128 x 256 tile.  The products and the fp32
 * accumulation order over K are the same in both forms.  Not synchronised
 * with work in flight: change it between calls. */
int32_t twell_set_pair_gemm(int32_t enable);

/* Fused sparse up + down projection.  Source: page 2, "¿Qué hace distinto a
 * TwELL frente a ELL clásico?" (one kernel reads the packed activations and
 * does both projections; the intermediate never reaches global memory) and,
 * for routed rows, the dense backup of the same section.
 * For every row m: y_m = sum over live j of g_mj * (x_m . Wu[:, j]) * Wd[j, :],
 * fp32 accumulation, y stored as bf16.
 * Exactly one of `tiles` (inference: reads TwELL directly; a tile with
 * cnt > C sets TWELL_ERR_CAPACITY in the device status word and its row
 * uses only the stored entries) and `route` (training: ELL rows by gather,
 * routed rows by a dense tensor-core gated FFN that recomputes their gate)
 * is non-NULL.  wgT is read only for routed rows (may be NULL with tiles).
 * ws/ws_bytes: with `route`, a workspace of at least
 * twell_workspace_bytes_capped(shape, W, route->dense_cap, 0) bytes (16-byte
 * aligned); besides the routed rows' buffers it carries the fp32 running y between passes when
 * the gathered Wu / Wd rows exceed L2 and the ELL gather is split into
 * L2-sized neuron passes (same result, bit for bit), and for rows wider than
 * 1024 the fp32 h of every live ELL entry between the up and down gathers.  With `tiles` the
 * workspace is optional: NULL keeps the fused gather; for d_model > 1024 a
 * workspace of at least twell_tiles_workspace_bytes(shape) bytes (16-byte
 * aligned; smaller returns TWELL_ERR_WORKSPACE) runs it as two gathers with
 * the same result, bit for bit; batches too small to fill the GPU split each
 * row over a thread-block cluster instead, which sums in another order. */
twell_status twell_ffn_fwd(const void* x, const void* wgT, const void* wuT, const void* wd,
                           const twell_shape* shape, const twell_tiles* tiles,
                           const twell_hybrid* route, void* y, void* ws, size_t ws_bytes,
                           void* stream);

/* Allocation-free variant of twell_ffn_fwd for the training (route) path.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory when they run the FFN -- a plugin whose host
 * runtime owns every allocation, a scheduler that must not call cudaMalloc
 * (which can synchronise the device) in the middle of a step, or a
 * deployment whose memory footprint is fixed up front.  It computes exactly
 * what twell_ffn_fwd(..., tiles = NULL, route, ...) computes, with the
 * routed-row scratch taken from a 32 MiB array compiled into the library
 * (held by every device that loads the library until the process exits)
 * instead of a caller workspace.  It allocates nothing and calls no
 * allocating routine.
 *   - Limit: twell_workspace_bytes_capped(shape, route->ell_width,
 *     route->dense_cap, 0) must not exceed 32 MiB (e.g. M <= 1408 at
 *     d_model = 1024, d_ff = 4096 with room for every row routed); larger
 *     needs return TWELL_ERR_WORKSPACE before any launch.
 *   - The array's device address is looked up on the first call on each
 *     device (with that device current) and cached; make that first call
 *     before any stream capture.  `stream` must belong to the current
 *     device, and the cached address does not survive cudaDeviceReset.
 *   - Every call on a device shares the one array and it keeps the previous
 *     call's contents; nothing in it needs to start at zero.  Calls that
 *     overlap on the GPU (on different streams, for example) race on it and
 *     must be serialised by the caller. */
twell_status twell_ffn_fwd_noalloc(const void* x, const void* wgT, const void* wuT,
                                   const void* wd, const twell_shape* shape,
                                   const twell_hybrid* route, void* y, void* stream);

/* Backward of the sparse FFN with the L1 activation term.  Source: the
 * training path of page 2, "¿Qué hace distinto a TwELL frente a ELL
 * clásico?" (hybrid rows) and "Receta de entrenamiento" (L1 with coefficient
 * l1_coeff on the gate activations).  With loss = sum(y * dy) + l1_coeff *
 * sum(g) it writes
 *   dx  = du Wu^T + da Wg^T                     (bf16 [M][d_model])
 *   dwd = h^T dy, dwuT = du^T x, dwgT = da^T x  (fp32 [d_ff][d_model], overwritten)
 * where dh = dy Wd^T, du = dh * g, da = (dh * u + l1_coeff) * 1[g > 0], h = g * u,
 * using only the live entries of ELL rows and a dense tensor-core path for the
 * routed rows.  The route must come from hybrid_route on the same x and Wg.
 * The reduction order is fixed, so results are bit-reproducible.
 * ws/ws_bytes: at least twell_workspace_bytes_capped(shape, W, route->dense_cap, 1)
 * bytes (16-byte aligned); it also carries the fp32 running dX when the row phase runs in
 * L2-sized neuron passes and, for rows wider than 1024 (split gathers, see
 * twell_set_split_gathers), dh of every live ELL entry.  When x
 * and dY together exceed 3/4 of L2 the weight gradients are formed in two
 * passes, over dY rows (dwd) and over x rows (dwuT, dwgT), with the same
 * per-element order. */
twell_status twell_ffn_bwd(const void* x, const void* wgT, const void* wuT, const void* wd,
                           const void* dy, const twell_shape* shape, const twell_hybrid* route,
                           float l1_coeff, void* dx, float* dwgT, float* dwuT, float* dwd,
                           void* ws, size_t ws_bytes, void* stream);

/* The library's own dense gated FFN (the comparator), same definitions, on
 * tcgen05 tensor cores throughout.  twell_dense_ffn_fwd writes y; with
 * training = 1 it also keeps what the backward needs (g, u, h) in `ws`, and
 * twell_dense_ffn_bwd must then get the same ws.  Shape fields tile_n and
 * tile_cap are ignored. */
size_t twell_dense_workspace_bytes(const twell_shape* shape, int32_t training);
twell_status twell_dense_ffn_fwd(const void* x, const void* wgT, const void* wuT, const void* wd,
                                 const twell_shape* shape, void* y, int32_t training, void* ws,
                                 size_t ws_bytes, void* stream);
twell_status twell_dense_ffn_bwd(const void* x, const void* wgT, const void* wuT, const void* wd,
                                 const void* dy, const twell_shape* shape, float l1_coeff,
                                 void* dx, float* dwgT, float* dwuT, float* dwd, void* ws,
                                 size_t ws_bytes, void* stream);

/* The dense comparator with a choice of gate activation.  TWELL_ACT_RELU is
 * exactly twell_dense_ffn_fwd / _bwd.  TWELL_ACT_SILU is the unmodified
 * gated FFN that page 2's "Receta de entrenamiento" replaces (its gate is
 * SiLU, s = a * sigmoid(a), before the switch to ReLU): h = s * u, and the
 * backward is du = dh * s, da = dh * u * s'(a) with s'(a) = sigmoid(a) *
 * (1 + a * (1 - sigmoid(a))); there is no L1 term, so l1_coeff must be 0
 * (else TWELL_ERR_INVALID_ARG).  With training = 1 the workspace keeps
 * bf16(a) in place of g.  Any other activation value is
 * TWELL_ERR_INVALID_ARG.  The fwd and bwd of one step must use the same
 * activation and workspace. */
enum { TWELL_ACT_RELU = 0, TWELL_ACT_SILU = 1 };
twell_status twell_dense_ffn_fwd_act(const void* x, const void* wgT, const void* wuT,
                                     const void* wd, const twell_shape* shape,
                                     int32_t activation, void* y, int32_t training, void* ws,
                                     size_t ws_bytes, void* stream);
twell_status twell_dense_ffn_bwd_act(const void* x, const void* wgT, const void* wuT,
                                     const void* wd, const void* dy, const twell_shape* shape,
                                     int32_t activation, float l1_coeff, void* dx, float* dwgT,
                                     float* dwuT, float* dwd, void* ws, size_t ws_bytes,
                                     void* stream);

/* The tcgen05 GEMM engine the entry points above are built on, exposed for
 * testing: C[m][n] = sum_k A(m, k) B(n, k), bf16 in, fp32 accumulate.
 *   a_mn_major = 0: A is [M][K] (K contiguous); 1: A is [K][M] (M contiguous).
 *   b_mn_major = 0: B is [N][K];                1: B is [K][N].
 *   c_dtype: 0 = bf16 [M][N], 1 = fp32 [M][N]; accumulate = 1 adds into an fp32 C.
 * Requires K % 8 == 0 and, for MN-major operands, M (or N) % 8 == 0. */
twell_status twell_gemm_bf16(const void* A, const void* B, void* C, int32_t M, int32_t N,
                             int32_t K, int32_t a_mn_major, int32_t b_mn_major, int32_t c_dtype,
                             int32_t accumulate, void* stream);

/* Failure-path self-test: one kernel waits on an mbarrier that nothing
 * completes, using the same bounded wait as the GEMM pipeline but with a
 * limit of limit_us microseconds (1 .. 10^7); when it gives up it records
 * TWELL_ERR_DEVICE_TIMEOUT in the device status word and returns, so the
 * error path is exercised without a fault and the context stays usable.
 * Read the result with twell_get_device_status.  Not part of the method. */
twell_status twell_selftest_wait_timeout(int32_t limit_us, void* stream);

/* Reads and clears the device status word of the current device after
 * synchronising `stream`.  *out receives TWELL_OK or the first error seen. */
twell_status twell_get_device_status(void* stream, int32_t* out);

/* Human-readable name of a status code (static string). */
const char* twell_status_string(int32_t status);

/* Number of SMs the library schedules persistent kernels over (0 if no device). */
int32_t twell_num_sms(void);

/* Number of CUDA kernels this library has launched in this process so far
 * (all devices, all streams).  Lets a caller count the kernels of a region. */
uint64_t twell_launch_count(void);

/* Built-in kernel timing.  twell_profile_begin(name) makes every later launch
 * of the kernel family `name` ("*" for all, NULL or "" to stop) record a CUDA
 * event pair on the stream it is launched on; twell_profile_end() stops,
 * synchronises those events and aggregates them per family, returning the
 * number of families (or -1 if an event could not be read); entry i is then
 * available from twell_profile_entry (name valid until the next begin/end).
 * Families: gemm_gate_pack (also the small-batch gate), gemm_gated,
 * gemm_dgate, gemm_store_kk/mk/km/mm, pack_dense, route_rows, route_list,
 * gather_rows, splitk_scatter, sparse_fwd, sparse_fwd_up, sparse_fwd_down,
 * csc_mark, csc_scan, csc_place, bwd_rows, bwd_dh, bwd_grad_dx,
 * bwd_neurons, bwd_neurons_dy, bwd_neurons_x.  Host-side state,
 * process-wide; not for use while another thread launches. */
twell_status twell_profile_begin(const char* kernel);
int32_t twell_profile_end(void);
twell_status twell_profile_entry(int32_t i, const char** name, int32_t* launches,
                                 double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* TWELL_H */
