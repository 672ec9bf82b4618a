// common.cuh -- device helpers shared by the library's kernels (sm_103a).
//
// Thin inline-PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor), the
// tcgen05 tensor-core instructions and TMEM, plus the bounded waits every
// pipeline uses.  A wait that does not complete within kWaitLimitNs records
// TWELL_ERR_DEVICE_TIMEOUT in the status word and returns false; no kernel
// traps or spins forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "twell.h"

#define TW_DEV __device__ __forceinline__

namespace tw {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

TW_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

TW_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// First error wins; later errors are dropped.
TW_DEV void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ checked build
// Built with -DTWELL_CHECKED (a debug library), every index a gather or
// index kernel reads from memory -- a column below d_ff, an in-tile column
// below T_n, a row below M, an entry position below M * W, an ELL length of
// at most W -- is tested before it is used: a bad one is replaced by 0 (an
// index that is always in bounds) and TWELL_ERR_INDEX is recorded in the
// device status word, with no trap.  In the normal build the checks vanish.
// Each translation unit keeps its own copy of the status word's address,
// set by checked_setup() (host) before its first launch on a device; that
// setup is a synchronous copy, so the first call on a device must not be
// inside a stream capture.
int* device_status_ptr();
#ifdef TWELL_CHECKED
static __device__ int* g_checked_status;
#define TW_CHECK_INDEX(v, ok)                                    \
  do {                                                           \
    if (!(ok)) {                                                 \
      ::tw::set_status(::tw::g_checked_status, TWELL_ERR_INDEX); \
      (v) = 0;                                                   \
    }                                                            \
  } while (0)
static inline cudaError_t checked_setup() {
  static int* done[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int* st = device_status_ptr();
  if (!st) return cudaErrorInvalidSymbol;
  if (done[dev] == st) return cudaSuccess;
  e = cudaMemcpyToSymbol(g_checked_status, &st, sizeof(st));
  if (e == cudaSuccess) done[dev] = st;
  return e;
}
#else
#define TW_CHECK_INDEX(v, ok) \
  do {                        \
  } while (0)
static inline cudaError_t checked_setup() { return cudaSuccess; }
#endif

// ------------------------------------------------------------------ mbarrier
TW_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
TW_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
TW_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

TW_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
TW_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
TW_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up (returns
// false) once the CTA-wide abort flag is raised or after kWaitLimitNs.
TW_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                      uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (abort_flag && *abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------------------ TMA
TW_DEV void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

TW_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// TMA stores from shared memory (bulk async-group completion).
TW_DEV void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1)
      : "memory");
}
TW_DEV void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1)
      : "memory");
}
TW_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N committed groups still read their shared-memory source
template <int N>
TW_DEV void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
TW_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------------ tcgen05
TW_DEV void tmem_alloc(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(holder)),
               "r"(ncols)
               : "memory");
}
TW_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
TW_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
TW_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
TW_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive once on `bar` when every tcgen05 op this thread issued so far is done.
TW_DEV void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one 128 x N x 16 bf16 step.
TW_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
TW_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  __syncwarp();  // .sync.aligned: the whole warp must arrive converged
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
TW_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start
// address, leading / stride byte offsets in 16-byte units, version 1).
TW_DEV uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, bf16 A and B,
// A / B K-major (0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Split-K plan shared by the GEMM and the kernel that reduces its partials:
// as many K splits (at most s_max) as fit when each split writes rows_eff
// (= the used rows rounded up to 128) rows of a buffer with buf_rows rows;
// kps k-blocks per split, splits = the number of non-empty splits.
__host__ __device__ inline void splitk_plan(int rows_eff, int buf_rows, int num_kb, int s_max,
                                            int& splits, int& kps) {
  int sp = rows_eff > 0 ? buf_rows / rows_eff : 1;
  sp = sp < s_max ? sp : s_max;
  sp = sp < num_kb ? sp : num_kb;
  sp = sp < 1 ? 1 : sp;
  kps = (num_kb + sp - 1) / sp;
  splits = kps > 0 ? (num_kb + kps - 1) / kps : 1;
}

// ------------------------------------------------------------------ numerics
TW_DEV float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// bf16 bits of ReLU(a) (round to nearest even); 0 or 0x8000 means dead.
TW_DEV uint32_t relu_bf16_bits(float a) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(fmaxf(a, 0.0f)));
}

TW_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

TW_DEV float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// 8 bf16 (one 16-byte vector) dot 8 bf16, fp32 accumulate.
TW_DEV float dot8(const uint4& a, const uint4& b, float acc) {
  float2 a0 = unpack_bf16x2(a.x), b0 = unpack_bf16x2(b.x);
  float2 a1 = unpack_bf16x2(a.y), b1 = unpack_bf16x2(b.y);
  float2 a2 = unpack_bf16x2(a.z), b2 = unpack_bf16x2(b.z);
  float2 a3 = unpack_bf16x2(a.w), b3 = unpack_bf16x2(b.w);
  acc = fmaf(a0.x, b0.x, acc);
  acc = fmaf(a0.y, b0.y, acc);
  acc = fmaf(a1.x, b1.x, acc);
  acc = fmaf(a1.y, b1.y, acc);
  acc = fmaf(a2.x, b2.x, acc);
  acc = fmaf(a2.y, b2.y, acc);
  acc = fmaf(a3.x, b3.x, acc);
  acc = fmaf(a3.y, b3.y, acc);
  return acc;
}

// acc[0..8) += s * (8 bf16)
TW_DEV void axpy8(float s, const uint4& w, float* acc) {
  float2 w0 = unpack_bf16x2(w.x), w1 = unpack_bf16x2(w.y);
  float2 w2 = unpack_bf16x2(w.z), w3 = unpack_bf16x2(w.w);
  acc[0] = fmaf(s, w0.x, acc[0]);
  acc[1] = fmaf(s, w0.y, acc[1]);
  acc[2] = fmaf(s, w1.x, acc[2]);
  acc[3] = fmaf(s, w1.y, acc[3]);
  acc[4] = fmaf(s, w2.x, acc[4]);
  acc[5] = fmaf(s, w2.y, acc[5]);
  acc[6] = fmaf(s, w3.x, acc[6]);
  acc[7] = fmaf(s, w3.y, acc[7]);
}

TW_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sums of two values over the warp, every lane gets both (7 shuffles
// instead of 10): the first exchange halves the work by letting lanes 0-15
// carry a and lanes 16-31 carry b.
TW_DEV void warp_sum2(float& a, float& b) {
  const int lane = threadIdx.x & 31;
  const bool lo = lane < 16;
  float keep = lo ? a : b;
  const float give = lo ? b : a;
  keep += __shfl_xor_sync(0xffffffffu, give, 16);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
  a = __shfl_sync(0xffffffffu, keep, 0);
  b = __shfl_sync(0xffffffffu, keep, 16);
}

// Sums of four values over the warp, every lane gets all four (10 shuffles
// instead of 20).
TW_DEV void warp_sum4(float& a, float& b, float& c, float& d) {
  const int lane = threadIdx.x & 31;
  const bool h16 = lane & 16, h8 = lane & 8;
  // step 1: lanes < 16 keep (a, b), lanes >= 16 keep (c, d)
  float k0 = h16 ? c : a, k1 = h16 ? d : b;
  const float g0 = h16 ? a : c, g1 = h16 ? b : d;
  k0 += __shfl_xor_sync(0xffffffffu, g0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, g1, 16);
  // step 2: within each half, lanes with bit 3 clear keep k0, set keep k1
  float k = h8 ? k1 : k0;
  const float g = h8 ? k0 : k1;
  k += __shfl_xor_sync(0xffffffffu, g, 8);
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
  // totals: a at lanes 0-7, b at 8-15, c at 16-23, d at 24-31
  a = __shfl_sync(0xffffffffu, k, 0);
  b = __shfl_sync(0xffffffffu, k, 8);
  c = __shfl_sync(0xffffffffu, k, 16);
  d = __shfl_sync(0xffffffffu, k, 24);
}

TW_DEV int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

TW_DEV uint4 ldg_v4(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// L2 policy that marks lines for early eviction: for results written once
// and not read again by the same kernel, so they do not push gathered
// operands out of L2.
TW_DEV uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
TW_DEV uint4 ldg_v4_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}
TW_DEV void st_v4_hint(void* p, const uint4& v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// ---- packed fp32 pairs (sm_100+ f32x2 arithmetic) --------------------------
// A uint64 holds two fp32 values: low word = element 2i, high word = 2i+1.
TW_DEV uint64_t f2_make(uint32_t lo_bits, uint32_t hi_bits) {
  return ((uint64_t)hi_bits << 32) | (uint64_t)lo_bits;
}
// bf16x2 word -> two fp32 (exact)
TW_DEV uint64_t bf2_to_f2(uint32_t v) { return f2_make(v << 16, v & 0xFFFF0000u); }
TW_DEV uint64_t f2_splat(float s) {
  const uint32_t b = __float_as_uint(s);
  return f2_make(b, b);
}
TW_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
TW_DEV float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
TW_DEV float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
TW_DEV float f2_sum(uint64_t v) { return f2_lo(v) + f2_hi(v); }

// 8 bf16 of a 16-byte vector as four fp32 pairs
TW_DEV void bf8_to_f2(const uint4& w, uint64_t (&o)[4]) {
  o[0] = bf2_to_f2(w.x);
  o[1] = bf2_to_f2(w.y);
  o[2] = bf2_to_f2(w.z);
  o[3] = bf2_to_f2(w.w);
}
// acc += a (fp32 pairs) * w (8 bf16), pairwise
TW_DEV uint64_t dot8_f2(const uint64_t (&a)[4], const uint4& w, uint64_t acc) {
  acc = f2_fma(a[0], bf2_to_f2(w.x), acc);
  acc = f2_fma(a[1], bf2_to_f2(w.y), acc);
  acc = f2_fma(a[2], bf2_to_f2(w.z), acc);
  acc = f2_fma(a[3], bf2_to_f2(w.w), acc);
  return acc;
}
// Mixed-precision dot of 8 bf16 x 8 bf16 with fp32 accumulation: the bf16
// halves feed the FMA directly (fma.rn.f32.bf16), no unpacking; two partial
// sums keep the dependency chains short.
TW_DEV void bf16_fma(float& acc, uint32_t a_word, uint32_t b_word, bool hi) {
  uint16_t a16, b16;
  if (hi) {
    asm("{ .reg .b16 t; mov.b32 {t, %0}, %1; }" : "=h"(a16) : "r"(a_word));
    asm("{ .reg .b16 t; mov.b32 {t, %0}, %1; }" : "=h"(b16) : "r"(b_word));
  } else {
    asm("{ .reg .b16 t; mov.b32 {%0, t}, %1; }" : "=h"(a16) : "r"(a_word));
    asm("{ .reg .b16 t; mov.b32 {%0, t}, %1; }" : "=h"(b16) : "r"(b_word));
  }
  asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a16), "h"(b16));
}
TW_DEV void dot8_bf16(const uint4& a, const uint4& b, float& acc0, float& acc1) {
  bf16_fma(acc0, a.x, b.x, false);
  bf16_fma(acc1, a.x, b.x, true);
  bf16_fma(acc0, a.y, b.y, false);
  bf16_fma(acc1, a.y, b.y, true);
  bf16_fma(acc0, a.z, b.z, false);
  bf16_fma(acc1, a.z, b.z, true);
  bf16_fma(acc0, a.w, b.w, false);
  bf16_fma(acc1, a.w, b.w, true);
}

// acc (fp32 pairs) += s * w (8 bf16)
TW_DEV void axpy8_f2(uint64_t s2, const uint4& w, uint64_t (&acc)[4]) {
  acc[0] = f2_fma(s2, bf2_to_f2(w.x), acc[0]);
  acc[1] = f2_fma(s2, bf2_to_f2(w.y), acc[1]);
  acc[2] = f2_fma(s2, bf2_to_f2(w.z), acc[2]);
  acc[3] = f2_fma(s2, bf2_to_f2(w.w), acc[3]);
}
TW_DEV uint4 f2x4_to_bf8(const uint64_t (&a)[4]) {
  return make_uint4(pack_bf16x2(f2_lo(a[0]), f2_hi(a[0])), pack_bf16x2(f2_lo(a[1]), f2_hi(a[1])),
                    pack_bf16x2(f2_lo(a[2]), f2_hi(a[2])), pack_bf16x2(f2_lo(a[3]), f2_hi(a[3])));
}

TW_DEV void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace tw
