// sv_device.cuh -- sm_103a device primitives for libspecverify: mbarriers,
// 1-D bulk (TMA engine) copies, bounded waits, bf16 unpacking, fast exp2 and
// warp reductions.  Every wait in this library is bounded by a wall-clock
// limit read from %globaltimer; on expiry the caller records an error and
// carries on, so no kernel can spin forever.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"

namespace sv {

constexpr float kPosInf = __builtin_huge_valf();
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed, for at most
// limit_ns nanoseconds.  Returns false when the limit expired.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// 1-D bulk copy global -> shared through the TMA engine; completion is
// signalled on `bar` as `bytes` transaction bytes.  Both addresses must be
// 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* gmem_src,
                                              uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Order this thread's earlier generic-proxy accesses to shared memory
// before later async-proxy ones (a bulk copy into a buffer just read).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_copy_g2s_hint(void* smem_dst, const void* gmem_src,
                                                   uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// Programmatic dependent launch.  wait: block until the grids this launch
// depends on have completed and their memory operations are visible.
// launch_dependents: let the next dependent grid begin launching; it still
// waits for this grid's completion before it touches memory.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// L2 prefetch of the line holding p (a hint: no value is read).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over the first `count` threads of the block (whole,
// converged warps: the caller reconverges after divergent code).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Arrive on a named barrier without waiting (the producer side of a
// hand-over: this warp's earlier writes are visible to the threads that
// wait on the barrier with named_sync).  The barrier counts whole warps,
// so the warp is reconverged first: a lane still inside a branch would
// otherwise be counted as arrived before its writes.
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t count) {
  __syncwarp();
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ values

// bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// 2^x through the MUFU.EX2 unit (relative error about 2^-22; flushes
// results below 2^-126 to zero).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x in fp64 for x <= 0 (x = -inf gives 0).  x = n + f with n = rint(x)
// and |f| <= 1/2; 2^f = e^t, t = f ln 2, |t| < 0.347, by the Taylor series
// of e^t to degree 13 (truncation below 4e-18 relative) in Horner form;
// 2^n is applied through the exponent field in two factors so that results
// down to the subnormal range come out right.  About 20 fp64 operations:
// much shorter than a general-purpose exp2 on a part whose fp64 rate is low.
__device__ __forceinline__ double exp2_nonpos(double x) {
  if (!(x > -1080.0)) return 0.0;
  const double n = rint(x);
  const double t = (x - n) * 0.69314718055994530942;
  // 1/k!, evaluated at compile time
  constexpr double f2 = 1.0 / 2, f3 = f2 / 3, f4 = f3 / 4, f5 = f4 / 5, f6 = f5 / 6;
  constexpr double f7 = f6 / 7, f8 = f7 / 8, f9 = f8 / 9, f10 = f9 / 10, f11 = f10 / 11;
  constexpr double f12 = f11 / 12, f13 = f12 / 13;
  double e = fma(f13, t, f12);
  e = fma(e, t, f11);
  e = fma(e, t, f10);
  e = fma(e, t, f9);
  e = fma(e, t, f8);
  e = fma(e, t, f7);
  e = fma(e, t, f6);
  e = fma(e, t, f5);
  e = fma(e, t, f4);
  e = fma(e, t, f3);
  e = fma(e, t, f2);
  e = fma(e, t, 1.0);
  e = fma(e, t, 1.0);
  const int ni = static_cast<int>(n);  // -1080 .. 0
  const int n1 = ni / 2, n2 = ni - n1;
  const double s1 = __longlong_as_double(static_cast<long long>(1023 + n1) << 52);
  const double s2 = __longlong_as_double(static_cast<long long>(1023 + n2) << 52);
  return (e * s1) * s2;
}

// 1/z for 2^-125 <= z <= 2^125 with fused multiply-adds only (no special-
// function unit, which the streaming reduction keeps busy): z = m 2^e with
// m in [1/2, 1), the linear start 48/17 - 32/17 m (relative error at most
// 1/17), three Newton-Raphson steps y += y (1 - m y) (error squared each
// step), then the exponent.  Accurate to about one ulp.
__device__ __forceinline__ float rcp_fma(float z) {
  const unsigned zb = __float_as_uint(z);
  const int e = static_cast<int>((zb >> 23) & 0xffu) - 126;
  const float m = __uint_as_float((zb & 0x007fffffu) | 0x3f000000u);
  float y = __fmaf_rn(-32.f / 17.f, m, 48.f / 17.f);
#pragma unroll
  for (int k = 0; k < 3; ++k) y = __fmaf_rn(y, __fmaf_rn(-m, y, 1.f), y);
  return __uint_as_float(__float_as_uint(y) - (static_cast<unsigned>(e) << 23));
}

// Packed max of two bf16 pairs, NaN-propagating.
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// log2(e)/t as an unevaluated float pair (hi + lo), so that the scaling of
// every exponent carries no systematic rounding of the constant.
struct Scale2 {
  float hi, lo;
};

// (x - m) * log2(e)/t with x - m exact for bf16 inputs.
__device__ __forceinline__ float scaled_arg(float x, float m, Scale2 c) {
  const float d = x - m;
  return fmaf(d, c.hi, d * c.lo);
}

// 2^((x - m) c) for x <= m to about 5e-7 relative, whatever the size of the
// exponent: the exponent is carried as an unevaluated pair -- x - m exactly
// (TwoSum), the product's rounding error by FMA -- the high part goes
// through ex2.approx and the low part (below 2^-23 of the high part) to
// first order.  a_hi returns the high part (exponents below -126 flush to
// zero).
__device__ __forceinline__ float exp2_scaled_pair(float x, float m, Scale2 c, float& a_hi) {
  const float d = x - m;
  const float bv = d - x;
  const float d_lo = (x - (d - bv)) + (-m - bv);
  const float p = d * c.hi;
  const float lo = fmaf(d, c.hi, -p) + fmaf(d_lo, c.hi, d * c.lo);
  a_hi = p;
  return fast_exp2(p) * fmaf(lo, 0.693147180559945f, 1.f);
}

// ------------------------------------------------- (max, sum) combination

// Online-softmax pair: the row max m and s = sum 2^((x - m) c).  m = -inf
// with s = 0 is the empty pair; m = NaN marks a row with a NaN / +inf.
struct MS {
  float m, s;
};

__device__ __forceinline__ MS ms_combine(MS a, MS b, Scale2 c) {
  if (a.m != a.m || b.m != b.m) return MS{__int_as_float(0x7fc00000), 0.f};
  const float m = fmaxf(a.m, b.m);
  if (m == kNegInf) return MS{kNegInf, 0.f};
  float s = 0.f;
  if (a.m != kNegInf) s += a.s * fast_exp2(scaled_arg(a.m, m, c));
  if (b.m != kNegInf) s += b.s * fast_exp2(scaled_arg(b.m, m, c));
  return MS{m, s};
}

// Warp-wide combination of (m, s) pairs: the maximum first, then each lane
// rescales its sum once to the common maximum and the sums are added.
__device__ __forceinline__ MS warp_reduce_ms(MS v, Scale2 c) {
  const bool bad = __any_sync(0xffffffffu, v.m != v.m);
  float m = v.m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (bad) return MS{__int_as_float(0x7fc00000), 0.f};
  if (m == kNegInf) return MS{kNegInf, 0.f};
  float s = v.m == kNegInf ? 0.f : v.s * fast_exp2(scaled_arg(v.m, m, c));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return MS{m, s};
}

// Argmax pair: value and lowest index attaining it.  NaN value marks a row
// with a NaN / +inf entry.
struct VI {
  float v;
  int i;
};

__device__ __forceinline__ VI vi_better(VI a, VI b) {
  if (a.v != a.v) return a;
  if (b.v != b.v) return b;
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}

__device__ __forceinline__ VI warp_reduce_vi(VI v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    VI w;
    w.v = __shfl_xor_sync(0xffffffffu, v.v, o);
    w.i = __shfl_xor_sync(0xffffffffu, v.i, o);
    v = vi_better(v, w);
  }
  return v;
}

// Inclusive warp scan (Kogge-Stone) of floats and doubles.
__device__ __forceinline__ float warp_incl_scan(float x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}
__device__ __forceinline__ unsigned warp_incl_scan_u(unsigned x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}
__device__ __forceinline__ double warp_incl_scan_d(double x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// ------------------------------------------------- float-pair (hi + lo) sums

// An unevaluated pair hi + lo for running sums that must stay far more
// accurate than fp32 rounding (about 2^-44 relative) without fp64, which is
// slow on this part.  Built on the error-free sum of two floats (Knuth's
// TwoSum) and on the fused multiply-add residual of a product; every step
// is an explicitly rounded intrinsic so the compiler cannot contract it.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
  return DF{s, e};
}

// (a + b) renormalised, for |a| >= |b| or a == 0
__device__ __forceinline__ DF quick_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return DF{s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ DF df_add(DF x, float y) {
  const DF s = two_sum(x.hi, y);
  return quick_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}

__device__ __forceinline__ DF df_add(DF x, DF y) {
  const DF s = two_sum(x.hi, y.hi);
  return quick_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}

// u * x for a float u
__device__ __forceinline__ DF df_mul(float u, DF x) {
  const float p = __fmul_rn(u, x.hi);
  const float e = __fmaf_rn(u, x.hi, -p);
  return quick_two_sum(p, __fmaf_rn(u, x.lo, e));
}

__device__ __forceinline__ bool df_lt(DF a, DF b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

__device__ __forceinline__ DF df_shfl(DF x, int src) {
  return DF{__shfl_sync(0xffffffffu, x.hi, src), __shfl_sync(0xffffffffu, x.lo, src)};
}

// Inclusive warp scan of pairs (Kogge-Stone).
__device__ __forceinline__ DF warp_incl_scan_df(DF x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF y{__shfl_up_sync(0xffffffffu, x.hi, o), __shfl_up_sync(0xffffffffu, x.lo, o)};
    if (lane >= o) x = df_add(y, x);
  }
  return x;
}

__device__ __forceinline__ void record_error(int* err, int flag) { atomicOr(err, flag); }

// Internal checks of debug builds (-DSV_CHECKS): SV_CHECK(cond, err) is
// true when cond holds; otherwise it sets SV_DERR_CHECK in the error word
// *err and is false, and the caller skips the access it guards.  Release
// builds compile every check to true.
#ifdef SV_CHECKS
__device__ __forceinline__ bool sv_check(bool ok, int* err) {
  if (!ok) record_error(err, SV_DERR_CHECK);
  return ok;
}
#define SV_CHECK(cond, err) ::sv::sv_check(static_cast<bool>(cond), (err))
#else
#define SV_CHECK(cond, err) true
#endif
// a 1-D bulk copy's requirements: both addresses 16-byte aligned, a size
// that is a positive multiple of 16 bytes
__device__ __forceinline__ bool bulk_args_ok(const void* dst, const void* src, uint32_t bytes) {
  return ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | bytes) & 15u) == 0 &&
         bytes > 0;
}

// Fetch-and-add with acquire-release semantics at GPU scope: orders this
// thread's earlier stores before the add (release) and, for the thread that
// reads the final count, makes every earlier releaser's stores visible
// (acquire).  No separate fence is needed on the hot path.
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// 64-bit words read and written whole (single-copy atomic), for values that
// other CTAs poll.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Four consecutive 32-bit words read with one relaxed GPU-scope load (each
// word single-copy atomic), for polling several words per round trip.
__device__ __forceinline__ uint4 ld_relaxed_v4(const unsigned* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

}  // namespace sv
