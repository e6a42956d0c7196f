// sv_device.cuh -- sm_103a device primitives for libspecverify: mbarriers,
// 1-D bulk (TMA engine) copies, bounded waits, bf16 unpacking, fast exp2 and
// warp reductions.  Every wait in this library is bounded by a wall-clock
// limit read from %globaltimer; on expiry the caller records an error and
// carries on, so no kernel can spin forever.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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

// Named barrier over the first `count` threads of the block.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
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
__device__ __forceinline__ double warp_incl_scan_d(double x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__device__ __forceinline__ void record_error(int* err, int flag) { atomicOr(err, flag); }

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

}  // namespace sv
