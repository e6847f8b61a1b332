// sv_device.cuh -- device-side building blocks of the verify-and-commit
// kernels: 16-byte streaming loads, bf16/fp32 element traits, base-2
// exponentials, double-float (hi + lo) accumulation and CTA reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

#ifndef SV_THREADS
#define SV_THREADS 256
#endif
constexpr int kThreads = SV_THREADS;     // threads per CTA of the verify kernel
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------
// 16-byte read-only load that does not allocate in L1: every logit is read
// once by the streaming pass, so L1 would only be polluted.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Element traits: DT 0 = fp32 (4 per 16-byte vector), DT 1 = bf16 (8 per vector).
template <int DT>
struct Elem;

template <>
struct Elem<0> {
  static constexpr int kEPV = 4;
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static float scalar(const void* row, int x) {
    return __ldg(reinterpret_cast<const float*>(row) + x);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[kEPV]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

template <>
struct Elem<1> {
  static constexpr int kEPV = 8;
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static float scalar(const void* row, int x) {
    unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(row) + x);
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
  // bf16 is the top half of an fp32: the low element of a 32-bit word is
  // shifted up, the high one is masked.
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[kEPV]) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xffff0000u);
  }
};

// Loads EPV consecutive elements starting at x (x a multiple of EPV).
// VEC: one 16-byte load (row 16-byte aligned, V a multiple of EPV, x < V).
// !VEC: scalar loads, elements at or past V read as -inf (zero mass).
template <int DT, bool VEC>
__device__ __forceinline__ void load_chunk(const void* row, int x, int V,
                                           float (&f)[Elem<DT>::kEPV]) {
  constexpr int EPV = Elem<DT>::kEPV;
  if constexpr (VEC) {
    if (x < V) {
      Elem<DT>::unpack(ld_stream16(static_cast<const char*>(row) + (size_t)x * Elem<DT>::kBytes), f);
    } else {
#pragma unroll
      for (int j = 0; j < EPV; ++j) f[j] = -INFINITY;
    }
  } else {
#pragma unroll
    for (int j = 0; j < EPV; ++j) f[j] = (x + j < V) ? Elem<DT>::scalar(row, x + j) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (the TMA engine) into shared memory, completed on
// an mbarrier. Addresses are 32-bit shared-window addresses.
// ---------------------------------------------------------------------------
// Upper bound on polls of one mbarrier phase. A healthy copy completes within
// microseconds; reaching the bound means the copy will never land, and the
// caller reports it instead of waiting forever.
constexpr int kSpinLimit = 1 << 22;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async (copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same buffers.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned); its completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The same copy with an L2 eviction-priority hint (a policy from
// l2_policy_*), for data that will soon be read again or never again.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with the given parity; false if it never came.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int it = 0; it < kSpinLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Global-memory flag accesses with acquire/release ordering at GPU scope.
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Read-modify-writes that release this thread's earlier writes and acquire
// the writes released before the values they read (GPU scope): a lighter
// ordering than a full fence (fence.sc) followed by a relaxed atomic.
__device__ __forceinline__ unsigned long long atom_or_acqrel_gpu(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_add_acqrel_gpu(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned atom_add_acqrel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16-byte shared-memory load.
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// ---------------------------------------------------------------------------
// Arithmetic
// ---------------------------------------------------------------------------
// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes in one 64-bit register, for the packed fp32 instructions of
// sm_100 and later (one instruction, two IEEE round-to-nearest results: each
// lane is bit-identical to the scalar instruction).
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
  f2_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ f2_t f2_splat(float x) { return f2_pack(x, x); }
__device__ __forceinline__ void f2_unpack(f2_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
  f2_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_ex2(f2_t v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  return f2_pack(ex2(lo), ex2(hi));
}

// Lane-wise maximum of two bf16 pairs (a NaN lane yields the other operand,
// like fmaxf). Exact, so the fp32 value of the result is the fp32 maximum.
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Double-float value hi + lo (|lo| <= ulp(hi)/2): error-free transformations
// keep sums of fp32 partials accurate to ~2^-44 relative without fp64 math.
struct alignas(8) DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s = a.hi + b.hi;                    // Knuth two-sum of the high parts
  float bb = s - a.hi;
  float e = (a.hi - (s - bb)) + (b.hi - bb);
  e += a.lo + b.lo;
  float hi = s + e;                         // renormalise (fast two-sum)
  float lo = e - (hi - s);
  return {hi, lo};
}

__device__ __forceinline__ DF df_add_f(DF a, float b) { return df_add(a, DF{b, 0.f}); }

// (hi + lo) * f with the product error of the high part kept.
__device__ __forceinline__ DF df_mul_f(DF a, float f) {
  float p = a.hi * f;
  float e = fmaf(a.hi, f, -p);
  e = fmaf(a.lo, f, e);
  float hi = p + e;
  float lo = e - (hi - p);
  return {hi, lo};
}

__device__ __forceinline__ DF df_neg(DF a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ DF df_sub(DF a, DF b) { return df_add(a, df_neg(b)); }

// a <= b for normalised pairs (|lo| <= ulp(hi) / 2).
__device__ __forceinline__ bool df_le(DF a, DF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo <= b.lo); }
__device__ __forceinline__ bool df_pos(DF a) { return a.hi > 0.f || (a.hi == 0.f && a.lo > 0.f); }

// a / b to about 2^-44 relative: a quotient in fp32, then its correction
// from the exact remainder (one more fp32 division). b must be nonzero.
__device__ __forceinline__ DF df_div(DF a, DF b) {
  const float q1 = __fdiv_rn(a.hi, b.hi);
  // remainder a - q1 * b, with q1 * b.hi split exactly
  const float p = q1 * b.hi;
  const float pe = fmaf(q1, b.hi, -p);
  DF r = df_sub(a, DF{p, pe});
  r = df_add_f(r, -q1 * b.lo);
  const float q2 = __fdiv_rn(r.hi, b.hi);
  const float hi = q1 + q2;
  return {hi, q2 - (hi - q1)};
}

__device__ __forceinline__ double df_to_d(DF a) { return (double)a.hi + (double)a.lo; }
__device__ __forceinline__ DF df_from_d(double d) {
  const float hi = (float)d;
  return {hi, (float)(d - (double)hi)};
}
// An 8-byte global load that bypasses L1 (data another CTA may have written).
__device__ __forceinline__ DF ldcg_df(const DF* p) {
  const float2 v = __ldcg(reinterpret_cast<const float2*>(p));
  return {v.x, v.y};
}

// ---------------------------------------------------------------------------
// Warp / CTA reductions (kThreads threads, all participating)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    DF w{__shfl_xor_sync(kFull, v.hi, o), __shfl_xor_sync(kFull, v.lo, o)};
    v = df_add(v, w);
  }
  return v;
}

// (value, index) argmax: larger value wins, equal values keep the lower index.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(kFull, v, o);
    int i2 = __shfl_xor_sync(kFull, i, o);
    argmax_merge(v, i, v2, i2);
  }
}

// Inclusive prefix sum across a warp (Kogge-Stone, fixed order).
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float u = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// The same scan in double-float.
__device__ __forceinline__ DF warp_incl_scan_df(DF v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF u{__shfl_up_sync(kFull, v.hi, o), __shfl_up_sync(kFull, v.lo, o)};
    if (lane >= o) v = df_add(u, v);
  }
  return v;
}

__device__ __forceinline__ double warp_incl_scan_d(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double u = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

}  // namespace sv
