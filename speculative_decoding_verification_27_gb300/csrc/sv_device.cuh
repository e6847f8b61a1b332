// sv_device.cuh -- device-side building blocks of the verify-and-commit
// kernels: 16-byte streaming loads, bf16/fp32 element traits, base-2
// exponentials, double-float (hi + lo) accumulation and CTA reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kThreads = 256;            // threads per CTA of the verify kernel
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
// Arithmetic
// ---------------------------------------------------------------------------
// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Double-float value hi + lo (|lo| <= ulp(hi)/2): error-free transformations
// keep sums of fp32 partials accurate to ~2^-44 relative without fp64 math.
struct DF {
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

__device__ __forceinline__ double warp_incl_scan_d(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double u = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

}  // namespace sv
