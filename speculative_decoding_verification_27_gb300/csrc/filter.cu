// filter.cu -- per-row thresholds of the top-k / top-p filters.
//
// "投机解码从零实现" (CSDN), §5.4 "采样策略对比": top-k and nucleus
// (top-p) rejection sampling keep the output distribution when the same
// filter is applied to the target and the draft distributions before the
// accept test and the residual. For every row this kernel finds a value
// threshold tau such that the filtered distribution keeps exactly the
// tokens with logit >= tau:
//   top-k (1 <= k < V): tau = the k-th largest logit (ties all kept);
//   then top-p (0 < p < 1): over the kept tokens, walking distinct logit
//     values from the largest down, the first value at which the cumulative
//     mass reaches p of the kept mass (its whole tie group is kept).
// tau = -inf keeps every token.
//
// Method: logits map to order-preserving unsigned keys (-0 folded into +0),
// and each threshold is a radix select over 8-bit digits of the key, most
// significant first. Every level is one pass over the row that histograms
// the next digit of the keys still in play: counts for top-k, masses
// 2^(z c - M c) (M the row maximum, c = log2(e) / T) for top-p. Each warp
// keeps its own histogram in shared memory, and a thread merges runs of
// equal digits in its vector before adding, because logits of one row share
// few leading digits.
//
// With top-k for k <= 256 a row is read from global memory once. Every
// logit at or above a floor is appended to a buffer in shared memory, and
// the floor never exceeds the k-th largest logit seen so far, so the buffer
// always holds the row's top-k set. The first floor is the k-th largest of
// the 256 threads' maxima over the first chunk (k of those maxima lie at or
// above it). If the buffer could overflow in the next chunk, the floor rises
// to the k-th largest value in the buffer and the buffer is compacted. After
// the pass, the radix levels above run on the buffer alone. A row whose tie
// group at the floor does not fit falls back to the passes over the row.
#include "../../include/spec_verify.h"
#include "sv_filter.cuh"

#include <cmath>
#include <cstdint>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sv {

constexpr int kFtThreads = 256;
constexpr int kFtWarps = kFtThreads / 32;
constexpr int kFtBatch = 4;  // 16-byte loads a thread issues before using them

// Order-preserving keys. bf16: the 16-bit pattern; fp32: the 32-bit pattern.
__device__ __forceinline__ uint32_t key16(uint32_t u) {
  if (u == 0x8000u) u = 0u;  // -0 -> +0
  return (u & 0x8000u) ? (~u & 0xffffu) : (u | 0x8000u);
}
__device__ __forceinline__ uint32_t key32(uint32_t u) {
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float value16(uint32_t k) {
  const uint32_t u = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
  return __uint_as_float(u << 16);
}
__device__ __forceinline__ float value32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr int kCand = 4096;      // logits that shared memory holds once few keys are left in play
constexpr int kStreamK = 256;    // top-k up to this collects its candidates in one pass
constexpr int kChunkWords = 4;   // 16-byte words a thread holds per chunk of the one-pass collection
// Chunks between checkpoints of the one-pass collection. Top-p alone and
// small top-k append few logits per chunk, so their checkpoints (barriers)
// can be sparse; a large k fills the buffer faster and needs its floor
// raised sooner. Measured on the benchmark batch: every 8 chunks for top-p
// alone and k = 50, every 2 for k = 256 (every 8 there overflows the buffer
// into the passes over the row).
constexpr int kCheckSparse = 8;
constexpr int kCheckDense = 2;
constexpr int kSparseMaxK = 64;
#ifndef SV_KTH_CHUNKS
#define SV_KTH_CHUNKS 0x808Bu
#endif
// Chunks (bit c, c < 16) after which top-k raises its floor to the k-th
// largest of the threads' running maxima: 0, 1, 3, 7 and 15 by default.
constexpr unsigned kKthChunks = SV_KTH_CHUNKS;

constexpr int kHistCopies = 2;  // per-pair-of-warps histogram copies
constexpr int kRing = 3;        // chunks of the one-pass collection in shared memory (two in flight)

struct FtSmem {
  uint4 ring[kRing][kChunkWords][kFtThreads];  // thread t's words of a chunk at [.][u][t]
  unsigned cnt[kHistCopies][256];
  // Mass bins in fixed point (units of 2^-44): every mass is at most ~1
  // (relative to the row maximum or the integer reference), so its fp32
  // value times 2^44 converts exactly (to the unit for masses below 2^-20),
  // a row of at most 2^19 logits fits in 64 bits, and the sums are exact in
  // any order. The nucleus cut compares them against the 1e-6 flag margin.
  unsigned long long mass[kHistCopies][256];
  unsigned tc[256];          // per-digit counts
  double tm[256];            // per-digit mass totals (mass levels only)
  float wmax[kFtWarps];
  unsigned wcount[kFtWarps];
  float cand[kCand];        // the logits still in play, once they fit
  unsigned ncand;
  float wm[2][kFtWarps];      // per-warp running reference and mass (one-pass top-p bound)
  float wsf[2][kFtWarps];
  double wsd[kFtWarps];       // per-warp mass in double (end of the one-pass top-p)
  double row_mass;            // one-pass top-p: mass left out of the buffer, relative to 2^row_ref
  float row_ref;              // one-pass top-p: the row's integer mass reference (log2 units)
  uint32_t digit;
  unsigned before_c;          // count of the digits above the chosen one
  double before_m;            // and their mass (mass levels)
  double total_m;
  float rowmax;
};

template <int DT>
__device__ __forceinline__ uint32_t key_of(float v) {
  return DT == 1 ? key16(__float_as_uint(v) >> 16) : key32(__float_as_uint(v));
}

// Visits every logit of a row as (key, value): 16-byte vectors when the row
// allows, element by element otherwise.
template <int DT>
struct RowSrc {
  const void* row;
  int V;
  bool vec;
  template <class F>
  __device__ __forceinline__ void each(F&& f) const {
    const int tid = threadIdx.x;
    if (DT == 1) {
      const uint16_t* r = static_cast<const uint16_t*>(row);
      if (vec) {
        const uint4* rv = reinterpret_cast<const uint4*>(row);
        const int nv = V / 8;
        // kFtBatch 16-byte loads in flight per thread, then their logits.
        for (int j0 = 0; j0 < nv; j0 += kFtBatch * kFtThreads) {
          uint4 w[kFtBatch];
#pragma unroll
          for (int u = 0; u < kFtBatch; ++u) {
            const int j = j0 + u * kFtThreads + tid;
            w[u] = j < nv ? __ldg(rv + j) : make_uint4(0xffffu, 0xffffu, 0xffffu, 0xffffu);
          }
#pragma unroll
          for (int u = 0; u < kFtBatch; ++u) {
            if (j0 + u * kFtThreads + tid >= nv) break;
            const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              f(key16(ws[q] & 0xffffu), __uint_as_float(ws[q] << 16));
              f(key16(ws[q] >> 16), __uint_as_float(ws[q] & 0xffff0000u));
            }
          }
        }
      } else {
        for (int x = tid; x < V; x += kFtThreads) {
          const uint32_t u = __ldg(r + x);
          f(key16(u), __uint_as_float(u << 16));
        }
      }
    } else {
      const float* r = static_cast<const float*>(row);
      if (vec) {
        const float4* rv = reinterpret_cast<const float4*>(row);
        const int nv = V / 4;
        for (int j0 = 0; j0 < nv; j0 += kFtBatch * kFtThreads) {
          float4 w[kFtBatch];
#pragma unroll
          for (int u = 0; u < kFtBatch; ++u) {
            const int j = j0 + u * kFtThreads + tid;
            w[u] = j < nv ? __ldg(rv + j) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < kFtBatch; ++u) {
            if (j0 + u * kFtThreads + tid >= nv) break;
            const float ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) f(key32(__float_as_uint(ws[q])), ws[q]);
          }
        }
      } else {
        for (int x = tid; x < V; x += kFtThreads) {
          const float z = __ldg(r + x);
          f(key32(__float_as_uint(z)), z);
        }
      }
    }
  }
};

// The collected logits in shared memory (any order).
template <int DT>
struct CandSrc {
  const float* v;
  int n;
  template <class F>
  __device__ __forceinline__ void each(F&& f) const {
    for (int j = threadIdx.x; j < n; j += kFtThreads) f(key_of<DT>(v[j]), v[j]);
  }
};

// Histogram of digit (key >> shift) & 255 over the keys >= floor whose
// higher digits equal `prefix` (all keys at the top level): counts always,
// masses 2^(v c - mc) when by_mass; with track_max also the largest value
// (into s.rowmax). Per-digit totals land in s.tc / s.tm, the mass total in
// s.total_m.
// kWarpBins: one bin copy per warp, kept in the one-pass collection's ring
// (idle outside it), for mass passes over a whole row: a flat row's keys
// crowd into few digits, and warps sharing bins serialize on their 64-bit
// atomics. Otherwise the kHistCopies copies in FtSmem (cheaper to clear and
// sum; enough for count passes and for the buffered candidates).
template <int DT, class Src, bool kWarpBins = false>
__device__ void histogram(FtSmem& s, const Src& src, int shift, uint32_t prefix, bool top_level,
                          uint32_t floor, bool by_mass, float c, float mc, bool track_max) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int ncp = kWarpBins ? kFtWarps : kHistCopies;
  static_assert(!kWarpBins || kFtWarps * 256 * (sizeof(unsigned) + sizeof(unsigned long long)) <= sizeof(s.ring),
                "the per-warp bins fit in the ring");
  unsigned* cnt;
  unsigned long long* mass;
  if constexpr (kWarpBins) {
    cnt = reinterpret_cast<unsigned*>(&s.ring[0][0][0]);
    mass = reinterpret_cast<unsigned long long*>(cnt + kFtWarps * 256);
  } else {
    cnt = &s.cnt[0][0];
    mass = &s.mass[0][0];
  }
  const int cp = (kWarpBins ? warp : (warp & (kHistCopies - 1))) * 256;
  for (int k = tid; k < ncp * 256; k += kFtThreads) {
    cnt[k] = 0u;
    mass[k] = 0ull;
  }
  __syncthreads();
  // Runs of one digit are merged in registers before they reach shared memory.
  uint32_t run_d = 0xffffffffu;
  unsigned run_n = 0;
  unsigned long long run_m = 0ull;
  float vmax = -INFINITY;
  auto flush = [&]() {
    if (run_n) {
      atomicAdd(&cnt[cp + run_d], run_n);
      if (by_mass) atomicAdd(&mass[cp + run_d], run_m);
    }
  };
  src.each([&](uint32_t key, float v) {
    if (track_max) vmax = fmaxf(vmax, v);
    if (key < floor) return;
    if (!top_level && (key >> (shift + 8)) != prefix) return;
    const uint32_t d = (key >> shift) & 255u;
    if (d != run_d) {
      flush();
      run_d = d;
      run_n = 0;
      run_m = 0ull;
    }
    ++run_n;
    if (by_mass) run_m += __float2ull_rn(exp2f(fmaf(v, c, -mc)) * 0x1p44f);
  });
  flush();
  if (track_max) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    if (lane == 0) s.wmax[warp] = vmax;
  }
  __syncthreads();
  // Counts stay integers; only mass levels pay for double precision (the
  // FP64 pipe is narrow on this part).
  unsigned tc = 0u;
#pragma unroll
  for (int w = 0; w < ncp; ++w) tc += cnt[w * 256 + tid];
  s.tc[tid] = tc;
  if (by_mass) {
    double tm = 0.0;
    unsigned long long tq = 0ull;
#pragma unroll
    for (int w = 0; w < ncp; ++w) tq += mass[w * 256 + tid];
    tm = (double)tq * 0x1p-44;
    s.tm[tid] = tm;
  }
  if (tid == 0 && track_max) {
    float r = s.wmax[0];
    for (int w = 1; w < kFtWarps; ++w) r = fmaxf(r, s.wmax[w]);
    s.rowmax = r;
  }
  __syncthreads();
  if (by_mass && tid < 32) {
    double t = 0.0;
    for (int j = tid; j < 256; j += 32) t += s.tm[j];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (tid == 0) s.total_m = t;
  }
  __syncthreads();
}

// The first digit from the top at which the running count reaches need_c
// (count levels) or the running mass reaches need_m (mass levels): s.digit,
// with the count and mass of the digits above it in s.before_c /
// s.before_m, taken from the warp's scans. If rounding leaves need_m
// unreached, the lowest digit is taken (everything in play stays).
__device__ void pick_digit(FtSmem& s, unsigned need_c, double need_m, bool by_mass) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    // Lane l covers digits 255 - 8l .. 248 - 8l (from the top).
    unsigned lc[8], csum = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      lc[j] = s.tc[255 - 8 * lane - j];
      csum += lc[j];
    }
    unsigned cincl = csum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned n = __shfl_up_sync(0xffffffffu, cincl, o);
      if (lane >= o) cincl += n;
    }
    unsigned cexcl = __shfl_up_sync(0xffffffffu, cincl, 1);
    if (lane == 0) cexcl = 0u;
    double lm[8], mincl = 0.0, mexcl = 0.0;
    if (by_mass) {
      double msum = 0.0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        lm[j] = s.tm[255 - 8 * lane - j];
        msum += lm[j];
      }
      mincl = msum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, mincl, o);
        if (lane >= o) mincl += n;
      }
      mexcl = __shfl_up_sync(0xffffffffu, mincl, 1);
      if (lane == 0) mexcl = 0.0;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) lm[j] = 0.0;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, by_mass ? mincl >= need_m : cincl >= need_c);
    const int first = hit ? __ffs(hit) - 1 : 31;
    if (lane == first) {
      unsigned bc = cexcl;
      double bm = mexcl;
      int j = 0;
      for (; j < 7; ++j) {
        if (by_mass ? bm + lm[j] >= need_m : bc + lc[j] >= need_c) break;
        bc += lc[j];
        bm += lm[j];
      }
      s.digit = 255u - 8u * (uint32_t)lane - (uint32_t)j;
      s.before_c = bc;
      s.before_m = bm;
    }
  }
  __syncthreads();
}

// Copies the row's logits with key >= lo into shared memory (the caller has
// checked that they fit).
template <int DT>
__device__ void collect(FtSmem& s, const RowSrc<DT>& row, uint32_t lo) {
  if (threadIdx.x == 0) s.ncand = 0u;
  __syncthreads();
  row.each([&](uint32_t key, float v) {
    if (key >= lo) {
      const unsigned slot = atomicAdd(&s.ncand, 1u);
      if (slot < (unsigned)kCand) s.cand[slot] = v;
    }
  });
  __syncthreads();
}

// Starts the copy of this thread's share of chunk c into ring stage
// c % kRing: kChunkWords 16-byte words, word u at index
// (c * kChunkWords + u) * kFtThreads + tid of the row viewed as 16-byte
// words; logits past V read as -inf. Vector rows copy asynchronously
// (cp.async, completed by the caller's wait); other rows load and store.
// Each thread reads back only its own words, so no barrier is involved.
template <int DT>
__device__ __forceinline__ void issue_chunk(FtSmem& s, const void* row, int V, bool vec, int c) {
  constexpr int EV = DT == 1 ? 8 : 4;  // logits per 16-byte word
  constexpr uint32_t kNegInf = DT == 1 ? 0xff80ff80u : 0xff800000u;
  const int tid = threadIdx.x;
#pragma unroll
  for (int u = 0; u < kChunkWords; ++u) {
    const int j = (c * kChunkWords + u) * kFtThreads + tid;
    const int e0 = j * EV;
    uint4* slot = &s.ring[c % kRing][u][tid];
    if (vec) {
      // V * s is a multiple of 16 bytes: a word is wholly inside or outside.
      if (e0 < V) {
        const unsigned dst = (unsigned)__cvta_generic_to_shared(slot);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst),
                     "l"(reinterpret_cast<const uint4*>(row) + j)
                     : "memory");
      } else {
        *slot = make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
      }
    } else {
      uint32_t ws[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (DT == 1) {
          const uint16_t* r = static_cast<const uint16_t*>(row);
          const int e = e0 + 2 * q;
          const uint32_t lo = e < V ? __ldg(r + e) : 0xff80u;
          const uint32_t hi = e + 1 < V ? __ldg(r + e + 1) : 0xff80u;
          ws[q] = lo | (hi << 16);
        } else {
          const float* r = static_cast<const float*>(row);
          const int e = e0 + q;
          ws[q] = e < V ? __float_as_uint(__ldg(r + e)) : kNegInf;
        }
      }
      *slot = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    }
  }
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// All but the most recent group of this thread's copies have landed.
__device__ __forceinline__ void cp_async_wait_but_one() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// The k-th largest key among one key per thread (1 <= k <= kFtThreads): the
// largest T with at least k keys >= T, one bit at a time from the top.
template <int DT>
__device__ __forceinline__ uint32_t kth_key_of_threads(uint32_t key, int k) {
  constexpr int KB = DT == 1 ? 16 : 32;
  uint32_t T = 0u;
  for (int bit = KB - 1; bit >= 0; --bit) {
    const uint32_t t = T | (1u << bit);
    if (__syncthreads_count(key >= t) >= k) T = t;
  }
  return T;
}

// A key as a floor value; keys below -inf's (NaN patterns) keep everything.
template <int DT>
__device__ __forceinline__ float floor_value(uint32_t T) {
  constexpr uint32_t kKeyNegInf = DT == 1 ? 0x007fu : 0x007fffffu;
  if (T <= kKeyNegInf) return -INFINITY;
  return DT == 1 ? value16(T) : value32(T);
}

// Exact k-th largest key of the buffer (s.cand[0, s.ncand)) by the radix
// levels, then a stable in-place compaction to the values >= it. The new
// floor goes to `fl`; returns the number of values kept (the same in every
// thread, so callers branch on it without reading shared memory again).
template <int DT>
__device__ int raise_floor(FtSmem& s, int k, float& fl_out) {
  constexpr int KB = DT == 1 ? 16 : 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = (int)s.ncand;
  const CandSrc<DT> cs{s.cand, n};
  uint32_t prefix = 0u;
  unsigned need = (unsigned)k;
  for (int sh = KB - 8; sh >= 0; sh -= 8) {
    histogram<DT>(s, cs, sh, prefix, sh == KB - 8, 0u, false, 0.f, 0.f, false);
    pick_digit(s, need, 0.0, false);
    need -= s.before_c;
    prefix = (prefix << 8) | s.digit;
  }
  const float fl = floor_value<DT>(prefix);
  // Round r reads entries [256 r, 256 r + 256) before any write of the round;
  // a kept entry moves to a position at or below its own.
  int out = 0;
  for (int base = 0; base < n; base += kFtThreads) {
    const int j = base + tid;
    const float v = j < n ? s.cand[j] : -INFINITY;
    const bool keep = j < n && v >= fl;
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s.wcount[warp] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kFtWarps; ++w) {
      const int c = (int)s.wcount[w];
      before += w < warp ? c : 0;
      total += c;
    }
    if (keep) s.cand[out + before + __popc(bal & ((1u << lane) - 1u))] = v;
    out += total;
    __syncthreads();
  }
  if (tid == 0) s.ncand = (unsigned)out;
  __syncthreads();
  fl_out = fl;
  return out;
}

// 32-bit word q of a thread's chunk share (two bf16 logits or one fp32).
__device__ __forceinline__ uint32_t word_at(const uint4 (&w)[kChunkWords], int q) {
  const uint4 x = w[q >> 2];
  const int r = q & 3;
  return r == 0 ? x.x : (r == 1 ? x.y : (r == 2 ? x.z : x.w));
}

// Packed bf16 pairs: per-half (a >= b) as 0xffff masks, and the per-half maximum.
__device__ __forceinline__ uint32_t bf2_ge_mask(uint32_t a, uint32_t b) {
  __nv_bfloat162 x, y;
  memcpy(&x, &a, 4);
  memcpy(&y, &b, 4);
  return __hge2_mask(x, y);
}
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  __nv_bfloat162 x, y;
  memcpy(&x, &a, 4);
  memcpy(&y, &b, 4);
  const __nv_bfloat162 r = __hmax2(x, y);
  uint32_t u;
  memcpy(&u, &r, 4);
  return u;
}

// Running state of the one-pass collection, per thread.
//   top-k: rmax is the running maximum.
//   top-p: masses are kept relative to 2^ref with ref an integer (log2
//   units, ref >= rmax * cc), so that moving to a larger reference is an
//   exact power-of-two rescale. sum_all is the mass of every logit seen (for
//   the floor); sum_rest the mass of those not appended, in double (the
//   row's mass is the buffer's, summed later exactly as the nucleus walk
//   sums it, plus this).
struct StreamState {
  float fl;         // floor: logits >= fl are appended
  uint32_t fl2;     // bf16: the floor in both halves
  float rmax;       // running maximum
  float ref;        // top-p: integer reference, or -inf before any finite logit
  float sum_all;    // top-p: mass of every logit seen, relative to 2^ref
  double sum_rest;  // top-p: mass of the logits not appended, relative to 2^ref
  unsigned my_end;  // largest buffer end of this thread's appends since the last checkpoint
  bool my_ovf;      // an append since the last checkpoint found the buffer full
};

// Raises the floor to f. bf16 rows round f down to a bf16 value first, so
// that the packed compare (fl2) and the float compare (fl) agree.
template <int DT>
__device__ __forceinline__ void set_floor(StreamState& st, float f) {
  if (DT == 1) {
    const uint32_t u = __float_as_uint(f);
    uint32_t hi = u & 0xffff0000u;
    if ((u & 0x80000000u) && (u & 0xffffu)) hi += 0x10000u;  // negative: away from zero
    f = __uint_as_float(hi);
  }
  st.fl = fmaxf(st.fl, f);
  const uint32_t fb = __float_as_uint(st.fl) >> 16;
  st.fl2 = fb | (fb << 16);
}

// (reference, mass) over the warp: the mass rescaled to the warp's largest
// reference by powers of two.
__device__ __forceinline__ void warp_ref_mass(float& ref, float& sm) {
  float wr = ref;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) wr = fmaxf(wr, __shfl_xor_sync(0xffffffffu, wr, o));
  sm = ref > -INFINITY ? ldexpf(sm, (int)(ref - wr)) : 0.f;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
  ref = wr;
}

// The top-p floor from the warps' (reference, mass) in slot `slot`: every
// logit whose mass is below (1 - p) S / V lies outside the nucleus
// (together they weigh less than (1 - p) S), and S only grows as the pass
// goes on. The 0.05 in log2 units keeps the bound below the exact one
// despite fp32 sums.
__device__ __forceinline__ float top_p_floor(const FtSmem& s, int slot, float p, float cc, int V) {
  float R = -INFINITY, S = 0.f;
#pragma unroll
  for (int w = 0; w < kFtWarps; ++w) R = fmaxf(R, s.wm[slot][w]);
  if (!(R > -INFINITY)) return -INFINITY;
#pragma unroll
  for (int w = 0; w < kFtWarps; ++w)
    if (s.wm[slot][w] > -INFINITY) S += ldexpf(s.wsf[slot][w], (int)(s.wm[slot][w] - R));
  return (R + log2f((1.f - p) * S / (float)V) - 0.05f) / cc;
}

// Appends this thread's logits of chunk c that are >= the floor (logits past
// V excepted). my_end: the largest buffer end this thread's appends reached;
// my_ovf: a logit found the buffer full and was dropped.
template <int DT>
__device__ __forceinline__ void append_chunk(FtSmem& s, const uint4 (&cur)[kChunkWords], int c, int V,
                                             const StreamState& st, unsigned& my_end, bool& my_ovf) {
  constexpr int EV = DT == 1 ? 8 : 4;
  constexpr int NW = kChunkWords * 4;
#pragma unroll
  for (int q = 0; q < NW; ++q) {
    const uint32_t wq = word_at(cur, q);
    const int j = (c * kChunkWords + (q >> 2)) * kFtThreads + threadIdx.x;  // 16-byte word
    if (DT == 1) {
      const uint32_t mk = bf2_ge_mask(wq, st.fl2);
      if (mk) {
        const int e = j * EV + 2 * (q & 3);
        const bool a = (mk & 0xffffu) && e < V, b = (mk >> 16) && e + 1 < V;
        const unsigned n = (unsigned)a + (unsigned)b;
        if (n) {
          unsigned pos = atomicAdd(&s.ncand, n);
          my_end = max(my_end, pos + n);
          if (pos + n <= (unsigned)kCand) {
            if (a) s.cand[pos++] = __uint_as_float(wq << 16);
            if (b) s.cand[pos] = __uint_as_float(wq & 0xffff0000u);
          } else {
            my_ovf = true;
          }
        }
      }
    } else {
      const float z = __uint_as_float(wq);
      if (z >= st.fl && j * EV + (q & 3) < V) {
        const unsigned pos = atomicAdd(&s.ncand, 1u);
        my_end = max(my_end, pos + 1u);
        if (pos < (unsigned)kCand)
          s.cand[pos] = z;
        else
          my_ovf = true;
      }
    }
  }
}

// Mass of this thread's chunk share relative to 2^ref: of every logit
// (all), and of those the floor leaves out (rest). Padding (-inf) weighs 0.
template <int DT>
__device__ __forceinline__ void chunk_mass(const uint4 (&cur)[kChunkWords], const StreamState& st,
                                           float cc, bool with_floor, float& all, float& rest) {
  constexpr int NW = kChunkWords * 4;
  all = 0.f;
  rest = 0.f;
#pragma unroll
  for (int q = 0; q < NW; ++q) {
    const uint32_t wq = word_at(cur, q);
#pragma unroll
    for (int h = 0; h < (DT == 1 ? 2 : 1); ++h) {
      const float z = DT == 1 ? __uint_as_float(h ? (wq & 0xffff0000u) : (wq << 16)) : __uint_as_float(wq);
      const float m = exp2f(fmaf(z, cc, -st.ref));
      all += m;
      // Padding is -inf (mass 0), so the V bound does not matter here.
      if (!with_floor || z < st.fl) rest += m;
    }
  }
}

// One step of the one-pass collection: chunk c, held in `cur`, while the
// next two chunks are on their way. Returns false when the collection must
// give up (the caller then takes the passes over the row).
template <int DT>
__device__ __forceinline__ bool stream_step(FtSmem& s, int V, int k, float p, float cc, int c, int nch,
                                            const uint4 (&cur)[kChunkWords], StreamState& st) {
  constexpr int NW = kChunkWords * 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // This thread's chunk maximum.
  float cmax;
  if (DT == 1) {
    uint32_t m2 = word_at(cur, 0);
#pragma unroll
    for (int q = 1; q < NW; ++q) m2 = bf2_max(m2, word_at(cur, q));
    cmax = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u));
  } else {
    cmax = __uint_as_float(word_at(cur, 0));
#pragma unroll
    for (int q = 1; q < NW; ++q) cmax = fmaxf(cmax, __uint_as_float(word_at(cur, q)));
  }
  if (k > 0) {
    // k of the threads' running maxima lie at or above their k-th largest.
    if (c < 16) {
      st.rmax = fmaxf(st.rmax, cmax);
      if ((kKthChunks >> c) & 1u) set_floor<DT>(st, floor_value<DT>(kth_key_of_threads<DT>(key_of<DT>(st.rmax), k)));
    }
  } else {
    // Move the reference up (an exact power-of-two rescale) if this chunk
    // holds a larger maximum.
    const float nm = fmaxf(st.rmax, cmax);
    if (nm > -INFINITY) {
      const float nref = ceilf(nm * cc);
      if (!(st.ref >= nref)) {
        if (st.ref > -INFINITY) {
          const int d = (int)(st.ref - nref);
          st.sum_all = ldexpf(st.sum_all, d);
          st.sum_rest = ldexp(st.sum_rest, d);
        }
        st.ref = nref;
      }
      st.rmax = nm;
    }
    if (c == 0) {
      // The first chunk's floor comes from the first chunk itself.
      float all = 0.f, rest = 0.f;
      if (st.ref > -INFINITY) chunk_mass<DT>(cur, st, cc, false, all, rest);
      float r = st.ref, sm = all;
      warp_ref_mass(r, sm);
      if (lane == 0) {
        s.wm[0][warp] = r;
        s.wsf[0][warp] = sm;
      }
      __syncthreads();
      set_floor<DT>(st, top_p_floor(s, 0, p, cc, V));
    }
    if (st.ref > -INFINITY) {
      float all, rest;
      chunk_mass<DT>(cur, st, cc, true, all, rest);
      st.sum_all += all;
      st.sum_rest += (double)rest;
    }
  }
  if (cmax >= st.fl) append_chunk<DT>(s, cur, c, V, st, st.my_end, st.my_ovf);
  // Checkpoints after every `every` chunks (and the last): the buffer's
  // fill, the floor raise and the top-p bound. An append between them that
  // finds the buffer full is caught here.
  const int every = k <= kSparseMaxK ? kCheckSparse : kCheckDense;  // k = 0: top-p alone
  if ((c + 1) % every != 0 && c + 1 < nch) return true;
  const int slot = (c / every + 1) & 1;  // chunk 0's own bound used slot 0
  if (k == 0 && c > 0) {
    float r = st.ref, sm = st.sum_all;
    warp_ref_mass(r, sm);
    if (lane == 0) {
      s.wm[slot][warp] = r;
      s.wsf[slot][warp] = sm;
    }
  }
  // Every decision below comes from a barrier's own result or from values
  // all threads hold: other threads may already be appending the next chunk
  // while a thread would still read the counter.
  if (__syncthreads_or(st.my_end > (unsigned)(kCand / 2))) {
    if (__syncthreads_or(st.my_ovf)) return false;
    if (k > 0 && c + 1 < nch) {
      float f;
      const int kept = raise_floor<DT>(s, k, f);
      set_floor<DT>(st, f);
      if (kept > kCand / 2) return false;
    }
  }
  st.my_end = 0u;
  st.my_ovf = false;
  if (k == 0 && c > 0 && c + 1 < nch) set_floor<DT>(st, top_p_floor(s, slot, p, cc, V));
  return true;
}

// One pass over the row that leaves in s.cand every logit at or above the
// final floor, the floor at most the row's threshold:
//   top-k (k >= 1, k <= kStreamK): the floor is raised after chunks 0, 1, 3,
//     7 and 15 to the k-th largest of the threads' running maxima, and to the
//     k-th largest value in the buffer when the buffer passes half full;
//   top-p alone (k = 0, 0 < p < 1): the floor is (R + log2((1-p) S / V)) / cc
//     from the running reference R and mass S. The row's maximum, its
//     reference and the mass of the logits left out of the buffer (double,
//     relative to 2^reference) land in s.rowmax, s.row_ref, s.row_mass.
// Returns false when the buffer cannot hold the logits at the floor.
template <int DT>
__device__ bool stream_collect(FtSmem& s, const void* row, int V, bool vec, int k, float p, float cc) {
  constexpr int EV = DT == 1 ? 8 : 4;
  constexpr int CH = kChunkWords * EV * kFtThreads;  // logits per chunk
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = (V + CH - 1) / CH;
  if (threadIdx.x == 0) s.ncand = 0u;
  StreamState st{-INFINITY, 0xff80ff80u, -INFINITY, -INFINITY, 0.f, 0.0, 0u, false};
  // Chunks c + 1 and c + 2 are in flight while chunk c is processed.
  issue_chunk<DT>(s, row, V, vec, 0);
  cp_async_commit();
  if (nch > 1) issue_chunk<DT>(s, row, V, vec, 1);
  cp_async_commit();
  for (int c = 0; c < nch; ++c) {
    cp_async_wait_but_one();
    uint4 cur[kChunkWords];
#pragma unroll
    for (int u = 0; u < kChunkWords; ++u) cur[u] = s.ring[c % kRing][u][threadIdx.x];
    if (c + 2 < nch) issue_chunk<DT>(s, row, V, vec, c + 2);
    cp_async_commit();
    if (!stream_step<DT>(s, V, k, p, cc, c, nch, cur, st)) {
      cp_async_wait_all();
      return false;
    }
  }
  if (k == 0) {
    float m = st.rmax, r = st.ref;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, o));
    }
    double d = st.ref > -INFINITY ? ldexp(st.sum_rest, (int)(st.ref - r)) : 0.0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0) {
      s.wm[0][warp] = m;
      s.wsf[0][warp] = r;
      s.wsd[warp] = d;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float M = -INFINITY, R = -INFINITY;
      for (int w = 0; w < kFtWarps; ++w) {
        M = fmaxf(M, s.wm[0][w]);
        R = fmaxf(R, s.wsf[0][w]);
      }
      double S = 0.0;
      for (int w = 0; w < kFtWarps; ++w)
        if (s.wsf[0][w] > -INFINITY) S += ldexp(s.wsd[w], (int)(s.wsf[0][w] - R));
      s.rowmax = M;
      s.row_ref = R;
      s.row_mass = S;
    }
    __syncthreads();
  }
  return true;
}

// Returns the row's threshold. kept_in_buf: s.cand[0, n_buf) holds every
// logit the threshold keeps (and maybe more below it); M_row: the row's
// maximum (when kept_in_buf).
template <int DT>
__device__ float row_threshold(FtSmem& s, const void* rowp, int V, bool vec, int top_k, float top_p,
                               float c, bool& kept_in_buf, int& n_buf, float& M_row) {
  constexpr int KB = DT == 1 ? 16 : 32;  // key bits
  const bool use_k = top_k >= 1 && top_k < V;
  const bool use_p = top_p > 0.f && top_p < 1.f;
  const RowSrc<DT> row{rowp, V, vec};
  CandSrc<DT> cs{s.cand, 0};
  bool in_smem = false;  // the candidates hold every key still in play
  kept_in_buf = false;
  uint32_t floor = 0u;   // keys >= floor are kept
  float M = -INFINITY;
  bool mass_known = false;  // s.row_mass holds the row's mass relative to M
  if (use_k) {
    if (top_k <= kStreamK && stream_collect<DT>(s, rowp, V, vec, top_k, 1.f, c)) {
      cs.n = (int)s.ncand;
      in_smem = true;
    }
    uint32_t prefix = 0u;
    unsigned need = (unsigned)top_k, above = 0u;
    for (int sh = KB - 8; sh >= 0; sh -= 8) {
      const bool top = sh == KB - 8;
      if (in_smem)
        histogram<DT>(s, cs, sh, prefix, top, 0u, false, 0.f, 0.f, top);
      else
        histogram<DT>(s, row, sh, prefix, top, 0u, false, 0.f, 0.f, top);
      if (top) M = s.rowmax;
      pick_digit(s, need, 0.0, false);
      need -= s.before_c;
      above += s.before_c;
      prefix = (prefix << 8) | s.digit;
      const unsigned in_play = above + s.tc[s.digit];
      if (!in_smem && in_play <= (unsigned)kCand && (sh > 0 || use_p)) {
        collect<DT>(s, row, prefix << sh);
        cs.n = (int)s.ncand;
        in_smem = true;
      }
    }
    floor = prefix;
    M_row = M;
  }
  if (use_p) {
    if (!use_k) {
      if (stream_collect<DT>(s, rowp, V, vec, 0, top_p, c)) {
        cs.n = (int)s.ncand;
        in_smem = true;
        mass_known = true;
      } else {
        histogram<DT>(s, row, KB - 8, 0u, true, 0u, false, 0.f, 0.f, true);  // the row maximum
      }
      M = s.rowmax;
    }
    if (!(M > -INFINITY)) return -INFINITY;
    M_row = M;
    // Masses are relative to 2^mc: the row maximum's scaled value, or the
    // one-pass collection's integer reference, which its left-out mass
    // shares.
    const float mc = mass_known ? s.row_ref : __fmul_rn(M, c);
    uint32_t prefix = 0u;
    double need = 0.0;
    unsigned above = 0u;
    for (int sh = KB - 8; sh >= 0; sh -= 8) {
      const bool top = sh == KB - 8;
      if (in_smem)
        histogram<DT>(s, cs, sh, prefix, top, floor, true, c, mc, false);
      else
        histogram<DT, RowSrc<DT>, true>(s, row, sh, prefix, top, floor, true, c, mc, false);
      // The buffer of the one-pass top-p holds only the logits near the
      // top: the mass the pass left out of it is added to the buffer's.
      if (top) need = (double)top_p * (mass_known ? s.total_m + s.row_mass : s.total_m);
      pick_digit(s, 0u, need, true);
      need -= s.before_m;
      above += s.before_c;
      prefix = (prefix << 8) | s.digit;
      const unsigned in_play = above + s.tc[s.digit];
      if (!in_smem && sh > 0 && in_play <= (unsigned)kCand) {
        collect<DT>(s, row, prefix << sh);
        cs.n = (int)s.ncand;
        in_smem = true;
      }
    }
    if (prefix > floor) floor = prefix;
  }
  // Every key >= floor is in the buffer once it holds the keys in play; a
  // threshold of -inf keeps the whole row, which it then holds only if it
  // holds all V logits.
  n_buf = cs.n;
  kept_in_buf = in_smem && M_row > -INFINITY && (floor != 0u || cs.n >= V);
  if (floor == 0u) return -INFINITY;
  return DT == 1 ? value16(floor) : value32(floor);
}

// Filtered softmax statistics of the row from the buffer (all threads; the
// result is valid in thread 0): mc = fp32(M c), S = sum over the buffered
// logits z >= tau of 2^(z c - mc), per thread in fp32, over the CTA in fp64.
__device__ FStat buffer_stats(FtSmem& s, int n, float tau, float M, float c) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float mc = __fmul_rn(M, c);
  float part = 0.f;
  for (int j = threadIdx.x; j < n; j += kFtThreads) {
    const float z = s.cand[j];
    if (z >= tau) part += exp2f(fmaf(z, c, -mc));
  }
  double d = (double)part;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
  if (lane == 0) s.wsd[warp] = d;
  __syncthreads();
  FStat f{};
  f.mc = mc;
  f.ok = 1;
  f.S = 0.0;
  for (int w = 0; w < kFtWarps; ++w) f.S += s.wsd[w];
  __syncthreads();
  return f;
}

// Rows [0, R_t) are target rows (request b at cu[b] + b + i); rows
// [R_t, R_t + R_d) draft rows. Greedy requests keep everything.
template <int DT>
__global__ void __launch_bounds__(kFtThreads, 3) threshold_kernel(FtParams P) {
  extern __shared__ __align__(16) unsigned char ft_smem[];
  FtSmem& s = *reinterpret_cast<FtSmem*>(ft_smem);
  // The warp kernel finished every row: nothing to do.
  if (P.after_warp && P.rows_left && __ldcg(P.rows_left) == 0u) return;
  // Rows past the caller's arrays (offsets that the verify kernel will
  // reject) are skipped.
  int R_d = P.cu[P.B], R_t = R_d + P.B;
  if (R_t > P.rows_t || R_d < 0) R_t = R_d = 0;
  const int rows = R_t + (P.draft ? R_d : 0);
  const size_t rowb = (size_t)P.V * (DT == 1 ? 2 : 4);
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const bool is_t = r < R_t;
    const int rr = is_t ? r : r - R_t;
    // The row's request, for its mode.
    int lo = 0, hi = P.mode ? P.B - 1 : 0;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((is_t ? P.cu[mid] + mid : P.cu[mid]) <= rr)
        lo = mid;
      else
        hi = mid - 1;
    }
    const bool greedy = P.mode && P.mode[lo] == SV_MODE_GREEDY;
    // Rows the warp kernel finished (ok) keep its threshold and statistics.
    if (P.after_warp && (greedy || (is_t ? P.fst_t : P.fst_d)[rr].ok)) continue;
    float tau = -INFINITY;
    FStat fs{};
    if (!greedy) {
      const char* row = static_cast<const char*>(is_t ? P.target : P.draft) + (size_t)rr * rowb;
      bool in_buf = false;
      int n_buf = 0;
      float M = -INFINITY;
      tau = row_threshold<DT>(s, row, P.V, P.vec, P.top_k, P.top_p, P.c, in_buf, n_buf, M);
      // The filtered row's softmax from the buffer: the verify kernel then
      // need not read the row again.
      if (in_buf && P.fst_t) fs = buffer_stats(s, n_buf, tau, M, P.c);
    }
    if (threadIdx.x == 0) {
      (is_t ? P.thr_t : P.thr_d)[rr] = tau;
      if (P.fst_t) (is_t ? P.fst_t : P.fst_d)[rr] = fs;
    }
    __syncthreads();
  }
}


// ---------------------------------------------------------------------------
// One warp per row (top-k up to kWarpMaxK, with or without top-p)
// ---------------------------------------------------------------------------
// Every row streams at once (one wave of warps), and each warp selects its
// row's threshold alone, with no CTA barrier. The warp keeps a buffer of the
// logits at or above a floor that never exceeds the k-th largest logit
// seen: the k-th largest of the lanes' kWTop largest vector maxima (k of
// those maxima, each a logit, lie at or above it), raised after iterations
// 0, 1, 3, 7, ... and to the k-th largest buffered logit when the buffer
// passes half full. After the pass the buffer holds every logit the
// threshold keeps:
//   top-k: the k-th largest buffered key (bit by bit, counts over the warp);
//   top-p: walking the distinct kept values from the largest down, summing
//     their masses 2^(z c - mc) (mc = fp32(M c), M the row maximum) in the
//     same 2^-44 fixed point as the CTA kernel's bins (exact, so its sums
//     and this walk agree), up to the first value at which the mass reaches
//     p times the kept mass.
// Rows the warp cannot finish (a buffer that stays more than half full: long
// tie groups, or no finite logit) are left with ok = 0 for the CTA kernel,
// which then skips the rows marked ok.
constexpr int kWarpMaxK = 128;
constexpr int kWTop = 4;          // vector maxima each lane tracks: k <= 32 * kWTop
constexpr int kWCap = 512;        // logits a warp's buffer holds
#ifndef SV_WLOADS
#define SV_WLOADS 8
#endif
constexpr int kWLoads = SV_WLOADS;  // 16-byte vectors a lane has in flight
#ifndef SV_WWARPS
#define SV_WWARPS 4
#endif
// Rows (warps) per CTA of the warp kernel. The rows of a batch make about
// one wave of warps; small CTAs spread them evenly over the SMs (on 3840
// rows of 151936 bf16 logits: 8 per CTA 259 µs per filtered call, 4 248 µs,
// 2 249 µs, 1 305 µs).
constexpr int kWWarps = SV_WWARPS;
constexpr int kWThreads = 32 * kWWarps;
#ifndef SV_WMINB
#define SV_WMINB (32 / SV_WWARPS)
#endif
constexpr int kWMinBlocks = SV_WMINB;  // resident CTAs per SM the register budget allows

static_assert(kWarpMaxK <= 32 * kWTop, "k of the tracked maxima must exist");

// 16-byte streaming load that does not allocate in L1 (read once).
__device__ __forceinline__ uint4 wt_ld16(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ float wt_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Largest key `x` such that at least k of the warp's values have key >= x
// (the k-th largest key), over n_per_lane values per lane (keys given).
template <int DT, int N>
__device__ __forceinline__ uint32_t warp_kth_key(const uint32_t (&keys)[N], int k) {
  constexpr int KB = DT == 1 ? 16 : 32;
  uint32_t prefix = 0u;
#pragma unroll 1
  for (int bit = KB - 1; bit >= 0; --bit) {
    const uint32_t cand = prefix | (1u << bit);
    unsigned c = 0;
#pragma unroll
    for (int j = 0; j < N; ++j) c += keys[j] >= cand ? 1u : 0u;
    if ((int)__reduce_add_sync(0xffffffffu, c) >= k) prefix = cand;
  }
  return prefix;
}

// The k-th largest key among the buffer's n logits (lane-strided).
template <int DT>
__device__ uint32_t buffer_kth_key(const float* buf, unsigned n, int k) {
  constexpr int KB = DT == 1 ? 16 : 32;
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0u;
#pragma unroll 1
  for (int bit = KB - 1; bit >= 0; --bit) {
    const uint32_t cand = prefix | (1u << bit);
    unsigned c = 0;
    for (unsigned j = lane; j < n; j += 32) c += key_of<DT>(buf[j]) >= cand ? 1u : 0u;
    if ((int)__reduce_add_sync(0xffffffffu, c) >= k) prefix = cand;
  }
  return prefix;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int DT>
__device__ __forceinline__ float value_of_key(uint32_t k) {
  return DT == 1 ? value16(k) : value32(k);
}

struct WarpRowSmem {
  float buf[kWWarps][kWCap];  // buffered logits
  int ix[kWWarps][kWCap];     // their tokens
  unsigned n[kWWarps];
};

template <int DT>
__global__ void __launch_bounds__(kWThreads, kWMinBlocks) threshold_warp_kernel(FtParams P) {
  constexpr int EV = DT == 1 ? 8 : 4;  // logits per 16-byte vector
  __shared__ WarpRowSmem sm;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* buf = sm.buf[warp];
  int* ix = sm.ix[warp];
  unsigned* nb = &sm.n[warp];
  int R_d = P.cu[P.B], R_t = R_d + P.B;
  if (R_t > P.rows_t || R_d < 0) R_t = R_d = 0;
  const int rows = R_t + (P.draft ? R_d : 0);
  const size_t rowb = (size_t)P.V * (DT == 1 ? 2 : 4);
  const int k = P.top_k;
  const bool use_p = P.top_p > 0.f && P.top_p < 1.f;
  const int nvec = P.V / EV;
  for (int r = blockIdx.x * kWWarps + warp; r < rows; r += gridDim.x * kWWarps) {
    const bool is_t = r < R_t;
    const int rr = is_t ? r : r - R_t;
    int greedy = 0;
    if (lane == 0 && P.mode) {
      int lo = 0, hi = P.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((is_t ? P.cu[mid] + mid : P.cu[mid]) <= rr) lo = mid; else hi = mid - 1;
      }
      greedy = P.mode[lo] == SV_MODE_GREEDY;
    }
    greedy = __shfl_sync(0xffffffffu, greedy, 0);
    FStat out{};
    float tau = -INFINITY;
    if (!greedy) {
      const uint4* row = reinterpret_cast<const uint4*>(static_cast<const char*>(is_t ? P.target : P.draft) +
                                                        (size_t)rr * rowb);
      if (lane == 0) *nb = 0u;
      __syncwarp();
      float top[kWTop];
#pragma unroll
      for (int j = 0; j < kWTop; ++j) top[j] = -INFINITY;
      float rmax = -INFINITY, fl = -INFINITY;
      bool ovf = false;
      int it = 0;
      for (int base = 0; base < nvec; base += 32 * kWLoads, ++it) {
        uint4 w[kWLoads];
#pragma unroll
        for (int u = 0; u < kWLoads; ++u) {
          const int j = base + u * 32 + lane;
          w[u] = j < nvec ? wt_ld16(row + j) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
          if (DT == 0 && j >= nvec) w[u] = make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
        }
        float vm[kWLoads];
#pragma unroll
        for (int u = 0; u < kWLoads; ++u) {
          if (DT == 1) {
            uint32_t m2 = bf2_max(bf2_max(w[u].x, w[u].y), bf2_max(w[u].z, w[u].w));
            vm[u] = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u));
          } else {
            vm[u] = fmaxf(fmaxf(__uint_as_float(w[u].x), __uint_as_float(w[u].y)),
                          fmaxf(__uint_as_float(w[u].z), __uint_as_float(w[u].w)));
          }
          rmax = fmaxf(rmax, vm[u]);
          // Keep this lane's kWTop largest vector maxima (sorted, largest first).
          if (vm[u] > top[kWTop - 1]) {
            float x = vm[u];
#pragma unroll
            for (int j = 0; j < kWTop; ++j) {
              const float hi = fmaxf(top[j], x);
              x = fminf(top[j], x);
              top[j] = hi;
            }
          }
        }
        // Raise the floor at iterations 0, 1, 3, 7, ...: k of the tracked
        // maxima lie at or above their k-th largest.
        if ((it & (it + 1)) == 0) {
          uint32_t keys[kWTop];
#pragma unroll
          for (int j = 0; j < kWTop; ++j) keys[j] = key_of<DT>(top[j]);
          fl = fmaxf(fl, value_of_key<DT>(warp_kth_key<DT, kWTop>(keys, k)));
        }
        // Append the logits at or above the floor, with their tokens.
#pragma unroll
        for (int u = 0; u < kWLoads; ++u) {
          if (vm[u] >= fl) {
            const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
            const int x0 = (base + u * 32 + lane) * EV;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
              for (int h = 0; h < (DT == 1 ? 2 : 1); ++h) {
                // bf16: the low half of a word is the lower token.
                const float z = DT == 1 ? __uint_as_float(h ? (ws[q] & 0xffff0000u) : (ws[q] << 16))
                                        : __uint_as_float(ws[q]);
                if (z >= fl) {
                  const unsigned pos = atomicAdd(nb, 1u);
                  if (pos < (unsigned)kWCap) {
                    buf[pos] = z;
                    ix[pos] = x0 + (DT == 1 ? 2 * q + h : q);
                  } else {
                    ovf = true;
                  }
                }
              }
            }
          }
        }
        __syncwarp();
        // Every branch below that leads to a warp collective is taken by the
        // whole warp: the overflow flag is made uniform first.
        ovf = __any_sync(0xffffffffu, ovf);
        if (ovf) break;
        unsigned n = *nb;
        if (n > (unsigned)(kWCap / 2)) {
          // Raise the floor to the k-th largest buffered logit and compact
          // in place, 32 entries at a time: an entry only moves down, past
          // entries already read.
          fl = fmaxf(fl, value_of_key<DT>(buffer_kth_key<DT>(buf, n, k)));
          __syncwarp();
          int total = 0;
          for (unsigned j0 = 0; j0 < n; j0 += 32) {
            const unsigned idx = j0 + lane;
            const float z = idx < n ? buf[idx] : -INFINITY;
            const int x = idx < n ? ix[idx] : 0;
            const bool kp = idx < n && z >= fl;
            const unsigned bal = __ballot_sync(0xffffffffu, kp);
            __syncwarp();
            if (kp) {
              const int pos = total + __popc(bal & ((1u << lane) - 1u));
              buf[pos] = z;
              ix[pos] = x;
            }
            total += __popc(bal);
            __syncwarp();
          }
          if (lane == 0) *nb = (unsigned)total;
          __syncwarp();
          if (total > kWCap / 2) {  // a tie group at the floor that does not fit
            ovf = true;
            break;
          }
        }
      }
      rmax = wt_max(rmax);
      const unsigned n = min(*nb, (unsigned)kWCap);
      if (!ovf && rmax > -INFINITY && (int)n >= k) {
        // Top-k: the k-th largest buffered key; every logit at or above it
        // is in the buffer.
        uint32_t tk = buffer_kth_key<DT>(buf, n, k);
        float tv = value_of_key<DT>(tk);
        const float mc = __fmul_rn(rmax, P.c);
        if (use_p) {
          // Top-p on the top-k set, distinct values from the largest down.
          unsigned long long tot = 0ull;
          for (unsigned j = lane; j < n; j += 32) {
            const float z = buf[j];
            if (z >= tv) tot += __float2ull_rn(exp2f(fmaf(z, P.c, -mc)) * 0x1p44f);
          }
          tot = warp_sum_u64(tot);
          const double need = (double)P.top_p * ((double)tot * 0x1p-44);
          unsigned long long cum = 0ull;
          float cur = INFINITY, pick = tv;
#pragma unroll 1
          for (;;) {
            float v = -INFINITY;
            for (unsigned j = lane; j < n; j += 32) {
              const float z = buf[j];
              if (z >= tv && z < cur) v = fmaxf(v, z);
            }
            v = wt_max(v);
            if (v == -INFINITY) break;  // no value left: everything in play stays
            unsigned long long g = 0ull;
            for (unsigned j = lane; j < n; j += 32) {
              const float z = buf[j];
              if (z == v) g += __float2ull_rn(exp2f(fmaf(z, P.c, -mc)) * 0x1p44f);
            }
            cum += warp_sum_u64(g);
            pick = v;
            if ((double)cum * 0x1p-44 >= need) break;
            cur = v;
          }
          if (pick > tv) tv = pick;
        }
        tau = tv;
        // The filtered row's softmax sum from the buffer.
        float part = 0.f;
        for (unsigned j = lane; j < n; j += 32) {
          const float z = buf[j];
          if (z >= tau) part += exp2f(fmaf(z, P.c, -mc));
        }
        double d = (double)part;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        out.mc = mc;
        out.ok = 1;
        out.S = d;
        if (is_t && P.list_t) {
          // The kept (token, logit) pairs of a target row, for its draw.
          int2* lst = P.list_t + (size_t)rr * kKeptListCap;
          int nk = 0;
          for (unsigned j0 = 0; j0 < n; j0 += 32) {
            const unsigned idx = j0 + lane;
            const float z = idx < n ? buf[idx] : -INFINITY;
            const bool kp = idx < n && z >= tau;
            const unsigned bal = __ballot_sync(0xffffffffu, kp);
            const int pos = nk + __popc(bal & ((1u << lane) - 1u));
            if (kp && pos < kKeptListCap) lst[pos] = make_int2(ix[idx], __float_as_int(z));
            nk += __popc(bal);
          }
          out.nl = nk <= kKeptListCap ? nk : 0;
        }
      }
    }
    if (lane == 0) {
      // Rows left with ok = 0 get their threshold from the CTA kernel.
      if (out.ok || greedy) (is_t ? P.thr_t : P.thr_d)[rr] = tau;
      (is_t ? P.fst_t : P.fst_d)[rr] = out;
      if (!out.ok && !greedy && P.rows_left) *P.rows_left = 1u;  // the CTA kernel has work
    }
    __syncwarp();
  }
}

template <int DT>
static cudaError_t launch_thresholds_t(const FtParams& P, int sms, cudaStream_t st) {
  const size_t smem = sizeof(FtSmem);
  cudaError_t e = cudaFuncSetAttribute(threshold_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, threshold_kernel<DT>, kFtThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  // One wave of resident CTAs walks the rows.
  const int rows = 2 * P.rows_t;
  int grid = rows < per_sm * sms ? rows : per_sm * sms;
  if (grid < 1) grid = 1;
  threshold_kernel<DT><<<grid, kFtThreads, smem, st>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_thresholds(const FtParams& P0, int dtype, cudaStream_t st, bool* warp_ran) {
  *warp_ran = false;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  FtParams P = P0;
  P.after_warp = false;
  // Top-k up to kWarpMaxK on vector rows: one warp per row first; the CTA
  // kernel then takes only the rows it left.
  if (P.fst_t && P.vec && P.top_k >= 1 && P.top_k <= kWarpMaxK) {
    const int rows = 2 * P.rows_t;
    int grid = (rows + kWWarps - 1) / kWWarps;
    if (grid < 1) grid = 1;
    if (dtype == SV_BF16)
      threshold_warp_kernel<1><<<grid, kWThreads, 0, st>>>(P);
    else
      threshold_warp_kernel<0><<<grid, kWThreads, 0, st>>>(P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    P.after_warp = true;
    *warp_ran = true;
  }
  return dtype == SV_BF16 ? launch_thresholds_t<1>(P, sms, st) : launch_thresholds_t<0>(P, sms, st);
}

}  // namespace sv
