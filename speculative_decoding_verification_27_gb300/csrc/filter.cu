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
#include "../../include/spec_verify.h"
#include "sv_filter.cuh"

#include <cmath>
#include <cstdint>
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

constexpr int kCand = 4096;  // logits that shared memory holds once few keys are left in play

struct FtSmem {
  unsigned cnt[kFtWarps][256];
  float mass[kFtWarps][256];
  double tc[256], tm[256];  // per-digit count and mass totals
  float wmax[kFtWarps];
  float cand[kCand];        // the logits still in play, once they fit
  unsigned ncand;
  uint32_t digit;
  double before_c, before_m;  // count and mass of the digits above the chosen one
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
template <int DT, class Src>
__device__ void histogram(FtSmem& s, const Src& src, int shift, uint32_t prefix, bool top_level,
                          uint32_t floor, bool by_mass, float c, float mc, bool track_max) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int k = tid; k < kFtWarps * 256; k += kFtThreads) {
    (&s.cnt[0][0])[k] = 0u;
    (&s.mass[0][0])[k] = 0.f;
  }
  __syncthreads();
  // Runs of one digit are merged in registers before they reach shared memory.
  uint32_t run_d = 0xffffffffu;
  unsigned run_n = 0;
  float run_m = 0.f, vmax = -INFINITY;
  auto flush = [&]() {
    if (run_n) {
      atomicAdd(&s.cnt[warp][run_d], run_n);
      if (by_mass) atomicAdd(&s.mass[warp][run_d], run_m);
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
      run_m = 0.f;
    }
    ++run_n;
    if (by_mass) run_m += exp2f(fmaf(v, c, -mc));
  });
  flush();
  if (track_max) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    if (lane == 0) s.wmax[warp] = vmax;
  }
  __syncthreads();
  double tc = 0.0, tm = 0.0;
  for (int w = 0; w < kFtWarps; ++w) {
    tc += (double)s.cnt[w][tid];
    tm += (double)s.mass[w][tid];
  }
  s.tc[tid] = tc;
  s.tm[tid] = tm;
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

// The first digit from the top at which the running count (or mass) reaches
// `need`: s.digit, with the count and mass of the digits above it in
// s.before_c / s.before_m. If rounding leaves `need` unreached, the lowest
// digit is taken (everything in play stays).
__device__ void pick_digit(FtSmem& s, double need, bool by_mass) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const double* t = by_mass ? s.tm : s.tc;
    // Lane l covers digits 255 - 8l .. 248 - 8l (from the top).
    double loc[8], sum = 0.0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      loc[j] = t[255 - 8 * lane - j];
      sum += loc[j];
    }
    double incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
    const int first = hit ? __ffs(hit) - 1 : 31;
    if (lane == first) {
      double run = incl - sum;
      int j = 0;
      for (; j < 7; ++j) {
        if (run + loc[j] >= need) break;
        run += loc[j];
      }
      const uint32_t d = 255u - 8u * (uint32_t)lane - (uint32_t)j;
      double bc = 0.0, bm = 0.0;
      for (uint32_t e = d + 1; e < 256; ++e) {
        bc += s.tc[e];
        bm += s.tm[e];
      }
      s.digit = d;
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

template <int DT>
__device__ float row_threshold(FtSmem& s, const void* rowp, int V, bool vec, int top_k, float top_p,
                               float c) {
  constexpr int KB = DT == 1 ? 16 : 32;  // key bits
  const bool use_k = top_k >= 1 && top_k < V;
  const bool use_p = top_p > 0.f && top_p < 1.f;
  const RowSrc<DT> row{rowp, V, vec};
  CandSrc<DT> cs{s.cand, 0};
  bool in_smem = false;  // the candidates hold every key still in play
  uint32_t floor = 0u;   // keys >= floor are kept
  float M = -INFINITY;
  if (use_k) {
    uint32_t prefix = 0u;
    double need = (double)top_k, above = 0.0;
    for (int sh = KB - 8; sh >= 0; sh -= 8) {
      const bool top = sh == KB - 8;
      if (in_smem)
        histogram<DT>(s, cs, sh, prefix, top, 0u, false, 0.f, 0.f, false);
      else
        histogram<DT>(s, row, sh, prefix, top, 0u, false, 0.f, 0.f, top);
      if (top) M = s.rowmax;
      pick_digit(s, need, false);
      need -= s.before_c;
      above += s.before_c;
      prefix = (prefix << 8) | s.digit;
      const double in_play = above + s.tc[s.digit];
      if (!in_smem && in_play <= (double)kCand && (sh > 0 || use_p)) {
        collect<DT>(s, row, prefix << sh);
        cs.n = (int)s.ncand;
        in_smem = true;
      }
    }
    floor = prefix;
  }
  if (use_p) {
    if (!use_k) {
      histogram<DT>(s, row, KB - 8, 0u, true, 0u, false, 0.f, 0.f, true);  // the row maximum
      M = s.rowmax;
    }
    if (!(M > -INFINITY)) return -INFINITY;
    const float mc = __fmul_rn(M, c);
    uint32_t prefix = 0u;
    double need = 0.0, above = 0.0;
    for (int sh = KB - 8; sh >= 0; sh -= 8) {
      const bool top = sh == KB - 8;
      if (in_smem)
        histogram<DT>(s, cs, sh, prefix, top, floor, true, c, mc, false);
      else
        histogram<DT>(s, row, sh, prefix, top, floor, true, c, mc, false);
      if (top) need = (double)top_p * s.total_m;
      pick_digit(s, need, true);
      need -= s.before_m;
      above += s.before_c;
      prefix = (prefix << 8) | s.digit;
      const double in_play = above + s.tc[s.digit];
      if (!in_smem && sh > 0 && in_play <= (double)kCand) {
        collect<DT>(s, row, prefix << sh);
        cs.n = (int)s.ncand;
        in_smem = true;
      }
    }
    if (prefix > floor) floor = prefix;
  }
  if (floor == 0u) return -INFINITY;
  return DT == 1 ? value16(floor) : value32(floor);
}

// Rows [0, R_t) are target rows (request b at cu[b] + b + i); rows
// [R_t, R_t + R_d) draft rows. Greedy requests keep everything.
template <int DT>
__global__ void __launch_bounds__(kFtThreads) threshold_kernel(FtParams P) {
  __shared__ FtSmem s;
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
    int lo = 0, hi = P.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((is_t ? P.cu[mid] + mid : P.cu[mid]) <= rr)
        lo = mid;
      else
        hi = mid - 1;
    }
    const bool greedy = P.mode && P.mode[lo] == SV_MODE_GREEDY;
    float tau = -INFINITY;
    if (!greedy) {
      const char* row = static_cast<const char*>(is_t ? P.target : P.draft) + (size_t)rr * rowb;
      tau = row_threshold<DT>(s, row, P.V, P.vec, P.top_k, P.top_p, P.c);
    }
    if (threadIdx.x == 0) (is_t ? P.thr_t : P.thr_d)[rr] = tau;
    __syncthreads();
  }
}

cudaError_t launch_thresholds(const FtParams& P, int dtype, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int rows = 2 * P.rows_t;
  int grid = rows < 4 * sms ? rows : 4 * sms;
  if (grid < 1) grid = 1;
  if (dtype == SV_BF16)
    threshold_kernel<1><<<grid, kFtThreads, 0, st>>>(P);
  else
    threshold_kernel<0><<<grid, kFtThreads, 0, st>>>(P);
  return cudaGetLastError();
}

}  // namespace sv
