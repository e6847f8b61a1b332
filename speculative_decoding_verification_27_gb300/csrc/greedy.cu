// greedy.cu -- strict (greedy) verify-and-commit, one CTA per target row.
//
// "Speculative Decoding在分布式推理中的应用" §二, strict verification: draft
// token x̂_i is accepted iff it equals the argmax of target row i (lowest
// index among ties); at the first mismatch, or at the bonus row, the row's
// argmax is emitted. No softmax, no uniform, no draw: a row only needs its
// argmax, so the step is one streaming pass per row and a commit.
//
// Layout of the work: CTA t streams target row t with sixteen 16-byte loads
// in flight per thread (no shared-memory ring, no barrier inside the pass),
// 64 KB per CTA, so that even a batch with fewer rows than twice the SMs
// keeps the memory busy (8 loads: 25.2 µs on a 64-request batch, 16: 25.0). The row's address needs only
// cu_draft[B] (for R_t): the first loads go out before the rest of the
// offsets check, and the request lookup runs while they are in flight. The CTA writes
// the row's argmax and sets its bits in the request's progress word (one
// "done" bit per row, one "accepted" bit per draft slot, for K <= 31); the
// request's last row reads the stop slot off the word and commits. No CTA
// waits on another.
#include "../../include/spec_verify.h"
#include "sv_device.cuh"
#include "sv_greedy.cuh"

#include <climits>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace gr {

#ifndef SV_GREEDY_LOADS
#define SV_GREEDY_LOADS 16
#endif
constexpr int kU = SV_GREEDY_LOADS;  // 16-byte loads in flight per thread
constexpr int kMaxTrackedSlots = 31;  // K up to this keeps per-slot bits in the progress word

// Largest b in [0, B) with cu[b] + b <= t, by every thread of the CTA: each
// round tests kThreads evenly spaced candidates, one barrier counts the
// passing prefix (one round up to B = kThreads).
__device__ __forceinline__ int find_request_cta(const int32_t* cu, int B, int t) {
  int lo = 0, n = B;
  while (n > 1) {
    const int step = (n + kThreads - 1) / kThreads;
    const int c = lo + (int)threadIdx.x * step;
    const bool pass = c < lo + n && cu[c] + c <= t;
    const int cnt = __syncthreads_count(pass);
    const int end = lo + n;
    lo += (cnt - 1) * step;
    n = min(step, end - lo);
  }
  return lo;
}

template <int DT>
__device__ __forceinline__ uint4 neg_inf_vec() {
  return DT == 1 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                 : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}

// Folds one 16-byte vector (elements x0 .. x0 + EPV - 1, in increasing
// order) into the thread's (value, first index) maximum.
template <int DT>
__device__ __forceinline__ void fold(const uint4& v, int x0, float& bv, int& bi) {
  constexpr int EPV = Elem<DT>::kEPV;
  float f[EPV];
  Elem<DT>::unpack(v, f);
#pragma unroll
  for (int j = 0; j < EPV; ++j)
    if (f[j] > bv) {  // strict: the first of equal values stays
      bv = f[j];
      bi = x0 + j;
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads) greedy_verify_kernel(GParams P) {
  constexpr int EPV = Elem<DT>::kEPV;
  __shared__ float s_v[kWarps];
  __shared__ int s_i[kWarps];
  __shared__ int s_b, s_t0, s_d0, s_K, s_xhat;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x;

  // Offsets: every CTA checks and all take the same decision. The row's
  // first loads need only R_t = cu[B] + B (the rows the layout claims,
  // within the workspace): they go out before the rest of the check.
  const int R_d = P.cu[P.B];
  const long long R_t = (long long)R_d + P.B;
  const bool rows_ok = R_d >= 0 && R_t <= P.row_cap;
  const bool live = rows_ok && t < R_t;
  const uint4* row = reinterpret_cast<const uint4*>(static_cast<const char*>(P.target) + (size_t)t * P.nvec * 16);
  const int stride = kThreads * kU;  // vectors per pass of the CTA
  uint4 raw[kU];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int v = u * kThreads + tid;
    raw[u] = (live && v < P.nvec) ? ld_stream16(row + v) : neg_inf_vec<DT>();
  }
  bool bad = !rows_ok;
  for (int k = tid; k < P.B; k += kThreads)
    if (P.cu[k + 1] < P.cu[k]) bad = true;
  if (tid == 0 && P.cu[0] != 0) bad = true;
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(P.status, SV_DATA_BAD_OFFSETS);
    return;
  }
  if (!live) return;
  const int b = find_request_cta(P.cu, P.B, t);
  if (tid == 0) {
    const int t0 = P.cu[b] + b, d0 = P.cu[b];
    const int K = P.cu[b + 1] - d0, i = t - t0;
    int xhat = -1;
    if (i < K && P.draft_tokens) {
      xhat = P.draft_tokens[d0 + i];
      if (xhat < 0 || xhat >= P.V) {
        atomicOr(P.status, SV_DATA_BAD_TOKEN);
        xhat = -1;
      }
    }
    s_b = b;
    s_t0 = t0;
    s_d0 = d0;
    s_K = K;
    s_xhat = xhat;
  }

  float bv = -INFINITY;
  int bi = INT_MAX;
#pragma unroll
  for (int u = 0; u < kU; ++u) fold<DT>(raw[u], (u * kThreads + tid) * EPV, bv, bi);
  for (int v0 = stride; v0 < P.nvec; v0 += stride) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = v0 + u * kThreads + tid;
      raw[u] = v < P.nvec ? ld_stream16(row + v) : neg_inf_vec<DT>();
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) fold<DT>(raw[u], (v0 + u * kThreads + tid) * EPV, bv, bi);
  }
  // The merge keeps the largest value and, among equal values, the lowest
  // index (each thread met its own elements in increasing order).
  warp_argmax(bv, bi);
  if (lane == 0) {
    s_v[warp] = bv;
    s_i[warp] = bi;
  }
  __syncthreads();

  if (warp == 0) {
    const int t0 = s_t0, d0 = s_d0, K = s_K, xhat = s_xhat;
    const int i = t - t0;
    const bool tracked = K <= kMaxTrackedSlots;
    unsigned long long old = 0, word = 0;
    int am = 0;
    if (lane == 0) {
      float v = s_v[0];
      int k = s_i[0];
      for (int w = 1; w < kWarps; ++w) argmax_merge(v, k, s_v[w], s_i[w]);
      am = k == INT_MAX ? 0 : k;  // all -inf: index 0, like argmax
      const bool acc = i < K && xhat == am;
      P.rows[t] = CRow{acc ? 1u : 0u, am, 0.f, 0.f};
      // Release the row's result with its bits; acquire the other rows'.
      const unsigned long long add = tracked ? ((1ull << i) | (acc ? 1ull << (32 + i) : 0ull)) : 1ull;
      old = tracked ? atom_or_acqrel_gpu(&P.arrive[s_b], add) : atom_add_acqrel_gpu(&P.arrive[s_b], add);
      word = old | add;
    }
    old = __shfl_sync(kFull, old, 0);
    word = __shfl_sync(kFull, word, 0);
    am = __shfl_sync(kFull, am, 0);
    const unsigned long long all = tracked ? (1ull << (K + 1)) - 1ull : 0ull;  // the rows' done bits
    const bool last = tracked ? ((word & all) == all && (old & all) != all) : old == (unsigned long long)K;
    if (last) {
      // The request's last row: first mismatch, drafts before it, its argmax.
      __threadfence();  // every lane reads the other rows' results after the count
      int stop = K;
      if (tracked) {
        const unsigned acc_bits = (unsigned)(word >> 32);
        const unsigned rej = ~acc_bits & (unsigned)((1ull << K) - 1ull);
        if (rej) stop = __ffs(rej) - 1;
      } else {
        for (int j0 = 0; j0 < K && stop == K; j0 += 32) {
          const int j = j0 + lane;
          const bool rej = j < K && (__ldcg(&P.rows[t0 + j].accept) & 1u) == 0u;
          const unsigned m = __ballot_sync(kFull, rej);
          if (m) stop = j0 + __ffs(m) - 1;
        }
      }
      for (int j = lane; j < stop; j += 32) P.out_tokens[t0 + j] = P.draft_tokens[d0 + j];
      if (lane == 0) {
        P.out_tokens[t0 + stop] = (t0 + stop == t) ? am : __ldcg(&P.rows[t0 + stop].y);
        P.out_len[s_b] = stop + 1;
        P.arrive[s_b] = 0ull;  // every row is in: ready for the next call
      }
    }
  }
}

}  // namespace gr

cudaError_t launch_greedy_verify(const GParams& P, int dtype, cudaStream_t st) {
  const long long rows = P.row_cap < 1 ? 1 : P.row_cap;
  if (dtype == 1)
    gr::greedy_verify_kernel<1><<<(unsigned)rows, kThreads, 0, st>>>(P);
  else
    gr::greedy_verify_kernel<0><<<(unsigned)rows, kThreads, 0, st>>>(P);
  return cudaGetLastError();
}

}  // namespace sv
