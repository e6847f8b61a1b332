// onehot.cu -- verify-and-commit with one CTA per target row, for batches
// of short rows whose proposals are one-hot (no draft rows, as from an
// n-gram or suffix proposer).
//
// The step is that of "Draft Model（草稿模型）" §2 with q = e_x̂
// ("5.2 Draft 模型与无模型方案" §4.3): accept draft token x̂_i with
// probability min(1, p(x̂_i)); at the first rejection emit a token drawn
// from p with x̂_i removed, renormalised; if all K are accepted emit one more
// from p_{K+1}. p is a softmax at temperature T ("投机解码从零实现" §3.2);
// strict (greedy) rows accept iff x̂ is the target's argmax
// ("Speculative Decoding在分布式推理中的应用" §二).
//
// On short rows the persistent kernel's time per row is its chain of
// dependent steps (claim, request lookup, ring fill, combine, decision), not
// bytes. Here every target row has its own CTA and nothing is claimed:
//   1. the CTA streams its row with register loads, sixteen 16-byte loads in
//      flight per thread (64 KB per CTA), the first ones before the request
//      is even known; z(x̂) comes from one scalar load;
//   2. the CTA combines the threads' online-softmax statistics (or argmax)
//      and takes the row's accept decision, then sets its bits in the
//      request's progress word (one "done" bit per row and one "accepted"
//      bit per slot for K <= 31, a count otherwise);
//   3. the request's last row commits: the first rejected slot, the drafts
//      before it, and the token drawn at the stop row. The draw streams the
//      stop row once more, from L2 at these batch sizes, for the tile sums
//      of r, then rescans the tile that holds u' * Z.
// No CTA waits on another. With draft rows the persistent kernel (or the
// cluster kernel) runs instead: a CTA streaming a row pair with as many
// loads in flight needs more registers than two CTAs per SM leave.
#include "../../include/spec_verify.h"
#include "sv_device.cuh"
#include "sv_onehot.cuh"

#include <climits>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace oh {

#ifndef SV_ONEHOT_LOADS
#define SV_ONEHOT_LOADS 16
#endif
constexpr int kU = SV_ONEHOT_LOADS;   // 16-byte loads in flight per thread
constexpr int kMaxTracked = 31;       // K up to this keeps per-slot bits in the progress word
constexpr int kMaxTiles = kThreads;   // a draw's tiles (one 16-byte vector per thread each)
static_assert(kOneHotMaxVec == kMaxTiles * kThreads, "tile count bound");

enum { kOneHot = 1, kBonus = 2 };

// Largest b in [0, B) with cu[b] + b <= t, by every thread of the CTA: each
// round tests kThreads evenly spaced candidates and one barrier counts the
// passing prefix (one round up to B = kThreads).
__device__ __forceinline__ int find_request(const int32_t* cu, int B, int t) {
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

// A thread's online softmax of its elements: running maximum m, its offset
// mc = fp32(m c), and the sum of 2^(z c - mc).
struct Soft {
  float m, mc, s;
};

template <int EPV>
__device__ __forceinline__ void soft_fold(Soft& a, const float (&f)[EPV], float c) {
  float vm = f[0];
#pragma unroll
  for (int j = 1; j < EPV; ++j) vm = fmaxf(vm, f[j]);
  if (vm > a.m) {
    const float nmc = __fmul_rn(vm, c);
    a.s = (a.m == -INFINITY) ? 0.f : a.s * ex2(a.mc - nmc);
    a.m = vm;
    a.mc = nmc;
  }
#pragma unroll
  for (int j = 0; j < EPV; ++j) a.s += ex2(fmaf(f[j], c, -a.mc));
}

// Folds one vector (elements x0 .. x0 + EPV - 1, in increasing order) into
// the thread's (value, first index) maximum.
template <int EPV>
__device__ __forceinline__ void amax_fold(const float (&f)[EPV], int x0, float& bv, int& bi) {
#pragma unroll
  for (int j = 0; j < EPV; ++j)
    if (f[j] > bv) {  // strict: the first of equal values stays
      bv = f[j];
      bi = x0 + j;
    }
}

struct Shm {
  float redf[kWarps];
  int redi[kWarps];
  DF redd[kWarps], redd2[kWarps];
  float wt[kMaxTiles * kWarps];  // a draw's per-warp tile sums
  DF tincl[kMaxTiles];           // inclusive prefix of the tile sums
  DF wexcl[kWarps + 1];
  int pick, pick2, tok;
  // the row's request
  int b, t0, d0, K, i, greedy, xhat;
  float u;
  // the commit
  int last, stop;
};

// The CTA's (m, S) of one row from the threads' online softmax: the largest
// m, then every thread's sum rescaled to that offset, in double-float in
// warp order. Every thread gets the result.
__device__ __forceinline__ void cta_soft(Shm& s, const Soft& a, float c, float& Mc, DF& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float wm = warp_max(a.m);
  if (lane == 0) s.redf[warp] = wm;
  __syncthreads();
  float M = s.redf[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s.redf[w]);
  Mc = (M == -INFINITY) ? 0.f : __fmul_rn(M, c);
  DF t = (a.m == -INFINITY) ? DF{0.f, 0.f} : df_mul_f(DF{a.s, 0.f}, ex2(a.mc - Mc));
  t = warp_sum_df(t);
  if (lane == 0) s.redd[warp] = t;
  __syncthreads();
  S = s.redd[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) S = df_add(S, s.redd[w]);
  __syncthreads();  // the scratch is free again
}

// Everything a draw needs about its stop row.
struct Draw {
  const uint4* trow;
  int kind, xhat;
  float mcp;
  float u2;
};

// r of one vector (elements x .. x + EPV - 1): e_p = S_p p, the rejected
// one-hot proposal removed (p itself, unnormalised, for a bonus draw).
template <int EPV>
__device__ __forceinline__ float residual(const Draw& d, float c, const float (&zp)[EPV], int x,
                                          float (&r)[EPV]) {
  float ts = 0.f;
#pragma unroll
  for (int j = 0; j < EPV; ++j) {
    const float ep = ex2(fmaf(zp[j], c, -d.mcp));
    r[j] = (d.kind == kOneHot && x + j == d.xhat) ? 0.f : ep;
    ts += r[j];
  }
  return ts;
}

// Inverse CDF of r over the row by the whole CTA: tile l is vector l *
// kThreads + tid of every thread; its sum goes to wt per warp, the tiles'
// sums are scanned in double-float, the tile that holds u' * Z is rescanned
// element by element. The token is the last index with mass whose lower
// edge is <= u' * Z (the smallest whose running sum exceeds it), or -1 if r
// has no mass.
template <int DT>
__device__ int draw_row(const RParams& P, Shm& s, const Draw& d) {
  constexpr int EPV = Elem<DT>::kEPV;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = P.nvec;
  const int ntiles = (nvec + kThreads - 1) / kThreads;
  for (int l0 = 0; l0 < ntiles; l0 += kU) {
    uint4 rp[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = (l0 + u) * kThreads + tid;
      rp[u] = (l0 + u < ntiles && v < nvec) ? ld_stream16(d.trow + v) : neg_inf_vec<DT>();
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (l0 + u < ntiles) {
        float zp[EPV], r[EPV];
        Elem<DT>::unpack(rp[u], zp);
        float ts = residual<EPV>(d, P.c, zp, ((l0 + u) * kThreads + tid) * EPV, r);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ts += __shfl_xor_sync(kFull, ts, o);
        if (lane == 0) s.wt[(l0 + u) * kWarps + warp] = ts;
      }
    }
  }
  __syncthreads();
  DF tt{0.f, 0.f};
  if (tid < ntiles)
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tt = df_add_f(tt, s.wt[tid * kWarps + w]);
  const DF inc = warp_incl_scan_df(tt, lane);
  if (lane == 31) s.redd[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    DF v = lane < kWarps ? s.redd[lane] : DF{0.f, 0.f};
    v = warp_incl_scan_df(v, lane);
    if (lane < kWarps) s.redd2[lane] = v;
  }
  __syncthreads();
  if (tid < ntiles) s.tincl[tid] = warp > 0 ? df_add(s.redd2[warp - 1], inc) : inc;
  if (tid == 0) s.pick = -1;
  __syncthreads();
  const DF Z = s.tincl[ntiles - 1];
  if (!df_pos(Z)) {
    __syncthreads();  // every thread has read Z before the scratch is reused
    return -1;
  }
  DF T = df_mul_f(Z, d.u2);
  if (!(T.hi >= 0.f)) T = DF{0.f, 0.f};  // a NaN or negative uniform draws the first token with mass
  if (tid < ntiles) {
    const DF lo = tid ? s.tincl[tid - 1] : DF{0.f, 0.f};
    if (df_pos(tt) && df_le(lo, T)) atomicMax(&s.pick, tid);
  }
  __syncthreads();
  const int kt = s.pick;  // >= 0: the first tile with mass has lower edge 0 <= T
  const DF Tk = kt > 0 ? df_sub(T, s.tincl[kt - 1]) : T;

  // The chosen tile: thread tid spans [wexcl[warp] + lane_lo, ... + ts).
  const int v = kt * kThreads + tid;
  const int x = v * EPV;
  float zp[EPV], r[EPV];
  const uint4 wp = v < nvec ? ld_stream16(d.trow + v) : neg_inf_vec<DT>();
  Elem<DT>::unpack(wp, zp);
  const float ts = residual<EPV>(d, P.c, zp, x, r);
  const float incl = warp_incl_scan(ts, lane);
  float lane_lo = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) lane_lo = 0.f;
  if (lane == 31) s.redf[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    DF acc{0.f, 0.f};
    s.wexcl[0] = acc;
    for (int w = 0; w < kWarps; ++w) {
      acc = df_add_f(acc, s.redf[w]);
      s.wexcl[w + 1] = acc;
    }
    s.pick2 = -1;
    s.tok = -1;
  }
  __syncthreads();
  const DF lo = df_add_f(s.wexcl[warp], lane_lo);
  if (ts > 0.f && df_le(lo, Tk)) atomicMax(&s.pick2, tid);
  __syncthreads();
  if (tid == s.pick2) {
    DF run = lo;
    int cand = x;
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      if (r[j] > 0.f && df_le(run, Tk)) cand = x + j;
      run = df_add_f(run, r[j]);
    }
    s.tok = cand;
  }
  __syncthreads();
  const int y = s.tok;
  __syncthreads();  // the scratch is free again
  return y;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) onehot_verify_kernel(RParams P) {
  constexpr int EPV = Elem<DT>::kEPV;
  __shared__ Shm s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x;
  const int nvec = P.nvec;
  const int stride = kThreads * kU;  // vectors per round of the CTA

  // Offsets: every CTA checks and all take the same decision. The row's
  // first loads need only R_t = cu[B] + B (the rows the layout claims,
  // within the workspace): they go out before the rest of the check.
  const int R_d = P.cu[P.B];
  const long long R_t = (long long)R_d + P.B;
  const bool rows_ok = R_d >= 0 && R_t <= P.row_cap;
  const bool live = rows_ok && t < R_t;
  const uint4* trow = reinterpret_cast<const uint4*>(static_cast<const char*>(P.target) + (size_t)t * nvec * 16);
  uint4 rt[kU];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int v = u * kThreads + tid;
    rt[u] = (live && v < nvec) ? ld_stream16(trow + v) : neg_inf_vec<DT>();
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

  // The row's request.
  const int bq = find_request(P.cu, P.B, t);
  if (tid == 0) {
    const int t0 = P.cu[bq] + bq, d0 = P.cu[bq];
    const int K = P.cu[bq + 1] - d0, i = t - t0;
    int greedy = P.greedy_all;
    if (!greedy && P.mode) {
      const uint8_t m = P.mode[bq];
      if (m == SV_MODE_GREEDY)
        greedy = 1;
      else if (m != SV_MODE_SAMPLE && i == 0)
        atomicOr(P.status, SV_DATA_BAD_MODE);
    }
    int xhat = -1;
    if (i < K) {
      xhat = P.draft_tokens[d0 + i];
      if (xhat < 0 || xhat >= P.V) {
        atomicOr(P.status, SV_DATA_BAD_TOKEN);
        xhat = -1;
      }
    }
    s.b = bq;
    s.t0 = t0;
    s.d0 = d0;
    s.K = K;
    s.i = i;
    s.greedy = greedy;
    s.xhat = xhat;
    s.u = (!greedy && i < K && P.uniforms) ? __ldg(&P.uniforms[2 * (size_t)t]) : 0.f;
    s.last = 0;
  }
  __syncthreads();
  const int b = s.b, t0 = s.t0, d0 = s.d0, K = s.K, i = s.i, xhat = s.xhat;
  const bool greedy = s.greedy != 0;

  RRow rec;
  if (greedy) {
    // Strict row: its argmax only.
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int v0 = 0; v0 < nvec; v0 += stride) {
      if (v0 > 0) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int v = v0 + u * kThreads + tid;
          rt[u] = v < nvec ? ld_stream16(trow + v) : neg_inf_vec<DT>();
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        float f[EPV];
        Elem<DT>::unpack(rt[u], f);
        amax_fold<EPV>(f, (v0 + u * kThreads + tid) * EPV, bv, bi);
      }
    }
    // The merge keeps the largest value and, among equal values, the lowest
    // index (each thread met its own elements in increasing order).
    warp_argmax(bv, bi);
    if (lane == 0) {
      s.redf[warp] = bv;
      s.redi[warp] = bi;
    }
    __syncthreads();
    float v = s.redf[0];
    int k = s.redi[0];
    for (int w = 1; w < kWarps; ++w) argmax_merge(v, k, s.redf[w], s.redi[w]);
    const int am = k == INT_MAX ? 0 : k;  // all -inf: index 0, like argmax
    rec.mc_p = rec.mc_q = 0.f;
    rec.S_p = rec.S_q = DF{0.f, 0.f};
    rec.am = am;
    rec.accept = (i < K && xhat == am) ? 1u : 0u;
    if (tid == 0 && P.out_probs && i < K) {
      P.out_probs[2 * (size_t)t] = -1.f;
      P.out_probs[2 * (size_t)t + 1] = -1.f;
    }
  } else {
    // Sampled row: (m, S) of the row, z(x̂) from one load.
    float zxp = -INFINITY;
    if (tid == 0 && i < K && xhat >= 0) zxp = Elem<DT>::scalar(trow, xhat);
    Soft at{-INFINITY, 0.f, 0.f};
    for (int v0 = 0; v0 < nvec; v0 += stride) {
      if (v0 > 0) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int v = v0 + u * kThreads + tid;
          rt[u] = v < nvec ? ld_stream16(trow + v) : neg_inf_vec<DT>();
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        float f[EPV];
        Elem<DT>::unpack(rt[u], f);
        soft_fold<EPV>(at, f, P.c);
      }
    }
    float mcp;
    DF Sp;
    cta_soft(s, at, P.c, mcp, Sp);
    rec.mc_p = mcp;
    rec.mc_q = 0.f;
    rec.S_p = Sp;
    rec.S_q = DF{0.f, 0.f};
    rec.am = 0;
    rec.accept = 1u;  // bonus rows count as accepted
    if (tid == 0) {
      if (!df_pos(Sp)) atomicOr(P.status, SV_DATA_EMPTY_ROW);
      if (i < K) {
        float ph = -1.f, qh = -1.f;
        unsigned acc = 0u;
        if (xhat >= 0) {
          // p(x̂) = 2^(z c - mc_p) / S_p and min(1, p(x̂) / 1), in fp32 as
          // the persistent kernel takes them; q(x̂) = 1.
          const float pd = __fdiv_rn(exp2f(fmaf(zxp, P.c, -mcp)), Sp.hi);
          acc = (s.u < fminf(1.f, pd)) ? 1u : 0u;
          ph = pd;
          qh = 1.f;
        }
        rec.accept = acc;
        if (P.out_probs) {
          P.out_probs[2 * (size_t)t] = ph;
          P.out_probs[2 * (size_t)t + 1] = qh;
        }
      }
    }
  }

  // The row's record and its bits in the request's progress word; the
  // update releases the record and acquires those of the rows before it.
  const bool tracked = K <= kMaxTracked;
  if (tid == 0) {
    P.rows[t] = rec;
    const bool acc = i < K && (rec.accept & 1u);
    const unsigned long long add = tracked ? ((1ull << i) | (acc ? 1ull << (32 + i) : 0ull)) : 1ull;
    const unsigned long long old =
        tracked ? atom_or_acqrel_gpu(&P.arrive[b], add) : atom_add_acqrel_gpu(&P.arrive[b], add);
    const unsigned long long word = old | add;
    const unsigned long long all = tracked ? (1ull << (K + 1)) - 1ull : 0ull;  // the rows' done bits
    const bool last = tracked ? ((word & all) == all && (old & all) != all) : old == (unsigned long long)K;
    if (last) {
      s.last = 1;
      int stop = K;
      if (tracked) {
        const unsigned rej = ~(unsigned)(word >> 32) & (unsigned)((1ull << K) - 1ull);
        if (rej) stop = __ffs(rej) - 1;
      }
      s.stop = stop;
      P.arrive[b] = 0ull;  // every row is in: ready for the next call
    }
  }
  __syncthreads();
  if (!s.last) return;

  // The request's last row: first rejection, the drafts before it, and the
  // stop row's token.
  __threadfence();  // every thread reads the other rows' records after the update
  int stop = s.stop;
  if (!tracked) {
    if (warp == 0) {
      stop = K;
      for (int j0 = 0; j0 < K && stop == K; j0 += 32) {
        const int j = j0 + lane;
        const bool rej = j < K && (__ldcg(&P.rows[t0 + j].accept) & 1u) == 0u;
        const unsigned m = __ballot_sync(kFull, rej);
        if (m) stop = j0 + __ffs(m) - 1;
      }
      if (lane == 0) s.stop = stop;
    }
    __syncthreads();
    stop = s.stop;
  }
  for (int j = tid; j < stop; j += kThreads) P.out_tokens[t0 + j] = P.draft_tokens[d0 + j];
  const int srow = t0 + stop;
  if (tid == 0) P.out_len[b] = stop + 1;
  if (greedy) {
    if (tid == 0) {
      P.out_tokens[srow] = (srow == t) ? rec.am : __ldcg(&P.rows[srow].am);
      if (P.out_probs) {
        P.out_probs[2 * (size_t)(t0 + K)] = -1.f;
        P.out_probs[2 * (size_t)(t0 + K) + 1] = -1.f;
      }
    }
    return;
  }
  // The draw at the stop row: p without the rejected proposal, or the
  // bonus row's p if all K are accepted.
  Draw d;
  int kind = kBonus, xs = -1;
  if (stop < K) {
    xs = P.draft_tokens[d0 + stop];
    if (xs < 0 || xs >= P.V) xs = -1;
    kind = kOneHot;
  }
  const float mcp = (srow == t) ? rec.mc_p : __ldcg(&P.rows[srow].mc_p);
  const DF Sp = (srow == t) ? rec.S_p : ldcg_df(&P.rows[srow].S_p);
  d.trow = reinterpret_cast<const uint4*>(static_cast<const char*>(P.target) + (size_t)srow * nvec * 16);
  d.kind = kind;
  d.xhat = xs;
  d.mcp = mcp;
  d.u2 = __ldg(&P.uniforms[2 * (size_t)srow + 1]);
  int y = draw_row<DT>(P, s, d);
  if (y < 0 && kind != kBonus) {
    // No mass besides the proposal's: draw from p instead.
    if (tid == 0) atomicOr(P.status, SV_DATA_DEGENERATE_RESIDUAL);
    Draw dp = d;
    dp.kind = kBonus;
    y = draw_row<DT>(P, s, dp);
  }
  if (tid == 0) {
    if (y < 0) {
      atomicOr(P.status, SV_DATA_EMPTY_ROW);
      y = 0;
    }
    const float zp = Elem<DT>::scalar(d.trow, y);
    const float py = __fdiv_rn(exp2f(fmaf(zp, P.c, -mcp)), Sp.hi);
    const float qy = (kind == kOneHot && y == xs) ? 1.f : 0.f;
    P.out_tokens[srow] = y;
    if (P.out_probs) {
      P.out_probs[2 * (size_t)(t0 + K)] = py;
      P.out_probs[2 * (size_t)(t0 + K) + 1] = qy;
    }
  }
}

}  // namespace oh

cudaError_t launch_onehot_verify(const RParams& P, int dtype, cudaStream_t st) {
  const long long rows = P.row_cap < 1 ? 1 : P.row_cap;
  if (dtype == 1)
    oh::onehot_verify_kernel<1><<<(unsigned)rows, kThreads, 0, st>>>(P);
  else
    oh::onehot_verify_kernel<0><<<(unsigned)rows, kThreads, 0, st>>>(P);
  return cudaGetLastError();
}

}  // namespace sv
