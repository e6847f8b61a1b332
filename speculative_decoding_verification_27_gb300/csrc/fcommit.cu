// fcommit.cu -- decisions, draws and commits of the top-k / top-p filtered
// step from the statistics the threshold kernels left, one CTA per request.
//
// "投机解码从零实现" §5.4: with the same filter applied to target and draft,
// the step of "Draft Model（草稿模型）" §2 runs on the filtered p' and q':
// accept x̂_i with probability min(1, p'(x̂_i)/q'(x̂_i)); at the first
// rejection draw from norm(max(0, p' - q')); if all K are accepted draw the
// bonus token from p'_{K+1}.
//
// When the threshold step left every row of a request its filtered softmax
// statistics (offset mc, sum S) and the stop row its kept (token, logit)
// list, nothing of the request's rows has to be read again but z(x̂) of each
// slot and, for a residual draw, the draft row at the listed tokens. So one
// CTA per request does the whole step: warp 0 decides every slot at once
// (lane j takes slot j), the first rejection comes from one ballot, and the
// CTA draws from the stop row's list (r at the listed tokens, put in
// vocabulary order, scanned in double-float). Requests it cannot finish are
// left to the streaming verify kernel, which then skips the others.
//
// Flags in the workspace, all written in stream order (no CTA waits): each
// CTA writes done[b] (1: committed here); a CTA that leaves its request sets
// need_slow, which the verify kernel reads on entry (0: it returns at once)
// and its last CTA clears; CTA 0 clears rows_left, the word through which the
// one-warp threshold kernel told the CTA threshold kernel of rows it left.
#include "../../include/spec_verify.h"
#include "sv_device.cuh"
#include "sv_filter.cuh"

#include <climits>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace fc {

enum { kResidual = 0, kOneHot = 1, kBonus = 2 };
constexpr int kMaxK = 31;  // slots per request decided by one warp

static_assert(kKeptListCap <= kThreads, "one listed token per thread");

template <int DT>
__device__ __forceinline__ float logit_at(const void* rows, size_t row, int V, int x) {
  return Elem<DT>::scalar(static_cast<const char*>(rows) + row * (size_t)V * Elem<DT>::kBytes, x);
}

// Logits below the row's threshold have no mass.
__device__ __forceinline__ float masked(float z, float tau) { return z >= tau ? z : -INFINITY; }

struct Smem {
  int lx[kThreads];     // listed tokens, in list order
  int ox[kThreads];     // the same in vocabulary order
  float orr[kThreads];  // r at them, in vocabulary order
  float oz[kThreads];   // their target logits
  float oq[kThreads];   // their draft logits (residual draws), masked below the draft threshold
  DF dred[kWarps], dred2[kWarps];
  int pick;
  // the request, as warp 0 decided it
  int go, stop, kind, xhat, srow, drow, brow, nl;
  float mcp, mcq, tau_p, tau_q, u2;
  DF Sp, Sq;
};

// The drawn token with its target logit and, for a residual draw, its
// draft logit (both as the step reads them), or y = -1.
struct Pick {
  int y;
  float zp, zq;
};

// Inverse CDF over the stop row's kept list (n <= kThreads entries): r at
// the listed tokens, ranked into vocabulary order, the smallest token whose
// running sum exceeds u' * Z. y = -1 if r has no mass.
template <int DT>
__device__ Pick draw_from_list(const FcParams& P, Smem& s, const int2* ent, int n, int kind, float bhi,
                               float blo) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int x = INT_MAX;
  float r = 0.f, zp = -INFINITY, zq = -INFINITY;
  if (tid < n) {
    const int2 e = __ldcg(ent + tid);
    x = e.x;
    zp = __int_as_float(e.y);
    const float ep = ex2(fmaf(zp, P.c, -s.mcp));
    if (kind == kResidual) {
      zq = masked(logit_at<DT>(P.draft, (size_t)s.drow, P.V, x), s.tau_q);
      const float eq = ex2(fmaf(zq, P.c, -s.mcq));
      float d = fmaf(-eq, bhi, ep);
      d = fmaf(-eq, blo, d);
      r = fmaxf(d, 0.f);
    } else {
      r = (kind == kOneHot && x == s.xhat) ? 0.f : ep;
    }
    s.lx[tid] = x;
  }
  if (tid == 0) s.pick = -1;
  __syncthreads();
  if (tid < n) {
    int rank = 0;  // listed tokens are distinct
    for (int j = 0; j < n; ++j) rank += s.lx[j] < x ? 1 : 0;
    s.ox[rank] = x;
    s.orr[rank] = r;
    s.oz[rank] = zp;
    s.oq[rank] = zq;
  }
  __syncthreads();
  const float rv = tid < n ? s.orr[tid] : 0.f;
  const DF inc = warp_incl_scan_df(DF{rv, 0.f}, lane);
  if (lane == 31) s.dred[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    DF v = lane < kWarps ? s.dred[lane] : DF{0.f, 0.f};
    v = warp_incl_scan_df(v, lane);
    if (lane < kWarps) s.dred2[lane] = v;
  }
  __syncthreads();
  DF lo{__shfl_up_sync(kFull, inc.hi, 1), __shfl_up_sync(kFull, inc.lo, 1)};
  if (lane == 0) lo = DF{0.f, 0.f};
  if (warp) lo = df_add(s.dred2[warp - 1], lo);
  const DF Z = s.dred2[kWarps - 1];
  Pick pk{-1, -INFINITY, -INFINITY};
  if (df_pos(Z)) {
    DF T = df_mul_f(Z, s.u2);
    if (!(T.hi >= 0.f)) T = DF{0.f, 0.f};  // a NaN or negative uniform draws the first token with mass
    if (tid < n && rv > 0.f && df_le(lo, T)) atomicMax(&s.pick, tid);
    __syncthreads();
    const int k = s.pick;
    if (k >= 0) pk = Pick{s.ox[k], s.oz[k], s.oq[k]};
  }
  __syncthreads();
  return pk;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) filtered_commit_kernel(FcParams P) {
  __shared__ Smem s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  // The threshold kernels have read their word: clear it for the next call.
  if (b == 0 && tid == 0 && P.rows_left) *P.rows_left = 0u;
  // Offsets of the whole batch, checked the way the verify kernel does so
  // that a bad layout is left whole to it (it reports and commits nothing).
  // The result is needed only before the first write; warp 0 meanwhile
  // reads its request's rows, which its own check keeps in bounds.
  bool bad = false;
  for (int k = tid; k < P.B; k += kThreads)
    if (P.cu[k + 1] < P.cu[k]) bad = true;
  if (tid == 0 && (P.cu[0] != 0 || (long long)P.cu[P.B] + P.B > P.rows_t)) bad = true;

  int go = 0, K = 0, t0 = 0, d0 = 0, stop = 0, xhat = -1;
  bool slot = false;
  float ph = -1.f, qh = -1.f;
  unsigned bits = 0u;
  if (warp == 0) {
    d0 = P.cu[b];
    const int d1 = P.cu[b + 1], dB = P.cu[P.B];
    // Rows t0 .. t0 + K and draft rows d0 .. d1 - 1 lie inside the batch.
    go = (d0 >= 0 && d1 >= d0 && d1 <= dB && (long long)dB + P.B <= P.rows_t) ? 1 : 0;
    K = go ? d1 - d0 : 0;
    if (K > kMaxK || (K > 0 && !P.draft_tokens)) go = 0;
    if (P.mode && P.mode[b] != SV_MODE_SAMPLE) go = 0;  // greedy (or invalid) requests: verify kernel
    t0 = d0 + b;
    const int j = lane, t = t0 + j;
    const bool row = go && j <= K, has_d = go && j < K && P.draft != nullptr;
    slot = go && j < K;
    // Every load of the slot's decision that depends on no other load goes
    // out at once; the logits at x̂ follow.
    FStat ft{}, fd{};
    ft.ok = fd.ok = 1;
    float tau_t = -INFINITY, tau_d = -INFINITY, u = 0.f, u2 = 0.f;
    if (row) {
      ft = P.fst_t[t];
      tau_t = __ldg(&P.thr_t[t]);
      u2 = __ldg(&P.uniforms[2 * (size_t)t + 1]);
    }
    if (has_d) {
      fd = P.fst_d[d0 + j];
      tau_d = __ldg(&P.thr_d[d0 + j]);
    }
    if (slot) {
      xhat = P.draft_tokens[d0 + j];
      u = __ldg(&P.uniforms[2 * (size_t)t]);
    }
    const bool xok = xhat >= 0 && xhat < P.V;
    float zp = -INFINITY, zq = -INFINITY;
    if (slot && xok) {
      zp = masked(logit_at<DT>(P.target, (size_t)t, P.V, xhat), tau_t);
      if (has_d) zq = masked(logit_at<DT>(P.draft, (size_t)(d0 + j), P.V, xhat), tau_d);
    }
    go = __all_sync(kFull, ft.ok && fd.ok) ? go : 0;
    // Slot j: p(x̂), q(x̂) and the accept test, in the verify kernel's operations.
    const DF Sp = df_from_d(ft.S), Sq = has_d ? df_from_d(fd.S) : DF{0.f, 0.f};
    bool acc = false;
    if (row && (!df_pos(Sp) || (has_d && !df_pos(Sq)))) bits |= SV_DATA_EMPTY_ROW;
    if (slot && !xok) {
      bits |= SV_DATA_BAD_TOKEN;
      xhat = -1;
    }
    if (slot && xok) {
      const float ap = fmaf(zp, P.c, -ft.mc);
      const float Spf = Sp.hi, Sqf = Sq.hi;
      const float pd = __fdiv_rn(exp2f(ap), Spf);
      float rho, qd = 1.f;
      if (has_d) {
        const float aq = fmaf(zq, P.c, -fd.mc);
        qd = __fdiv_rn(exp2f(aq), Sqf);
        rho = (zq == -INFINITY) ? 0.f : fminf(1.f, __fmul_rn(exp2f(ap - aq), __fdiv_rn(Sqf, Spf)));
      } else {
        rho = fminf(1.f, pd);
      }
      acc = u < rho;
      ph = pd;
      qh = qd;
    }
    const unsigned rej = __ballot_sync(kFull, slot && !acc);
    stop = rej ? __ffs(rej) - 1 : K;
    // The stop row's kept list: without one the request is left whole.
    const int nl = __shfl_sync(kFull, ft.nl, stop);
    if (nl < 1 || nl > kKeptListCap) go = 0;
    bits = __reduce_or_sync(kFull, bits);
    const DF Sps{__shfl_sync(kFull, Sp.hi, stop), __shfl_sync(kFull, Sp.lo, stop)};
    const DF Sqs{__shfl_sync(kFull, Sq.hi, stop), __shfl_sync(kFull, Sq.lo, stop)};
    const float mcp = __shfl_sync(kFull, ft.mc, stop), mcq = __shfl_sync(kFull, fd.mc, stop);
    const float tq = __shfl_sync(kFull, tau_d, stop), tp = __shfl_sync(kFull, tau_t, stop);
    const float us = __shfl_sync(kFull, u2, stop);
    const int xs = __shfl_sync(kFull, xhat, stop);
    if (lane == 0 && go) {
      const int srow = t0 + stop;
      const int kind = stop < K ? (P.draft ? kResidual : kOneHot) : kBonus;
      s.stop = stop;
      s.kind = kind;
      s.xhat = stop < K ? xs : -1;
      s.srow = srow;
      s.drow = d0 + stop;
      s.brow = t0 + K;
      s.nl = nl;
      s.mcp = mcp;
      s.mcq = kind == kResidual ? mcq : 0.f;
      s.Sp = Sps;
      s.Sq = kind == kResidual ? Sqs : DF{0.f, 0.f};
      s.u2 = us;
      s.tau_p = tp;
      s.tau_q = kind == kResidual ? tq : -INFINITY;
    }
  }
  const bool bad_any = __syncthreads_or(bad);
  if (warp == 0) {
    if (bad_any) go = 0;
    if (go) {
      if (lane == 0 && bits) atomicOr(P.status, bits);
      const int t = t0 + lane;
      if (slot && P.out_probs) {
        P.out_probs[2 * (size_t)t] = ph;
        P.out_probs[2 * (size_t)t + 1] = qh;
      }
      if (lane < stop) P.out_tokens[t] = xhat;  // accepted slots hold valid tokens
      if (lane == 0) P.out_len[b] = stop + 1;
    }
    if (lane == 0) {
      s.go = go;
      if (!go) {
        P.done[b] = 0;
        atomicOr(P.need_slow, 1u);
      }
    }
  }
  __syncthreads();
  if (!s.go) return;

  // The draw at the stop row, from its kept list.
  const int kind = s.kind, srow = s.srow;
  const DF beta = (kind == kResidual && df_pos(s.Sq)) ? df_div(s.Sp, s.Sq) : DF{1.f, 0.f};
  const int2* ent = P.list_t + (size_t)srow * kKeptListCap;
  Pick pk = draw_from_list<DT>(P, s, ent, s.nl, kind, beta.hi, beta.lo);
  bool have_q = kind == kResidual;
  if (pk.y < 0 && kind != kBonus) {
    // No residual mass (p' == q' in fp32): draw from p' instead.
    if (tid == 0) atomicOr(P.status, SV_DATA_DEGENERATE_RESIDUAL);
    pk = draw_from_list<DT>(P, s, ent, s.nl, kBonus, 1.f, 0.f);
    have_q = false;
  }
  if (tid == 0) {
    int y = pk.y;
    float zp = pk.zp, zq = pk.zq;
    if (y < 0) {
      atomicOr(P.status, SV_DATA_EMPTY_ROW);
      y = 0;
      zp = masked(logit_at<DT>(P.target, (size_t)srow, P.V, 0), s.tau_p);
      have_q = false;
    }
    const float py = __fdiv_rn(exp2f(fmaf(zp, P.c, -s.mcp)), s.Sp.hi);
    float qy = 0.f;
    if (kind == kResidual) {
      if (!have_q) zq = masked(logit_at<DT>(P.draft, (size_t)s.drow, P.V, y), s.tau_q);
      qy = __fdiv_rn(exp2f(fmaf(zq, P.c, -s.mcq)), s.Sq.hi);
    } else if (kind == kOneHot) {
      qy = (y == s.xhat) ? 1.f : 0.f;
    }
    P.out_tokens[srow] = y;
    if (P.out_probs) {
      P.out_probs[2 * (size_t)s.brow] = py;
      P.out_probs[2 * (size_t)s.brow + 1] = qy;
    }
    P.done[b] = 1;
  }
}

}  // namespace fc

cudaError_t launch_filtered_commit(const FcParams& P, int dtype, cudaStream_t st) {
  if (P.B < 1) return cudaSuccess;
  if (dtype == 1)
    fc::filtered_commit_kernel<1><<<(unsigned)P.B, kThreads, 0, st>>>(P);
  else
    fc::filtered_commit_kernel<0><<<(unsigned)P.B, kThreads, 0, st>>>(P);
  return cudaGetLastError();
}

}  // namespace sv
