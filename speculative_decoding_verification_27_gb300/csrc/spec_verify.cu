// spec_verify.cu -- verify-and-commit of speculative decoding on sm_103a.
//
// One persistent kernel does the whole step:
//
//   1. Row pass. Work items are target rows t = (request b, slot i), handed
//      out in request order by an atomic counter. The CTA streams the target
//      row (and, for a sampled draft slot, the paired draft row) once with
//      16-byte loads and keeps a single-pass online softmax: per thread a
//      running maximum and one fp32 partial sum per vector lane, rescaled when
//      the maximum grows. Sums are combined in double-float arithmetic, so
//      S = sum_x 2^(z_x c - Mc) (c = log2(e)/T, Mc = fp32(max z * c)) is
//      accurate to ~1e-9 relative. Greedy rows compute the argmax instead
//      (lowest index among ties). The CTA then gathers z[x̂] and decides the
//      slot: accept iff u < min(1, p(x̂)/q(x̂)) ("Draft Model（草稿模型）",
//      §2 "接受-拒绝准则"; a zero draft probability rejects, "投机解码从零实现"
//      §4.3), or, strict mode, iff x̂ == argmax ("Speculative Decoding在分布式
//      推理中的应用", §二). The per-row record goes to the workspace.
//   2. Commit. Each finished row bumps its request's counter; the CTA that
//      finishes the request's last row (last-CTA-done: nobody waits) finds the
//      first rejected slot, writes the accepted drafts ("算法：Speculative
//      Decoding (一步)", step 3) and makes the final draw at the stop row s:
//        after a rejection  r = max(0, p - q)     ("接受-拒绝准则")
//        one-hot proposal   r = p without x̂       ("5.2 Draft 模型与无模型方案" §4.3)
//        all accepted       r = p                  (bonus token, algorithm box)
//        greedy request     the argmax of row s
//      The draw is the inverse CDF in vocabulary order: the smallest k whose
//      running sum of r exceeds u' * sum(r). It re-reads the stop row pair
//      (usually still in L2): pass A computes per-warp sums of r for every
//      tile, pass B rescans only the tile that holds the target.
//   The last CTA to leave resets the work counter, and each request's counter
//   is reset by its commit, so the workspace is left zeroed.
#include <atomic>
#include <cmath>
#include <cstring>

#include "../../include/spec_verify.h"
#include "sv_device.cuh"

namespace sv {

struct WsHeader {
  unsigned int status;     // SV_DATA_* bits (sticky until sv_check_status)
  unsigned int next_item;  // work counter of the persistent kernel
  unsigned int exited;     // CTAs that left the work loop
  unsigned int pad[13];
};
static_assert(sizeof(WsHeader) == 64, "workspace header is 64 bytes");

// Per target row result of the row pass (32 bytes).
struct alignas(16) RowRec {
  float mc_p;        // fp32(max z_target * c): exponent offset of the target row
  float mc_q;        // same for the paired draft row (sampled draft slots)
  double S_p;        // sum_x 2^(z_x c - mc_p) over the target row
  double S_q;        // same over the draft row
  int argmax;        // greedy rows: first index of the maximum
  unsigned accept;   // 1 if the slot's draft token is accepted
};
static_assert(sizeof(RowRec) == 32, "row record is 32 bytes");

constexpr int kMaxScanTiles = kThreads;   // the draw scans at most one tile per thread
// Largest vocabulary for each element type: kMaxScanTiles tiles of one
// 16-byte vector per thread (fp32 262144, bf16 524288).
constexpr int max_vocab(int dtype) { return kMaxScanTiles * kThreads * (dtype == 0 ? 4 : 8); }
constexpr int kScanUnroll = 4;            // tiles loaded ahead in the draw passes

enum DrawKind { kResidual = 0, kOneHot = 1, kBonus = 2 };

struct Params {
  const void* target;
  const void* draft;  // NULL: one-hot proposals
  int V, B;
  const int32_t* draft_tokens;
  const int32_t* cu;
  const uint8_t* mode;
  const float* uniforms;
  float c;  // log2(e) / T
  int32_t* out_tokens;
  int32_t* out_len;
  float* out_probs;
  WsHeader* ws;
  unsigned int* req_done;
  RowRec* rows;
  long long row_cap;
  int greedy_all;
};

struct Smem {
  int item, b, t0, d0, K, i, greedy, xhat, last, stop, pick, pick2, tok;
  float redf[kWarps];
  float redf2[kWarps];
  int redi[kWarps];
  DF reddf_p[kWarps];
  DF reddf_q[kWarps];
  float bcast_f[2];
  double dred[kWarps];
  double dred2[kWarps];
  double wexcl[kWarps + 1];
  double tincl[kMaxScanTiles];
  float wtot[kMaxScanTiles * kWarps];
};

// Online softmax state of one thread: running maximum m, its fp32 exponent
// offset mc = fp32(m * c) (0 while m is -inf) and one partial sum per lane of
// the 16-byte vector. Every term is 2^(z c - mc).
template <int EPV>
struct SoftAcc {
  float m, mc;
  float a[EPV];
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    mc = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) a[j] = 0.f;
  }
  __device__ __forceinline__ void add(const float (&f)[EPV], float c) {
    float vm = f[0];
#pragma unroll
    for (int j = 1; j < EPV; ++j) vm = fmaxf(vm, f[j]);
    if (vm > m) {
      float nmc = __fmul_rn(vm, c);
      float s = (m == -INFINITY) ? 0.f : ex2(mc - nmc);
#pragma unroll
      for (int j = 0; j < EPV; ++j) a[j] *= s;
      m = vm;
      mc = nmc;
    }
#pragma unroll
    for (int j = 0; j < EPV; ++j) a[j] += ex2(fmaf(f[j], c, -mc));
  }
};

// Streams one row (and optionally its draft row) through the online softmax.
template <int DT, bool VEC, bool HAS_D>
__device__ __forceinline__ void stats_pass(const void* trow, const void* drow, int V, float c,
                                           SoftAcc<Elem<DT>::kEPV>& at,
                                           SoftAcc<Elem<DT>::kEPV>& ad) {
  constexpr int EPV = Elem<DT>::kEPV;
  constexpr int TILE = kThreads * EPV;
  constexpr int U = HAS_D ? 4 : 8;
  int x = threadIdx.x * EPV;
  if constexpr (VEC) {
    const char* tb = static_cast<const char*>(trow);
    const char* db = static_cast<const char*>(drow);
    for (; x + (U - 1) * TILE < V; x += U * TILE) {
      uint4 rt[U], rd[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        rt[u] = ld_stream16(tb + (size_t)(x + u * TILE) * Elem<DT>::kBytes);
        if constexpr (HAS_D) rd[u] = ld_stream16(db + (size_t)(x + u * TILE) * Elem<DT>::kBytes);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[EPV];
        Elem<DT>::unpack(rt[u], f);
        at.add(f, c);
        if constexpr (HAS_D) {
          Elem<DT>::unpack(rd[u], f);
          ad.add(f, c);
        }
      }
    }
  }
  for (; x < V; x += TILE) {
    float f[EPV];
    load_chunk<DT, VEC>(trow, x, V, f);
    at.add(f, c);
    if constexpr (HAS_D) {
      load_chunk<DT, VEC>(drow, x, V, f);
      ad.add(f, c);
    }
  }
}

template <int DT, bool VEC>
__device__ __forceinline__ void argmax_pass(const void* trow, int V, float& bv, int& bi) {
  constexpr int EPV = Elem<DT>::kEPV;
  constexpr int TILE = kThreads * EPV;
  constexpr int U = 8;
  int x = threadIdx.x * EPV;
  if constexpr (VEC) {
    const char* tb = static_cast<const char*>(trow);
    for (; x + (U - 1) * TILE < V; x += U * TILE) {
      uint4 rt[U];
#pragma unroll
      for (int u = 0; u < U; ++u) rt[u] = ld_stream16(tb + (size_t)(x + u * TILE) * Elem<DT>::kBytes);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[EPV];
        Elem<DT>::unpack(rt[u], f);
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if (f[j] > bv) {
            bv = f[j];
            bi = x + u * TILE + j;
          }
      }
    }
  }
  for (; x < V; x += TILE) {
    float f[EPV];
    load_chunk<DT, VEC>(trow, x, V, f);
#pragma unroll
    for (int j = 0; j < EPV; ++j)
      if (f[j] > bv) {
        bv = f[j];
        bi = x + j;
      }
  }
}

// CTA combine of the online-softmax states into (Mc, S) for the target row
// and, if has_d, the draft row. Results are valid in thread 0.
template <int EPV>
__device__ void combine_softmax(SoftAcc<EPV>& at, SoftAcc<EPV>& ad, bool has_d, float c, Smem& s,
                                float& Mc_p, double& S_p, float& Mc_q, double& S_q) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float mp = warp_max(at.m);
  float mq = has_d ? warp_max(ad.m) : -INFINITY;
  if (lane == 0) {
    s.redf[warp] = mp;
    s.redf2[warp] = mq;
  }
  __syncthreads();
  if (warp == 0) {
    float v = lane < kWarps ? s.redf[lane] : -INFINITY;
    float w = lane < kWarps ? s.redf2[lane] : -INFINITY;
    v = warp_max(v);
    w = warp_max(w);
    if (lane == 0) {
      s.bcast_f[0] = v;
      s.bcast_f[1] = w;
    }
  }
  __syncthreads();
  const float Mp = s.bcast_f[0], Mq = s.bcast_f[1];
  const float mcp = (Mp == -INFINITY) ? 0.f : __fmul_rn(Mp, c);
  const float mcq = (Mq == -INFINITY) ? 0.f : __fmul_rn(Mq, c);
  DF tp{0.f, 0.f}, tq{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < EPV; ++j) tp = df_add_f(tp, at.a[j]);
  tp = df_mul_f(tp, (at.m == -INFINITY) ? 0.f : ex2(at.mc - mcp));
  tp = warp_sum_df(tp);
  if (has_d) {
#pragma unroll
    for (int j = 0; j < EPV; ++j) tq = df_add_f(tq, ad.a[j]);
    tq = df_mul_f(tq, (ad.m == -INFINITY) ? 0.f : ex2(ad.mc - mcq));
    tq = warp_sum_df(tq);
  }
  if (lane == 0) {
    s.reddf_p[warp] = tp;
    s.reddf_q[warp] = tq;
  }
  __syncthreads();
  if (warp == 0) {
    DF v = lane < kWarps ? s.reddf_p[lane] : DF{0.f, 0.f};
    DF w = lane < kWarps ? s.reddf_q[lane] : DF{0.f, 0.f};
    v = warp_sum_df(v);
    w = warp_sum_df(w);
    if (lane == 0) {
      Mc_p = mcp;
      Mc_q = mcq;
      S_p = (double)v.hi + (double)v.lo;
      S_q = (double)w.hi + (double)w.lo;
    }
  }
}

__device__ __forceinline__ int find_request(const int32_t* cu, int B, int t) {
  int lo = 0, hi = B - 1;  // largest b with cu[b] + b <= t
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cu[mid] + mid <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Inverse-CDF draw at a stop row. Returns the token, or -1 if r has no mass.
template <int DT, bool VEC>
__device__ int draw_token(const Params& P, Smem& s, int kind, const void* trow, const void* drow,
                          int xhat, float mcp, float mcq, double beta, double u2) {
  constexpr int EPV = Elem<DT>::kEPV;
  constexpr int TILE = kThreads * EPV;
  const int V = P.V;
  const float c = P.c;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntiles = (V + TILE - 1) / TILE;
  const float bhi = (float)beta;
  const float blo = (float)(beta - (double)bhi);

  // r for the EPV elements starting at x. kResidual: max(0, e_p - beta e_q)
  // with beta = S_p / S_q, i.e. S_p * max(0, p - q); otherwise e_p = S_p * p.
  auto r_of = [&](const float (&zp)[EPV], const float (&zq)[EPV], int x, float (&r)[EPV]) {
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      float ep = ex2(fmaf(zp[j], c, -mcp));
      if (kind == kResidual) {
        float eq = ex2(fmaf(zq[j], c, -mcq));
        float d = fmaf(-eq, bhi, ep);
        d = fmaf(-eq, blo, d);
        r[j] = fmaxf(d, 0.f);
      } else {
        r[j] = (kind == kOneHot && x + j == xhat) ? 0.f : ep;
      }
    }
  };

  // Pass A: per (tile, warp) sums of r, the warp sum being the last value of
  // the same Kogge-Stone scan that pass B repeats. The vector path keeps
  // kScanUnroll tiles of raw 16-byte loads in flight.
  auto tile_sum = [&](int k, const float (&zp)[EPV], const float (&zq)[EPV]) {
    const int x = k * TILE + tid * EPV;
    float r[EPV];
    r_of(zp, zq, x, r);
    float ts = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) ts += r[j];
    const float inc = warp_incl_scan(ts, lane);
    if (lane == 31) s.wtot[k * kWarps + warp] = inc;
  };
  if constexpr (VEC) {
    const char* tb = static_cast<const char*>(trow);
    const char* db = static_cast<const char*>(drow);
    for (int k0 = 0; k0 < ntiles; k0 += kScanUnroll) {
      uint4 vt[kScanUnroll], vd[kScanUnroll];
#pragma unroll
      for (int u = 0; u < kScanUnroll; ++u) {
        const int x = (k0 + u) * TILE + tid * EPV;
        if (x < V) {
          vt[u] = ld_stream16(tb + (size_t)x * Elem<DT>::kBytes);
          if (kind == kResidual) vd[u] = ld_stream16(db + (size_t)x * Elem<DT>::kBytes);
        }
      }
#pragma unroll
      for (int u = 0; u < kScanUnroll; ++u) {
        if (k0 + u < ntiles) {
          const int x = (k0 + u) * TILE + tid * EPV;
          float zp[EPV], zq[EPV];
          if (x < V) {
            Elem<DT>::unpack(vt[u], zp);
            if (kind == kResidual) Elem<DT>::unpack(vd[u], zq);
          } else {
#pragma unroll
            for (int j = 0; j < EPV; ++j) zp[j] = zq[j] = -INFINITY;
          }
          tile_sum(k0 + u, zp, zq);
        }
      }
    }
  } else {
    for (int k = 0; k < ntiles; ++k) {
      const int x = k * TILE + tid * EPV;
      float zp[EPV], zq[EPV];
      load_chunk<DT, VEC>(trow, x, V, zp);
      if (kind == kResidual) load_chunk<DT, VEC>(drow, x, V, zq);
      tile_sum(k, zp, zq);
    }
  }
  __syncthreads();

  // Tile sums (warps in order, fp64) and their inclusive prefix over tiles.
  double tt = 0.0;
  if (tid < ntiles) {
    for (int w = 0; w < kWarps; ++w) tt += (double)s.wtot[tid * kWarps + w];
  }
  double inc = warp_incl_scan_d(tt, lane);
  if (lane == 31) s.dred[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    double v = lane < kWarps ? s.dred[lane] : 0.0;
    v = warp_incl_scan_d(v, lane);
    if (lane < kWarps) s.dred2[lane] = v;
  }
  __syncthreads();
  if (tid < ntiles) s.tincl[tid] = inc + (warp > 0 ? s.dred2[warp - 1] : 0.0);
  if (tid == 0) s.pick = -1;
  __syncthreads();
  const double Z = s.tincl[ntiles - 1];
  if (!(Z > 0.0)) return -1;
  double T = u2 * Z;
  if (!(T >= 0.0)) T = 0.0;  // a NaN or negative uniform draws the first token with mass

  // Tile holding T: the last tile with mass whose lower edge is <= T. Tile k
  // spans [tincl[k-1], tincl[k]), so adjacent tiles share their edge.
  if (tid < ntiles) {
    double lo = tid ? s.tincl[tid - 1] : 0.0;
    if (tt > 0.0 && lo <= T) atomicMax(&s.pick, tid);
  }
  __syncthreads();
  const int kt = s.pick;
  if (kt < 0) return -1;  // unreachable: the first tile with mass has lower edge 0 <= T
  const double Tk = T - (kt ? s.tincl[kt - 1] : 0.0);

  // Pass B over that tile: thread k spans [wexcl[w] + lane_lo, wexcl[w] + inc).
  {
    const int x = kt * TILE + tid * EPV;
    float zp[EPV], zq[EPV], r[EPV];
    load_chunk<DT, VEC>(trow, x, V, zp);
    if (kind == kResidual) load_chunk<DT, VEC>(drow, x, V, zq);
    r_of(zp, zq, x, r);
    float ts = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) ts += r[j];
    float incl = warp_incl_scan(ts, lane);
    float lane_lo = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) lane_lo = 0.f;
    if (tid == 0) {
      double acc = 0.0;
      s.wexcl[0] = 0.0;
      for (int w = 0; w < kWarps; ++w) {
        acc = acc + (double)s.wtot[kt * kWarps + w];
        s.wexcl[w + 1] = acc;
      }
      s.pick2 = -1;
      s.tok = -1;
    }
    __syncthreads();
    const double lo = s.wexcl[warp] + (double)lane_lo;
    if (ts > 0.f && lo <= Tk) atomicMax(&s.pick2, tid);
    __syncthreads();
    if (tid == s.pick2) {
      double run = lo;
      int cand = x;
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        if (r[j] > 0.f && run <= Tk) cand = x + j;
        run += (double)r[j];
      }
      s.tok = cand;
    }
    __syncthreads();
  }
  return s.tok;
}

template <int DT, bool VEC>
__device__ __noinline__ void commit_request(const Params& P, Smem& s, int b, int t0, int d0, int K, bool greedy) {
  const int tid = threadIdx.x;
  const size_t rowb = (size_t)P.V * Elem<DT>::kBytes;
  if (tid == 0) {
    __threadfence();
    int stop = K;
    for (int i = 0; i < K; ++i) {
      if (__ldcg(&P.rows[t0 + i].accept) == 0u) {
        stop = i;
        break;
      }
    }
    s.stop = stop;
  }
  __syncthreads();
  const int stop = s.stop;
  for (int j = tid; j < stop; j += kThreads) P.out_tokens[t0 + j] = P.draft_tokens[d0 + j];
  const int srow = t0 + stop;
  int y;
  float py = -1.f, qy = -1.f;
  if (greedy) {
    y = __ldcg(&P.rows[srow].argmax);
  } else {
    const float mcp = __ldcg(&P.rows[srow].mc_p);
    const float mcq = __ldcg(&P.rows[srow].mc_q);
    const double Sp = __ldcg(&P.rows[srow].S_p);
    const double Sq = __ldcg(&P.rows[srow].S_q);
    const char* trow = static_cast<const char*>(P.target) + (size_t)srow * rowb;
    const char* drow = nullptr;
    int kind = kBonus, xhat = -1;
    if (stop < K) {
      xhat = P.draft_tokens[d0 + stop];
      if (xhat < 0 || xhat >= P.V) xhat = -1;
      if (P.draft) {
        kind = kResidual;
        drow = static_cast<const char*>(P.draft) + (size_t)(d0 + stop) * rowb;
      } else {
        kind = kOneHot;
      }
    }
    const double u2 = (double)__ldg(&P.uniforms[2 * (size_t)srow + 1]);
    y = draw_token<DT, VEC>(P, s, kind, trow, drow, xhat, mcp, mcq,
                            kind == kResidual ? Sp / Sq : 1.0, u2);
    if (y < 0 && kind != kBonus) {
      // No residual mass (p == q in fp32): draw from p instead.
      if (tid == 0) atomicOr(&P.ws->status, SV_DATA_DEGENERATE_RESIDUAL);
      kind = kBonus;
      y = draw_token<DT, VEC>(P, s, kind, trow, drow, xhat, mcp, mcq, 1.0, u2);
    }
    if (y < 0) {
      if (tid == 0) atomicOr(&P.ws->status, SV_DATA_EMPTY_ROW);
      y = 0;
    }
    if (tid == 0) {
      float zp = Elem<DT>::scalar(trow, y);
      py = (float)((double)exp2f(fmaf(zp, P.c, -mcp)) / Sp);
      if (kind == kResidual) {
        float zq = Elem<DT>::scalar(drow, y);
        qy = (float)((double)exp2f(fmaf(zq, P.c, -mcq)) / Sq);
      } else if (kind == kOneHot) {
        qy = (y == xhat) ? 1.f : 0.f;
      } else {
        qy = 0.f;
      }
    }
  }
  if (tid == 0) {
    P.out_tokens[srow] = y;
    P.out_len[b] = stop + 1;
    if (P.out_probs) {
      P.out_probs[2 * (size_t)(t0 + K)] = py;
      P.out_probs[2 * (size_t)(t0 + K) + 1] = qy;
    }
    P.req_done[b] = 0u;
  }
}

template <int DT, bool VEC>
__device__ void process_row(const Params& P, Smem& s, int t) {
  constexpr int EPV = Elem<DT>::kEPV;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    const int b = find_request(P.cu, P.B, t);
    const int t0 = P.cu[b] + b, d0 = P.cu[b];
    const int K = P.cu[b + 1] - d0;
    const int i = t - t0;
    int greedy = P.greedy_all;
    if (!greedy && P.mode) {
      const uint8_t m = P.mode[b];
      if (m == SV_MODE_GREEDY)
        greedy = 1;
      else if (m != SV_MODE_SAMPLE && i == 0)
        atomicOr(&P.ws->status, SV_DATA_BAD_MODE);
    }
    int xhat = -1;
    if (i < K) {
      xhat = P.draft_tokens[d0 + i];
      if (xhat < 0 || xhat >= P.V) {
        atomicOr(&P.ws->status, SV_DATA_BAD_TOKEN);
        xhat = -1;
      }
    }
    s.b = b;
    s.t0 = t0;
    s.d0 = d0;
    s.K = K;
    s.i = i;
    s.greedy = greedy;
    s.xhat = xhat;
  }
  __syncthreads();
  const int b = s.b, t0 = s.t0, d0 = s.d0, K = s.K, i = s.i, xhat = s.xhat;
  const bool greedy = s.greedy != 0;
  const size_t rowb = (size_t)P.V * Elem<DT>::kBytes;
  const char* trow = static_cast<const char*>(P.target) + (size_t)t * rowb;
  RowRec rec;
  if (greedy) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    argmax_pass<DT, VEC>(trow, P.V, bv, bi);
    warp_argmax(bv, bi);
    if (lane == 0) {
      s.redf[warp] = bv;
      s.redi[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
      float v = lane < kWarps ? s.redf[lane] : -INFINITY;
      int ix = lane < kWarps ? s.redi[lane] : 0x7fffffff;
      warp_argmax(v, ix);
      if (lane == 0) {
        const int am = (ix == 0x7fffffff) ? 0 : ix;  // all -inf: index 0, like argmax
        rec.mc_p = rec.mc_q = 0.f;
        rec.S_p = rec.S_q = 0.0;
        rec.argmax = am;
        rec.accept = (i < K && xhat == am) ? 1u : 0u;
        if (P.out_probs && i < K) {
          P.out_probs[2 * (size_t)t] = -1.f;
          P.out_probs[2 * (size_t)t + 1] = -1.f;
        }
      }
    }
  } else {
    const bool has_d = (i < K) && (P.draft != nullptr);
    const char* drow = has_d ? static_cast<const char*>(P.draft) + (size_t)(d0 + i) * rowb : nullptr;
    SoftAcc<EPV> at, ad;
    at.init();
    ad.init();
    if (has_d)
      stats_pass<DT, VEC, true>(trow, drow, P.V, P.c, at, ad);
    else
      stats_pass<DT, VEC, false>(trow, drow, P.V, P.c, at, ad);
    float mcp, mcq;
    double Sp, Sq;
    combine_softmax<EPV>(at, ad, has_d, P.c, s, mcp, Sp, mcq, Sq);
    if (tid == 0) {
      rec.mc_p = mcp;
      rec.mc_q = mcq;
      rec.S_p = Sp;
      rec.S_q = Sq;
      rec.argmax = 0;
      rec.accept = 1u;
      if (!(Sp > 0.0) || (has_d && !(Sq > 0.0))) atomicOr(&P.ws->status, SV_DATA_EMPTY_ROW);
      if (i < K) {
        float ph = -1.f, qh = -1.f;
        unsigned acc = 0u;
        if (xhat >= 0) {
          // p(x̂) = 2^(z c - mc_p) / S_p, and min(1, p/q) with q from the
          // draft row or q = 1 for a one-hot proposal.
          const float zp = Elem<DT>::scalar(trow, xhat);
          const float ap = fmaf(zp, P.c, -mcp);
          const double pd = (double)exp2f(ap) / Sp;
          double rho;
          double qd = 1.0;
          if (has_d) {
            const float zq = Elem<DT>::scalar(drow, xhat);
            const float aq = fmaf(zq, P.c, -mcq);
            qd = (double)exp2f(aq) / Sq;
            rho = (zq == -INFINITY) ? 0.0 : fmin(1.0, (double)exp2f(ap - aq) * (Sq / Sp));
          } else {
            rho = fmin(1.0, pd);
          }
          const double u = (double)__ldg(&P.uniforms[2 * (size_t)t]);
          acc = (u < rho) ? 1u : 0u;
          ph = (float)pd;
          qh = (float)qd;
        }
        rec.accept = acc;
        if (P.out_probs) {
          P.out_probs[2 * (size_t)t] = ph;
          P.out_probs[2 * (size_t)t + 1] = qh;
        }
      }
    }
  }
  if (tid == 0) {
    P.rows[t] = rec;
    __threadfence();
    const unsigned old = atomicAdd(&P.req_done[b], 1u);
    s.last = (old == (unsigned)K) ? 1 : 0;
  }
  __syncthreads();
  if (s.last) commit_request<DT, VEC>(P, s, b, t0, d0, K, greedy);
  __syncthreads();
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(Params P) {
  __shared__ Smem s;
  const int tid = threadIdx.x;
  // Offsets must be a valid packed layout that fits the workspace; every CTA
  // checks and all of them take the same decision.
  bool bad = false;
  for (int k = tid; k < P.B; k += kThreads)
    if (P.cu[k + 1] < P.cu[k]) bad = true;
  if (tid == 0) {
    if (P.cu[0] != 0) bad = true;
    if ((long long)P.cu[P.B] + P.B > P.row_cap) bad = true;
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(&P.ws->status, SV_DATA_BAD_OFFSETS);
    return;
  }
  const int R_t = P.cu[P.B] + P.B;
  for (;;) {
    if (tid == 0) s.item = (int)atomicAdd(&P.ws->next_item, 1u);
    __syncthreads();
    const int t = s.item;
    __syncthreads();
    if (t >= R_t) break;
    process_row<DT, VEC>(P, s, t);
  }
  if (tid == 0) {
    const unsigned old = atomicAdd(&P.ws->exited, 1u);
    if (old == gridDim.x - 1) {
      P.ws->next_item = 0u;
      P.ws->exited = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

static size_t ws_size(long long B, long long R_t) {
  return sizeof(WsHeader) + align16((size_t)B * sizeof(unsigned)) + (size_t)R_t * sizeof(RowRec);
}

// Resident CTAs per device for each kernel variant, filled on first use.
constexpr int kMaxDevices = 64;
static std::atomic<int> g_resident[kMaxDevices][2][2];

template <int DT, bool VEC>
static cudaError_t resident_ctas(int dev, int* out) {
  int cached = dev < kMaxDevices ? g_resident[dev][DT][VEC].load(std::memory_order_relaxed) : 0;
  if (cached > 0) {
    *out = cached;
    return cudaSuccess;
  }
  int sms = 0, per_sm = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<DT, VEC>, kThreads, 0);
  if (e != cudaSuccess) return e;
  const int n = sms * (per_sm > 0 ? per_sm : 1);
  if (dev < kMaxDevices) g_resident[dev][DT][VEC].store(n, std::memory_order_relaxed);
  *out = n;
  return cudaSuccess;
}

template <int DT, bool VEC>
static cudaError_t launch(const Params& P, cudaStream_t st) {
  int dev = 0, resident = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = resident_ctas<DT, VEC>(dev, &resident);
  if (e != cudaSuccess) return e;
  long long grid = resident;
  if (grid > P.row_cap) grid = P.row_cap;
  if (grid < 1) grid = 1;
  verify_kernel<DT, VEC><<<(unsigned)grid, kThreads, 0, st>>>(P);
  return cudaGetLastError();
}

static sv_status run_verify(const void* target, const void* draft, sv_dtype dtype, int32_t V,
                            int32_t B, const int32_t* draft_tokens, const int32_t* cu_draft,
                            const uint8_t* mode, const float* uniforms, float temperature,
                            int32_t* out_tokens, int32_t* out_len, float* out_probs,
                            void* workspace, size_t workspace_bytes, void* stream,
                            int greedy_all) {
  if (dtype != SV_FP32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (B < 0 || V < 1 || V > max_vocab(dtype)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target || !cu_draft || !out_tokens || !out_len || !workspace) return SV_ERR_INVALID_ARG;
  if (!greedy_all) {
    if (!uniforms) return SV_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  }
  const size_t es = dtype == SV_FP32 ? 4 : 2;
  if ((uintptr_t)target % es || (draft && (uintptr_t)draft % es)) return SV_ERR_INVALID_ARG;
  if ((uintptr_t)workspace % 16 || (uintptr_t)cu_draft % 4 || (uintptr_t)out_tokens % 4 ||
      (uintptr_t)out_len % 4 || (out_probs && (uintptr_t)out_probs % 4) ||
      (uniforms && (uintptr_t)uniforms % 4) || (draft_tokens && (uintptr_t)draft_tokens % 4))
    return SV_ERR_INVALID_ARG;
  const size_t fixed = sizeof(WsHeader) + align16((size_t)B * sizeof(unsigned));
  if (workspace_bytes < fixed + sizeof(RowRec)) return SV_ERR_INVALID_ARG;

  Params P;
  P.target = target;
  P.draft = greedy_all ? nullptr : draft;
  P.V = V;
  P.B = B;
  P.draft_tokens = draft_tokens;
  P.cu = cu_draft;
  P.mode = greedy_all ? nullptr : mode;
  P.uniforms = uniforms;
  P.c = greedy_all ? 1.f : (float)(1.4426950408889634 / (double)temperature);
  P.out_tokens = out_tokens;
  P.out_len = out_len;
  P.out_probs = greedy_all ? nullptr : out_probs;
  P.ws = static_cast<WsHeader*>(workspace);
  P.req_done = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + sizeof(WsHeader));
  P.rows = reinterpret_cast<RowRec*>(static_cast<char*>(workspace) + fixed);
  P.row_cap = (long long)((workspace_bytes - fixed) / sizeof(RowRec));
  P.greedy_all = greedy_all;

  const bool vec = ((uintptr_t)target % 16 == 0) && (!P.draft || (uintptr_t)P.draft % 16 == 0) &&
                   (((size_t)V * es) % 16 == 0);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == SV_BF16)
    e = vec ? launch<1, true>(P, st) : launch<1, false>(P, st);
  else
    e = vec ? launch<0, true>(P, st) : launch<0, false>(P, st);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv

extern "C" {

size_t spec_verify_workspace_size(int32_t B, int32_t R_t) {
  if (B < 0 || R_t < 0) return 0;
  return sv::ws_size(B, R_t > 0 ? R_t : 1);
}

sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      int32_t V, int32_t B, const int32_t* draft_tokens,
                      const int32_t* cu_draft, const uint8_t* mode, const float* uniforms,
                      float temperature, int32_t* out_tokens, int32_t* out_len,
                      float* out_probs, void* workspace, size_t workspace_bytes,
                      void* cuda_stream) {
  return sv::run_verify(target_logits, draft_logits, dtype, V, B, draft_tokens, cu_draft, mode,
                        uniforms, temperature, out_tokens, out_len, out_probs, workspace,
                        workspace_bytes, cuda_stream, 0);
}

sv_status spec_verify_greedy(const void* target_logits, sv_dtype dtype, int32_t V, int32_t B,
                             const int32_t* draft_tokens, const int32_t* cu_draft,
                             int32_t* out_tokens, int32_t* out_len, void* workspace,
                             size_t workspace_bytes, void* cuda_stream) {
  return sv::run_verify(target_logits, nullptr, dtype, V, B, draft_tokens, cu_draft, nullptr,
                        nullptr, 1.f, out_tokens, out_len, nullptr, workspace, workspace_bytes,
                        cuda_stream, 1);
}

sv_status sv_check_status(void* workspace, void* cuda_stream, uint32_t* out_bits) {
  if (!workspace || !out_bits) return SV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  uint32_t bits = 0;
  if (cudaMemcpyAsync(&bits, workspace, sizeof bits, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof bits, st) != cudaSuccess) return SV_ERR_CUDA;
  *out_bits = bits;
  return (bits & ~SV_DATA_DEGENERATE_RESIDUAL) ? SV_ERR_DATA : SV_OK;
}

const char* sv_status_string(sv_status status) {
  switch (status) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG";
    case SV_ERR_CUDA: return "SV_ERR_CUDA";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT";
    case SV_ERR_UNIMPLEMENTED: return "SV_ERR_UNIMPLEMENTED";
    case SV_ERR_DATA: return "SV_ERR_DATA";
  }
  return "SV_ERR_UNKNOWN";
}

}  // extern "C"
