// vshard.cu -- verify-and-commit with the vocabulary split over shards.
//
// A tensor-parallel target (and draft) hands each rank the logits of a
// contiguous slice [v0, v0 + Vs) of the vocabulary for every row. The step
// of "Draft Model（草稿模型）" §2 (accept x̂_i with probability
// min(1, p(x̂_i)/q(x̂_i)); at the first rejection draw from
// norm(max(0, p - q)); if all are accepted draw from p_{K+1}) then needs
// two exchanges between the shards, both done by the caller between these
// kernels:
//   1. every shard's per-row statistics of its slice (sv_vshard_stats): the
//      exponent offset mc and sum S of its softmax terms, the proposed
//      token's logit if the shard holds it, and the slice's argmax. Gathered
//      from all shards, they give every rank the whole-vocabulary p(x̂) and
//      q(x̂), so every rank takes the same decisions (sv_vshard_decide);
//   2. every shard's mass of the residual r = max(0, p - q) (or of p, for a
//      bonus draw) over its slice (sv_vshard_masses). Gathered in shard
//      order they are an exclusive scan of the mass over the vocabulary:
//      the shard whose range of the scan holds u' * Z draws the token inside
//      its slice (sv_vshard_draw), and a max over the shards' answers (-1
//      from the others) gives it to every rank (sv_vshard_finish writes it).
// Shards must cover [0, V) in rank order without overlap.
//
// Arithmetic follows the one-launch kernel: per thread fp32 partial sums of
// 2^(z c - mc) with c = log2(e) / T, combined in fp64; the accept test in
// fp32; the draw as an inverse CDF in vocabulary order over fp64 tile sums,
// then a rescan of the chosen tile.
#include "../../include/spec_verify.h"
#include "sv_device.cuh"

#include <climits>
#include <cmath>
#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

namespace sv {
namespace vs {

constexpr int kT = kThreads;           // threads per CTA
constexpr int kW = kT / 32;            // warps per CTA
constexpr int kMaxTiles = kT;          // one tile per thread in the draw's scan
constexpr int kStatGrid = 4 * 152;     // CTAs of the row-statistics kernel, at most
// Tiles whose 16-byte loads (per row of the pair) a thread keeps in flight
// in the residual-mass and draw passes: one CTA per request streams its two
// stop-row slices, so the depth sets the pass's bandwidth (4 tiles: 0.378 ms
// per sharded call on config 3 over two shards, 8: 0.368 ms).
#ifndef SV_VS_LOADS
#define SV_VS_LOADS 8
#endif

static_assert(sizeof(sv_shard_stat) == 32, "shard statistics are 32 bytes");

// One request's draw, as every rank decided it (64 bytes).
struct Job {
  int row;        // stop row (target row index), or -1: nothing to draw
  int drow;       // paired draft row (residual draws), or -1
  int kind;       // 0 residual, 1 one-hot, 2 from p (bonus)
  int xhat;       // the rejected one-hot proposal, or -1
  float mcp, mcq; // whole-vocabulary exponent offsets of the stop rows
  double Sp, Sq;  // whole-vocabulary sums of the stop rows
  int bonus_row;  // row that receives (p(y), q(y)) of the drawn token
  int pad[5];
};
static_assert(sizeof(Job) == 64, "draw job is 64 bytes");
enum { kResidual = 0, kOneHot = 1, kBonus = 2 };

// The slice of one row: base pointer, its length and first global index.
struct Slice {
  const char* p;   // target row
  const char* q;   // draft row (residual draws), or null
  int Vs, v0;
};

template <int DT, bool VEC>
__device__ __forceinline__ void load_elems(const char* row, int x, int Vs, float (&f)[Elem<DT>::kEPV]) {
  load_chunk<DT, VEC>(row, x, Vs, f);
}

// Largest b in [0, B) with cu[b] + b <= t (the request owning target row t),
// by every thread of the CTA at once: each round tests kT evenly spaced
// candidates and one barrier counts the passing prefix (one round up to
// B = kT).
__device__ __forceinline__ int find_request_cta(const int32_t* cu, int B, int t) {
  int lo = 0, n = B;
  while (n > 1) {
    const int step = (n + kT - 1) / kT;
    const int c = lo + (int)threadIdx.x * step;
    const bool pass = c < lo + n && cu[c] + c <= t;
    const int cnt = __syncthreads_count(pass);
    const int end = lo + n;
    lo += (cnt - 1) * step;
    n = min(step, end - lo);
  }
  return lo;
}

// Offsets of a packed ragged layout are valid for R_t target rows. Every
// thread of the CTA calls it: each checks a strided share of the pairs and
// one barrier combines them.
__device__ __forceinline__ bool offsets_ok(const int32_t* cu, int B, long long R_t) {
  bool bad = false;
  for (int b = threadIdx.x; b < B; b += kT)
    if (cu[b + 1] < cu[b]) bad = true;
  if (threadIdx.x == 0 && (cu[0] != 0 || (long long)cu[B] + B != R_t)) bad = true;
  return !__syncthreads_or(bad);
}

// ---------------------------------------------------------------------------
// 1. Row statistics of one shard
// ---------------------------------------------------------------------------
struct StatParams {
  const char* logits;
  long long ld_bytes;  // row stride
  int rows, Vs, v0, V, B, is_draft;
  const int32_t* cu;
  const int32_t* tokens;
  float c;
  sv_shard_stat* out;
  uint32_t* status;
};

template <int DT, bool VEC>
__global__ void __launch_bounds__(kT) stats_kernel(StatParams P) {
  constexpr int EPV = Elem<DT>::kEPV;
  __shared__ float s_m[kW], s_zx;
  __shared__ DF s_S[kW];
  __shared__ float s_av[kW];
  __shared__ int s_ai[kW], s_hx;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Token lookups go through the offsets: they must be a valid layout of
  // these rows (R_t target rows, or R_d = R_t - B draft rows).
  if (!offsets_ok(P.cu, P.B, P.is_draft ? (long long)P.rows + P.B : (long long)P.rows)) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(P.status, SV_DATA_BAD_OFFSETS);
    return;
  }
  for (int r = blockIdx.x; r < P.rows; r += gridDim.x) {
    // The row's proposed token: draft rows carry their own; target row
    // (b, i) carries draft slot i's when i < K_b (none for the bonus row).
    // The whole CTA finds the request of a target row.
    const int rb = P.is_draft ? 0 : find_request_cta(P.cu, P.B, r);
    if (tid == 0) {
      int x = -1;
      if (P.is_draft) {
        x = P.tokens[r];
      } else {
        const int i = r - (P.cu[rb] + rb), K = P.cu[rb + 1] - P.cu[rb];
        x = (i < K && P.tokens) ? P.tokens[P.cu[rb] + i] : -1;
      }
      // The proposed token's logit, if this shard holds it: one load.
      const char* row = P.logits + (long long)r * P.ld_bytes;
      const bool here = x >= P.v0 && x < P.v0 + P.Vs;
      s_zx = here ? Elem<DT>::scalar(row, x - P.v0) : NAN;
      s_hx = here ? 1 : 0;
    }
    const char* row = P.logits + (long long)r * P.ld_bytes;
    float m = -INFINITY, mc = 0.f, sum = 0.f, av = -INFINITY;
    int ai = INT_MAX;
    auto fold = [&](const float (&f)[EPV], int e) {
      float vm = f[0];
#pragma unroll
      for (int j = 1; j < EPV; ++j) vm = fmaxf(vm, f[j]);
      if (vm > m) {
        const float nmc = __fmul_rn(vm, P.c);
        sum = (m == -INFINITY) ? 0.f : sum * ex2(mc - nmc);
        m = vm;
        mc = nmc;
      }
#pragma unroll
      for (int j = 0; j < EPV; ++j) sum += ex2(fmaf(f[j], P.c, -mc));
      if (vm > av) {  // elements visited in increasing index order: the first of equal values stays
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if (f[j] > av) {
            av = f[j];
            ai = P.v0 + e + j;
          }
      }
    };
    if constexpr (VEC) {
      // kU 16-byte loads in flight per thread before any is used.
      constexpr int kU = 8;
      for (int e0 = tid * EPV; e0 < P.Vs; e0 += kT * EPV * kU) {
        uint4 raw[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int e = e0 + u * kT * EPV;
          raw[u] = e < P.Vs ? ld_stream16(row + (size_t)e * Elem<DT>::kBytes)
                            : (DT == 1 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                                       : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u));
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int e = e0 + u * kT * EPV;
          if (e < P.Vs) {
            float f[EPV];
            Elem<DT>::unpack(raw[u], f);
            fold(f, e);
          }
        }
      }
    } else {
      for (int e = tid * EPV; e < P.Vs; e += kT * EPV) {
        float f[EPV];
        load_elems<DT, VEC>(row, e, P.Vs, f);
        fold(f, e);
      }
    }
    // CTA combine: maximum, then every thread's sum rescaled to its offset.
    const float wm = warp_max(m);
    warp_argmax(av, ai);
    if (lane == 0) {
      s_m[warp] = wm;
      s_av[warp] = av;
      s_ai[warp] = ai;
    }
    __syncthreads();
    float M = s_m[0];
#pragma unroll
    for (int w = 1; w < kW; ++w) M = fmaxf(M, s_m[w]);
    const float Mc = (M == -INFINITY) ? 0.f : __fmul_rn(M, P.c);
    // Sums in double-float: a dependent fp64 operation costs about 14 fp32
    // ones on this part.
    DF t = (m == -INFINITY) ? DF{0.f, 0.f} : df_mul_f(DF{sum, 0.f}, ex2(mc - Mc));
    t = warp_sum_df(t);
    if (lane == 0) s_S[warp] = t;
    __syncthreads();
    if (tid == 0) {
      DF Sd = s_S[0];
      float bv = s_av[0];
      int bi = s_ai[0];
      for (int w = 1; w < kW; ++w) {
        Sd = df_add(Sd, s_S[w]);
        argmax_merge(bv, bi, s_av[w], s_ai[w]);
      }
      const double S = df_to_d(Sd);
      sv_shard_stat st;
      st.mc = Mc;
      st.zx = s_zx;
      st.S = S;
      st.amax_v = bv;
      st.amax_i = bi;
      st.has_x = s_hx;
      st.pad = 0;
      P.out[r] = st;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// 2. Decisions from all shards' statistics (one warp per request)
// ---------------------------------------------------------------------------
struct DecideParams {
  const sv_shard_stat* ts;  // [S, R_t]
  const sv_shard_stat* ds;  // [S, R_d] or null (one-hot proposals)
  int S, V, B;
  long long R_t;
  const int32_t* cu;
  const int32_t* tokens;
  const uint8_t* mode;
  const float* uniforms;
  float c;
  int32_t* out_tokens;
  int32_t* out_len;
  float* out_probs;
  Job* jobs;
  uint32_t* status;
};

// Whole-vocabulary statistics of one row from its S shard records: the
// largest offset of the shards with mass, their sums rescaled to it, the
// proposed token's logit from the shard that holds it (-inf if none does),
// and the argmax (largest logit, lowest index among ties).
struct RowComb {
  float Mc;
  double S;
  float zx;
  float av;
  int ai;
};

__device__ RowComb combine_row(const sv_shard_stat* st, long long stride, long long row, int S) {
  RowComb r;
  r.Mc = -INFINITY;
  r.zx = -INFINITY;
  r.av = -INFINITY;
  r.ai = INT_MAX;
  for (int s = 0; s < S; ++s) {
    const sv_shard_stat& a = st[s * stride + row];
    if (a.S > 0.0) r.Mc = fmaxf(r.Mc, a.mc);
    if (a.has_x) r.zx = a.zx;
    argmax_merge(r.av, r.ai, a.amax_v, a.amax_i);
  }
  r.S = 0.0;
  for (int s = 0; s < S; ++s) {
    const sv_shard_stat& a = st[s * stride + row];
    if (a.S > 0.0) r.S += a.S * (double)ex2(a.mc - r.Mc);
  }
  if (r.Mc == -INFINITY) r.Mc = 0.f;
  return r;
}

__global__ void __launch_bounds__(kT) decide_kernel(DecideParams P) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kW + (threadIdx.x >> 5), nw = gridDim.x * kW;
  if (!offsets_ok(P.cu, P.B, P.R_t)) {
    // No decision, and no draw for the later kernels to make.
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(P.status, SV_DATA_BAD_OFFSETS);
    for (int b = blockIdx.x * kT + threadIdx.x; b < P.B; b += gridDim.x * kT) P.jobs[b].row = -1;
    return;
  }
  const long long R_d = P.cu[P.B];
  // One warp per request: lane i decides draft slot j0 + i; the first
  // rejection comes from a ballot.
  for (int b = gw; b < P.B; b += nw) {
    const int d0 = P.cu[b], K = P.cu[b + 1] - d0, t0 = d0 + b;
    int greedy = 0;
    if (P.mode) {
      const uint8_t m = P.mode[b];
      if (m == SV_MODE_GREEDY) greedy = 1;
      else if (m != SV_MODE_SAMPLE && lane == 0) atomicOr(P.status, SV_DATA_BAD_MODE);
    }
    int stop = K;
    for (int j0 = 0; j0 < K; j0 += 32) {
      const int i = j0 + lane;
      bool rej = false;
      if (i < K) {
        const int x = P.tokens[d0 + i];
        const bool bad = x < 0 || x >= P.V;
        if (bad) atomicOr(P.status, SV_DATA_BAD_TOKEN);
        bool acc;
        if (greedy) {
          const RowComb tr = combine_row(P.ts, P.R_t, t0 + i, P.S);
          const int am = tr.ai == INT_MAX ? 0 : tr.ai;
          acc = !bad && x == am;
        } else {
          // p(x̂) = 2^(z c - Mc_p) / S_p; rho = min(1, p/q), q from the draft
          // row or 1 for a one-hot proposal; q(x̂) = 0 rejects.
          const RowComb tr = combine_row(P.ts, P.R_t, t0 + i, P.S);
          if (!(tr.S > 0.0)) atomicOr(P.status, SV_DATA_EMPTY_ROW);
          float ph = -1.f, qh = -1.f;
          acc = false;
          if (!bad) {
            const float ap = fmaf(tr.zx, P.c, -tr.Mc);
            const float pd = __fdiv_rn(exp2f(ap), (float)tr.S);
            float rho, qd = 1.f;
            if (P.ds) {
              const RowComb dr = combine_row(P.ds, R_d, d0 + i, P.S);
              if (!(dr.S > 0.0)) atomicOr(P.status, SV_DATA_EMPTY_ROW);
              const float aq = fmaf(dr.zx, P.c, -dr.Mc);
              qd = __fdiv_rn(exp2f(aq), (float)dr.S);
              rho = (dr.zx == -INFINITY) ? 0.f
                                         : fminf(1.f, __fmul_rn(exp2f(ap - aq), __fdiv_rn((float)dr.S, (float)tr.S)));
            } else {
              rho = fminf(1.f, pd);
            }
            acc = P.uniforms[2 * (size_t)(t0 + i)] < rho;
            ph = pd;
            qh = qd;
          }
          if (P.out_probs) {
            P.out_probs[2 * (size_t)(t0 + i)] = ph;
            P.out_probs[2 * (size_t)(t0 + i) + 1] = qh;
          }
        }
        rej = !acc;
      }
      const unsigned m = __ballot_sync(kFull, rej);
      if (m) {
        stop = j0 + __ffs(m) - 1;
        if (greedy) break;  // greedy rows carry no probabilities to fill in
        // sampled slots after the stop still write their probabilities
        for (j0 += 32; j0 < K; j0 += 32) {
          const int i2 = j0 + lane;
          if (i2 >= K) continue;
          const int x = P.tokens[d0 + i2];
          const bool bad = x < 0 || x >= P.V;
          if (bad) atomicOr(P.status, SV_DATA_BAD_TOKEN);
          const RowComb tr = combine_row(P.ts, P.R_t, t0 + i2, P.S);
          if (!(tr.S > 0.0)) atomicOr(P.status, SV_DATA_EMPTY_ROW);
          float ph = -1.f, qh = -1.f;
          if (!bad) {
            const float ap = fmaf(tr.zx, P.c, -tr.Mc);
            ph = __fdiv_rn(exp2f(ap), (float)tr.S);
            qh = 1.f;
            if (P.ds) {
              const RowComb dr = combine_row(P.ds, R_d, d0 + i2, P.S);
              if (!(dr.S > 0.0)) atomicOr(P.status, SV_DATA_EMPTY_ROW);
              qh = __fdiv_rn(exp2f(fmaf(dr.zx, P.c, -dr.Mc)), (float)dr.S);
            }
          }
          if (P.out_probs) {
            P.out_probs[2 * (size_t)(t0 + i2)] = ph;
            P.out_probs[2 * (size_t)(t0 + i2) + 1] = qh;
          }
        }
        break;
      }
    }
    for (int j = lane; j < stop; j += 32) P.out_tokens[t0 + j] = P.tokens[d0 + j];
    if (greedy && P.out_probs)
      for (int j = lane; j <= K; j += 32) {  // greedy rows, the bonus row included
        P.out_probs[2 * (size_t)(t0 + j)] = -1.f;
        P.out_probs[2 * (size_t)(t0 + j) + 1] = -1.f;
      }
    if (lane != 0) continue;
    P.out_len[b] = stop + 1;
    Job job;
    job.row = -1;
    job.drow = -1;
    job.kind = kBonus;
    job.xhat = -1;
    job.mcp = job.mcq = 0.f;
    job.Sp = job.Sq = 0.0;
    job.bonus_row = t0 + K;
    for (int k = 0; k < 5; ++k) job.pad[k] = 0;
    if (greedy) {
      const RowComb tr = combine_row(P.ts, P.R_t, t0 + stop, P.S);
      P.out_tokens[t0 + stop] = tr.ai == INT_MAX ? 0 : tr.ai;
    } else {
      const RowComb tr = combine_row(P.ts, P.R_t, t0 + stop, P.S);
      job.row = t0 + stop;
      job.mcp = tr.Mc;
      job.Sp = tr.S;
      if (stop < K) {
        const int x = P.tokens[d0 + stop];
        job.xhat = (x >= 0 && x < P.V) ? x : -1;
        if (P.ds) {
          const RowComb dr = combine_row(P.ds, R_d, d0 + stop, P.S);
          job.kind = kResidual;
          job.drow = d0 + stop;
          job.mcq = dr.Mc;
          job.Sq = dr.S;
        } else {
          job.kind = kOneHot;
        }
      }
    }
    P.jobs[b] = job;
  }
}

// ---------------------------------------------------------------------------
// 3 and 4. Residual masses of one shard and the draw inside the owning shard
// ---------------------------------------------------------------------------
// r for EPV elements starting at slice element e (global index v0 + e).
template <int EPV>
__device__ __forceinline__ void residual(const Job& J, int kind, float c, float bhi, float blo,
                                         const float (&zp)[EPV], const float (&zq)[EPV], int gx,
                                         float (&r)[EPV]) {
#pragma unroll
  for (int j = 0; j < EPV; ++j) {
    const float ep = ex2(fmaf(zp[j], c, -J.mcp));
    if (kind == kResidual) {
      const float eq = ex2(fmaf(zq[j], c, -J.mcq));
      float d = fmaf(-eq, bhi, ep);
      d = fmaf(-eq, blo, d);
      r[j] = fmaxf(d, 0.f);
    } else {
      r[j] = (kind == kOneHot && gx + j == J.xhat) ? 0.f : ep;
    }
  }
}

// Sums of r over each tile of kT * EPV elements of the slice, in
// double-float, into tt[0, ntiles) (shared); per thread fp32 over its EPV
// elements, per warp fp32, over the warps double-float in warp order. The
// 16-byte path keeps kU tiles' loads in flight before using any.
template <int DT, bool VEC>
__device__ void tile_totals(const Slice& sl, const Job& J, int kind, float c, float bhi, float blo,
                            float* wt, DF* tt, int ntiles) {
  constexpr int EPV = Elem<DT>::kEPV;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto one = [&](int l, const float (&zp)[EPV], const float (&zq)[EPV], int e) {
    float r[EPV];
    residual<EPV>(J, kind, c, bhi, blo, zp, zq, sl.v0 + e, r);
    float ts = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) ts += r[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ts += __shfl_xor_sync(kFull, ts, o);
    if (lane == 0) wt[l * kW + warp] = ts;
  };
  if constexpr (VEC) {
    constexpr int kU = SV_VS_LOADS;
    const uint4 ninf = DT == 1 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                               : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
    for (int l0 = 0; l0 < ntiles; l0 += kU) {
      uint4 rp[kU], rq[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = (l0 + u) * kT * EPV + tid * EPV;
        const bool in = l0 + u < ntiles && e < sl.Vs;
        rp[u] = in ? ld_stream16(sl.p + (size_t)e * Elem<DT>::kBytes) : ninf;
        rq[u] = (in && kind == kResidual) ? ld_stream16(sl.q + (size_t)e * Elem<DT>::kBytes) : ninf;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (l0 + u >= ntiles) break;
        float zp[EPV], zq[EPV];
        Elem<DT>::unpack(rp[u], zp);
        Elem<DT>::unpack(rq[u], zq);
        one(l0 + u, zp, zq, (l0 + u) * kT * EPV + tid * EPV);
      }
    }
  } else {
    for (int l = 0; l < ntiles; ++l) {
      const int e = l * kT * EPV + tid * EPV;
      float zp[EPV], zq[EPV];
      load_elems<DT, VEC>(sl.p, e, sl.Vs, zp);
      if (kind == kResidual) load_elems<DT, VEC>(sl.q, e, sl.Vs, zq);
      one(l, zp, zq, e);
    }
  }
  __syncthreads();
  for (int l = tid; l < ntiles; l += kT) {
    DF t{0.f, 0.f};
    for (int w = 0; w < kW; ++w) t = df_add_f(t, wt[l * kW + w]);
    tt[l] = t;
  }
  __syncthreads();
}

struct MassParams {
  const char* target;
  const char* draft;
  long long ld_bytes;
  int Vs, v0, B;
  long long R_t;
  const int32_t* cu;
  const sv_shard_stat* ts_local;  // [R_t] this shard's statistics
  const Job* jobs;
  float c;
  double* mass;  // [B]
};

__device__ __forceinline__ void beta_of(const Job& J, float& bhi, float& blo) {
  const double beta = J.kind == kResidual ? J.Sp / J.Sq : 1.0;
  bhi = (float)beta;
  blo = (float)(beta - (double)bhi);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kT) mass_kernel(MassParams P) {
  constexpr int EPV = Elem<DT>::kEPV;
  __shared__ float wt[kMaxTiles * kW];
  __shared__ DF tt[kMaxTiles];
  if (!offsets_ok(P.cu, P.B, P.R_t)) return;
  const int ntiles = (P.Vs + kT * EPV - 1) / (kT * EPV);
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    const Job J = P.jobs[b];
    if (J.row < 0) {
      if (threadIdx.x == 0) P.mass[b] = 0.0;
      continue;
    }
    if (J.kind == kBonus) {
      // Mass of p over the slice, in units of 2^(z c - Mc_p): its own sum.
      if (threadIdx.x == 0) {
        const sv_shard_stat& a = P.ts_local[J.row];
        P.mass[b] = a.S > 0.0 ? a.S * (double)ex2(a.mc - J.mcp) : 0.0;
      }
      continue;
    }
    Slice sl;
    sl.p = P.target + (long long)J.row * P.ld_bytes;
    sl.q = J.kind == kResidual ? P.draft + (long long)J.drow * P.ld_bytes : nullptr;
    sl.Vs = P.Vs;
    sl.v0 = P.v0;
    float bhi, blo;
    beta_of(J, bhi, blo);
    tile_totals<DT, VEC>(sl, J, J.kind, P.c, bhi, blo, wt, tt, ntiles);
    if (threadIdx.x < 32) {  // the slice's mass: warp 0 sums the tiles in double-float
      DF z{0.f, 0.f};
      for (int l = threadIdx.x; l < ntiles; l += 32) z = df_add(z, tt[l]);
      z = warp_sum_df(z);
      if (threadIdx.x == 0) P.mass[b] = df_to_d(z);
    }
    __syncthreads();
  }
}

struct DrawParams {
  const char* target;
  const char* draft;
  long long ld_bytes;
  int Vs, v0, shard, S, B;
  long long R_t;
  const int32_t* cu;
  const double* masses;        // [S, B]
  const sv_shard_stat* ts;     // [S, R_t] all shards' target statistics
  const Job* jobs;
  const float* uniforms;
  float c;
  int32_t* draw_tok;           // [B]
  float* draw_prob;            // [B, 2]
  uint32_t* status;
};

template <int DT, bool VEC>
__global__ void __launch_bounds__(kT) draw_kernel(DrawParams P) {
  constexpr int EPV = Elem<DT>::kEPV;
  constexpr int TILE = kT * EPV;
  __shared__ float wt[kMaxTiles * kW];
  __shared__ DF tt[kMaxTiles], tincl[kMaxTiles], dred[kW], dred2[kW], wexcl[kW + 1];
  __shared__ float redf[kW];
  __shared__ int s_owner, s_kind, pick, pick2, tok;
  __shared__ DF s_T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!offsets_ok(P.cu, P.B, P.R_t)) return;
  const int ntiles = (P.Vs + TILE - 1) / TILE;
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    const Job J = P.jobs[b];
    if (J.row < 0) continue;
    if (tid == 0) {
      // The scan of the shards' masses in vocabulary order; the owner is the
      // first shard with mass whose range reaches past u' * Z, else (u' * Z
      // at or past the total through rounding) the last shard with mass.
      int kind = J.kind;
      double Z = 0.0;
      for (int s = 0; s < P.S; ++s) Z += P.masses[(size_t)s * P.B + b];
      auto mass_of = [&](int s) -> double {
        if (kind == J.kind) return P.masses[(size_t)s * P.B + b];
        const sv_shard_stat& a = P.ts[(size_t)s * P.R_t + J.row];  // p's own mass
        return a.S > 0.0 ? a.S * (double)ex2(a.mc - J.mcp) : 0.0;
      };
      if (!(Z > 0.0) && kind != kBonus) {
        // No residual mass (p == q in fp32): draw from p instead.
        atomicOr(P.status, SV_DATA_DEGENERATE_RESIDUAL);
        kind = kBonus;
        Z = 0.0;
        for (int s = 0; s < P.S; ++s) Z += mass_of(s);
      }
      double T = (double)P.uniforms[2 * (size_t)J.row + 1] * Z;
      if (!(T >= 0.0)) T = 0.0;
      int owner = -1, last = -1;
      double pre = 0.0, pre_last = 0.0, Tl = 0.0;
      for (int s = 0; s < P.S; ++s) {
        const double m = mass_of(s);
        if (m > 0.0) {
          if (owner < 0 && pre + m > T) {
            owner = s;
            Tl = T - pre;
          }
          last = s;
          pre_last = pre;
        }
        pre += m;
      }
      if (owner < 0 && last >= 0) {
        owner = last;
        Tl = T - pre_last;
      }
      s_owner = owner;
      s_kind = kind;
      s_T = df_from_d(Tl);
      if (owner != P.shard) {
        P.draw_tok[b] = -1;
        P.draw_prob[2 * (size_t)b] = -1.f;
        P.draw_prob[2 * (size_t)b + 1] = -1.f;
      }
      if (owner < 0) atomicOr(P.status, SV_DATA_EMPTY_ROW);
    }
    __syncthreads();
    if (s_owner != P.shard) {
      __syncthreads();
      continue;
    }
    const int kind = s_kind;
    const DF T = s_T;
    Slice sl;
    sl.p = P.target + (long long)J.row * P.ld_bytes;
    sl.q = J.kind == kResidual ? P.draft + (long long)J.drow * P.ld_bytes : nullptr;
    sl.Vs = P.Vs;
    sl.v0 = P.v0;
    Job Jk = J;
    Jk.kind = kind;
    float bhi, blo;
    beta_of(Jk, bhi, blo);
    tile_totals<DT, VEC>(sl, Jk, kind, P.c, bhi, blo, wt, tt, ntiles);
    // The tile holding T: the last tile with mass whose lower edge is <= T
    // (scans in double-float).
    const DF mine = tid < ntiles ? tt[tid] : DF{0.f, 0.f};
    const DF inc = warp_incl_scan_df(mine, lane);
    if (lane == 31) dred[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      DF v = lane < kW ? dred[lane] : DF{0.f, 0.f};
      v = warp_incl_scan_df(v, lane);
      if (lane < kW) dred2[lane] = v;
    }
    __syncthreads();
    if (tid < ntiles) tincl[tid] = warp > 0 ? df_add(dred2[warp - 1], inc) : inc;
    if (tid == 0) pick = -1;
    __syncthreads();
    if (tid < ntiles) {
      const DF lo = tid ? tincl[tid - 1] : DF{0.f, 0.f};
      if (df_pos(mine) && df_le(lo, T)) atomicMax(&pick, tid);
    }
    __syncthreads();
    const int kt = pick;
    int y = -1;
    if (kt >= 0) {
      const DF Tk = kt ? df_sub(T, tincl[kt - 1]) : T;
      const int e = kt * TILE + tid * EPV;
      float zp[EPV], zq[EPV], r[EPV];
      load_elems<DT, VEC>(sl.p, e, sl.Vs, zp);
      if (kind == kResidual) load_elems<DT, VEC>(sl.q, e, sl.Vs, zq);
      residual<EPV>(Jk, kind, P.c, bhi, blo, zp, zq, sl.v0 + e, r);
      float ts = 0.f;
#pragma unroll
      for (int j = 0; j < EPV; ++j) ts += r[j];
      const float incl = warp_incl_scan(ts, lane);
      float lane_lo = __shfl_up_sync(kFull, incl, 1);
      if (lane == 0) lane_lo = 0.f;
      if (lane == 31) redf[warp] = incl;
      __syncthreads();
      if (tid == 0) {
        DF a{0.f, 0.f};
        wexcl[0] = a;
        for (int w = 0; w < kW; ++w) {
          a = df_add_f(a, redf[w]);
          wexcl[w + 1] = a;
        }
        pick2 = -1;
        tok = -1;
      }
      __syncthreads();
      const DF lo = df_add_f(wexcl[warp], lane_lo);
      if (ts > 0.f && df_le(lo, Tk)) atomicMax(&pick2, tid);
      __syncthreads();
      if (tid == pick2) {
        DF run = lo;
        int cand = e;
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          if (r[j] > 0.f && df_le(run, Tk)) cand = e + j;
          run = df_add_f(run, r[j]);
        }
        tok = cand;
      }
      __syncthreads();
      y = tok;
    }
    if (tid == 0) {
      if (y < 0) {
        atomicOr(P.status, SV_DATA_EMPTY_ROW);
        y = 0;
      }
      // (p(y), q(y)) of the drawn token; y is in this shard's slice.
      float zpy[1] = {0.f}, zqy[1] = {0.f};
      zpy[0] = Elem<DT>::scalar(sl.p, y);
      const float py = __fdiv_rn(exp2f(fmaf(zpy[0], P.c, -J.mcp)), (float)J.Sp);
      // q of the stop slot (also when a residual without mass fell back to p).
      float qy = 0.f;
      if (J.kind == kResidual) {
        zqy[0] = Elem<DT>::scalar(sl.q, y);
        qy = __fdiv_rn(exp2f(fmaf(zqy[0], P.c, -J.mcq)), (float)J.Sq);
      } else if (J.kind == kOneHot) {
        qy = (P.v0 + y == J.xhat) ? 1.f : 0.f;
      }
      P.draw_tok[b] = P.v0 + y;
      P.draw_prob[2 * (size_t)b] = py;
      P.draw_prob[2 * (size_t)b + 1] = qy;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// 5. The drawn tokens into the outputs
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kT) finish_kernel(const Job* jobs, int B, int R_t, const int32_t* draw_tok,
                                                     const float* draw_prob, int32_t* out_tokens,
                                                     float* out_probs, uint32_t* status) {
  for (int b = blockIdx.x * kT + threadIdx.x; b < B; b += gridDim.x * kT) {
    const Job J = jobs[b];
    if (J.row < 0) continue;
    if (J.row >= R_t || J.bonus_row < 0 || J.bonus_row >= R_t) {  // never from sv_vshard_decide
      atomicOr(status, SV_DATA_BAD_OFFSETS);
      continue;
    }
    int y = draw_tok[b];
    if (y < 0) {
      atomicOr(status, SV_DATA_EMPTY_ROW);
      y = 0;
    }
    out_tokens[J.row] = y;
    if (out_probs) {
      out_probs[2 * (size_t)J.bonus_row] = draw_prob[2 * (size_t)b];
      out_probs[2 * (size_t)J.bonus_row + 1] = draw_prob[2 * (size_t)b + 1];
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int max_vocab(sv_dtype dt) { return kMaxTiles * kT * (dt == SV_FP32 ? 4 : 8); }

static bool vec_ok(const void* p, long long ld_bytes) {
  return ((uintptr_t)p % 16 == 0) && (ld_bytes % 16 == 0);
}

static int grid_for(long long n, int cap) { return (int)(n < 1 ? 1 : (n < cap ? n : cap)); }

template <class L>
static cudaError_t dispatch(sv_dtype dt, bool vec, L&& launch) {
  if (dt == SV_BF16) {
    if (vec) launch(std::integral_constant<int, 1>{}, std::true_type{});
    else launch(std::integral_constant<int, 1>{}, std::false_type{});
  } else {
    if (vec) launch(std::integral_constant<int, 0>{}, std::true_type{});
    else launch(std::integral_constant<int, 0>{}, std::false_type{});
  }
  return cudaGetLastError();
}

}  // namespace vs
}  // namespace sv

extern "C" {

size_t sv_vshard_jobs_bytes(int32_t B) { return B < 0 ? 0 : (size_t)B * sizeof(sv::vs::Job); }

sv_status sv_vshard_stats(const void* logits, sv_dtype dtype, int32_t rows, int32_t Vs, int64_t ld,
                          int32_t v0, int32_t V, int32_t is_draft, int32_t B, const int32_t* cu_draft,
                          const int32_t* draft_tokens, float temperature, sv_shard_stat* out,
                          uint32_t* status, void* cuda_stream) {
  using namespace sv::vs;
  if (dtype != SV_FP32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (rows < 0 || B < 0 || Vs < 1 || Vs > max_vocab(dtype) || ld < Vs || v0 < 0 || V < 1 ||
      (long long)v0 + Vs > V)
    return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (!is_draft && rows > 0 && B < 1) return SV_ERR_INVALID_ARG;
  if (rows == 0) return SV_OK;
  const size_t es = dtype == SV_FP32 ? 4 : 2;
  if (!logits || !out || !status || !cu_draft || (is_draft && !draft_tokens) || (uintptr_t)logits % es ||
      (uintptr_t)out % 16 || (uintptr_t)status % 4)
    return SV_ERR_INVALID_ARG;
  StatParams P;
  P.logits = static_cast<const char*>(logits);
  P.ld_bytes = (long long)ld * (long long)es;
  P.rows = rows;
  P.Vs = Vs;
  P.v0 = v0;
  P.V = V;
  P.B = B;
  P.is_draft = is_draft;
  P.cu = cu_draft;
  P.tokens = draft_tokens;
  P.c = (float)(1.4426950408889634 / (double)temperature);
  P.out = out;
  P.status = status;
  const bool vec = vec_ok(logits, P.ld_bytes) && ((size_t)Vs * es) % 16 == 0;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int grid = grid_for(rows, kStatGrid);
  const cudaError_t e = dispatch(dtype, vec, [&](auto dt, auto v) {
    stats_kernel<decltype(dt)::value, decltype(v)::value><<<grid, kT, 0, st>>>(P);
  });
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_vshard_decide(const sv_shard_stat* target_stats, const sv_shard_stat* draft_stats,
                           int32_t S, int32_t V, int32_t B, int32_t R_t, const int32_t* cu_draft,
                           const int32_t* draft_tokens, const uint8_t* mode, const float* uniforms,
                           float temperature, int32_t* out_tokens, int32_t* out_len, float* out_probs,
                           void* jobs, uint32_t* status, void* cuda_stream) {
  using namespace sv::vs;
  if (S < 1 || V < 1 || B < 0 || R_t < B) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (!target_stats || !cu_draft || !uniforms || !out_tokens || !out_len || !jobs || !status ||
      (R_t > B && !draft_tokens) || (uintptr_t)jobs % 16 || (uintptr_t)target_stats % 16 ||
      (draft_stats && (uintptr_t)draft_stats % 16))
    return SV_ERR_INVALID_ARG;
  DecideParams P;
  P.ts = target_stats;
  P.ds = draft_stats;
  P.S = S;
  P.V = V;
  P.B = B;
  P.R_t = R_t;
  P.cu = cu_draft;
  P.tokens = draft_tokens;
  P.mode = mode;
  P.uniforms = uniforms;
  P.c = (float)(1.4426950408889634 / (double)temperature);
  P.out_tokens = out_tokens;
  P.out_len = out_len;
  P.out_probs = out_probs;
  P.jobs = static_cast<Job*>(jobs);
  P.status = status;
  decide_kernel<<<grid_for((B + kW - 1) / kW, kStatGrid), kT, 0, static_cast<cudaStream_t>(cuda_stream)>>>(P);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_vshard_masses(const void* target, const void* draft, sv_dtype dtype, int32_t Vs, int64_t ld,
                           int32_t v0, int32_t B, int32_t R_t, const int32_t* cu_draft,
                           const sv_shard_stat* target_stats, const void* jobs, float temperature,
                           double* masses, void* cuda_stream) {
  using namespace sv::vs;
  if (dtype != SV_FP32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (B < 0 || R_t < B || Vs < 1 || Vs > max_vocab(dtype) || ld < Vs || v0 < 0) return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  const size_t es = dtype == SV_FP32 ? 4 : 2;
  if (!target || !cu_draft || !target_stats || !jobs || !masses || (uintptr_t)target % es ||
      (draft && (uintptr_t)draft % es) || (uintptr_t)masses % 8)
    return SV_ERR_INVALID_ARG;
  MassParams P;
  P.target = static_cast<const char*>(target);
  P.draft = static_cast<const char*>(draft);
  P.ld_bytes = (long long)ld * (long long)es;
  P.Vs = Vs;
  P.v0 = v0;
  P.B = B;
  P.R_t = R_t;
  P.cu = cu_draft;
  P.ts_local = target_stats;
  P.jobs = static_cast<const Job*>(jobs);
  P.c = (float)(1.4426950408889634 / (double)temperature);
  P.mass = masses;
  const bool vec = vec_ok(target, P.ld_bytes) && (!draft || vec_ok(draft, P.ld_bytes)) &&
                   ((size_t)Vs * es) % 16 == 0;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int grid = grid_for(B, kStatGrid);
  const cudaError_t e = dispatch(dtype, vec, [&](auto dt, auto v) {
    mass_kernel<decltype(dt)::value, decltype(v)::value><<<grid, kT, 0, st>>>(P);
  });
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_vshard_draw(const void* target, const void* draft, sv_dtype dtype, int32_t Vs, int64_t ld,
                         int32_t v0, int32_t shard, int32_t S, int32_t B, int32_t R_t,
                         const int32_t* cu_draft, const double* masses, const sv_shard_stat* target_stats,
                         const void* jobs, const float* uniforms, float temperature, int32_t* draw_tok,
                         float* draw_prob, uint32_t* status, void* cuda_stream) {
  using namespace sv::vs;
  if (dtype != SV_FP32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (S < 1 || shard < 0 || shard >= S || B < 0 || R_t < B || Vs < 1 || Vs > max_vocab(dtype) || ld < Vs ||
      v0 < 0)
    return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  const size_t es = dtype == SV_FP32 ? 4 : 2;
  if (!target || !cu_draft || !masses || !target_stats || !jobs || !uniforms || !draw_tok || !draw_prob ||
      !status || (uintptr_t)target % es || (draft && (uintptr_t)draft % es))
    return SV_ERR_INVALID_ARG;
  DrawParams P;
  P.target = static_cast<const char*>(target);
  P.draft = static_cast<const char*>(draft);
  P.ld_bytes = (long long)ld * (long long)es;
  P.Vs = Vs;
  P.v0 = v0;
  P.shard = shard;
  P.S = S;
  P.B = B;
  P.R_t = R_t;
  P.cu = cu_draft;
  P.masses = masses;
  P.ts = target_stats;
  P.jobs = static_cast<const Job*>(jobs);
  P.uniforms = uniforms;
  P.c = (float)(1.4426950408889634 / (double)temperature);
  P.draw_tok = draw_tok;
  P.draw_prob = draw_prob;
  P.status = status;
  const bool vec = vec_ok(target, P.ld_bytes) && (!draft || vec_ok(draft, P.ld_bytes)) &&
                   ((size_t)Vs * es) % 16 == 0;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int grid = grid_for(B, kStatGrid);
  const cudaError_t e = dispatch(dtype, vec, [&](auto dt, auto v) {
    draw_kernel<decltype(dt)::value, decltype(v)::value><<<grid, kT, 0, st>>>(P);
  });
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_vshard_finish(const void* jobs, int32_t B, int32_t R_t, const int32_t* draw_tok,
                           const float* draw_prob, int32_t* out_tokens, float* out_probs, uint32_t* status,
                           void* cuda_stream) {
  using namespace sv::vs;
  if (B < 0 || R_t < B) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!jobs || !draw_tok || !draw_prob || !out_tokens || !status) return SV_ERR_INVALID_ARG;
  finish_kernel<<<grid_for((B + kT - 1) / kT, 152), kT, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      static_cast<const Job*>(jobs), B, R_t, draw_tok, draw_prob, out_tokens, out_probs, status);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
