// cluster.cu -- verify-and-commit for batches of few rows, one thread-block
// cluster per target row.
//
// The step is that of "Draft Model（草稿模型）" §2, one request at a time:
// accept draft token x̂_i with probability min(1, p(x̂_i)/q(x̂_i)); at the
// first rejection emit a token drawn from norm(max(0, p - q)); if all K are
// accepted emit one more from p_{K+1}. Both rows are softmaxes at
// temperature T ("投机解码从零实现" §3.2); strict rows accept iff x̂ is the
// target's argmax ("Speculative Decoding在分布式推理中的应用" §二).
//
// When a batch has few rows, the persistent kernel's time is a chain of
// dependent steps per row (claim, lookup, stream, combine, decide, commit,
// draw in parts). Here every row gets its own cluster of kCluster CTAs and
// nothing is claimed, merged through global memory or re-read:
//   1. each CTA copies its slice of the target row (and of the paired draft
//      row) into shared memory with bulk copies, the target slice before the
//      request is even known;
//   2. the slices' softmax statistics (or argmax) are exchanged through
//      distributed shared memory, so every CTA of the cluster holds the
//      row's p(x̂) and q(x̂) and takes the same accept decision;
//   3. a row that rejects (and every bonus row) draws its token at once,
//      whether or not it turns out to be the request's stop row: the slices'
//      masses of r are exchanged the same way, which gives each slice its
//      range of the inverse CDF, and the slice that holds u' * Z locates the
//      token in its shared memory;
//   4. the row's result goes to global memory, and the last row of a
//      request to finish (one atomic per row) commits it: the first
//      rejected slot, the draft tokens before it and that row's token.
// Synchronisation: one cluster barrier, right after the CTAs' mbarriers are
// initialised and reached by every thread of every CTA of the cluster
// without a condition (a cluster leaves before it only as a whole). Each
// exchange after it is a write into every peer's shared memory followed by
// a remote arrive on the peer's mbarrier for that exchange; every CTA waits
// on its own mbarrier with a bounded wait, so a peer that never arrives is
// reported (SV_DEV_COPY_TIMEOUT) instead of hanging the kernel. Which
// exchanges run depends only on values every CTA of the cluster shares.
#include "../../include/spec_verify.h"
#include "sv_device.cuh"
#include "sv_cluster.cuh"

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace cl {

constexpr size_t kMaxSmem = 200 * 1024;   // dynamic shared memory per CTA, at most
constexpr uint32_t kCopyPiece = 32 * 1024;  // bytes per bulk copy instruction

// ---------------------------------------------------------------------------
// Cluster primitives (inline PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// The shared::cluster address of `p` (in this CTA's shared memory) in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* p, unsigned rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void st_cluster(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster64(uint32_t a, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this
// thread's earlier writes (into that CTA's shared memory) at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Bounded wait, acquiring at cluster scope what the arrivals released.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  for (int it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// ---------------------------------------------------------------------------
// Shared state
// ---------------------------------------------------------------------------
// One slice's statistics, as exchanged between the CTAs of a cluster.
struct alignas(16) SliceRec {
  DF Sp, Sq;       // sums of 2^(z c - mc) over the slice, mc = fp32(m c) (0 if m = -inf)
  float mp, mq;    // slice maxima of the target and draft rows
  float zxp, zxq;  // z(x̂) of both rows if the slice holds x̂
  float av;        // greedy: the slice's largest logit
  int ai;          // and its first index (INT_MAX if none)
  int has_x;       // the slice holds x̂
  int pad;
};
static_assert(sizeof(SliceRec) == 48, "slice record is 48 bytes");

enum { kX1 = 0, kX2 = 1, kX3 = 2, kExchanges = 3 };

struct Smem {
  unsigned long long bar_t, bar_d;  // bulk-copy completion of the two slices
  unsigned long long xbar[kExchanges];  // one arrival per CTA of the cluster per exchange
  // request of this row
  int b, t0, d0, K, i, greedy, xhat, has_d;
  float u_acc, u2;
  // this CTA's slice statistics, then the merged row
  SliceRec mine;
  SliceRec rec[kCluster];           // written by every CTA of the cluster
  DF mass[kCluster];                // slices' masses of r (first pass)
  DF mass2[kCluster];               // second pass (draw from p after an empty residual)
  float mcp, mcq;
  DF Sp, Sq;
  int acc, am, need_draw, kind;
  // reductions
  float redf[kWarps], redf2[kWarps];
  DF reddf_p[kWarps], reddf_q[kWarps];
  int redi[kWarps];
  DF redx[kWarps];
  int pick;
  int copy_timeout;
  int x_timeout;
};

enum { kResidual = 0, kOneHot = 1, kBonus = 2 };

template <int DT>
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[Elem<DT>::kEPV]) {
  Elem<DT>::unpack(v, f);
}

// Largest b with cu[b] + b <= t, by one warp in rounds of 32 probes.
__device__ __forceinline__ int find_request(const int32_t* cu, int B, int t, int lane) {
  int lo = 0, n = B;
  while (n > 1) {
    const int step = (n + 31) >> 5;
    const int c = lo + lane * step;
    const bool pass = c < lo + n && cu[c] + c <= t;
    const unsigned m = __ballot_sync(kFull, pass);
    const int k = 31 - __clz(m);
    const int end = lo + n;
    lo += k * step;
    n = min(step, end - lo);
  }
  return lo;
}

// Issues the bulk copies of `bytes` (a multiple of 16) from src into dst,
// completing on bar (thread 0).
__device__ __forceinline__ void copy_slice(uint32_t dst, const char* src, uint32_t bytes, uint32_t bar) {
  mbar_arrive_expect_tx(bar, bytes);
  for (uint32_t off = 0; off < bytes; off += kCopyPiece) {
    const uint32_t n = bytes - off < kCopyPiece ? bytes - off : kCopyPiece;
    bulk_g2s(dst + off, src + off, n, bar);
  }
}

// r of one element: kResidual max(0, e_p - beta e_q) with beta = S_p / S_q
// as a double-float pair (bhi, blo); kOneHot e_p except at x̂; kBonus e_p.
__device__ __forceinline__ float r_of(int kind, float zp, float zq, int x, int xhat, float c, float mcp,
                                      float mcq, float bhi, float blo) {
  const float ep = ex2(fmaf(zp, c, -mcp));
  if (kind == kResidual) {
    const float eq = ex2(fmaf(zq, c, -mcq));
    float d = fmaf(-eq, bhi, ep);
    d = fmaf(-eq, blo, d);
    return fmaxf(d, 0.f);
  }
  return (kind == kOneHot && x == xhat) ? 0.f : ep;
}

// This thread's contiguous run of slice vectors, [a, e).
__device__ __forceinline__ void thread_run(int nv, int& a, int& e) {
  const int q = (nv + kThreads - 1) / kThreads;
  a = min(nv, (int)threadIdx.x * q);
  e = min(nv, a + q);
}

// Sum of r over this thread's run, in element order (fp32).
template <int DT>
__device__ float run_mass(const unsigned char* tsl, const unsigned char* dsl, int nv, int x0, int kind,
                          int xhat, float c, float mcp, float mcq, float bhi, float blo) {
  constexpr int EPV = Elem<DT>::kEPV;
  int a, e;
  thread_run(nv, a, e);
  float acc = 0.f;
  for (int v = a; v < e; ++v) {
    float zp[EPV], zq[EPV];
    unpack<DT>(lds16(smem_addr(tsl + (size_t)v * 16)), zp);
    if (kind == kResidual) unpack<DT>(lds16(smem_addr(dsl + (size_t)v * 16)), zq);
#pragma unroll
    for (int j = 0; j < EPV; ++j)
      acc += r_of(kind, zp[j], kind == kResidual ? zq[j] : 0.f, x0 + v * EPV + j, xhat, c, mcp, mcq, bhi, blo);
  }
  return acc;
}

// CTA sum of one fp32 value per thread (all threads), in double-float;
// the result in every thread. Sums here stay out of fp64, whose dependent
// operations take about 14 times as long as fp32 ones on this part.
__device__ DF cta_sum_df(Smem& s, float v) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const DF w = warp_sum_df(DF{v, 0.f});
  if (lane == 0) s.redx[warp] = w;
  __syncthreads();
  DF tot = s.redx[0];
#pragma unroll
  for (int k = 1; k < kWarps; ++k) tot = df_add(tot, s.redx[k]);
  __syncthreads();
  return tot;
}

// Ends exchange x: thread k < kCluster arrives on CTA k's mbarrier for it
// (after writing into CTA k), then every thread waits for this CTA's
// mbarrier to collect all kCluster arrivals (bounded).
__device__ __forceinline__ void exchange_done(Smem& s, int x) {
  const int tid = threadIdx.x;
  if (tid < kCluster) mbar_arrive_remote(peer_addr(&s.xbar[x], (unsigned)tid));
  if (!mbar_wait_cluster(smem_addr(&s.xbar[x]), 0)) s.x_timeout = 1;
}

// Writes this CTA's value into slot `rank` of arr in every CTA of the cluster.
__device__ __forceinline__ void broadcast_df(DF* arr, unsigned rank, DF v) {
  const int tid = threadIdx.x;
  if (tid < kCluster)
    st_cluster64(peer_addr(&arr[rank], (unsigned)tid),
                 (uint64_t)__float_as_uint(v.hi) | ((uint64_t)__float_as_uint(v.lo) << 32));
}

// The draw's mass exchange (exchange x): this slice's mass into `arr`
// everywhere. Returns Z and sets the owner slice (the last one with mass
// whose lower edge is <= T = u' Z) and that edge.
__device__ DF exchange_mass(Smem& s, int x, DF* arr, unsigned rank, DF mine, float u2, int& owner,
                            DF& lo_owner, DF& T) {
  broadcast_df(arr, rank, mine);
  exchange_done(s, x);
  DF Z = arr[0];
#pragma unroll
  for (int k = 1; k < kCluster; ++k) Z = df_add(Z, arr[k]);
  T = df_mul_f(Z, u2);
  if (!(T.hi >= 0.f)) T = DF{0.f, 0.f};  // a NaN or negative uniform draws the first token with mass
  owner = -1;
  lo_owner = DF{0.f, 0.f};
  DF pre{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kCluster; ++k) {
    if (df_pos(arr[k]) && df_le(pre, T)) {
      owner = k;
      lo_owner = pre;
    }
    pre = df_add(pre, arr[k]);
  }
  return Z;
}

// In the owner slice: the largest token x with r(x) > 0 whose lower CDF edge
// (from the slice's start) is <= Tc. Returns it in every thread (-1: none).
template <int DT>
__device__ int locate_in_slice(Smem& s, const unsigned char* tsl, const unsigned char* dsl, int nv, int x0,
                               int kind, int xhat, float c, float mcp, float mcq, float bhi, float blo,
                               DF Tc) {
  constexpr int EPV = Elem<DT>::kEPV;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float m = run_mass<DT>(tsl, dsl, nv, x0, kind, xhat, c, mcp, mcq, bhi, blo);
  const DF inc = warp_incl_scan_df(DF{m, 0.f}, lane);
  if (lane == 31) s.redx[warp] = inc;
  if (tid == 0) s.pick = -1;
  __syncthreads();
  DF lo{__shfl_up_sync(kFull, inc.hi, 1), __shfl_up_sync(kFull, inc.lo, 1)};
  if (lane == 0) lo = DF{0.f, 0.f};
  for (int w = 0; w < warp; ++w) lo = df_add(lo, s.redx[w]);
  if (m > 0.f && df_le(lo, Tc)) atomicMax(&s.pick, tid);
  __syncthreads();
  if (tid == s.pick) {
    int a, e;
    thread_run(nv, a, e);
    DF run = lo;
    int cand = -1;
    for (int v = a; v < e; ++v) {
      float zp[EPV], zq[EPV];
      unpack<DT>(lds16(smem_addr(tsl + (size_t)v * 16)), zp);
      if (kind == kResidual) unpack<DT>(lds16(smem_addr(dsl + (size_t)v * 16)), zq);
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        const int x = x0 + v * EPV + j;
        const float r = r_of(kind, zp[j], kind == kResidual ? zq[j] : 0.f, x, xhat, c, mcp, mcq, bhi, blo);
        if (r > 0.f && df_le(run, Tc)) cand = x;
        run = df_add_f(run, r);
      }
    }
    s.redi[0] = cand;
  }
  __syncthreads();
  const int y = s.pick >= 0 ? s.redi[0] : -1;
  __syncthreads();
  return y;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) cluster_verify_kernel(CParams P) {
  constexpr int EPV = Elem<DT>::kEPV;
  extern __shared__ __align__(128) unsigned char slices[];
  __shared__ Smem s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned rank = cluster_rank();
  const int t = (int)(blockIdx.x / kCluster);

  // Offsets: every CTA checks and all take the same decision.
  bool bad = false;
  for (int k = tid; k < P.B; k += kThreads)
    if (P.cu[k + 1] < P.cu[k]) bad = true;
  if (tid == 0 && (P.cu[0] != 0 || (long long)P.cu[P.B] + P.B > P.row_cap)) bad = true;
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(P.status, SV_DATA_BAD_OFFSETS);
    return;
  }
  if (t >= P.cu[P.B] + P.B) return;  // the whole cluster: t is the same in all its CTAs

  // This CTA's slice: 16-byte vectors [v0, v0 + nv) of the row.
  const int v0 = min(P.nvec, (int)rank * P.vp);
  const int nv = min(P.nvec, v0 + P.vp) - v0;
  const int x0 = v0 * EPV;  // first token of the slice
  unsigned char* tsl = slices;
  unsigned char* dsl = slices + (size_t)P.vp * 16;
  const size_t rowb = (size_t)P.nvec * 16;
  const uint32_t bar_t = smem_addr(&s.bar_t), bar_d = smem_addr(&s.bar_d);
  if (tid == 0) {
    mbar_init(bar_t, 1);
    mbar_init(bar_d, 1);
    for (int x = 0; x < kExchanges; ++x) mbar_init(smem_addr(&s.xbar[x]), kCluster);
    fence_mbar_init();
    s.copy_timeout = 0;
    s.x_timeout = 0;
    if (nv > 0)
      copy_slice(smem_addr(tsl), static_cast<const char*>(P.target) + (size_t)t * rowb + (size_t)v0 * 16,
                 (uint32_t)nv * 16u, bar_t);
  }
  // Every CTA of the cluster must have started, and initialised its
  // mbarriers, before any write or arrive into its shared memory: arrive now
  // (releasing the initialisation), wait just before the first exchange.
  cluster_arrive();

  if (warp == 0) {
    const int b = find_request(P.cu, P.B, t, lane);
    if (lane == 0) {
      const int t0 = P.cu[b] + b, d0 = P.cu[b];
      const int K = P.cu[b + 1] - d0, i = t - t0;
      int greedy = P.greedy_all;
      if (!greedy && P.mode) {
        const uint8_t m = P.mode[b];
        if (m == SV_MODE_GREEDY)
          greedy = 1;
        else if (m != SV_MODE_SAMPLE && i == 0 && rank == 0)
          atomicOr(P.status, SV_DATA_BAD_MODE);
      }
      int xhat = -1;
      if (i < K && P.draft_tokens) {
        xhat = P.draft_tokens[d0 + i];
        if (xhat < 0 || xhat >= P.V) {
          if (rank == 0) atomicOr(P.status, SV_DATA_BAD_TOKEN);
          xhat = -1;
        }
      }
      const int has_d = !greedy && i < K && P.draft != nullptr;
      if (has_d && nv > 0)
        copy_slice(smem_addr(dsl), static_cast<const char*>(P.draft) + (size_t)(d0 + i) * rowb + (size_t)v0 * 16,
                   (uint32_t)nv * 16u, bar_d);
      s.b = b;
      s.t0 = t0;
      s.d0 = d0;
      s.K = K;
      s.i = i;
      s.greedy = greedy;
      s.xhat = xhat;
      s.has_d = has_d;
      s.u_acc = greedy ? 0.f : __ldg(&P.uniforms[2 * (size_t)t]);
      s.u2 = greedy ? 0.f : __ldg(&P.uniforms[2 * (size_t)t + 1]);
    }
  }
  __syncthreads();
  const int K = s.K, i = s.i, xhat = s.xhat;
  const bool greedy = s.greedy != 0, has_d = s.has_d != 0;

  // Wait for the slices (bounded; a copy that never lands is reported).
  if (nv > 0) {
    bool ok = mbar_wait(bar_t, 0);
    if (has_d) ok = mbar_wait(bar_d, 0) && ok;
    if (!ok) s.copy_timeout = 1;
  }
  __syncthreads();
  if (tid == 0 && s.copy_timeout) atomicOr(P.status, SV_DEV_COPY_TIMEOUT);

  // Slice statistics.
  const float c = P.c;
  if (greedy) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int v = tid; v < nv; v += kThreads) {
      float z[EPV];
      unpack<DT>(lds16(smem_addr(tsl + (size_t)v * 16)), z);
#pragma unroll
      for (int j = 0; j < EPV; ++j)
        if (z[j] > bv) {  // elements of a thread come in increasing order: keep the first
          bv = z[j];
          bi = x0 + v * EPV + j;
        }
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      s.redf[warp] = bv;
      s.redi[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      float v = s.redf[0];
      int k = s.redi[0];
      for (int w = 1; w < kWarps; ++w) argmax_merge(v, k, s.redf[w], s.redi[w]);
      s.mine = SliceRec{DF{0.f, 0.f}, DF{0.f, 0.f}, -INFINITY, -INFINITY, 0.f, 0.f, v, k, 0, 0};
    }
  } else {
    // Maxima, then sums relative to them (the slice is in shared memory).
    float mp = -INFINITY, mq = -INFINITY;
    for (int v = tid; v < nv; v += kThreads) {
      float z[EPV];
      unpack<DT>(lds16(smem_addr(tsl + (size_t)v * 16)), z);
#pragma unroll
      for (int j = 0; j < EPV; ++j) mp = fmaxf(mp, z[j]);
      if (has_d) {
        unpack<DT>(lds16(smem_addr(dsl + (size_t)v * 16)), z);
#pragma unroll
        for (int j = 0; j < EPV; ++j) mq = fmaxf(mq, z[j]);
      }
    }
    mp = warp_max(mp);
    mq = warp_max(mq);
    if (lane == 0) {
      s.redf[warp] = mp;
      s.redf2[warp] = mq;
    }
    __syncthreads();
    mp = s.redf[0];
    mq = s.redf2[0];
    for (int w = 1; w < kWarps; ++w) {
      mp = fmaxf(mp, s.redf[w]);
      mq = fmaxf(mq, s.redf2[w]);
    }
    const float mcp = mp == -INFINITY ? 0.f : __fmul_rn(mp, c);
    const float mcq = mq == -INFINITY ? 0.f : __fmul_rn(mq, c);
    float ap[EPV], aq[EPV];
#pragma unroll
    for (int j = 0; j < EPV; ++j) ap[j] = aq[j] = 0.f;
    for (int v = tid; v < nv; v += kThreads) {
      float z[EPV];
      unpack<DT>(lds16(smem_addr(tsl + (size_t)v * 16)), z);
#pragma unroll
      for (int j = 0; j < EPV; ++j) ap[j] += ex2(fmaf(z[j], c, -mcp));
      if (has_d) {
        unpack<DT>(lds16(smem_addr(dsl + (size_t)v * 16)), z);
#pragma unroll
        for (int j = 0; j < EPV; ++j) aq[j] += ex2(fmaf(z[j], c, -mcq));
      }
    }
    DF tp{0.f, 0.f}, tq{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      tp = df_add_f(tp, ap[j]);
      tq = df_add_f(tq, aq[j]);
    }
    tp = warp_sum_df(tp);
    tq = warp_sum_df(tq);
    if (lane == 0) {
      s.reddf_p[warp] = tp;
      s.reddf_q[warp] = tq;
    }
    __syncthreads();
    if (tid == 0) {
      DF sp = s.reddf_p[0], sq = s.reddf_q[0];
      for (int w = 1; w < kWarps; ++w) {
        sp = df_add(sp, s.reddf_p[w]);
        sq = df_add(sq, s.reddf_q[w]);
      }
      SliceRec r{sp, sq, mp, mq, 0.f, 0.f, -INFINITY, INT_MAX, 0, 0};
      if (xhat >= x0 && xhat < x0 + nv * EPV) {
        const int o = xhat - x0;
        float z[EPV];
        unpack<DT>(lds16(smem_addr(tsl + (size_t)(o / EPV) * 16)), z);
        r.zxp = z[o % EPV];
        if (has_d) {
          unpack<DT>(lds16(smem_addr(dsl + (size_t)(o / EPV) * 16)), z);
          r.zxq = z[o % EPV];
        }
        r.has_x = 1;
      }
      s.mine = r;
    }
  }
  __syncthreads();

  // Exchange 1: every slice's record to every CTA of the cluster.
  cluster_wait();  // every CTA has started
  if (tid < kCluster) {
    const uint32_t dst = peer_addr(&s.rec[rank], (unsigned)tid);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&s.mine);
#pragma unroll
    for (int w = 0; w < (int)(sizeof(SliceRec) / 4); ++w) st_cluster(dst + 4u * w, src[w]);
  }
  exchange_done(s, kX1);

  // The row, merged in rank order (the same in every CTA), and its decision.
  if (tid == 0) {
    if (greedy) {
      float v = s.rec[0].av;
      int k = s.rec[0].ai;
      for (int r = 1; r < kCluster; ++r) argmax_merge(v, k, s.rec[r].av, s.rec[r].ai);
      const int am = k == INT_MAX ? 0 : k;  // all -inf: index 0, like argmax
      s.am = am;
      s.acc = (i < K && xhat == am) ? 1 : 0;
      s.need_draw = 0;
      if (rank == 0 && P.out_probs) {
        P.out_probs[2 * (size_t)t] = -1.f;
        P.out_probs[2 * (size_t)t + 1] = -1.f;
      }
    } else {
      float Mp = -INFINITY, Mq = -INFINITY;
      for (int r = 0; r < kCluster; ++r) {
        Mp = fmaxf(Mp, s.rec[r].mp);
        Mq = fmaxf(Mq, s.rec[r].mq);
      }
      const float mcp = Mp == -INFINITY ? 0.f : __fmul_rn(Mp, c);
      const float mcq = Mq == -INFINITY ? 0.f : __fmul_rn(Mq, c);
      DF Sp{0.f, 0.f}, Sq{0.f, 0.f};
      float zxp = -INFINITY, zxq = -INFINITY;
      for (int r = 0; r < kCluster; ++r) {
        const SliceRec& q = s.rec[r];
        if (df_pos(q.Sp)) Sp = df_add(Sp, df_mul_f(q.Sp, ex2(__fmul_rn(q.mp, c) - mcp)));
        if (df_pos(q.Sq)) Sq = df_add(Sq, df_mul_f(q.Sq, ex2(__fmul_rn(q.mq, c) - mcq)));
        if (q.has_x) {
          zxp = q.zxp;
          zxq = q.zxq;
        }
      }
      s.mcp = mcp;
      s.mcq = mcq;
      s.Sp = Sp;
      s.Sq = Sq;
      if (rank == 0 && (!df_pos(Sp) || (has_d && !df_pos(Sq)))) atomicOr(P.status, SV_DATA_EMPTY_ROW);
      int acc = 0;
      if (i < K) {
        float ph = -1.f, qh = -1.f;
        if (xhat >= 0) {
          // p(x̂) = 2^(z c - mc_p) / S_p and min(1, p/q), q from the draft
          // row or 1 for a one-hot proposal, in fp32 as in the streaming kernel.
          const float a_p = fmaf(zxp, c, -mcp);
          const float Spf = Sp.hi, Sqf = Sq.hi;
          const float pd = __fdiv_rn(exp2f(a_p), Spf);
          float rho, qd = 1.f;
          if (has_d) {
            const float a_q = fmaf(zxq, c, -mcq);
            qd = __fdiv_rn(exp2f(a_q), Sqf);
            rho = (zxq == -INFINITY) ? 0.f : fminf(1.f, __fmul_rn(exp2f(a_p - a_q), __fdiv_rn(Sqf, Spf)));
          } else {
            rho = fminf(1.f, pd);
          }
          acc = (s.u_acc < rho) ? 1 : 0;
          ph = pd;
          qh = qd;
        }
        if (rank == 0 && P.out_probs) {
          P.out_probs[2 * (size_t)t] = ph;
          P.out_probs[2 * (size_t)t + 1] = qh;
        }
      }
      s.acc = acc;
      s.am = -1;
      s.need_draw = (i == K || !acc) ? 1 : 0;
      s.kind = i == K ? kBonus : (has_d ? kResidual : kOneHot);
    }
  }
  __syncthreads();

  // One CTA of the cluster writes the row's result and counts the row in:
  // the one that drew the token, else rank 0.
  bool writer = rank == 0;
  if (s.need_draw) {
    // A token from r over the whole row: every slice's mass, then the slice
    // that holds u' * Z finds it. The same in every CTA of the cluster.
    const int kind0 = s.kind;
    const float mcp = s.mcp, mcq = s.mcq;
    const DF Sp = s.Sp, Sq = s.Sq;
    // beta = S_p / S_q as a double-float pair (r needs it to ~2^-44).
    const DF beta = (kind0 == kResidual && df_pos(Sq)) ? df_div(Sp, Sq) : DF{1.f, 0.f};
    const float bhi = beta.hi, blo = beta.lo;
    int kind = kind0;
    DF m = cta_sum_df(s, run_mass<DT>(tsl, dsl, nv, x0, kind, xhat, c, mcp, mcq, bhi, blo));
    int owner;
    DF lo, T;
    DF Z = exchange_mass(s, kX2, s.mass, rank, m, s.u2, owner, lo, T);
    if (!df_pos(Z) && kind != kBonus) {
      // No residual mass (p == q in fp32): draw from p instead.
      if (rank == 0 && tid == 0) atomicOr(P.status, SV_DATA_DEGENERATE_RESIDUAL);
      kind = kBonus;
      m = cta_sum_df(s, run_mass<DT>(tsl, dsl, nv, x0, kind, xhat, c, mcp, mcq, 1.f, 0.f));
      Z = exchange_mass(s, kX3, s.mass2, rank, m, s.u2, owner, lo, T);
    }
    const float bh = kind == kResidual ? bhi : 1.f, bl = kind == kResidual ? blo : 0.f;
    int y = -1;
    if ((int)rank == owner) y = locate_in_slice<DT>(s, tsl, dsl, nv, x0, kind, xhat, c, mcp, mcq, bh, bl, df_sub(T, lo));
    writer = owner < 0 ? rank == 0 : (int)rank == owner;
    if (writer && tid == 0) {
      if (y < 0) {  // no mass at all (or a lost rescan): token 0, like the streaming kernel
        if (owner < 0) atomicOr(P.status, SV_DATA_EMPTY_ROW);
        y = 0;
      }
      // p(y), q(y) as the streaming kernel reports them (q by the row's own
      // rule, also after a fall back to p).
      float zpy, zqy = -INFINITY;
      {
        const int o = y - x0;
        float z[EPV];
        if (o >= 0 && o < nv * EPV) {
          unpack<DT>(lds16(smem_addr(tsl + (size_t)(o / EPV) * 16)), z);
          zpy = z[o % EPV];
          if (kind0 == kResidual) {
            unpack<DT>(lds16(smem_addr(dsl + (size_t)(o / EPV) * 16)), z);
            zqy = z[o % EPV];
          }
        } else {
          zpy = Elem<DT>::scalar(static_cast<const char*>(P.target) + (size_t)t * rowb, y);
          if (kind0 == kResidual)
            zqy = Elem<DT>::scalar(static_cast<const char*>(P.draft) + (size_t)(s.d0 + i) * rowb, y);
        }
      }
      const float py = __fdiv_rn(exp2f(fmaf(zpy, c, -mcp)), Sp.hi);
      float qy = 0.f;
      if (kind0 == kResidual)
        qy = __fdiv_rn(exp2f(fmaf(zqy, c, -mcq)), Sq.hi);
      else if (kind0 == kOneHot)
        qy = (y == xhat) ? 1.f : 0.f;
      P.rows[t] = CRow{(unsigned)s.acc, y, py, qy};
      __threadfence();
    }
  } else if (rank == 0 && tid == 0) {
    P.rows[t] = CRow{(unsigned)s.acc, greedy ? s.am : -1, 0.f, 0.f};
    __threadfence();
  }

  // Every write into this CTA's shared memory came before the last exchange
  // it waited for, and no CTA writes into another after its own last one.
  __syncthreads();
  if (tid == 0 && s.x_timeout) atomicOr(P.status, SV_DEV_COPY_TIMEOUT);

  // The request's last row to finish commits it. The writer's fence above
  // released the row's result before the count.
  if (writer && warp == 0) {
    const int b = s.b, t0 = s.t0, d0 = s.d0;
    unsigned long long old = 0;
    if (lane == 0) old = atomicAdd(&P.arrive[b], 1ull);
    old = __shfl_sync(kFull, old, 0);
    if (old == (unsigned long long)K) {
      __threadfence();
      int stop = K;
      for (int j0 = 0; j0 < K && stop == K; j0 += 32) {
        const int j = j0 + lane;
        const bool rej = j < K && __ldcg(&P.rows[t0 + j].accept) == 0u;
        const unsigned m = __ballot_sync(kFull, rej);
        if (m) stop = j0 + __ffs(m) - 1;
      }
      for (int j = lane; j < stop; j += 32) P.out_tokens[t0 + j] = P.draft_tokens[d0 + j];
      if (lane == 0) {
        const int4 w = __ldcg(reinterpret_cast<const int4*>(&P.rows[t0 + stop]));
        const CRow r{(unsigned)w.x, w.y, __int_as_float(w.z), __int_as_float(w.w)};
        P.out_tokens[t0 + stop] = r.y;
        P.out_len[b] = stop + 1;
        if (P.out_probs) {
          P.out_probs[2 * (size_t)(t0 + K)] = greedy ? -1.f : r.py;
          P.out_probs[2 * (size_t)(t0 + K) + 1] = greedy ? -1.f : r.qy;
        }
        P.arrive[b] = 0ull;  // every row is in: ready for the next call
      }
    }
  }
}

static std::atomic<int> g_smem_set[64][2];

}  // namespace cl

size_t cluster_smem_bytes(size_t row_bytes, bool has_draft) {
  const size_t vp = ((row_bytes / 16) + kCluster - 1) / kCluster;
  const size_t need = (has_draft ? 2 : 1) * vp * 16;
  return need <= cl::kMaxSmem ? (need > 0 ? need : 16) : 0;
}

cudaError_t launch_cluster_verify(const CParams& P0, int dtype, cudaStream_t st) {
  CParams P = P0;
  P.vp = (P.nvec + kCluster - 1) / kCluster;
  const size_t smem = cluster_smem_bytes((size_t)P.nvec * 16, P.draft != nullptr);
  if (smem == 0) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const void* fn = dtype == 1 ? (const void*)cl::cluster_verify_kernel<1> : (const void*)cl::cluster_verify_kernel<0>;
  if (dev < 64 && cl::g_smem_set[dev][dtype].load(std::memory_order_relaxed) < (int)smem) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cl::kMaxSmem);
    if (e != cudaSuccess) return e;
    cl::g_smem_set[dev][dtype].store((int)cl::kMaxSmem, std::memory_order_relaxed);
  }
  long long rows = P.row_cap < 1 ? 1 : P.row_cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * kCluster));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (dtype == 1)
    e = cudaLaunchKernelEx(&cfg, cl::cluster_verify_kernel<1>, P);
  else
    e = cudaLaunchKernelEx(&cfg, cl::cluster_verify_kernel<0>, P);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sv
