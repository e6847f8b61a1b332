// spec_verify.cu -- verify-and-commit of speculative decoding on sm_103a.
//
// One persistent kernel does the whole step:
//
//   1. Row pass. Work items are target rows t = (request b, slot i), handed
//      out in request order by an atomic counter. The CTA streams the target
//      row (and, for a sampled draft slot, the paired draft row) once through
//      a ring of shared-memory stages filled by bulk asynchronous copies (the
//      TMA engine), and keeps a single-pass online softmax: per thread a running
//      maximum and one fp32 partial sum per vector lane, rescaled when the
//      maximum grows. Sums are combined, kept and scanned in double-float
//      arithmetic (fp32 pairs), so S = sum_x 2^(z_x c - Mc) (c = log2(e)/T,
//      Mc = fp32(max z * c)) is accurate to ~1e-9 relative. No fp64 sits on
//      a dependent path: on this part a dependent fp64 operation takes about
//      14 times as long as an fp32 one, and a division about 6 times as long
//      as an fp32 division. Greedy rows compute the argmax instead
//      (lowest index among ties). The CTA then gathers z[x̂] and decides the
//      slot: accept iff u < min(1, p(x̂)/q(x̂)) ("Draft Model（草稿模型）", §2
//      "接受-拒绝准则"; a zero draft probability rejects, "投机解码从零实现"
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
//      running sum of r exceeds u' * sum(r). The stop row (pair) is streamed
//      through the ring once, last chunk first, to sum r over every tile;
//      only the tile that holds the target is rescanned.
//   The last CTA to leave resets the work counter, and each request's counter
//   is reset by its commit, so the workspace is left zeroed.
//
// Rows whose base is not 16-byte aligned (or whose byte length is not a
// multiple of 16) take the same steps with scalar global loads.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <cuda_bf16.h>

#include "../../include/spec_verify.h"
#include "sv_device.cuh"
#include "sv_filter.cuh"
#include "sv_cluster.cuh"
#include "sv_greedy.cuh"
#include "sv_onehot.cuh"

namespace sv {

struct WsHeader {
  unsigned int status;     // SV_DATA_* bits (sticky until sv_check_status)
  unsigned int next_item;  // items handed out by claims (every CTA's first item, blockIdx.x, is not claimed)
  unsigned int exited;     // CTAs that left the work loop
  unsigned int n_draws;    // draw slots reserved
  unsigned int draw_head;  // slots before this one are fully handed out
  unsigned int committed;  // requests committed
  unsigned int pad[10];
};
static_assert(sizeof(WsHeader) == 64, "workspace header is 64 bytes");

// Per target row result of the row pass (32 bytes).
struct alignas(16) RowRec {
  float mc_p;        // fp32(max z_target * c): exponent offset of the target row
  float mc_q;        // same for the paired draft row (sampled draft slots)
  DF S_p;            // sum_x 2^(z_x c - mc_p) over the target row (double-float)
  DF S_q;            // same over the draft row
  int argmax;        // greedy rows: first index of the maximum
  unsigned accept;   // bit 0: the slot's draft token is accepted; bit 1: the
                     // row's tile sums of its draw's r are stored (rows streamed
                     // alone: bonus rows r = 2^(z c - mc_p), one-hot rows the same
                     // without x̂)
};
static_assert(sizeof(RowRec) == 32, "row record is 32 bytes");

// Statistics of one part of a split row (32 bytes): the same quantities as
// RowRec over the part's slice, S = 0 for a slice without a finite logit.
struct alignas(16) PartRec {
  float mc_p, mc_q;
  DF S_p, S_q;
  float amax_v;      // greedy: largest logit of the slice
  int amax_i;        // and its first index (0x7fffffff if none)
};
static_assert(sizeof(PartRec) == 32, "part record is 32 bytes");

// A draw published in parts (64 bytes); `done` counts finished parts. The
// slot's state word packs the part count (bits 20..31, 0 = not published)
// and the parts handed out (bits 0..19), so one load checks a slot and one
// atomic claims a part.
constexpr unsigned kSlotCountBits = 20;
constexpr unsigned kSlotCountMask = (1u << kSlotCountBits) - 1u;
struct alignas(16) DrawDesc {
  int b;            // request
  int row;          // stop row (target row index)
  int drow;         // paired draft row index, or -1
  int kind;         // DrawKind
  int xhat;         // the rejected one-hot proposal, or -1
  float mcp, mcq;   // exponent offsets of the stop rows
  int nparts;       // parts the draw is split into
  DF Sp, Sq;        // sums of the stop rows
  unsigned unused;
  unsigned done;    // parts finished
  int bonus_row;    // row that receives (p(y), q(y)) of the drawn token
  int pad;
};
static_assert(sizeof(DrawDesc) == 64, "draw descriptor is 64 bytes");

constexpr int kMaxScanTiles = kThreads;   // the draw scans at most one tile per thread
// Largest vocabulary for each element type: kMaxScanTiles tiles of one
// 16-byte vector per thread (fp32 262144, bf16 524288).
constexpr int max_vocab(int dtype) { return kMaxScanTiles * kThreads * (dtype == 0 ? 4 : 8); }

// Shared-memory ring of the bulk-copy streams.
#ifndef SV_STAGES
#define SV_STAGES 2
#endif
#ifndef SV_VPT
#define SV_VPT 4
#endif
#ifndef SV_MINBLOCKS
#define SV_MINBLOCKS 3
#endif
#ifndef SV_PART_CHUNKS
#define SV_PART_CHUNKS 1
#endif
#ifndef SV_PUBLISH_PCT
#define SV_PUBLISH_PCT 0
#endif
#ifndef SV_ROW_PARTS
#define SV_ROW_PARTS 1
#endif
#ifndef SV_TAIL_WAVES
#define SV_TAIL_WAVES 1
#endif
constexpr int kStages = SV_STAGES;                  // stages (kStages - 1 in flight)
constexpr int kVPT = SV_VPT;                        // 16-byte vectors per thread per chunk
constexpr int kChunkBytes = kThreads * 16 * kVPT;   // bytes of one row per stage
static_assert((kVPT & (kVPT - 1)) == 0, "vectors per thread must be a power of two");
// Kernel variants: DT & 1 is the logit type (0 fp32, 1 bf16); DT & kFilt
// marks the top-k / top-p filtered form, in which a logit below its row's
// threshold counts as -inf everywhere it is read.
constexpr int kFilt = 2;
constexpr int kStageBytes = 2 * kChunkBytes;        // target + draft chunk
constexpr int kRingBytes = kStages * kStageBytes;   // dynamic shared memory per CTA
constexpr int kPartChunks = SV_PART_CHUNKS;         // ring chunks per draw part
constexpr int kMaxParts = 16;                       // parts a draw is split into, at most
constexpr size_t kMinPublishBytes = 192 * 1024;      // smallest draw worth splitting
constexpr int kMaxDrawSlots = 4096;                 // draws that can be published per call
// Draws are split into parts once the rows still to be handed out number at
// most kPublishPct percent of the grid (0: once all rows are handed out).
constexpr unsigned kPublishPct = SV_PUBLISH_PCT;
// Rows may be split into parts that different CTAs stream; the CTA that
// finishes a row's last part merges the parts' statistics. Every row is
// split when there are fewer rows than CTAs (small batches); the last
// kTailWaves waves of a large batch are split when kRowParts > 1 (measured
// slower on the benchmark workload, so off by default).
constexpr unsigned kRowParts = SV_ROW_PARTS;        // parts per split row (large batches)
constexpr unsigned kTailWaves = SV_TAIL_WAVES;
constexpr unsigned kMaxRowParts = 16;
constexpr unsigned kMaxTailRows = 4096;             // split rows per call, at most
constexpr unsigned kMaxPartRecs = 16384;            // part records, at most
// A CTA with no rows left looks for draw parts until every request has
// committed, sleeping kLingerNs between looks, at most kLingerPolls times.
// Giving up early is harmless: a draw's owner takes its remaining parts.
#ifndef SV_BONUS_LAST
#define SV_BONUS_LAST 1
#endif
#ifndef SV_LINGER_NS
#define SV_LINGER_NS 500
#endif
constexpr unsigned kLingerNs = SV_LINGER_NS;
// Work order: rows in target-row order, or (kBonusLast) every draft-slot row
// first and the requests' bonus rows last.
constexpr bool kBonusLast = SV_BONUS_LAST != 0;
constexpr unsigned kLingerPolls = 1u << 16;

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
  unsigned long long* req_state;  // [B] rows finished (and accepted) per request
  unsigned int* slot_state; // [n_slots] nparts << 20 | parts handed out (0: unpublished)
  DrawDesc* descs;          // [n_slots]
  DF* tsum;                 // [n_slots, tsum_stride] per-tile sums of r
  float* rtile;             // [row_cap, tsum_stride] tile sums of r of rows streamed alone, or NULL
  const float* thr;         // [R_t] filter thresholds of the target rows, or NULL
  const float* thr_d;       // [R_d] filter thresholds of the draft rows, or NULL
  const FStat* fst;         // [R_t] filtered softmax statistics of the target rows, or NULL
  const FStat* fst_d;       // [R_d] of the draft rows, or NULL
  const int2* flist;        // [R_t, kKeptListCap] kept (token, logit bits) per target row, or NULL
  unsigned* fc_need;        // the filtered commit left requests (nonzero), or NULL: no such commit ran
  const unsigned char* fc_done;  // [B] 1: request committed by the filtered commit
  int n_slots, tsum_stride;
  unsigned int* part_done;  // [kMaxTailRows] parts finished per split row
  PartRec* parts;           // [kMaxPartRecs]
  RowRec* rows;             // [R_t]
  long long row_cap;
  int greedy_all;
  int may_publish;          // some draw of this call may be published in parts
};

struct Smem {
  unsigned long long full[kStages];   // stage holds its chunk (bulk-copy bytes landed)
  unsigned long long empty[kStages];  // every warp has finished reading the stage
  unsigned ring_seq;                  // chunks this CTA has streamed so far
  int wk, item, slot, part;
  unsigned n_items, r_full, row_parts;  // work-item layout of this launch
  int b, t, t0, d0, K, i, greedy, xhat, last, stop, merge, pick, pick2, tok, R_d;
  int zx_ok;        // z_p(x̂) (and z_q(x̂)) were taken from the ring during the row pass
  int pre;          // filtered row: its statistics came from the threshold kernel
  int claims;       // work items this CTA has asked for (thread 0)
  int btile_ok;     // this row's tile sums of r were stored during its pass
  float tau_t, tau_d;  // filter thresholds of the row pair (-inf: unfiltered)
  float zx_p, zx_q, u_acc;
  float redf[kWarps];
  float redf2[kWarps];
  int redi[kWarps];
  DF reddf_p[kWarps];
  DF reddf_q[kWarps];
  float bcast_f[2];
  DF dred[kWarps];
  DF dred2[kWarps];
  DF wexcl[kWarps + 1];
  DF tincl[kMaxScanTiles];
  float wtot[kMaxScanTiles * kWarps];
};

// Raw 16-byte vectors of logits as the ring holds them: the all -inf vector,
// the elements as fp32 pairs (lanes 2i, 2i+1) and the maximum over N vectors.
template <int DT>
struct Raw;

template <>
struct Raw<0> {
  static constexpr uint32_t kNegInf = 0xff800000u;
  __device__ __forceinline__ static void pairs(const uint4& v, f2_t (&z)[2]) {
    z[0] = f2_pack(__uint_as_float(v.x), __uint_as_float(v.y));
    z[1] = f2_pack(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  template <int N>
  __device__ __forceinline__ static float max_of(const uint4 (&v)[N]) {
    float t[4 * N];
#pragma unroll
    for (int u = 0; u < N; ++u) {
      t[4 * u] = __uint_as_float(v[u].x);
      t[4 * u + 1] = __uint_as_float(v[u].y);
      t[4 * u + 2] = __uint_as_float(v[u].z);
      t[4 * u + 3] = __uint_as_float(v[u].w);
    }
#pragma unroll
    for (int w = 2 * N; w >= 1; w /= 2)
#pragma unroll
      for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
    return t[0];
  }
};

template <>
struct Raw<1> {
  static constexpr uint32_t kNegInf = 0xff80ff80u;
  // bf16 is the top half of an fp32: the low element of a word is shifted
  // up, the high one masked.
  __device__ __forceinline__ static void pairs(const uint4& v, f2_t (&z)[4]) {
    z[0] = f2_pack(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
    z[1] = f2_pack(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    z[2] = f2_pack(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u));
    z[3] = f2_pack(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
  }
  // Pairwise bf16x2 maxima down to one word, then its two halves.
  template <int N>
  __device__ __forceinline__ static float max_of(const uint4 (&v)[N]) {
    uint32_t t[4 * N];
#pragma unroll
    for (int u = 0; u < N; ++u) {
      t[4 * u] = v[u].x;
      t[4 * u + 1] = v[u].y;
      t[4 * u + 2] = v[u].z;
      t[4 * u + 3] = v[u].w;
    }
#pragma unroll
    for (int w = 2 * N; w >= 1; w /= 2)
#pragma unroll
      for (int j = 0; j < w; ++j) t[j] = bf2_max(t[j], t[j + w]);
    return fmaxf(__uint_as_float(t[0] << 16), __uint_as_float(t[0] & 0xffff0000u));
  }
};

// Online softmax state of one thread: running maximum m, its fp32 exponent
// offset mc = fp32(m * c) (0 while m is -inf) and one partial sum per lane of
// the 16-byte vector, kept as fp32 pairs. Every term is 2^(z c - mc).
template <int EPV>
struct SoftAcc {
  static constexpr int kPairs = EPV / 2;
  float m, mc;
  f2_t a[kPairs];
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    mc = 0.f;
#pragma unroll
    for (int i = 0; i < kPairs; ++i) a[i] = 0ull;  // two +0.0f
  }
  __device__ __forceinline__ float lane(int j) const {
    float lo, hi;
    f2_unpack(a[j >> 1], lo, hi);
    return (j & 1) ? hi : lo;
  }
  // Raises the running maximum to vm (if larger), rescaling the partial sums.
  __device__ __forceinline__ void raise(float vm, float c) {
    if (vm > m) {
      float nmc = __fmul_rn(vm, c);
      const f2_t s = f2_splat((m == -INFINITY) ? 0.f : ex2(mc - nmc));
#pragma unroll
      for (int i = 0; i < kPairs; ++i) a[i] = f2_mul(a[i], s);
      m = vm;
      mc = nmc;
    }
  }
  __device__ __forceinline__ void accumulate(const f2_t (&z)[kPairs], f2_t cc, f2_t nmc) {
#pragma unroll
    for (int i = 0; i < kPairs; ++i) a[i] = f2_add(a[i], f2_ex2(f2_fma(z[i], cc, nmc)));
  }
  __device__ __forceinline__ void add(const float (&f)[EPV], float c) {
    float vm = f[0];
#pragma unroll
    for (int j = 1; j < EPV; ++j) vm = fmaxf(vm, f[j]);
    raise(vm, c);
    f2_t z[kPairs];
#pragma unroll
    for (int i = 0; i < kPairs; ++i) z[i] = f2_pack(f[2 * i], f[2 * i + 1]);
    accumulate(z, f2_splat(c), f2_splat(-mc));
  }
  // As add_raw, also returning each vector's own sum of terms (relative to
  // this thread's offset mc after the chunk); the running sums are the same.
  template <int DT, int N>
  __device__ __forceinline__ void add_raw_tiles(const uint4 (&v)[N], float c, float (&tv)[N]) {
    raise(Raw<DT & 1>::template max_of<N>(v), c);
    const f2_t cc = f2_splat(c), nmc = f2_splat(-mc);
#pragma unroll
    for (int u = 0; u < N; ++u) {
      f2_t z[kPairs], acc = 0ull;
      Raw<DT & 1>::pairs(v[u], z);
#pragma unroll
      for (int i = 0; i < kPairs; ++i) {
        const f2_t e = f2_ex2(f2_fma(z[i], cc, nmc));
        a[i] = f2_add(a[i], e);
        acc = f2_add(acc, e);
      }
      float lo, hi;
      f2_unpack(acc, lo, hi);
      tv[u] = lo + hi;
    }
  }
  // N raw vectors at once: one maximum and one rescale check.
  template <int DT, int N>
  __device__ __forceinline__ void add_raw(const uint4 (&v)[N], float c) {
    raise(Raw<DT & 1>::template max_of<N>(v), c);
    const f2_t cc = f2_splat(c), nmc = f2_splat(-mc);
#pragma unroll
    for (int u = 0; u < N; ++u) {
      f2_t z[kPairs];
      Raw<DT & 1>::pairs(v[u], z);
      accumulate(z, cc, nmc);
    }
  }
};

// Per-half (a >= b) of two bf16 pairs as 0xffff masks.
__device__ __forceinline__ uint32_t bf16x2_ge_mask(uint32_t a, uint32_t b) {
  __nv_bfloat162 x, y;
  memcpy(&x, &a, 4);
  memcpy(&y, &b, 4);
  return __hge2_mask(x, y);
}

// The kVPT vectors this thread consumes from a ring stage holding elements
// [x, x + kVPT * kThreads * EPV) of a row: whole vectors inside the row are
// read, those at or past V read as -inf.
// Filtered variants: logits below tau become -inf (zero mass).
template <int DT>
__device__ __forceinline__ uint4 mask_below(uint4 v, float tau) {
  if constexpr ((DT & kFilt) == 0) {
    return v;
  } else if constexpr ((DT & 1) == 1) {
    // Packed compare of bf16 pairs against tau in both halves (a bf16 row's
    // threshold is an exact bf16 value), then -inf where it fails.
    const uint32_t tb = __float_as_uint(tau) >> 16, t2 = tb | (tb << 16);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t mk = bf16x2_ge_mask(w[q], t2);
      w[q] = (w[q] & mk) | (0xff80ff80u & ~mk);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = __uint_as_float(w[q]) >= tau ? w[q] : 0xff800000u;
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}
template <int DT, int N>
__device__ __forceinline__ void mask_below(float (&f)[N], float tau) {
  if constexpr ((DT & kFilt) != 0) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (!(f[j] >= tau)) f[j] = -INFINITY;
  }
}
template <int DT>
__device__ __forceinline__ float mask_below(float z, float tau) {
  if constexpr ((DT & kFilt) != 0) return z >= tau ? z : -INFINITY;
  return z;
}

template <int DT>
__device__ __forceinline__ uint4 stage_vector(uint32_t stage, int x, int V, int v, bool whole,
                                              float tau) {
  constexpr int EPV = Elem<DT & 1>::kEPV;
  const int vi = v * kThreads + threadIdx.x;
  const uint32_t n = Raw<DT & 1>::kNegInf;
  return (whole || x + vi * EPV < V) ? mask_below<DT>(lds16(stage + 16u * vi), tau)
                                     : make_uint4(n, n, n, n);
}

template <int DT>
__device__ __forceinline__ void stage_vectors(uint32_t stage, int x, int V, uint4 (&rv)[kVPT],
                                              float tau) {
  constexpr int EPV = Elem<DT & 1>::kEPV;
  const int tid = threadIdx.x;
  if (x + kVPT * kThreads * EPV <= V) {
#pragma unroll
    for (int v = 0; v < kVPT; ++v) rv[v] = mask_below<DT>(lds16(stage + 16u * (v * kThreads + tid)), tau);
  } else {
    const uint32_t n = Raw<DT & 1>::kNegInf;
#pragma unroll
    for (int v = 0; v < kVPT; ++v) {
      const int vi = v * kThreads + tid;
      rv[v] = (x + vi * EPV < V) ? mask_below<DT>(lds16(stage + 16u * vi), tau) : make_uint4(n, n, n, n);
    }
  }
}

// Filtered variants: whether any of this thread's vectors kept a logit (a
// vector whose logits all fall below the threshold adds no mass and no
// maximum, so its softmax update can be skipped). Always true otherwise.
template <int DT>
__device__ __forceinline__ bool any_kept(const uint4 (&rv)[kVPT]) {
  if constexpr ((DT & kFilt) == 0) {
    return true;
  } else {
    constexpr uint32_t n = Raw<DT & 1>::kNegInf;
    bool any = false;
#pragma unroll
    for (int v = 0; v < kVPT; ++v)
      any |= (rv[v].x != n) | (rv[v].y != n) | (rv[v].z != n) | (rv[v].w != n);
    return any;
  }
}

// Warp totals of kVPT per-lane values (one per tile of a chunk): each
// halving step trades half of the tiles with the partner lane, then a plain
// butterfly. Returns the total of tile `t`, valid in lanes whose low
// log2(32 / kVPT) bits are zero (lane j * (32 / kVPT) holds tile j).
__device__ __forceinline__ float warp_tile_totals(float (&ts)[kVPT], int lane, int& t) {
  t = 0;
#pragma unroll
  for (int half = kVPT / 2, o = 16; half >= 1; half /= 2, o /= 2) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? ts[i] : ts[i + half];
      const float keep = up ? ts[i + half] : ts[i];
      ts[i] = keep + __shfl_xor_sync(kFull, send, o);
    }
    if (up) t += half;
  }
#pragma unroll
  for (int o = 16 / kVPT; o >= 1; o /= 2) ts[0] += __shfl_xor_sync(kFull, ts[0], o);
  return ts[0];
}

// Element j of vector v of rv (run once per row, by one thread).
template <int DT>
__device__ __forceinline__ float pick_element(const uint4 (&rv)[kVPT], int v, int j) {
  constexpr int EPV = Elem<DT & 1>::kEPV;
  float out = 0.f;
#pragma unroll
  for (int u = 0; u < kVPT; ++u) {
    if (u == v) {
      float f[EPV];
      Elem<DT & 1>::unpack(rv[u], f);
#pragma unroll
      for (int q = 0; q < EPV; ++q)
        if (q == j) out = f[q];
    }
  }
  return out;
}

// ---------------------------------------------------------------------------
// Bulk-copy ring
// ---------------------------------------------------------------------------
// Streams `nbytes` of a row (and the same span of its paired row) through the
// ring, first chunk first or (reverse) last chunk first; consume() gets the
// chunk's index in the span and its shared-memory address. A stage holds a
// chunk of each row, or, for a row streamed alone, two consecutive chunks of
// it (one copy of twice the size, so a lone row keeps as many bytes in
// flight as a pair). The k-th copy streamed lands in stage (seq + k) %
// kStages and completes on that stage's full barrier; every thread consumes
// the stage once it has arrived, after which each warp releases it on its
// empty barrier. Thread 0 refills a stage only once all warps have released
// its previous copy, so warps never wait for each other inside the stream.
// Every wait is bounded: a warp that gives up leaves the loop (warp-uniformly)
// and the CTA then agrees on the failure; the copies still in flight are
// waited for (bounded) and the ring must not be used again. Returns false on
// such a failure.
template <class Consume>
__device__ __forceinline__ bool ring_stream(Smem& s, unsigned char* ring, const char* tptr,
                                            const char* dptr, size_t nbytes, bool reverse,
                                            Consume&& consume) {
  const int tid = threadIdx.x, lane = tid & 31;
  const bool alone = dptr == nullptr;
  const size_t copy_bytes = alone ? 2 * (size_t)kChunkBytes : (size_t)kChunkBytes;
  const int nch = (int)((nbytes + copy_bytes - 1) / copy_bytes);
  const int nlog = (int)((nbytes + kChunkBytes - 1) / kChunkBytes);  // chunks of the span
  const unsigned seq0 = s.ring_seq;
  const uint32_t ring_base = smem_addr(ring);
  const uint32_t full_base = smem_addr(&s.full[0]);
  const uint32_t empty_base = smem_addr(&s.empty[0]);
  int issued = 0;    // copies issued (thread 0)
  bool ok = true;    // thread 0's refill waits
  // L2 priority: a row pass reads its bytes once, so they go first and the
  // small data every CTA keeps touching (offsets, tokens, uniforms, row
  // records) stays in L2; a draw's bytes stay, because the draw rescans the
  // chosen tile right after its pass.
  const uint64_t pol = (tid == 0) ? (reverse ? l2_policy_evict_last() : l2_policy_evict_first()) : 0ull;
  auto issue = [&](int k) {
    const unsigned q = seq0 + (unsigned)k;
    const int st = (int)(q % kStages);
    // The stage's previous copy (q - kStages) must have been released.
    if (q >= (unsigned)kStages && !mbar_wait(empty_base + 8u * st, ((q / kStages) - 1u) & 1u)) {
      ok = false;
      return;
    }
    const uint32_t bar = full_base + 8u * st;
    const size_t off = (size_t)(reverse ? nch - 1 - k : k) * copy_bytes;
    const size_t left = nbytes - off;
    const uint32_t bytes = (uint32_t)(left < copy_bytes ? left : copy_bytes);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, alone ? bytes : 2u * bytes);
    bulk_g2s_hint(ring_base + (uint32_t)st * kStageBytes, tptr + off, bytes, bar, pol);
    if (!alone)
      bulk_g2s_hint(ring_base + (uint32_t)st * kStageBytes + kChunkBytes, dptr + off, bytes, bar, pol);
    issued = k + 1;
  };
  if (tid == 0)
    for (int k = 0; k < kStages - 1 && k < nch && ok; ++k) issue(k);
  bool failed = false;
  for (int k = 0; k < nch; ++k) {
    if (tid == 0 && ok && k + kStages - 1 < nch) issue(k + kStages - 1);
    const unsigned q = seq0 + (unsigned)k;
    const int st = (int)(q % kStages);
    const bool arrived = mbar_wait(full_base + 8u * st, (q / kStages) & 1u) && ok;
    if (!__all_sync(kFull, arrived)) {
      failed = true;
      break;
    }
    const int c = reverse ? nch - 1 - k : k;
    const uint32_t stage = ring_base + (uint32_t)st * kStageBytes;
    if (!alone) {
      consume(c, stage);
    } else {
      consume(2 * c, stage);
      if (2 * c + 1 < nlog) consume(2 * c + 1, stage + kChunkBytes);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_base + 8u * st);
  }
  if (__syncthreads_or(failed)) {
    if (tid == 0) {
      // Wait (bounded) for every copy this stream issued before giving up.
      for (int j = 0; j < issued; ++j) {
        const unsigned q = seq0 + (unsigned)j;
        mbar_wait(full_base + 8u * (q % kStages), (q / kStages) & 1u);
      }
    }
    return false;
  }
  if (tid == 0) s.ring_seq = seq0 + (unsigned)nch;
  __syncthreads();
  return true;
}

// ---------------------------------------------------------------------------
// Row passes
// ---------------------------------------------------------------------------
// Scalar-load variants for rows that are not 16-byte aligned.
template <int DT, bool HAS_D>
__device__ __forceinline__ void stats_pass_scalar(const void* trow, const void* drow, int V, float c,
                                                  SoftAcc<Elem<DT & 1>::kEPV>& at,
                                                  SoftAcc<Elem<DT & 1>::kEPV>& ad, float tau_t,
                                                  float tau_d) {
  constexpr int EPV = Elem<DT & 1>::kEPV;
  constexpr int TILE = kThreads * EPV;
  for (int x = threadIdx.x * EPV; x < V; x += TILE) {
    float f[EPV];
    load_chunk<DT & 1, false>(trow, x, V, f);
    mask_below<DT>(f, tau_t);
    at.add(f, c);
    if constexpr (HAS_D) {
      load_chunk<DT & 1, false>(drow, x, V, f);
      mask_below<DT>(f, tau_d);
      ad.add(f, c);
    }
  }
}

template <int DT>
__device__ __forceinline__ void argmax_scalar(const void* trow, int V, float& bv, int& bi) {
  constexpr int EPV = Elem<DT & 1>::kEPV;
  constexpr int TILE = kThreads * EPV;
  for (int x = threadIdx.x * EPV; x < V; x += TILE) {
    float f[EPV];
    load_chunk<DT & 1, false>(trow, x, V, f);
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
                                float& Mc_p, DF& S_p, float& Mc_q, DF& S_q) {
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
  for (int j = 0; j < EPV; ++j) tp = df_add_f(tp, at.lane(j));
  tp = df_mul_f(tp, (at.m == -INFINITY) ? 0.f : ex2(at.mc - mcp));
  tp = warp_sum_df(tp);
  if (has_d) {
#pragma unroll
    for (int j = 0; j < EPV; ++j) tq = df_add_f(tq, ad.lane(j));
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
      S_p = v;
      S_q = w;
    }
  }
}

// Largest b in [0, B) with cu[b] (+ b when plus_b) <= j: the request that
// owns target row j (plus_b) or draft slot j. The keys do not decrease with
// b and key(0) = 0 <= j. Every thread of the CTA calls it: each round tests
// kThreads evenly spaced candidates of the remaining range at once, and the
// candidates that pass form a prefix whose length one barrier counts. One
// round (one memory round trip) up to B = kThreads, two up to kThreads^2.
__device__ __forceinline__ int find_request_cta(const int32_t* cu, int B, int j, bool plus_b) {
  int lo = 0, n = B;  // the answer lies in [lo, lo + n); key(lo) <= j
  while (n > 1) {
    const int step = (n + kThreads - 1) / kThreads;
    const int c = lo + (int)threadIdx.x * step;
    const bool pass = c < lo + n && cu[c] + (plus_b ? c : 0) <= j;
    const int cnt = __syncthreads_count(pass);  // >= 1: candidate lo passes
    const int end = lo + n;
    lo += (cnt - 1) * step;
    n = min(step, end - lo);
  }
  return lo;
}

// ---------------------------------------------------------------------------
// The draw at a stop row
// ---------------------------------------------------------------------------
// Everything the draw needs about its stop row.
struct DrawArgs {
  const char* trow;
  const char* drow;  // kResidual only
  int row, kind, xhat;
  float mcp, mcq;
  float bhi, blo;    // beta = S_p / S_q as a double-float pair
  float u2;
  float tau_p, tau_q;  // filter thresholds of the two rows (-inf: unfiltered)
};

__device__ __forceinline__ DrawArgs make_draw_args(const Params& P, size_t rowb, int row, int drow,
                                                   int kind, int xhat, float mcp, float mcq,
                                                   DF Sp, DF Sq) {
  DrawArgs a;
  a.row = row;
  a.trow = static_cast<const char*>(P.target) + (size_t)row * rowb;
  a.drow = kind == kResidual ? static_cast<const char*>(P.draft) + (size_t)drow * rowb : nullptr;
  a.kind = kind;
  a.xhat = xhat;
  a.mcp = mcp;
  a.mcq = mcq;
  const DF beta = (kind == kResidual && df_pos(Sq)) ? df_div(Sp, Sq) : DF{1.f, 0.f};
  a.bhi = beta.hi;
  a.blo = beta.lo;
  a.u2 = __ldg(&P.uniforms[2 * (size_t)row + 1]);
  a.tau_p = P.thr ? __ldg(&P.thr[row]) : -INFINITY;
  a.tau_q = (P.thr_d && kind == kResidual) ? __ldg(&P.thr_d[drow]) : -INFINITY;
  return a;
}

// r for the EPV elements starting at x. kResidual: max(0, e_p - beta e_q)
// with beta = S_p / S_q, i.e. S_p * max(0, p - q); otherwise e_p = S_p * p
// (the rejected one-hot proposal removed).
template <int EPV>
__device__ __forceinline__ void residual_of(const DrawArgs& a, float c, const float (&zp)[EPV],
                                            const float (&zq)[EPV], int x, float (&r)[EPV]) {
#pragma unroll
  for (int j = 0; j < EPV; ++j) {
    const float ep = ex2(fmaf(zp[j], c, -a.mcp));
    if (a.kind == kResidual) {
      const float eq = ex2(fmaf(zq[j], c, -a.mcq));
      float d = fmaf(-eq, a.bhi, ep);
      d = fmaf(-eq, a.blo, d);
      r[j] = fmaxf(d, 0.f);
    } else {
      r[j] = (a.kind == kOneHot && x + j == a.xhat) ? 0.f : ep;
    }
  }
}

// Sums of r over the warp-sized pieces of tiles [tile0, tile0 + ntl): the
// total of tile tile0 + l by warp w goes to s.wtot[l * kWarps + w]. Ends with
// a CTA barrier. Returns false if a bulk copy timed out.
template <int DT, bool VEC>
__device__ bool tile_sums(const Params& P, Smem& s, unsigned char* ring, const DrawArgs& a,
                          int tile0, int ntl) {
  constexpr int EPV = Elem<DT & 1>::kEPV;
  constexpr int TILE = kThreads * EPV;
  const int V = P.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto one_tile = [&](int l, const float (&zp)[EPV], const float (&zq)[EPV]) {
    const int x = (tile0 + l) * TILE + tid * EPV;
    float r[EPV];
    residual_of<EPV>(a, P.c, zp, zq, x, r);
    float ts = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) ts += r[j];
    const float inc = warp_incl_scan(ts, lane);
    if (lane == 31) s.wtot[l * kWarps + warp] = inc;
  };
  if constexpr (VEC) {
    // Tiles of a chunk are kVPT consecutive tiles; tile0 is chunk aligned.
    const size_t off = (size_t)tile0 * TILE * Elem<DT & 1>::kBytes;
    const size_t row_bytes = (size_t)V * Elem<DT & 1>::kBytes;
    size_t len = (size_t)ntl * TILE * Elem<DT & 1>::kBytes;
    if (off + len > row_bytes) len = row_bytes - off;
    const bool res = a.kind == kResidual;
    const bool onehot = a.kind == kOneHot;
    const f2_t cc = f2_splat(P.c), nmcp = f2_splat(-a.mcp), nmcq = f2_splat(-a.mcq);
    const f2_t nbhi = f2_splat(-a.bhi), nblo = f2_splat(-a.blo);
    constexpr int NP = EPV / 2;
    // Last chunk first: the end of the stop row was streamed most recently by
    // the CTA that processed it, so it is the part most likely still in L2.
    return ring_stream(s, ring, a.trow + off, res ? a.drow + off : nullptr, len, true,
                       [&](int k, uint32_t stage) {
      const int xc = (tile0 + k * kVPT) * TILE;  // first element of the chunk
      const bool whole = xc + kVPT * TILE <= V;
      float ts[kVPT];
#pragma unroll
      for (int v = 0; v < kVPT; ++v) {
        f2_t zp[NP], acc = 0ull;
        Raw<DT & 1>::pairs(stage_vector<DT>(stage, xc, V, v, whole, a.tau_p), zp);
        if (res) {
          f2_t zq[NP];
          Raw<DT & 1>::pairs(stage_vector<DT>(stage + kChunkBytes, xc, V, v, whole, a.tau_q), zq);
#pragma unroll
          for (int i = 0; i < NP; ++i) {
            const f2_t ep = f2_ex2(f2_fma(zp[i], cc, nmcp));
            const f2_t eq = f2_ex2(f2_fma(zq[i], cc, nmcq));
            float lo, hi;
            f2_unpack(f2_fma(eq, nblo, f2_fma(eq, nbhi, ep)), lo, hi);
            acc = f2_add(acc, f2_pack(fmaxf(lo, 0.f), fmaxf(hi, 0.f)));
          }
        } else {
          const int xv = xc + (v * kThreads + tid) * EPV;
          const int drop = (onehot && (unsigned)(a.xhat - xv) < (unsigned)EPV) ? a.xhat - xv : -1;
#pragma unroll
          for (int i = 0; i < NP; ++i) {
            f2_t ep = f2_ex2(f2_fma(zp[i], cc, nmcp));
            if ((drop >> 1) == i) {  // the rejected one-hot proposal has no mass
              float lo, hi;
              f2_unpack(ep, lo, hi);
              ep = (drop & 1) ? f2_pack(lo, 0.f) : f2_pack(0.f, hi);
            }
            acc = f2_add(acc, ep);
          }
        }
        float lo, hi;
        f2_unpack(acc, lo, hi);
        ts[v] = lo + hi;
      }
      int t;
      const float tot = warp_tile_totals(ts, lane, t);
      const int l = k * kVPT + t;
      if ((lane & (32 / kVPT - 1)) == 0 && l < ntl) s.wtot[l * kWarps + warp] = tot;
    });
  } else {
    for (int l = 0; l < ntl; ++l) {
      const int x = (tile0 + l) * TILE + tid * EPV;
      float zp[EPV], zq[EPV];
      load_chunk<DT & 1, false>(a.trow, x, V, zp);
      mask_below<DT>(zp, a.tau_p);
      if (a.kind == kResidual) {
        load_chunk<DT & 1, false>(a.drow, x, V, zq);
        mask_below<DT>(zq, a.tau_q);
      }
      one_tile(l, zp, zq);
    }
    __syncthreads();
    return true;
  }
}

// Given this thread's tile sum tt (tile tid < ntiles), finds the tile holding
// u' * Z and rescans it. Returns the token, or -1 if r has no mass.
// Tile k spans [tincl[k-1], tincl[k]) of the inclusive prefix of tile sums,
// so adjacent tiles share their edge; the chosen token is the last index with
// mass whose lower edge is <= u' * Z, which is the smallest k whose running
// sum exceeds u' * Z.
template <int DT, bool VEC>
__device__ int locate_token(const Params& P, Smem& s, const DrawArgs& a, DF tt, int ntiles) {
  constexpr int EPV = Elem<DT & 1>::kEPV;
  constexpr int TILE = kThreads * EPV;
  const int V = P.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const DF inc = warp_incl_scan_df(tt, lane);
  if (lane == 31) s.dred[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    DF v = lane < kWarps ? s.dred[lane] : DF{0.f, 0.f};
    v = warp_incl_scan_df(v, lane);
    if (lane < kWarps) s.dred2[lane] = v;
  }
  __syncthreads();
  if (tid < ntiles) s.tincl[tid] = warp > 0 ? df_add(s.dred2[warp - 1], inc) : inc;
  if (tid == 0) s.pick = -1;
  __syncthreads();
  const DF Z = s.tincl[ntiles - 1];
  if (!df_pos(Z)) return -1;
  DF T = df_mul_f(Z, a.u2);
  if (!(T.hi >= 0.f)) T = DF{0.f, 0.f};  // a NaN or negative uniform draws the first token with mass
  if (tid < ntiles) {
    const DF lo = tid ? s.tincl[tid - 1] : DF{0.f, 0.f};
    if (df_pos(tt) && df_le(lo, T)) atomicMax(&s.pick, tid);
  }
  __syncthreads();
  const int kt = s.pick;
  if (kt < 0) return -1;  // unreachable: the first tile with mass has lower edge 0 <= T
  const DF Tk = kt ? df_sub(T, s.tincl[kt - 1]) : T;

  // The chosen tile: thread k spans [wexcl[w] + lane_lo, wexcl[w] + incl).
  const int x = kt * TILE + tid * EPV;
  float zp[EPV], zq[EPV], r[EPV];
  load_chunk<DT & 1, VEC>(a.trow, x, V, zp);
  mask_below<DT>(zp, a.tau_p);
  if (a.kind == kResidual) {
    load_chunk<DT & 1, VEC>(a.drow, x, V, zq);
    mask_below<DT>(zq, a.tau_q);
  }
  residual_of<EPV>(a, P.c, zp, zq, x, r);
  float ts = 0.f;
#pragma unroll
  for (int j = 0; j < EPV; ++j) ts += r[j];
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
  return s.tok;
}

// Whole draw by one CTA. Returns the token, -1 if r has no mass, -2 on a
// copy timeout.
template <int DT, bool VEC>
__device__ int draw_whole(const Params& P, Smem& s, unsigned char* ring, const DrawArgs& a) {
  constexpr int TILE = kThreads * Elem<DT & 1>::kEPV;
  const int ntiles = (P.V + TILE - 1) / TILE;
  if (!tile_sums<DT, VEC>(P, s, ring, a, 0, ntiles)) return -2;
  DF tt{0.f, 0.f};
  if (threadIdx.x < ntiles)
    for (int w = 0; w < kWarps; ++w) tt = df_add_f(tt, s.wtot[threadIdx.x * kWarps + w]);
  return locate_token<DT, VEC>(P, s, a, tt, ntiles);
}

// Whole draw from a filtered row whose kept logits are listed (n <= one per
// thread): r at the listed tokens (r is 0 off the list, where p is 0), put
// in vocabulary order by rank, then the inverse CDF of locate_token over
// those n values. Returns the token, or -1 if r has no mass.
template <int DT>
__device__ int draw_list(const Params& P, Smem& s, const DrawArgs& a, const int2* ent, int n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Scratch in the tile-sum area, idle outside a streamed draw.
  int* lx = reinterpret_cast<int*>(s.wtot);  // [n] listed tokens
  int* ox = lx + kThreads;                   // [n] tokens in vocabulary order
  float* orr = s.wtot + 2 * kThreads;        // [n] r in vocabulary order
  int x = INT_MAX;
  float r = 0.f;
  if (tid < n) {
    const int2 e = __ldcg(ent + tid);
    x = e.x;
    const float ep = ex2(fmaf(__int_as_float(e.y), P.c, -a.mcp));
    if (a.kind == kResidual) {
      const float zq = mask_below<DT>(Elem<DT & 1>::scalar(a.drow, x), a.tau_q);
      const float eq = ex2(fmaf(zq, P.c, -a.mcq));
      float d = fmaf(-eq, a.bhi, ep);
      d = fmaf(-eq, a.blo, d);
      r = fmaxf(d, 0.f);
    } else {
      r = (a.kind == kOneHot && x == a.xhat) ? 0.f : ep;
    }
    lx[tid] = x;
  }
  if (tid == 0) s.pick = -1;
  __syncthreads();
  if (tid < n) {
    int rank = 0;  // tokens are distinct
    for (int j = 0; j < n; ++j) rank += lx[j] < x ? 1 : 0;
    ox[rank] = x;
    orr[rank] = r;
  }
  __syncthreads();
  const float rv = tid < n ? orr[tid] : 0.f;
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
  int y = -1;
  if (df_pos(Z)) {
    DF T = df_mul_f(Z, a.u2);
    if (!(T.hi >= 0.f)) T = DF{0.f, 0.f};  // a NaN or negative uniform draws the first token with mass
    if (tid < n && rv > 0.f && df_le(lo, T)) atomicMax(&s.pick, tid);
    __syncthreads();
    y = s.pick >= 0 ? ox[s.pick] : -1;
  }
  __syncthreads();  // the scratch is free again
  return y;
}

// Writes the drawn token and (p(y), q(y)) (thread 0).
template <int DT>
__device__ void finish_draw(const Params& P, const DrawArgs& a, DF Sp, DF Sq, int y,
                            int bonus_row) {
  float qy;
  const float zp = mask_below<DT>(Elem<DT & 1>::scalar(a.trow, y), a.tau_p);
  const float py = __fdiv_rn(exp2f(fmaf(zp, P.c, -a.mcp)), Sp.hi);
  if (a.kind == kResidual) {
    const float zq = mask_below<DT>(Elem<DT & 1>::scalar(a.drow, y), a.tau_q);
    qy = __fdiv_rn(exp2f(fmaf(zq, P.c, -a.mcq)), Sq.hi);
  } else if (a.kind == kOneHot) {
    qy = (y == a.xhat) ? 1.f : 0.f;
  } else {
    qy = 0.f;
  }
  P.out_tokens[a.row] = y;
  if (P.out_probs) {
    P.out_probs[2 * (size_t)bonus_row] = py;
    P.out_probs[2 * (size_t)bonus_row + 1] = qy;
  }
}

// Hands out one part of a published draw (thread 0); nothing here waits.
// Slots are scanned from the head, which moves past every leading slot whose
// parts are all handed out.
__device__ bool claim_draw_part(const Params& P, int& slot_out, int& part_out) {
  unsigned n = ld_relaxed_gpu(&P.ws->n_draws);
  if (n > (unsigned)P.n_slots) n = (unsigned)P.n_slots;
  const unsigned h = ld_relaxed_gpu(&P.ws->draw_head);
  unsigned adv = h;
  bool leading = true;
  for (unsigned i = h; i < n; ++i) {
    const unsigned v = ld_acquire_gpu(&P.slot_state[i]);
    const unsigned np = v >> kSlotCountBits;
    if (np == 0u) {  // reserved, not yet published
      leading = false;
      continue;
    }
    if ((v & kSlotCountMask) < np) {
      const unsigned pt = atomicAdd(&P.slot_state[i], 1u) & kSlotCountMask;
      if (pt < np) {
        if (leading && pt + 1u == np) adv = i + 1;
        if (adv > h) atomicMax(&P.ws->draw_head, adv);
        slot_out = (int)i;
        part_out = (int)pt;
        return true;
      }
    }
    if (leading) adv = i + 1;
  }
  if (adv > h) atomicMax(&P.ws->draw_head, adv);
  return false;
}

// One part of the draw in `slot`: sums of r over the part's tiles go to the
// workspace; the CTA that finishes the draw's last part locates the token.
// Returns false if a bulk copy timed out.
template <int DT, bool VEC>
__device__ __noinline__ bool draw_part(const Params& P, Smem& s, unsigned char* ring, int slot,
                                       int part) {
  constexpr int TILE = kThreads * Elem<DT & 1>::kEPV;
  const int tid = threadIdx.x;
  const DrawDesc* d = &P.descs[slot];
  const DF Sp = ldcg_df(&d->Sp), Sq = ldcg_df(&d->Sq);
  const int kind = __ldcg(&d->kind);
  const DrawArgs a = make_draw_args(P, (size_t)P.V * Elem<DT & 1>::kBytes, __ldcg(&d->row),
                                    __ldcg(&d->drow), kind, __ldcg(&d->xhat), __ldcg(&d->mcp),
                                    __ldcg(&d->mcq), Sp, Sq);
  const int nparts = __ldcg(&d->nparts);
  const int ntiles = (P.V + TILE - 1) / TILE;
  // Parts are whole ring chunks (kVPT tiles each).
  const int nchunks = (ntiles + kVPT - 1) / kVPT;
  const int cpp = (nchunks + nparts - 1) / nparts;
  const int tile0 = part * cpp * kVPT;
  const int tile1 = min(ntiles, (part + 1) * cpp * kVPT);
  const int ntl = tile1 - tile0;
  DF* tsum = P.tsum + (size_t)slot * P.tsum_stride;
  if (ntl > 0) {
    if (!tile_sums<DT, VEC>(P, s, ring, a, tile0, ntl)) return false;
    if (tid < ntl) {
      DF tt{0.f, 0.f};
      for (int w = 0; w < kWarps; ++w) tt = df_add_f(tt, s.wtot[tid * kWarps + w]);
      tsum[tile0 + tid] = tt;
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&P.descs[slot].done, 1u);
    s.last = (old == (unsigned)nparts - 1u) ? 1 : 0;
  }
  __syncthreads();
  if (!s.last) return true;
  // Last part: every tile sum is in the workspace.
  __threadfence();
  const DF tt = tid < ntiles ? ldcg_df(&tsum[tid]) : DF{0.f, 0.f};
  int y = locate_token<DT, VEC>(P, s, a, tt, ntiles);
  DrawArgs used = a;
  if (y < 0 && kind != kBonus) {
    // No residual mass (p == q in fp32): draw from p instead.
    if (tid == 0) atomicOr(&P.ws->status, SV_DATA_DEGENERATE_RESIDUAL);
    used.kind = kBonus;
    used.bhi = 1.f;
    used.blo = 0.f;
    y = draw_whole<DT, VEC>(P, s, ring, used);
    if (y == -2) return false;
  }
  if (y < 0) {
    if (tid == 0) atomicOr(&P.ws->status, SV_DATA_EMPTY_ROW);
    y = 0;
  }
  if (tid == 0) finish_draw<DT>(P, a, Sp, Sq, y, __ldcg(&d->bonus_row));
  return true;
}

// Commit of request b by the CTA that finished its last row: stop slot,
// accepted drafts, length and the final token (the argmax for a greedy
// request, the draw for a sampled one). Returns false if a bulk copy timed out.
template <int DT, bool VEC>
__device__ __noinline__ bool commit_request(const Params& P, Smem& s, unsigned char* ring, int b,
                                            int t0, int d0, int K, bool greedy) {
  const int tid = threadIdx.x;
  const int stop = s.stop;  // set by the row that decided it (its update acquired the rows' records)
  for (int j = tid; j < stop; j += kThreads) P.out_tokens[t0 + j] = P.draft_tokens[d0 + j];
  const int srow = t0 + stop;
  if (tid == 0) P.out_len[b] = stop + 1;
  if (greedy) {
    if (tid == 0) {
      atomicAdd(&P.ws->committed, 1u);
      P.out_tokens[srow] = __ldcg(&P.rows[srow].argmax);
      if (P.out_probs) {
        P.out_probs[2 * (size_t)(t0 + K)] = -1.f;
        P.out_probs[2 * (size_t)(t0 + K) + 1] = -1.f;
      }
    }
    return true;
  }
  int kind = kBonus, xhat = -1, drow = -1;
  if (stop < K) {
    xhat = P.draft_tokens[d0 + stop];
    if (xhat < 0 || xhat >= P.V) xhat = -1;
    if (P.draft) {
      kind = kResidual;
      drow = d0 + stop;
    } else {
      kind = kOneHot;
    }
  }
  const DF Sp = ldcg_df(&P.rows[srow].S_p), Sq = ldcg_df(&P.rows[srow].S_q);
  const float mcp = __ldcg(&P.rows[srow].mc_p), mcq = __ldcg(&P.rows[srow].mc_q);
  if constexpr (VEC && (DT & kFilt) != 0) {
    // A filtered stop row with its kept logits listed: the draw reads the
    // list (and the draft row at the listed tokens), not the rows.
    const int nl = P.flist ? __ldcg(&P.fst[srow].nl) : 0;
    if (nl > 0 && nl <= kThreads) {
      if (tid == 0) atomicAdd(&P.ws->committed, 1u);
      const DrawArgs a = make_draw_args(P, (size_t)P.V * Elem<DT & 1>::kBytes, srow, drow, kind, xhat,
                                        mcp, mcq, Sp, Sq);
      const int2* ent = P.flist + (size_t)srow * kKeptListCap;
      int y = draw_list<DT>(P, s, a, ent, nl);
      if (y < 0 && kind != kBonus) {
        // No residual mass (p == q in fp32): draw from p instead.
        if (tid == 0) atomicOr(&P.ws->status, SV_DATA_DEGENERATE_RESIDUAL);
        DrawArgs used = a;
        used.kind = kBonus;
        used.bhi = 1.f;
        used.blo = 0.f;
        y = draw_list<DT>(P, s, used, ent, nl);
      }
      if (y < 0) {
        if (tid == 0) atomicOr(&P.ws->status, SV_DATA_EMPTY_ROW);
        y = 0;
      }
      if (tid == 0) finish_draw<DT>(P, a, Sp, Sq, y, t0 + K);
      return true;
    }
  }
  if (VEC && (kind == kBonus || kind == kOneHot) && (__ldcg(&P.rows[srow].accept) & 2u)) {
    // The stop row left the tile sums of r (a bonus row: p; a one-hot row:
    // p without x̂): only the chosen tile is read again.
    if (tid == 0) atomicAdd(&P.ws->committed, 1u);
    const DrawArgs a = make_draw_args(P, (size_t)P.V * Elem<DT & 1>::kBytes, srow, drow, kind, xhat,
                                      mcp, mcq, Sp, Sq);
    constexpr int EPV = Elem<DT & 1>::kEPV;
    constexpr int TILE = kThreads * EPV;
    const int ntiles = (P.V + TILE - 1) / TILE;
    DF tt{tid < ntiles ? __ldcg(&P.rtile[(size_t)srow * P.tsum_stride + tid]) : 0.f, 0.f};
    if (kind == kOneHot && xhat >= 0) {
      // The row's tiles hold every term of p; x̂'s tile is summed again
      // without x̂ (afresh, so a dominant x̂ leaves no rounding behind).
      const int lx = xhat / TILE;
      float z[EPV], r[EPV];
      load_chunk<DT & 1, VEC>(a.trow, lx * TILE + tid * EPV, P.V, z);
      mask_below<DT>(z, a.tau_p);
      residual_of<EPV>(a, P.c, z, z, lx * TILE + tid * EPV, r);
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < EPV; ++j) m += r[j];
      const DF w = warp_sum_df(DF{m, 0.f});
      if ((tid & 31) == 0) s.reddf_p[tid >> 5] = w;
      __syncthreads();
      if (tid == lx) {
        DF sum = s.reddf_p[0];
        for (int k = 1; k < kWarps; ++k) sum = df_add(sum, s.reddf_p[k]);
        tt = sum;
      }
      __syncthreads();
    }
    int y = locate_token<DT, VEC>(P, s, a, tt, ntiles);
    if (y < 0 && kind == kOneHot) {
      // No mass besides x̂: draw from p instead.
      if (tid == 0) atomicOr(&P.ws->status, SV_DATA_DEGENERATE_RESIDUAL);
      DrawArgs used = a;
      used.kind = kBonus;
      y = draw_whole<DT, VEC>(P, s, ring, used);
      if (y == -2) return false;
    }
    if (y < 0) {
      if (tid == 0) atomicOr(&P.ws->status, SV_DATA_EMPTY_ROW);
      y = 0;
    }
    if (tid == 0) finish_draw<DT>(P, a, Sp, Sq, y, t0 + K);
    return true;
  }
  // Once the rows left fit in one wave, CTAs are about to fall idle: publish
  // the draw in parts so that they can share it, and take parts of it here.
  // The request counts as committed only once its draw is published (or
  // kept whole here), so that idle CTAs linger until they can take parts.
  if (tid == 0) {
    constexpr int TILE = kThreads * Elem<DT & 1>::kEPV;
    const int nchunks = ((P.V + TILE - 1) / TILE + kVPT - 1) / kVPT;
    // Draws published here come due after the last rows are handed out, when
    // CTAs fall idle: single-chunk parts spread them widest (kPartChunks; 4
    // measured 0.6% slower on the benchmark batch), up to kMaxParts.
    int nparts = (nchunks + kPartChunks - 1) / kPartChunks;
    nparts = nparts > kMaxParts ? kMaxParts : nparts;
    // Parts carry a fixed cost (descriptor, ring start, a global merge); a
    // draw that streams less than kMinPublishBytes is faster kept whole.
    const size_t draw_bytes = (size_t)P.V * Elem<DT & 1>::kBytes * (kind == kResidual ? 2 : 1);
    s.slot = -1;
    if (nparts > 1 && draw_bytes >= kMinPublishBytes &&
        ld_relaxed_gpu(&P.ws->next_item) + gridDim.x + kPublishPct * gridDim.x / 100u >= s.n_items) {
      const unsigned slot = atomicAdd(&P.ws->n_draws, 1u);
      if (slot < (unsigned)P.n_slots) {
        DrawDesc* d = &P.descs[slot];
        d->b = b;
        d->row = srow;
        d->drow = drow;
        d->kind = kind;
        d->xhat = xhat;
        d->mcp = mcp;
        d->mcq = mcq;
        d->nparts = nparts;
        d->Sp = Sp;
        d->Sq = Sq;
        d->bonus_row = t0 + K;
        __threadfence();
        st_release_gpu(&P.slot_state[slot], (unsigned)nparts << kSlotCountBits);
        s.slot = (int)slot;
      }
    }
    atomicAdd(&P.ws->committed, 1u);
  }
  __syncthreads();
  if (s.slot >= 0) {
    const int slot = s.slot;
    for (;;) {
      __syncthreads();
      if (tid == 0) s.part = (int)(atomicAdd(&P.slot_state[slot], 1u) & kSlotCountMask);
      __syncthreads();
      const int part = s.part;
      if (part >= __ldcg(&P.descs[slot].nparts)) break;
      if (!draw_part<DT, VEC>(P, s, ring, slot, part)) return false;
    }
    return true;
  }
  const DrawArgs a = make_draw_args(P, (size_t)P.V * Elem<DT & 1>::kBytes, srow, drow, kind, xhat, mcp,
                                    mcq, Sp, Sq);
  int y = draw_whole<DT, VEC>(P, s, ring, a);
  if (y == -2) return false;
  DrawArgs used = a;
  if (y < 0 && kind != kBonus) {
    // No residual mass (p == q in fp32): draw from p instead.
    if (tid == 0) atomicOr(&P.ws->status, SV_DATA_DEGENERATE_RESIDUAL);
    used.kind = kBonus;
    used.bhi = 1.f;
    used.blo = 0.f;
    y = draw_whole<DT, VEC>(P, s, ring, used);
    if (y == -2) return false;
  }
  if (y < 0) {
    if (tid == 0) atomicOr(&P.ws->status, SV_DATA_EMPTY_ROW);
    y = 0;
  }
  if (tid == 0) finish_draw<DT>(P, a, Sp, Sq, y, t0 + K);
  return true;
}

__device__ __forceinline__ int t0_of(const Params& P, int b) { return P.cu[b] + b; }

// Request progress. With K <= kMaxTrackedK draft slots the word holds one
// "done" bit per target row (bits 0..K) and one "accepted" bit per draft
// slot (bits 32..32+K-1), so the stop slot is known as soon as the rows up to
// it are done -- later rows may still be streaming. With more slots it
// counts finished rows and the request commits when all are done.
constexpr int kMaxTrackedK = 31;

// Stop slot decided by a progress word (tracked requests), or -1.
__device__ __forceinline__ int stop_from_state(unsigned long long st, int K) {
  for (int i = 0; i < K; ++i) {
    if (!((st >> i) & 1ull)) return -1;         // slot i not decided yet
    if (!((st >> (32 + i)) & 1ull)) return i;   // first rejection
  }
  return ((st >> K) & 1ull) ? K : -1;           // all accepted: needs the bonus row
}

// Run by warp 0: the row at position o of the work order, of request b.
__device__ __noinline__ void row_meta(const Params& P, Smem& s, int o, int b) {
  const int lane = threadIdx.x & 31;
  int t;
  if (!kBonusLast)
    t = o;
  else if (o < s.R_d)  // draft-slot rows first, in order
    t = o + b;
  else                 // then the bonus rows
    t = P.cu[b + 1] + b;
  // The accept uniform is needed only after the row pass: load it now.
  const float u = (lane == 0 && P.uniforms) ? __ldg(&P.uniforms[2 * (size_t)t]) : 0.f;
  if (lane != 0) return;
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
  s.u_acc = u;
  s.zx_ok = 0;
  s.tau_t = P.thr ? __ldg(&P.thr[t]) : -INFINITY;
  s.tau_d = (P.thr_d && i < K) ? __ldg(&P.thr_d[d0 + i]) : -INFINITY;
  s.btile_ok = 0;
  s.b = b;
  s.t = t;
  s.t0 = t0;
  s.d0 = d0;
  s.K = K;
  s.i = i;
  s.greedy = greedy;
  s.xhat = xhat;
}

// Statistics of chunks [c0, c1) of a row (and its paired draft row): the
// online softmax (sampled rows) or the argmax (greedy rows), combined over
// the CTA into `st` (valid in thread 0). Returns false on a copy timeout.
template <int DT, bool VEC>
__device__ bool slice_stats(const Params& P, Smem& s, unsigned char* ring, const char* trow,
                            const char* drow, bool greedy, int c0, int c1, PartRec& st,
                            bool btiles, int t) {
  constexpr int EPV = Elem<DT & 1>::kEPV;
  constexpr int CH = kChunkBytes / Elem<DT & 1>::kBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V;
  const size_t rowb = (size_t)V * Elem<DT & 1>::kBytes;
  const size_t off = (size_t)c0 * kChunkBytes;
  const size_t end = (size_t)c1 * kChunkBytes < rowb ? (size_t)c1 * kChunkBytes : rowb;
  const size_t len = end > off ? end - off : 0;
  const int x0 = c0 * CH;  // first element of the slice
  bool ok = true;
  if (greedy) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if constexpr (VEC) {
      ok = ring_stream(s, ring, trow + off, nullptr, len, false, [&](int k, uint32_t stage) {
        uint4 rv[kVPT];
        stage_vectors<DT>(stage, x0 + k * CH, V, rv, s.tau_t);
        const float cm = Raw<DT & 1>::template max_of<kVPT>(rv);
        if (cm > bv) {
          // A new maximum: its first occurrence in this thread's elements,
          // which it visits in increasing index order.
          int first = 0x7fffffff;
#pragma unroll
          for (int v = kVPT - 1; v >= 0; --v) {
            float f[EPV];
            Elem<DT & 1>::unpack(rv[v], f);
#pragma unroll
            for (int j = EPV - 1; j >= 0; --j)
              if (f[j] == cm) first = x0 + k * CH + (v * kThreads + tid) * EPV + j;
          }
          bv = cm;
          bi = first;
        }
      });
    } else {
      argmax_scalar<DT>(trow, V, bv, bi);
    }
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
        st.mc_p = st.mc_q = 0.f;
        st.S_p = st.S_q = DF{0.f, 0.f};
        st.amax_v = v;
        st.amax_i = ix;
      }
    }
  } else {
    SoftAcc<EPV> at, ad;
    at.init();
    ad.init();
    const bool has_d = drow != nullptr;
    if constexpr (VEC) {
      // The thread whose vector holds the proposed token keeps its logits
      // for the accept test, so that test needs no global load.
      const int xh = s.xhat;
      int kx = -1, vx = 0, jx = 0;
      if (xh >= x0 && (size_t)(xh - x0) < len / Elem<DT & 1>::kBytes) {
        const int e = xh - x0;
        kx = e / CH;
        const int vi = (e - kx * CH) / EPV;
        vx = vi / kThreads;
        jx = (e - kx * CH) % EPV;
        if (vi % kThreads != tid) kx = -1;
      }
      // A row streamed alone (a bonus row, or a one-hot draft slot) also
      // leaves, per tile and warp, the sum of its draw's terms relative to a
      // per-chunk warp offset, in the draw's scratch (idle during a row pass):
      // r = 2^(z c - mc), without x̂ for a one-hot slot, so that a draw at
      // this row reads none of it again.
      float* bref = reinterpret_cast<float*>(s.tincl);  // [chunk][warp] offsets
      constexpr int TILE = kThreads * EPV;
      const int ntiles = (V + TILE - 1) / TILE;
      if (btiles) {
        ok = ring_stream(s, ring, trow + off, nullptr, len, false, [&](int k, uint32_t stage) {
          uint4 rv[kVPT];
          stage_vectors<DT>(stage, x0 + k * CH, V, rv, s.tau_t);
          float tv[kVPT];
          at.template add_raw_tiles<DT, kVPT>(rv, P.c, tv);
          const bool live = at.m != -INFINITY;
          const float ref = warp_max(live ? at.mc : -INFINITY);
          const float f = live ? ex2(at.mc - ref) : 0.f;
#pragma unroll
          for (int v = 0; v < kVPT; ++v) tv[v] *= f;
          int t;
          const float tot = warp_tile_totals(tv, lane, t);
          const int l = (c0 + k) * kVPT + t;  // tile of the row (a part starts at chunk c0)
          if ((lane & (32 / kVPT - 1)) == 0 && l < ntiles) s.wtot[l * kWarps + warp] = tot;
          if (lane == 0) bref[k * kWarps + warp] = ref;
        });
      } else {
        ok = ring_stream(s, ring, trow + off, has_d ? drow + off : nullptr, len, false,
                         [&](int k, uint32_t stage) {
          uint4 rv[kVPT];
          stage_vectors<DT>(stage, x0 + k * CH, V, rv, s.tau_t);
          if (k == kx) {
            s.zx_p = pick_element<DT>(rv, vx, jx);
            s.zx_ok = 1;
          }
          if (any_kept<DT>(rv)) at.template add_raw<DT, kVPT>(rv, P.c);
          if (has_d) {
            stage_vectors<DT>(stage + kChunkBytes, x0 + k * CH, V, rv, s.tau_d);
            if (k == kx) s.zx_q = pick_element<DT>(rv, vx, jx);
            if (any_kept<DT>(rv)) ad.template add_raw<DT, kVPT>(rv, P.c);
          }
        });
      }
    } else {
      if (has_d)
        stats_pass_scalar<DT, true>(trow, drow, V, P.c, at, ad, s.tau_t, s.tau_d);
      else
        stats_pass_scalar<DT, false>(trow, drow, V, P.c, at, ad, s.tau_t, s.tau_d);
    }
    float mcp, mcq;
    DF Sp, Sq;
    combine_softmax<EPV>(at, ad, has_d, P.c, s, mcp, Sp, mcq, Sq);
    if (VEC && btiles && ok) {
      // Tile sums of r = 2^(z c - mc_p) over this slice's tiles: each warp's
      // part rescaled from its chunk offset to the slice's, summed over the
      // warps in double-float. (A split row's merge rescales them to the row's.)
      if (tid == 0) s.bcast_f[0] = mcp;
      __syncthreads();
      const float M = s.bcast_f[0];
      constexpr int TILE = kThreads * EPV;
      const int ntiles = (V + TILE - 1) / TILE;
      const float* bref = reinterpret_cast<const float*>(s.tincl);
      const int l = c0 * kVPT + tid;
      if (tid < (c1 - c0) * kVPT && l < ntiles) {
        const int k = tid / kVPT;
        DF T{0.f, 0.f};
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float r = bref[k * kWarps + w];
          if (r > -INFINITY) T = df_add_f(T, s.wtot[l * kWarps + w] * ex2(r - M));
        }
        P.rtile[(size_t)t * P.tsum_stride + l] = T.hi + T.lo;
        __threadfence();  // visible to a split row's merging CTA before this part counts as done
      }
      if (tid == 0) s.btile_ok = 1;
      __syncthreads();
    }
    if (tid == 0) {
      st.mc_p = mcp;
      st.mc_q = mcq;
      st.S_p = Sp;
      st.S_q = Sq;
      st.amax_v = -INFINITY;
      st.amax_i = 0x7fffffff;
    }
  }
  return ok;
}

// Merges the statistics of a split row's n <= 32 parts, one part per lane of
// the calling warp; the result is valid in lane 0. The offset is the largest
// exponent offset of the parts with mass, each part's sum is rescaled to it
// by 2^(mc_r - mc) (the fp32 exponential the whole-row combine also uses) and
// summed in double-float; greedy rows take the largest logit, lowest index on ties.
__device__ __noinline__ PartRec merge_parts(const PartRec* parts, int n) {
  const int lane = threadIdx.x & 31;
  float mp = 0.f, mq = 0.f, av = -INFINITY;
  DF sp{0.f, 0.f}, sq{0.f, 0.f};
  int ai = 0x7fffffff;
  if (lane < n) {
    mp = __ldcg(&parts[lane].mc_p);
    mq = __ldcg(&parts[lane].mc_q);
    sp = ldcg_df(&parts[lane].S_p);
    sq = ldcg_df(&parts[lane].S_q);
    av = __ldcg(&parts[lane].amax_v);
    ai = __ldcg(&parts[lane].amax_i);
  }
  const bool hp = df_pos(sp), hq = df_pos(sq);
  const float Mp = warp_max(hp ? mp : -INFINITY), Mq = warp_max(hq ? mq : -INFINITY);
  DF wp = hp ? df_mul_f(sp, ex2(mp - Mp)) : DF{0.f, 0.f};
  DF wq = hq ? df_mul_f(sq, ex2(mq - Mq)) : DF{0.f, 0.f};
  wp = warp_sum_df(wp);
  wq = warp_sum_df(wq);
  warp_argmax(av, ai);
  PartRec m;
  m.mc_p = Mp == -INFINITY ? 0.f : Mp;
  m.mc_q = Mq == -INFINITY ? 0.f : Mq;
  m.S_p = wp;
  m.S_q = wq;
  m.amax_v = av;
  m.amax_i = ai;
  return m;
}

template <int DT>
__device__ __noinline__ void decide_row(const Params& P, Smem& s, int t, const PartRec& st) {
  const int b = s.b, d0 = s.d0, K = s.K, i = s.i, xhat = s.xhat;
  const bool greedy = s.greedy != 0;
  const size_t rowb = (size_t)P.V * Elem<DT & 1>::kBytes;
  const char* trow = static_cast<const char*>(P.target) + (size_t)t * rowb;
  const bool has_d = !greedy && i < K && P.draft != nullptr;
  const char* drow = has_d ? static_cast<const char*>(P.draft) + (size_t)(d0 + i) * rowb : nullptr;
  RowRec rec;
  if (greedy) {
    const int am = (st.amax_i == 0x7fffffff) ? 0 : st.amax_i;  // all -inf: index 0, like argmax
    rec.mc_p = rec.mc_q = 0.f;
    rec.S_p = rec.S_q = DF{0.f, 0.f};
    rec.argmax = am;
    rec.accept = (i < K && xhat == am) ? 1u : 0u;
    if (P.out_probs && i < K) {
      P.out_probs[2 * (size_t)t] = -1.f;
      P.out_probs[2 * (size_t)t + 1] = -1.f;
    }
  } else {
    const float mcp = st.mc_p, mcq = st.mc_q;
    const DF Sp = st.S_p, Sq = st.S_q;
    rec.mc_p = mcp;
    rec.mc_q = mcq;
    rec.S_p = Sp;
    rec.S_q = Sq;
    rec.argmax = 0;
    rec.accept = (i == K && s.btile_ok) ? 3u : 1u;  // bonus rows count as accepted
    if (!df_pos(Sp) || (has_d && !df_pos(Sq))) atomicOr(&P.ws->status, SV_DATA_EMPTY_ROW);
    if (i < K) {
      float ph = -1.f, qh = -1.f;
      unsigned acc = 0u;
      if (xhat >= 0) {
        // p(x̂) = 2^(z c - mc_p) / S_p, and min(1, p/q) with q from the
        // draft row or q = 1 for a one-hot proposal.
        const float zp = s.zx_ok ? s.zx_p : mask_below<DT>(Elem<DT & 1>::scalar(trow, xhat), s.tau_t);
        const float ap = fmaf(zp, P.c, -mcp);
        // In fp32: p(x̂), q(x̂) and rho come out to a few ulp (about 2e-7 at
        // most), far inside the 1e-6 within which a decision counts as a tie
        // with the float64 evaluation; fp64 divisions cost this step more on
        // this part than the bytes it saves.
        const float Spf = Sp.hi, Sqf = Sq.hi;
        const float pd = __fdiv_rn(exp2f(ap), Spf);
        float rho, qd = 1.f;
        if (has_d) {
          const float zq = s.zx_ok ? s.zx_q : mask_below<DT>(Elem<DT & 1>::scalar(drow, xhat), s.tau_d);
          const float aq = fmaf(zq, P.c, -mcq);
          qd = __fdiv_rn(exp2f(aq), Sqf);
          rho = (zq == -INFINITY) ? 0.f : fminf(1.f, __fmul_rn(exp2f(ap - aq), __fdiv_rn(Sqf, Spf)));
        } else {
          rho = fminf(1.f, pd);
        }
        acc = (s.u_acc < rho) ? 1u : 0u;
        ph = pd;
        qh = qd;
      }
      rec.accept = acc | (s.btile_ok ? 2u : 0u);
      if (P.out_probs) {
        P.out_probs[2 * (size_t)t] = ph;
        P.out_probs[2 * (size_t)t + 1] = qh;
      }
    }
  }
  P.rows[t] = rec;
  // s.last: this row makes the request's stop slot known (commit here);
  // s.stop: that slot. The progress update releases this row's record and
  // acquires those of the rows counted before it (read by the commit).
  s.last = 0;
  if (K <= kMaxTrackedK) {
    const unsigned long long add = (1ull << i) | ((rec.accept & 1u) && i < K ? 1ull << (32 + i) : 0ull);
    const unsigned long long old = atom_or_acqrel_gpu(&P.req_state[b], add);
    const unsigned long long now = old | add;
    const int stop = stop_from_state(now, K);
    if (stop >= 0 && stop_from_state(old, K) < 0) {
      s.last = 1;
      s.stop = stop;
    }
    const unsigned long long all = (K + 1 == 64) ? ~0ull : ((1ull << (K + 1)) - 1ull);
    if ((now & all) == all) P.req_state[b] = 0ull;  // every row is in: reset for the next call
  } else {
    const unsigned long long old = atom_add_acqrel_gpu(&P.req_state[b], 1ull);
    if (old == (unsigned long long)K) {
      int stop = K;
      for (int j = 0; j < K; ++j)
        if ((__ldcg(&P.rows[t0_of(P, b) + j].accept) & 1u) == 0u) {
          stop = j;
          break;
        }
      s.last = 1;
      s.stop = stop;
      P.req_state[b] = 0ull;
    }
  }
}

// One work item: a whole row (part < 0) or part `part` of split row t, whose
// index among the split rows is `split`. Returns false on a copy timeout.
template <int DT, bool VEC>
__device__ bool process_item(const Params& P, Smem& s, unsigned char* ring, int o, int part,
                             int split) {
  const int tid = threadIdx.x;
  // The row's request: the whole CTA searches the offsets.
  const int bq = !kBonusLast ? find_request_cta(P.cu, P.B, o, true)
                 : (o < s.R_d ? find_request_cta(P.cu, P.B, o, false) : o - s.R_d);
  if (tid < 32) row_meta(P, s, o, bq);
  __syncthreads();
  const int b = s.b, t = s.t, t0 = s.t0, d0 = s.d0, K = s.K, i = s.i;
  if constexpr ((DT & kFilt) != 0) {
    if (P.fc_done && P.fc_done[b]) {
      // Committed by the filtered commit: counted once, by its first row.
      if (tid == 0 && i == 0 && part <= 0) atomicAdd(&P.ws->committed, 1u);
      return true;
    }
  }
  const bool greedy = s.greedy != 0;
  const size_t rowb = (size_t)P.V * Elem<DT & 1>::kBytes;
  const char* trow = static_cast<const char*>(P.target) + (size_t)t * rowb;
  const bool has_d = !greedy && i < K && P.draft != nullptr;
  const char* drow = has_d ? static_cast<const char*>(P.draft) + (size_t)(d0 + i) * rowb : nullptr;
  const int nch = (int)((rowb + kChunkBytes - 1) / kChunkBytes);
  int c0 = 0, c1 = nch;
  const int np = (int)s.row_parts;
  if (part >= 0) {
    const int cpp = (nch + np - 1) / np;
    c0 = min(nch, part * cpp);
    c1 = min(nch, c0 + cpp);
  }
  PartRec st;
  // Rows streamed alone keep their draw's tile sums: bonus rows, and draft
  // slots with one-hot proposals (no draft row).
  const bool btiles = VEC && P.rtile != nullptr && !greedy && (i == K || !has_d);
  bool pre = false;
  if constexpr ((DT & kFilt) != 0) {
    // A whole filtered row whose threshold kernel left its statistics (and
    // its draft row's) is not read again: the accept test needs only z(x̂)
    // of each row, two scalar loads.
    if (part < 0 && P.fst) {
      if (tid == 0) {
        const FStat ft = P.fst[t];
        FStat fd{};
        fd.ok = 1;
        if (has_d) fd = P.fst_d[d0 + i];
        int ok = !greedy && ft.ok && fd.ok;
        if (ok) {
          st.mc_p = ft.mc;
          st.S_p = df_from_d(ft.S);
          st.mc_q = has_d ? fd.mc : 0.f;
          st.S_q = has_d ? df_from_d(fd.S) : DF{0.f, 0.f};
          st.amax_v = -INFINITY;
          st.amax_i = 0x7fffffff;
          const int xh = s.xhat;
          if (i < K && xh >= 0) {
            s.zx_p = mask_below<DT>(Elem<DT & 1>::scalar(trow, xh), s.tau_t);
            if (has_d) s.zx_q = mask_below<DT>(Elem<DT & 1>::scalar(drow, xh), s.tau_d);
            s.zx_ok = 1;
          }
        }
        s.pre = ok;
      }
      __syncthreads();
      pre = s.pre != 0;
    }
  }
  if (!pre && !slice_stats<DT, VEC>(P, s, ring, trow, drow, greedy, c0, c1, st, btiles, t)) return false;
  if (part >= 0) {
    if (tid == 0) {
      P.parts[(size_t)split * np + part] = st;
      const unsigned old = atom_add_acqrel_gpu(&P.part_done[split], 1u);
      s.merge = (old == (unsigned)np - 1u) ? 1 : 0;  // this CTA merges the row
      if (s.merge) P.part_done[split] = 0u;
    }
    __syncthreads();
    if (!s.merge) return true;
    if (tid < 32) {
      const PartRec m = merge_parts(P.parts + (size_t)split * np, np);
      if (tid == 0) {
        st = m;
        s.bcast_f[0] = m.mc_p;
      }
    }
    if (btiles) {
      // Each part left its tiles' sums relative to its own offset: rescale
      // them to the merged one, as merge_parts does with the parts' sums.
      __syncthreads();
      const float M = s.bcast_f[0];
      constexpr int TILE = kThreads * Elem<DT & 1>::kEPV;
      const int ntiles = (P.V + TILE - 1) / TILE;
      const int cpp = (nch + np - 1) / np;
      for (int l = tid; l < ntiles; l += kThreads) {
        const PartRec* pr = P.parts + (size_t)split * np + (l / kVPT) / cpp;
        const DF Sp_part = ldcg_df(&pr->S_p);
        const float f = df_pos(Sp_part) ? ex2(__ldcg(&pr->mc_p) - M) : 0.f;
        float* bt = P.rtile + (size_t)t * P.tsum_stride + l;
        *bt = __ldcg(bt) * f;
      }
      if (tid == 0) s.btile_ok = 1;
    }
  }
  if (tid == 0) decide_row<DT>(P, s, t, st);
  __syncthreads();
  bool ok = true;
  if (s.last) ok = commit_request<DT, VEC>(P, s, ring, b, t0, d0, K, greedy);
  __syncthreads();
  return ok;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, SV_MINBLOCKS) verify_kernel(Params P) {
  __shared__ Smem s;
  extern __shared__ __align__(128) unsigned char ring[];
  const int tid = threadIdx.x;
  // The filtered commit finished every request: nothing is left.
  if ((DT & kFilt) != 0 && P.fc_need && __ldcg(P.fc_need) == 0u) return;
  // Offsets must be a valid packed layout that fits the workspace; every CTA
  // checks and all of them take the same decision.
  bool bad = false;
  for (int k = tid; k < P.B; k += kThreads)
    if (P.cu[k + 1] < P.cu[k]) bad = true;
  if (tid == 0) {
    if (P.cu[0] != 0) bad = true;
    if ((long long)P.cu[P.B] + P.B > P.row_cap) bad = true;
    if constexpr (VEC) {
      for (int j = 0; j < kStages; ++j) {
        mbar_init(smem_addr(&s.full[j]), 1);
        mbar_init(smem_addr(&s.empty[j]), kWarps);
      }
      fence_mbar_init();
    }
    s.ring_seq = 0;
    s.claims = 0;
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(&P.ws->status, SV_DATA_BAD_OFFSETS);
    return;
  }
  const unsigned R_t = (unsigned)(P.cu[P.B] + P.B);
  if (tid == 0) {
    s.R_d = P.cu[P.B];
    // Work items: whole rows, then the last rows split into parts.
    unsigned W = 0, np = 1;
    if (VEC) {
      W = min(R_t, min(kTailWaves * gridDim.x, kMaxTailRows));
      np = kRowParts;
      if (R_t < gridDim.x) np = max(np, gridDim.x / R_t);  // few rows: spread each row out
      const unsigned nch = (unsigned)(((size_t)P.V * Elem<DT & 1>::kBytes + kChunkBytes - 1) / kChunkBytes);
      np = min(np, min(kMaxRowParts, nch));
      if (W > 0) np = min(np, kMaxPartRecs / W);
      if (np < 2) W = 0, np = 1;
    }
    s.row_parts = np;
    s.r_full = R_t - W;
    s.n_items = (R_t - W) + W * np;
  }
  __syncthreads();
  const unsigned n_items = s.n_items, r_full = s.r_full, row_parts = s.row_parts;
  for (;;) {
    if (tid == 0) {
      // Rows first; once they are all handed out, parts of published draws.
      int slot = -1, part = -1;
      // A CTA's first item is its own index; later ones come from the counter.
      const unsigned t = s.claims++ == 0 ? blockIdx.x : atomicAdd(&P.ws->next_item, 1u) + gridDim.x;
      s.wk = 0;
      if (t < n_items) {
        s.wk = 2;
        s.item = (int)t;
      } else if (P.may_publish) {
        // Rows are all handed out: stay for parts of draws published later
        // (none can be when every draw is too small to split or the batch
        // is greedy; then leave at once).
        for (unsigned poll = 0; poll < kLingerPolls; ++poll) {
          if (claim_draw_part(P, slot, part)) {
            s.wk = 1;
            break;
          }
          if (ld_relaxed_gpu(&P.ws->committed) >= (unsigned)P.B) {
            if (claim_draw_part(P, slot, part)) s.wk = 1;
            break;
          }
          __nanosleep(kLingerNs);
        }
      }
      s.slot = slot;
      s.part = part;
    }
    __syncthreads();
    const int wk = s.wk, item = s.item, slot = s.slot, part = s.part;
    __syncthreads();
    if (wk == 0) break;
    bool ok;
    if (wk == 1) {
      ok = draw_part<DT, VEC>(P, s, ring, slot, part);
    } else if ((unsigned)item < r_full) {
      ok = process_item<DT, VEC>(P, s, ring, item, -1, 0);
    } else {
      const unsigned j = (unsigned)item - r_full;
      ok = process_item<DT, VEC>(P, s, ring, (int)(r_full + j / row_parts), (int)(j % row_parts),
                                 (int)(j / row_parts));
    }
    if (!ok) {
      // A bulk copy never completed: report it and leave without touching
      // the shared counters (the workspace must be zero-filled again).
      if (tid == 0) atomicOr(&P.ws->status, SV_DEV_COPY_TIMEOUT);
      return;
    }
  }
  // The last CTA to leave clears the draw slots and the counters.
  if (tid == 0) {
    const unsigned old = atom_add_acqrel_gpu(&P.ws->exited, 1u);
    s.last = (old == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s.last) return;
  unsigned n = __ldcg(&P.ws->n_draws);
  if (n > (unsigned)P.n_slots) n = (unsigned)P.n_slots;
  for (unsigned k = tid; k < n; k += kThreads) {
    P.slot_state[k] = 0u;
    P.descs[k].done = 0u;
  }
  if (tid == 0) {
    P.ws->next_item = 0u;
    P.ws->n_draws = 0u;
    P.ws->draw_head = 0u;
    P.ws->committed = 0u;
    P.ws->exited = 0u;
    if (P.fc_need) *P.fc_need = 0u;  // every CTA read it on entry
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Draw slots (parts of draws published near the end of a call), and tile
// sums per slot counted with the smaller fp32 tile so one size fits both types.
static int n_draw_slots(long long B) { return (int)(B < kMaxDrawSlots ? B : kMaxDrawSlots); }
static int tsum_stride(int V) { return (V + kThreads * 4 - 1) / (kThreads * 4); }

// header | req_state[B] | slot_state[S] | descs[S] | tsum[S][stride] |
// part_done[kMaxTailRows] | parts[kMaxPartRecs] | rows[R_t] | rtile[R_t][stride]
struct WsLayout {
  size_t req_done, slot_state, descs, tsum, part_done, parts, rows;
};

static WsLayout ws_layout(long long B, int V) {
  const size_t S = (size_t)n_draw_slots(B);
  WsLayout L;
  L.req_done = sizeof(WsHeader);
  L.slot_state = L.req_done + align16((size_t)B * sizeof(unsigned long long));
  L.descs = L.slot_state + align16(S * sizeof(unsigned));
  L.tsum = L.descs + S * sizeof(DrawDesc);
  L.part_done = L.tsum + align16(S * (size_t)tsum_stride(V) * sizeof(DF));
  L.parts = L.part_done + align16((size_t)kMaxTailRows * sizeof(unsigned));
  L.rows = L.parts + (size_t)kMaxPartRecs * sizeof(PartRec);
  return L;
}

// Bytes per target row: its record and its tile sums.
static size_t row_bytes(int V) { return sizeof(RowRec) + (size_t)tsum_stride(V) * sizeof(float); }

static size_t ws_size(long long B, long long R_t, int V) {
  return ws_layout(B, V).rows + (size_t)R_t * row_bytes(V);
}

// Resident CTAs per device for each kernel variant, filled on first use
// (which also raises the variant's dynamic shared-memory limit).
constexpr int kMaxDevices = 64;
static std::atomic<int> g_resident[kMaxDevices][4][2];

template <bool VEC>
static constexpr int dyn_smem() { return VEC ? kRingBytes : 0; }

template <int DT, bool VEC>
static cudaError_t resident_ctas(int dev, int* out) {
  int cached = dev < kMaxDevices ? g_resident[dev][DT][VEC].load(std::memory_order_relaxed) : 0;
  if (cached > 0) {
    *out = cached;
    return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<DT, VEC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<VEC>());
  if (e != cudaSuccess) return e;
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<DT, VEC>, kThreads,
                                                    dyn_smem<VEC>());
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
  // At most one CTA per possible work item (rows may be split into parts).
  long long grid = resident;
  if (grid > P.row_cap * (long long)kMaxRowParts) grid = P.row_cap * (long long)kMaxRowParts;
  if (grid < 1) grid = 1;
  verify_kernel<DT, VEC><<<(unsigned)grid, kThreads, dyn_smem<VEC>(), st>>>(P);
  return cudaGetLastError();
}

// The host checks of every verify entry point except those of the
// workspace; makes no CUDA call. B == 0 passes (the call is then a no-op).
static sv_status check_verify_args(const void* target, const void* draft, sv_dtype dtype, int32_t V,
                                   int32_t B, const int32_t* draft_tokens, const int32_t* cu_draft,
                                   const float* uniforms, float temperature, const int32_t* out_tokens,
                                   const int32_t* out_len, const float* out_probs, int greedy_all) {
  if (dtype != SV_FP32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (B < 0 || V < 1 || V > max_vocab(dtype)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target || !cu_draft || !out_tokens || !out_len) return SV_ERR_INVALID_ARG;
  if (!greedy_all) {
    if (!uniforms) return SV_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  }
  const size_t es = dtype == SV_FP32 ? 4 : 2;
  if ((uintptr_t)target % es || (draft && (uintptr_t)draft % es)) return SV_ERR_INVALID_ARG;
  if ((uintptr_t)cu_draft % 4 || (uintptr_t)out_tokens % 4 || (uintptr_t)out_len % 4 ||
      (out_probs && (uintptr_t)out_probs % 4) || (uniforms && (uintptr_t)uniforms % 4) ||
      (draft_tokens && (uintptr_t)draft_tokens % 4))
    return SV_ERR_INVALID_ARG;
  return SV_OK;
}

// Workspaces holding at most this many target rows take the cluster kernel.
static std::atomic<int> g_cluster_rows{SV_CLUSTER_ROWS_DEFAULT};

// One-hot batches (no draft rows) with rows of at most this many bytes take
// the one-CTA-per-row kernel when the cluster kernel does not.
static std::atomic<int> g_onehot_row_bytes{SV_ONEHOT_ROW_BYTES_DEFAULT};

static sv_status run_verify(const void* target, const void* draft, sv_dtype dtype, int32_t V,
                            int32_t B, const int32_t* draft_tokens, const int32_t* cu_draft,
                            const uint8_t* mode, const float* uniforms, float temperature,
                            int32_t* out_tokens, int32_t* out_len, float* out_probs,
                            void* workspace, size_t workspace_bytes, void* stream,
                            int greedy_all, const float* thr = nullptr,
                            const float* thr_d = nullptr, const FStat* fst = nullptr,
                            const FStat* fst_d = nullptr, const int2* flist = nullptr,
                            int row_tiles = 1, FcParams* fc = nullptr) {
  const sv_status chk = check_verify_args(target, draft, dtype, V, B, draft_tokens, cu_draft, uniforms,
                                          temperature, out_tokens, out_len, out_probs, greedy_all);
  if (chk != SV_OK || B == 0) return chk;
  if (!workspace || (uintptr_t)workspace % 16) return SV_ERR_INVALID_ARG;
  const size_t es = dtype == SV_FP32 ? 4 : 2;
  const WsLayout L = ws_layout(B, V);
  if (workspace_bytes < L.rows + sizeof(RowRec)) return SV_ERR_INVALID_ARG;

  char* ws = static_cast<char*>(workspace);
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
  P.ws = reinterpret_cast<WsHeader*>(ws);
  P.req_state = reinterpret_cast<unsigned long long*>(ws + L.req_done);
  P.slot_state = reinterpret_cast<unsigned*>(ws + L.slot_state);
  P.descs = reinterpret_cast<DrawDesc*>(ws + L.descs);
  P.tsum = reinterpret_cast<DF*>(ws + L.tsum);

  P.n_slots = n_draw_slots(B);
  P.part_done = reinterpret_cast<unsigned*>(ws + L.part_done);
  P.parts = reinterpret_cast<PartRec*>(ws + L.parts);
  P.tsum_stride = tsum_stride(V);
  P.rows = reinterpret_cast<RowRec*>(ws + L.rows);
  // Rows and their tile sums share what follows the fixed part; without
  // tiles (row_tiles == 0) the records alone fill it.
  P.row_cap = (long long)((workspace_bytes - L.rows) / (row_tiles ? row_bytes(V) : sizeof(RowRec)));
  P.rtile = row_tiles ? reinterpret_cast<float*>(ws + L.rows + (size_t)P.row_cap * sizeof(RowRec)) : nullptr;
  P.greedy_all = greedy_all;
  // Draws are published in parts only if they stream kMinPublishBytes or more.
  P.may_publish = !greedy_all && (size_t)V * es * (P.draft ? 2 : 1) >= kMinPublishBytes;
  P.thr = thr;
  P.thr_d = thr_d;
  P.fst = fst;
  P.fst_d = fst_d;
  P.flist = flist;
  P.fc_need = nullptr;
  P.fc_done = nullptr;

  // Bulk copies need 16-byte aligned row starts and 16-byte multiples.
  const bool vec = ((uintptr_t)target % 16 == 0) && (!P.draft || (uintptr_t)P.draft % 16 == 0) &&
                   (((size_t)V * es) % 16 == 0);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (greedy_all && vec && !thr) {
    // Strict verification needs only each row's argmax: one CTA per row.
    GParams G;
    G.target = target;
    G.V = V;
    G.B = B;
    G.draft_tokens = draft_tokens;
    G.cu = cu_draft;
    G.out_tokens = out_tokens;
    G.out_len = out_len;
    G.status = &P.ws->status;
    G.arrive = P.req_state;
    G.rows = reinterpret_cast<CRow*>(P.rows);
    G.row_cap = P.row_cap;
    G.nvec = (int)(((size_t)V * es) / 16);
    e = launch_greedy_verify(G, dtype == SV_BF16 ? 1 : 0, st);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
  }
  if (vec && !thr && P.row_cap <= (long long)g_cluster_rows.load(std::memory_order_relaxed) &&
      cluster_smem_bytes((size_t)V * es, P.draft != nullptr) > 0) {
    CParams C;
    C.target = target;
    C.draft = P.draft;
    C.V = V;
    C.B = B;
    C.draft_tokens = draft_tokens;
    C.cu = cu_draft;
    C.mode = P.mode;
    C.uniforms = uniforms;
    C.c = P.c;
    C.out_tokens = out_tokens;
    C.out_len = out_len;
    C.out_probs = P.out_probs;
    C.status = &P.ws->status;
    C.arrive = P.req_state;
    C.rows = reinterpret_cast<CRow*>(P.rows);
    C.row_cap = P.row_cap;
    C.greedy_all = greedy_all;
    C.nvec = (int)(((size_t)V * es) / 16);
    C.vp = 0;
    e = launch_cluster_verify(C, dtype == SV_BF16 ? 1 : 0, st);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
  }
  if (vec && !thr && !P.draft && row_tiles &&
      (long long)V * (long long)es <= (long long)g_onehot_row_bytes.load(std::memory_order_relaxed) &&
      (size_t)V * es / 16 <= (size_t)kOneHotMaxVec) {
    // Short rows and one-hot proposals: one CTA per row, no claims, no ring.
    RParams R;
    R.target = target;
    R.V = V;
    R.B = B;
    R.draft_tokens = draft_tokens;
    R.cu = cu_draft;
    R.mode = P.mode;
    R.uniforms = uniforms;
    R.c = P.c;
    R.out_tokens = out_tokens;
    R.out_len = out_len;
    R.out_probs = P.out_probs;
    R.status = &P.ws->status;
    R.arrive = P.req_state;
    R.rows = reinterpret_cast<RRow*>(P.rows);
    R.row_cap = P.row_cap;
    R.greedy_all = greedy_all;
    R.nvec = (int)(((size_t)V * es) / 16);
    e = launch_onehot_verify(R, dtype == SV_BF16 ? 1 : 0, st);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
  }
  if (thr) {
    if (fc) {
      // Requests whose rows all carry their statistics are decided, drawn
      // and committed first, one CTA each; the verify kernel takes the rest.
      fc->out_tokens = out_tokens;
      fc->out_len = out_len;
      fc->out_probs = P.out_probs;
      fc->status = &P.ws->status;
      if (fc->rows_t > P.row_cap) fc->rows_t = (int)P.row_cap;
      e = launch_filtered_commit(*fc, dtype == SV_BF16 ? 1 : 0, st);
      if (e != cudaSuccess) return SV_ERR_CUDA;
      P.fc_need = fc->need_slow;
      P.fc_done = fc->done;
    }
    if (dtype == SV_BF16)
      e = vec ? launch<1 | kFilt, true>(P, st) : launch<1 | kFilt, false>(P, st);
    else
      e = vec ? launch<0 | kFilt, true>(P, st) : launch<0 | kFilt, false>(P, st);
  } else if (dtype == SV_BF16) {
    e = vec ? launch<1, true>(P, st) : launch<1, false>(P, st);
  } else {
    e = vec ? launch<0, true>(P, st) : launch<0, false>(P, st);
  }
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Verify without a caller workspace: scratch in a fixed device block
// ---------------------------------------------------------------------------
// The block is part of the module image, so using it needs no allocation.
// Its address is looked up once per device, with that device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];
static std::atomic<void*> g_noalloc_ptr[kMaxDevices];

static cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  void* p = dev < kMaxDevices ? g_noalloc_ptr[dev].load(std::memory_order_acquire) : nullptr;
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) g_noalloc_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace sv

extern "C" {

sv_status spec_verify_noalloc(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                              int32_t V, int32_t B, const int32_t* draft_tokens,
                              const int32_t* cu_draft, const uint8_t* mode,
                              const float* uniforms, float temperature, int32_t* out_tokens,
                              int32_t* out_len, float* out_probs, uint32_t* status_out,
                              void* cuda_stream) {
  // Every host check comes before the first CUDA call, so a rejected call
  // enqueues nothing (not even the clearing of the block).
  if (status_out && (uintptr_t)status_out % 4) return SV_ERR_INVALID_ARG;
  const sv_status chk = sv::check_verify_args(target_logits, draft_logits, dtype, V, B, draft_tokens,
                                              cu_draft, uniforms, temperature, out_tokens, out_len,
                                              out_probs, 0);
  if (chk != SV_OK || B == 0) return chk;
  // The row count lives on the device; size the check by the largest R_t the
  // block could hold for this B and V, and let the kernel flag offsets past it.
  const sv::WsLayout L = sv::ws_layout(B, V);
  if (L.rows + sizeof(sv::RowRec) > SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (sv::noalloc_scratch(&scratch) != cudaSuccess) return SV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // Counters, per-request state, draw slots and split-row counters start at
  // zero; the per-row records after them are written before they are read.
  if (cudaMemsetAsync(scratch, 0, L.rows, st) != cudaSuccess) return SV_ERR_CUDA;
  const sv_status s = sv::run_verify(target_logits, draft_logits, dtype, V, B, draft_tokens,
                                     cu_draft, mode, uniforms, temperature, out_tokens, out_len,
                                     out_probs, scratch, SV_NOALLOC_SCRATCH_BYTES, cuda_stream, 0,
                                     nullptr, nullptr, nullptr, nullptr, nullptr, 0);
  if (s != SV_OK) return s;
  if (status_out && cudaMemcpyAsync(status_out, scratch, sizeof(uint32_t),
                                    cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

// Filtered form: the per-row thresholds and filtered statistics come first
// in the workspace, then the verify kernel's own workspace.
static size_t filter_thr_bytes(int64_t R_t, int64_t B) {
  return sv::align16((size_t)R_t * 4) + sv::align16((size_t)(R_t - B) * 4 + 4);
}
static size_t filter_fst_bytes(int64_t R_t, int64_t B) {
  return (size_t)R_t * sizeof(sv::FStat) + (size_t)(R_t - B + 1) * sizeof(sv::FStat);
}
static size_t filter_list_bytes(int64_t R_t) { return (size_t)R_t * sv::kKeptListCap * sizeof(int2); }
// Flags of the filtered commit: rows left to the CTA threshold kernel,
// requests left to the verify kernel, then one "committed" byte per request.
static size_t filter_flag_bytes(int64_t B) { return sv::align16(8 + (size_t)B); }
static size_t filter_bytes(int64_t R_t, int64_t B) {
  return filter_thr_bytes(R_t, B) + filter_fst_bytes(R_t, B) + filter_list_bytes(R_t) + filter_flag_bytes(B);
}

size_t spec_verify_filtered_workspace_size(int32_t B, int32_t R_t, int32_t V) {
  if (B < 0 || R_t < B || V < 1) return 0;
  return filter_bytes(R_t, B) + sv::ws_size(B, R_t > 0 ? R_t : 1, V);
}

sv_status spec_verify_filtered(const void* target_logits, const void* draft_logits,
                               sv_dtype dtype, int32_t V, int32_t B, int32_t R_t,
                               const int32_t* draft_tokens, const int32_t* cu_draft,
                               const uint8_t* mode, const float* uniforms, float temperature,
                               int32_t top_k, float top_p, int32_t* out_tokens,
                               int32_t* out_len, float* out_probs, void* workspace,
                               size_t workspace_bytes, void* cuda_stream) {
  if (B < 0 || R_t < B || top_k < 0 || !(top_p > 0.f) || top_p != top_p) return SV_ERR_INVALID_ARG;
  if (dtype != SV_FP32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!workspace || (uintptr_t)workspace % 16 || !cu_draft || !target_logits) return SV_ERR_INVALID_ARG;
  const size_t fb = filter_bytes(R_t, B);
  if (workspace_bytes < fb) return SV_ERR_INVALID_ARG;
  const bool use_k = top_k >= 1 && top_k < V, use_p = top_p < 1.f;
  char* ws = static_cast<char*>(workspace);
  if (!use_k && !use_p)  // nothing to filter: the plain step
    return sv::run_verify(target_logits, draft_logits, dtype, V, B, draft_tokens, cu_draft, mode,
                          uniforms, temperature, out_tokens, out_len, out_probs, ws + fb,
                          workspace_bytes - fb, cuda_stream, 0);
  if (!(temperature > 0.f) || !std::isfinite(temperature) || V < 1 || V > sv::max_vocab(dtype))
    return SV_ERR_INVALID_ARG;
  const size_t es = dtype == SV_FP32 ? 4 : 2;
  if ((uintptr_t)target_logits % es || (draft_logits && (uintptr_t)draft_logits % es))
    return SV_ERR_INVALID_ARG;
  // Every check of the verify step too, before the thresholds are enqueued:
  // a rejected call enqueues nothing.
  const sv_status chk = sv::check_verify_args(target_logits, draft_logits, dtype, V, B, draft_tokens,
                                              cu_draft, uniforms, temperature, out_tokens, out_len,
                                              out_probs, 0);
  if (chk != SV_OK) return chk;
  if (workspace_bytes - fb < sv::ws_layout(B, V).rows + sizeof(sv::RowRec)) return SV_ERR_INVALID_ARG;
  sv::FtParams fp;
  fp.target = target_logits;
  fp.draft = draft_logits;
  fp.V = V;
  fp.B = B;
  fp.rows_t = R_t;
  fp.cu = cu_draft;
  fp.mode = mode;
  fp.c = (float)(1.4426950408889634 / (double)temperature);
  fp.top_k = use_k ? top_k : 0;
  fp.top_p = use_p ? top_p : 1.f;
  fp.vec = ((uintptr_t)target_logits % 16 == 0) && (!draft_logits || (uintptr_t)draft_logits % 16 == 0) &&
           (((size_t)V * es) % 16 == 0);
  fp.thr_t = reinterpret_cast<float*>(ws);
  fp.thr_d = reinterpret_cast<float*>(ws + sv::align16((size_t)R_t * 4));
  fp.fst_t = reinterpret_cast<sv::FStat*>(ws + filter_thr_bytes(R_t, B));
  fp.fst_d = fp.fst_t + R_t;
  fp.list_t = reinterpret_cast<int2*>(ws + filter_thr_bytes(R_t, B) + filter_fst_bytes(R_t, B));
  unsigned* flags = reinterpret_cast<unsigned*>(ws + filter_thr_bytes(R_t, B) + filter_fst_bytes(R_t, B) +
                                                filter_list_bytes(R_t));
  fp.rows_left = flags;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  bool warp_ran = false;
  if (sv::launch_thresholds(fp, dtype, st, &warp_ran) != cudaSuccess) return SV_ERR_CUDA;
  // The one-warp-per-row thresholds leave statistics and kept lists that
  // let most requests commit without the verify kernel.
  sv::FcParams fc;
  fc.target = target_logits;
  fc.draft = draft_logits;
  fc.V = V;
  fc.B = B;
  fc.rows_t = R_t;
  fc.draft_tokens = draft_tokens;
  fc.cu = cu_draft;
  fc.mode = mode;
  fc.uniforms = uniforms;
  fc.c = fp.c;
  fc.thr_t = fp.thr_t;
  fc.thr_d = draft_logits ? fp.thr_d : nullptr;
  fc.fst_t = fp.fst_t;
  fc.fst_d = draft_logits ? fp.fst_d : nullptr;
  fc.list_t = fp.list_t;
  fc.need_slow = flags + 1;
  fc.done = reinterpret_cast<unsigned char*>(flags + 2);
  fc.rows_left = flags;
  return sv::run_verify(target_logits, draft_logits, dtype, V, B, draft_tokens, cu_draft, mode,
                        uniforms, temperature, out_tokens, out_len, out_probs, ws + fb,
                        workspace_bytes - fb, cuda_stream, 0, fp.thr_t,
                        draft_logits ? fp.thr_d : nullptr, fp.fst_t, draft_logits ? fp.fst_d : nullptr,
                        fp.list_t, 1, warp_ran ? &fc : nullptr);
}

size_t spec_verify_workspace_size(int32_t B, int32_t R_t, int32_t V) {
  if (B < 0 || R_t < 0 || V < 1) return 0;
  return sv::ws_size(B, R_t > 0 ? R_t : 1, V);
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
  if (bits & SV_DEV_COPY_TIMEOUT) return SV_ERR_TIMEOUT;
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

int32_t sv_set_onehot_row_bytes(int32_t bytes) {
  if (bytes < 0) return sv::g_onehot_row_bytes.load();
  return sv::g_onehot_row_bytes.exchange(bytes);
}

int32_t sv_set_cluster_rows(int32_t rows) {
  if (rows < 0) return sv::g_cluster_rows.load();
  return sv::g_cluster_rows.exchange(rows);
}

}  // extern "C"
