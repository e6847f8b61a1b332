// suffix.cu -- frequency-ranked suffix proposer on sm_103a.
//
// "5.2 Draft 模型与无模型方案：怎样便宜地猜得更准", §5 "Suffix Decoding":
// where the n-gram proposer copies what followed the single most recent
// occurrence of the history's tail, the suffix proposer lets the earlier
// occurrences vote. Counts of the continuations rank the candidates (§5.1:
// "return" 20 times against "raise" twice), and the proposal is only as long
// as the continuations agree (§5.2: the configured length is a ceiling).
//
// Reading, per history h of length L:
//   * the tail is the longest h[L-n, L), n from min(max_n, L) down to min_n,
//     with an earlier occurrence at a start s, 0 <= s <= L-2n-1 (the starts
//     the n-gram proposer admits: the match ends before the tail and leaves a
//     token after it); the max_occ occurrences with the largest s vote;
//   * step j: every voter whose continuation h[s+n+j] lies before the tail
//     votes for that token; the most frequent token wins, the most recent
//     voter's token among equal counts; from the second step on the proposal
//     ends when the winner has less than min_share of the votes; only the
//     voters for the winner take part in the next step.
//
// One CTA per history, the history staged in shared memory when it fits.
// Matching starts are collected in most-recent-first order by an ordered
// block compaction over tiles of 4 x 256 candidates; a tile with no match
// costs one barrier. Each voting step counts every voter's token against the
// other voters (at most 256 of them), takes the (count, start) maximum over
// the first voter of each token, and compacts the winner's voters in order.
// Integer work only: the result is bit-exact.
#include "../../include/spec_verify.h"

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kSfThreads = 256;
constexpr int kSfWarps = kSfThreads / 32;
constexpr int kSfTile = 4;               // candidate starts per thread per tile
constexpr int kSfSmemInts = 16384;       // 64 KB: histories up to this stride are staged
static_assert(SV_SUFFIX_MAX_OCC <= kSfThreads, "one voter per thread");

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__global__ void __launch_bounds__(kSfThreads) suffix_kernel(
    const int32_t* __restrict__ hist, long long stride, const int32_t* __restrict__ hist_len,
    int min_n, int max_n, int max_tokens, float min_share, int max_occ,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_count, int32_t* __restrict__ out_n,
    int staged) {
  extern __shared__ __align__(16) int32_t sh_hist[];
  __shared__ int s_occ[kSfThreads];        // voters' starts, most recent first
  __shared__ int s_tok[kSfThreads];        // their tokens at the current step
  __shared__ int s_wcnt[kSfTile][kSfWarps];
  __shared__ unsigned long long s_wkey[kSfWarps];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int32_t* g = hist + (long long)b * stride;
  int L = hist_len[b];
  if (L < 0) L = 0;
  if ((long long)L > stride) L = (int)stride;
  const int32_t* h = g;
  if (staged) {
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(g) & 15) == 0) {
      const int nv = L >> 2;
      const int4* gv = reinterpret_cast<const int4*>(g);
      int4* sv = reinterpret_cast<int4*>(sh_hist);
#pragma unroll 4
      for (int k = tid; k < nv; k += kSfThreads) sv[k] = __ldg(gv + k);
      done = nv << 2;
    }
    for (int k = done + tid; k < L; k += kSfThreads) sh_hist[k] = g[k];
    __syncthreads();
    h = sh_hist;
  }

  // ---- the longest recurring tail and its most recent occurrences ----
  int n_found = 0, A = 0;
  const int nhi = max_n < L ? max_n : L;
  for (int n = nhi; n >= min_n && n_found == 0; --n) {
    const int tail = L - n;
    int found = 0;  // occurrences seen so far (all threads agree)
    for (int top = tail - n - 1; top >= 0 && found < max_occ; top -= kSfTile * kSfThreads) {
      unsigned mine = 0;  // bit k: start top - (k*256 + tid) matches
#pragma unroll
      for (int k = 0; k < kSfTile; ++k) {
        const int st = top - (k * kSfThreads + tid);
        if (st >= 0) {
          bool match = true;
          for (int j = 0; j < n; ++j) {
            if (h[st + j] != h[tail + j]) {
              match = false;
              break;
            }
          }
          if (match) mine |= 1u << k;
        }
      }
      if (!__syncthreads_or(mine != 0u)) continue;
      unsigned bal[kSfTile];
#pragma unroll
      for (int k = 0; k < kSfTile; ++k) {
        bal[k] = __ballot_sync(0xffffffffu, (mine >> k) & 1u);
        if (lane == 0) s_wcnt[k][warp] = __popc(bal[k]);
      }
      __syncthreads();
      int base = found;
#pragma unroll
      for (int k = 0; k < kSfTile; ++k) {
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kSfWarps; ++w) {
          const int c = s_wcnt[k][w];
          before += w < warp ? c : 0;
          total += c;
        }
        if ((mine >> k) & 1u) {
          const int pos = base + before + __popc(bal[k] & lt_mask);
          if (pos < max_occ) s_occ[pos] = top - (k * kSfThreads + tid);
        }
        base += total;
      }
      found = base;
      __syncthreads();  // s_wcnt is reused by the next tile; s_occ is complete
    }
    if (found > 0) {
      n_found = n;
      A = found < max_occ ? found : max_occ;
    }
  }

  // ---- voting, one proposal token per step ----
  int32_t* out = out_tokens + (long long)b * max_tokens;
  int cnt = 0;
  if (n_found > 0) {
    const int n = n_found;
    const double share = (double)min_share;
    for (int j = 0; j < max_tokens; ++j) {
      // Voters run most recent (largest start) first, so the ones whose
      // continuation would reach into the tail form a prefix of the list.
      const int limit = L - 2 * n - j;  // voter s is valid iff s < limit
      const int my_s = tid < A ? s_occ[tid] : 0;
      const bool in_list = tid < A;
      const int invalid = __syncthreads_count(in_list && my_s >= limit);
      const int first = invalid, nvotes = A - invalid;
      if (nvotes <= 0) break;
      const bool voter = in_list && tid >= first;
      const int my_t = voter ? h[my_s + n + j] : 0;
      if (voter) s_tok[tid] = my_t;
      __syncthreads();
      unsigned long long key = 0;
      if (voter) {
        int c = 0;
        bool is_first = true;
        for (int k = first; k < A; ++k) {
          if (s_tok[k] == my_t) {
            ++c;
            if (k < tid) is_first = false;
          }
        }
        // The first voter of a token is its most recent one: (count, start)
        // orders the tokens by count, then by recency.
        if (is_first) key = ((unsigned long long)c << 32) | (unsigned)my_s;
      }
      key = warp_max_u64(key);
      if (lane == 0) s_wkey[warp] = key;
      __syncthreads();
      key = s_wkey[0];
#pragma unroll
      for (int w = 1; w < kSfWarps; ++w) key = s_wkey[w] > key ? s_wkey[w] : key;
      const int win_count = (int)(key >> 32);
      const int win_s = (int)(unsigned)(key & 0xffffffffu);
      const int win_t = h[win_s + n + j];
      if (j > 0 && (double)win_count < share * (double)nvotes) break;
      if (tid == 0) out[j] = win_t;
      cnt = j + 1;
      // The winner's voters, in order, are the next step's list.
      const bool keep = voter && my_t == win_t;
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (lane == 0) s_wcnt[0][warp] = __popc(bal);
      __syncthreads();  // every read of s_occ and s_tok of this step is done
      int before = 0;
#pragma unroll
      for (int w = 0; w < kSfWarps; ++w) before += w < warp ? s_wcnt[0][w] : 0;
      if (keep) s_occ[before + __popc(bal & lt_mask)] = my_s;
      A = win_count;
      __syncthreads();
    }
  }
  for (int j = cnt + tid; j < max_tokens; j += kSfThreads) out[j] = -1;
  if (tid == 0) {
    out_count[b] = cnt;
    out_n[b] = n_found;
  }
}

}  // namespace sv

extern "C" {

sv_status suffix_propose(const int32_t* histories, int64_t hist_stride, const int32_t* hist_len,
                         int32_t B, int32_t min_n, int32_t max_n, int32_t max_tokens,
                         float min_share, int32_t max_occ, int32_t* out_tokens,
                         int32_t* out_count, int32_t* out_n, void* cuda_stream) {
  if (B < 0 || min_n < 1 || max_n < min_n || max_tokens < 0 || hist_stride < 0)
    return SV_ERR_INVALID_ARG;
  if (max_occ < 1 || max_occ > SV_SUFFIX_MAX_OCC || !(min_share >= 0.0f && min_share <= 1.0f))
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!hist_len || !out_count || !out_n || (max_tokens > 0 && !out_tokens) ||
      (hist_stride > 0 && !histories))
    return SV_ERR_INVALID_ARG;
  if ((uintptr_t)histories % 4 || (uintptr_t)hist_len % 4 || (uintptr_t)out_tokens % 4 ||
      (uintptr_t)out_count % 4 || (uintptr_t)out_n % 4)
    return SV_ERR_INVALID_ARG;
  if (hist_stride > 0x7fffffffLL) return SV_ERR_INVALID_ARG;
  const int staged = hist_stride <= sv::kSfSmemInts ? 1 : 0;
  const size_t smem = staged ? (size_t)hist_stride * sizeof(int32_t) : 0;
  // Above 48 KB a block's dynamic shared memory needs the function's opt-in.
  if (smem > 0 && cudaFuncSetAttribute(sv::suffix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(sv::kSfSmemInts * sizeof(int32_t))) != cudaSuccess)
    return SV_ERR_CUDA;
  sv::suffix_kernel<<<(unsigned)B, sv::kSfThreads, smem, static_cast<cudaStream_t>(cuda_stream)>>>(
      histories, (long long)hist_stride, hist_len, min_n, max_n, max_tokens, min_share, max_occ,
      out_tokens, out_count, out_n, staged);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
