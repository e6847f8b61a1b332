// ngram.cu -- model-free n-gram (prompt-lookup) proposer on sm_103a.
//
// "5.2 Draft 模型与无模型方案：怎样便宜地猜得更准", §4 "N-gram" and §6
// "动手实验": for window lengths n from min(max_n, L) down to min_n, take the
// last n tokens of the history as the tail and look for its most recent
// earlier occurrence that ends before the tail begins and leaves at least one
// token after it; propose what followed, cut to max_tokens.
//
// One CTA per history. The history is staged in shared memory when it fits;
// for each n every thread tests its own candidate starts from the most recent
// down and stops at its first match; the largest over the threads wins. All
// comparisons are on integers, so the result is bit-exact.
#include "../../include/spec_verify.h"

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kNgThreads = 256;
constexpr int kNgSmemInts = 12288;  // 48 KB: histories up to this length are staged

__global__ void __launch_bounds__(kNgThreads) ngram_kernel(
    const int32_t* __restrict__ hist, long long stride, const int32_t* __restrict__ hist_len,
    int min_n, int max_n, int max_tokens, int32_t* __restrict__ out_tokens,
    int32_t* __restrict__ out_count, int32_t* __restrict__ out_n, int staged) {
  extern __shared__ __align__(16) int32_t sh_hist[];
  __shared__ int s_warp_best[kNgThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x;
  const int32_t* g = hist + (long long)b * stride;
  int L = hist_len[b];
  if (L < 0) L = 0;
  if ((long long)L > stride) L = (int)stride;
  const int32_t* h = g;
  if (staged) {
    // 16-byte loads when the row allows them, several in flight per thread.
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(g) & 15) == 0) {
      const int nv = L >> 2;
      const int4* gv = reinterpret_cast<const int4*>(g);
      int4* sv = reinterpret_cast<int4*>(sh_hist);
#pragma unroll 4
      for (int k = tid; k < nv; k += kNgThreads) sv[k] = __ldg(gv + k);
      done = nv << 2;
    }
    for (int k = done + tid; k < L; k += kNgThreads) sh_hist[k] = g[k];
    __syncthreads();
    h = sh_hist;
  }
  int found_n = 0, found_s = -1;
  const int nhi = max_n < L ? max_n : L;
  for (int n = nhi; n >= min_n && found_n == 0; --n) {
    const int tail = L - n;
    // Largest start whose match ends before the tail and leaves a token.
    // Each thread walks its own candidates downwards, so its first match is
    // its largest; the CTA then takes the largest over the threads.
    int best = -1;
    for (int st = tail - n - 1 - tid; st >= 0; st -= kNgThreads) {
      bool match = true;
      for (int j = 0; j < n; ++j) {
        if (h[st + j] != h[tail + j]) {
          match = false;
          break;
        }
      }
      if (match) {
        best = st;
        break;
      }
    }
    best = __reduce_max_sync(0xffffffffu, best);
    if ((tid & 31) == 0) s_warp_best[tid >> 5] = best;
    __syncthreads();
    best = s_warp_best[0];
#pragma unroll
    for (int w = 1; w < kNgThreads / 32; ++w) best = max(best, s_warp_best[w]);
    __syncthreads();  // s_warp_best is reused by the next window length
    if (best >= 0) {
      found_n = n;
      found_s = best;
    }
  }
  int cnt = 0;
  if (found_n > 0) {
    const int cont = (L - found_n) - (found_s + found_n);
    cnt = cont < max_tokens ? cont : max_tokens;
  }
  int32_t* out = out_tokens + (long long)b * max_tokens;
  for (int j = tid; j < max_tokens; j += kNgThreads) out[j] = j < cnt ? h[found_s + found_n + j] : -1;
  if (tid == 0) {
    out_count[b] = cnt;
    out_n[b] = found_n;
  }
}

// cu_draft = exclusive prefix sums of the clamped counts; proposals packed
// back to back. One CTA walks the batch in chunks of kPackThreads.
constexpr int kPackThreads = 1024;

__global__ void __launch_bounds__(kPackThreads) pack_kernel(
    const int32_t* __restrict__ tokens, const int32_t* __restrict__ counts, int B, int max_tokens,
    int32_t* __restrict__ cu, int32_t* __restrict__ packed) {
  __shared__ int s_warp[kPackThreads / 32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < B; base += kPackThreads) {
    const int b = base + tid;
    int k = 0;
    if (b < B) {
      k = counts[b];
      k = k < 0 ? 0 : (k > max_tokens ? max_tokens : k);
    }
    int v = k;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += u;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int carry = s_carry;
    const int excl = carry + (warp ? s_warp[warp - 1] : 0) + v - k;
    if (b < B) {
      cu[b] = excl;
      for (int j = 0; j < k; ++j) packed[excl + j] = tokens[(long long)b * max_tokens + j];
    }
    __syncthreads();
    if (tid == 0) s_carry = carry + s_warp[kPackThreads / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) cu[B] = s_carry;
}

}  // namespace sv

extern "C" {

sv_status ngram_propose(const int32_t* histories, int64_t hist_stride, const int32_t* hist_len,
                        int32_t B, int32_t min_n, int32_t max_n, int32_t max_tokens,
                        int32_t* out_tokens, int32_t* out_count, int32_t* out_n,
                        void* cuda_stream) {
  if (B < 0 || min_n < 1 || max_n < min_n || max_tokens < 0 || hist_stride < 0)
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!hist_len || !out_count || !out_n || (max_tokens > 0 && !out_tokens) ||
      (hist_stride > 0 && !histories))
    return SV_ERR_INVALID_ARG;
  if ((uintptr_t)histories % 4 || (uintptr_t)hist_len % 4 || (uintptr_t)out_tokens % 4 ||
      (uintptr_t)out_count % 4 || (uintptr_t)out_n % 4)
    return SV_ERR_INVALID_ARG;
  if (hist_stride > 0x7fffffffLL) return SV_ERR_INVALID_ARG;
  const int staged = hist_stride <= sv::kNgSmemInts ? 1 : 0;
  const size_t smem = staged ? (size_t)hist_stride * sizeof(int32_t) : 0;
  // Static and dynamic shared memory together above 48 KB need the
  // function's opt-in (a full 12288-token stage plus the static words).
  if (smem > 0 && cudaFuncSetAttribute(sv::ngram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(sv::kNgSmemInts * sizeof(int32_t))) != cudaSuccess)
    return SV_ERR_CUDA;
  sv::ngram_kernel<<<(unsigned)B, sv::kNgThreads, smem, static_cast<cudaStream_t>(cuda_stream)>>>(
      histories, (long long)hist_stride, hist_len, min_n, max_n, max_tokens, out_tokens, out_count,
      out_n, staged);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_pack_drafts(const int32_t* tokens, const int32_t* counts, int32_t B,
                         int32_t max_tokens, int32_t* cu_draft, int32_t* packed,
                         void* cuda_stream) {
  if (B < 0 || max_tokens < 0) return SV_ERR_INVALID_ARG;
  if (!cu_draft) return SV_ERR_INVALID_ARG;
  if (B > 0 && (!counts || (max_tokens > 0 && (!tokens || !packed)))) return SV_ERR_INVALID_ARG;
  if ((uintptr_t)tokens % 4 || (uintptr_t)counts % 4 || (uintptr_t)cu_draft % 4 ||
      (uintptr_t)packed % 4)
    return SV_ERR_INVALID_ARG;
  sv::pack_kernel<<<1, sv::kPackThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      tokens, counts, B, max_tokens, cu_draft, packed);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
