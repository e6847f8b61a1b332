// metrics.cu -- acceptance statistics of verify rounds, accumulated on the
// device, and the host-side sliding-window draft-length controller.
//
// "5.2 Draft 模型与无模型方案：怎样便宜地猜得更准", §7.1 and §7.2: over an
// observation window with D proposed draft tokens, C of them accepted and R
// verify rounds, the draft acceptance rate is C / D and the mean acceptance
// length 1 + C / R; candidate coverage counts the rounds that had any
// proposal at all; the conditional acceptance rate of slot i (given that
// every earlier slot was accepted) differs from the probability of
// accepting every slot up to i.
//
// "投机解码从零实现" (CSDN), §5.2 "动态草稿长度策略": the draft length is
// moved by one step when the mean accepted fraction over a sliding window of
// recent rounds leaves a band of +-0.1 around a target.
#include "../../include/spec_verify.h"

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kMetThreads = 256;
constexpr int kMetCounters = 5 + 3 * SV_METRICS_MAX_POS;
static_assert(sizeof(sv_metrics) == kMetCounters * sizeof(unsigned long long),
              "sv_metrics is a flat array of 64-bit counters");

// One request per thread. Each warp sums its 32 requests' counts with warp
// reductions, one lane per warp adds them to the CTA's counters in shared
// memory, and each CTA then adds its counters to the caller's block.
__global__ void __launch_bounds__(kMetThreads) metrics_kernel(const int32_t* __restrict__ cu,
                                                              const int32_t* __restrict__ out_len,
                                                              int B, unsigned long long* __restrict__ g) {
  __shared__ unsigned long long c[kMetCounters];
  const int lane = threadIdx.x & 31;
  for (int k = threadIdx.x; k < kMetCounters; k += kMetThreads) c[k] = 0ull;
  __syncthreads();
  for (int base = blockIdx.x * kMetThreads; base < B; base += gridDim.x * kMetThreads) {
    const int b = base + threadIdx.x;
    int K = 0, stop = 0;
    const bool live = b < B;
    if (live) {
      K = max(0, cu[b + 1] - cu[b]);
      stop = min(max(out_len[b], 1), K + 1) - 1;  // slots before it accepted
    }
    const unsigned full = 0xffffffffu;
    // K and stop are below 2^31 / 32 for any valid batch, so 32-bit warp sums fit.
    const unsigned r = __reduce_add_sync(full, live ? 1u : 0u);
    const unsigned w = __reduce_add_sync(full, K > 0 ? 1u : 0u);
    const unsigned d = __reduce_add_sync(full, (unsigned)K);
    const unsigned a = __reduce_add_sync(full, (unsigned)stop);
    const unsigned kmax = __reduce_max_sync(full, (unsigned)min(K, SV_METRICS_MAX_POS));
    if (lane == 0 && r) {
      atomicAdd(&c[0], (unsigned long long)r);
      atomicAdd(&c[1], (unsigned long long)w);
      atomicAdd(&c[2], (unsigned long long)d);
      atomicAdd(&c[3], (unsigned long long)a);
      atomicAdd(&c[4], (unsigned long long)(a + r));  // committed = stop + 1 per round
    }
    // Slot i is offered if i < K, tested if every earlier slot was accepted
    // (i <= stop), and accepted (with all before it) if i < stop.
    for (int i = 0; i < (int)kmax; ++i) {
      const unsigned off = __reduce_add_sync(full, i < K ? 1u : 0u);
      const unsigned rea = __reduce_add_sync(full, (i < K && i <= stop) ? 1u : 0u);
      const unsigned acc = __reduce_add_sync(full, (i < K && i < stop) ? 1u : 0u);
      if (lane == 0) {
        if (off) atomicAdd(&c[5 + i], (unsigned long long)off);
        if (rea) atomicAdd(&c[5 + SV_METRICS_MAX_POS + i], (unsigned long long)rea);
        if (acc) atomicAdd(&c[5 + 2 * SV_METRICS_MAX_POS + i], (unsigned long long)acc);
      }
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < kMetCounters; k += kMetThreads)
    if (c[k]) atomicAdd(&g[k], c[k]);
}

}  // namespace sv

extern "C" {

sv_status sv_accumulate_metrics(const int32_t* cu_draft, const int32_t* out_len, int32_t B,
                                sv_metrics* metrics, void* cuda_stream) {
  if (B < 0 || !metrics || (uintptr_t)metrics % 8) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!cu_draft || !out_len || (uintptr_t)cu_draft % 4 || (uintptr_t)out_len % 4)
    return SV_ERR_INVALID_ARG;
  int grid = (B + sv::kMetThreads * 4 - 1) / (sv::kMetThreads * 4);  // ~4 requests per thread
  grid = grid < 1 ? 1 : (grid > 152 ? 152 : grid);
  sv::metrics_kernel<<<grid, sv::kMetThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      cu_draft, out_len, B, reinterpret_cast<unsigned long long*>(metrics));
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_adapt_init(sv_adapt* a, int32_t window, int32_t min_k, int32_t max_k, double target,
                        int32_t initial_k) {
  if (!a || window < 1 || window > SV_ADAPT_MAX_WINDOW || min_k < 0 || max_k < min_k ||
      initial_k < min_k || initial_k > max_k || !(target == target))
    return SV_ERR_INVALID_ARG;
  a->window = window;
  a->min_k = min_k;
  a->max_k = max_k;
  a->target = target;
  a->k = initial_k;
  a->count = 0;
  a->next = 0;
  for (int i = 0; i < SV_ADAPT_MAX_WINDOW; ++i) a->ratio[i] = 0.0;
  return SV_OK;
}

sv_status sv_adapt_update(sv_adapt* a, int32_t draft_len, int32_t accepted_len) {
  if (!a || draft_len < 0 || accepted_len < 0 || accepted_len > draft_len) return SV_ERR_INVALID_ARG;
  // The round's accepted fraction enters the ring, replacing the oldest once
  // the window is full.
  a->ratio[a->next] = (double)accepted_len / (double)(draft_len > 0 ? draft_len : 1);
  a->next = (a->next + 1) % a->window;
  if (a->count < a->window) ++a->count;
  if (a->count < SV_ADAPT_MIN_ROUNDS) return SV_OK;
  // Mean over the window, oldest entry first.
  const int first = (a->next - a->count + a->window) % a->window;
  double sum = 0.0;
  for (int j = 0; j < a->count; ++j) sum += a->ratio[(first + j) % a->window];
  const double mean = sum / (double)a->count;
  if (mean > a->target + SV_ADAPT_BAND) {
    if (a->k < a->max_k) ++a->k;
  } else if (mean < a->target - SV_ADAPT_BAND) {
    if (a->k > a->min_k) --a->k;
  }
  return SV_OK;
}

int32_t sv_adapt_draft_length(const sv_adapt* a) { return a ? a->k : -1; }

}  // extern "C"
