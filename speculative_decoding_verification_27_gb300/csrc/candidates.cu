// candidates.cu -- keep one of several verified draft candidates per request.
//
// "投机解码从零实现" (CSDN), §5.1 "批量验证": one target pass verifies several
// draft candidates that share a prefix, each returning its accepted tokens
// and gain. Here every candidate is verified as its own request of a
// spec_verify call; this kernel keeps one candidate per request, by one of
// two rules (SV_SELECT_* in the header):
//   uniform          candidate min(n - 1, floor(u * n)) of the request's n,
//                    u its selection uniform: independent of the outcomes,
//                    so the kept commit is distributed as one candidate's;
//   longest (biased) the longest committed length, lowest index among ties.
#include "../../include/spec_verify.h"

#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kSelThreads = 256;

__global__ void __launch_bounds__(kSelThreads) select_kernel(const int32_t* __restrict__ cu_cand,
                                                             const int32_t* __restrict__ out_len, int B,
                                                             int policy, const float* __restrict__ u_sel,
                                                             int32_t* __restrict__ best,
                                                             int32_t* __restrict__ best_len) {
  for (int b = blockIdx.x * kSelThreads + threadIdx.x; b < B; b += gridDim.x * kSelThreads) {
    const int c0 = cu_cand[b], c1 = cu_cand[b + 1];
    int bi = -1, bl = 0;
    if (c1 > c0 && policy == SV_SELECT_UNIFORM) {
      // floor(u * n) is exact in fp64 (a float times an int below 2^31).
      const int n = c1 - c0;
      const double u = (double)u_sel[b];
      const double j = u >= 0.0 ? floor(u * (double)n) : 0.0;
      bi = c0 + (j < (double)(n - 1) ? (int)j : n - 1);
      bl = out_len[bi];
    } else {
      for (int c = c0; c < c1; ++c) {
        const int l = out_len[c];
        if (bi < 0 || l > bl) {
          bi = c;
          bl = l;
        }
      }
    }
    best[b] = bi;
    best_len[b] = bl;
  }
}

}  // namespace sv

extern "C" {

sv_status sv_select_candidates(const int32_t* cu_cand, const int32_t* out_len, int32_t B,
                               int32_t policy, const float* u_select, int32_t* best,
                               int32_t* best_len, void* cuda_stream) {
  if (B < 0) return SV_ERR_INVALID_ARG;
  if (policy != SV_SELECT_UNIFORM && policy != SV_SELECT_LONGEST_BIASED) return SV_ERR_INVALID_ARG;
  if (policy == SV_SELECT_UNIFORM && (!u_select || (uintptr_t)u_select % 4)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!cu_cand || !out_len || !best || !best_len || (uintptr_t)cu_cand % 4 || (uintptr_t)out_len % 4 ||
      (uintptr_t)best % 4 || (uintptr_t)best_len % 4)
    return SV_ERR_INVALID_ARG;
  int grid = (B + sv::kSelThreads - 1) / sv::kSelThreads;
  grid = grid > 152 ? 152 : grid;
  sv::select_kernel<<<grid, sv::kSelThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      cu_cand, out_len, B, policy, u_select, best, best_len);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
