// candidates.cu -- keep one of several verified draft candidates per request.
//
// "投机解码从零实现" (CSDN), §5.1 "批量验证": one target pass verifies several
// draft candidates that share a prefix, each returning its accepted tokens
// and gain. Here every candidate is verified as its own request of a
// spec_verify call; this kernel keeps, per request, the candidate with the
// longest committed length (the lowest candidate index among ties).
#include "../../include/spec_verify.h"

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kSelThreads = 256;

__global__ void __launch_bounds__(kSelThreads) select_kernel(const int32_t* __restrict__ cu_cand,
                                                             const int32_t* __restrict__ out_len, int B,
                                                             int32_t* __restrict__ best,
                                                             int32_t* __restrict__ best_len) {
  for (int b = blockIdx.x * kSelThreads + threadIdx.x; b < B; b += gridDim.x * kSelThreads) {
    const int c0 = cu_cand[b], c1 = cu_cand[b + 1];
    int bi = -1, bl = 0;
    for (int c = c0; c < c1; ++c) {
      const int l = out_len[c];
      if (bi < 0 || l > bl) {
        bi = c;
        bl = l;
      }
    }
    best[b] = bi;
    best_len[b] = bl;
  }
}

}  // namespace sv

extern "C" {

sv_status sv_select_candidates(const int32_t* cu_cand, const int32_t* out_len, int32_t B,
                               int32_t* best, int32_t* best_len, void* cuda_stream) {
  if (B < 0) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!cu_cand || !out_len || !best || !best_len || (uintptr_t)cu_cand % 4 || (uintptr_t)out_len % 4 ||
      (uintptr_t)best % 4 || (uintptr_t)best_len % 4)
    return SV_ERR_INVALID_ARG;
  int grid = (B + sv::kSelThreads - 1) / sv::kSelThreads;
  grid = grid > 152 ? 152 : grid;
  sv::select_kernel<<<grid, sv::kSelThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      cu_cand, out_len, B, best, best_len);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
