// sv_greedy.cuh -- launcher of the strict-verification kernel (greedy.cu),
// the path run_verify takes for spec_verify_greedy on 16-byte vector rows.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "sv_cluster.cuh"  // CRow: a row's result for its request's commit

namespace sv {

struct GParams {
  const void* target;           // [R_t, V], 16-byte aligned rows
  int V, B;
  const int32_t* draft_tokens;  // [R_d]
  const int32_t* cu;            // [B + 1]
  int32_t* out_tokens;
  int32_t* out_len;
  unsigned* status;             // SV_DATA_* bits
  unsigned long long* arrive;   // [B] rows of each request finished; 0 between calls
  CRow* rows;                   // [row_cap]: accept bit and argmax per target row
  long long row_cap;            // target rows the workspace holds
  int nvec;                     // 16-byte vectors per row
};

// One CTA per row the workspace holds (rows past R_t = cu[B] + B leave at
// once). dtype: 0 fp32, 1 bf16.
cudaError_t launch_greedy_verify(const GParams& P, int dtype, cudaStream_t st);

}  // namespace sv
