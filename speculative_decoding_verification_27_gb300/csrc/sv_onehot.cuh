// sv_onehot.cuh -- launcher of the one-CTA-per-row verify kernel for one-hot
// proposals (onehot.cu), the path run_verify takes for batches of short rows
// without draft rows.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "sv_device.cuh"  // DF

namespace sv {

// Result of one target row for its request's commit (32 bytes; the
// workspace's per-row record).
struct alignas(16) RRow {
  float mc_p, mc_q;  // fp32(max z * c) of the row (0 if no finite logit); mc_q = 0
  DF S_p, S_q;       // sum of 2^(z c - mc_p); S_q = 0 (no draft rows)
  int am;            // greedy rows: the argmax
  unsigned accept;   // the slot's draft token is accepted (bonus rows: 1)
};
static_assert(sizeof(RRow) == 32, "row record is 32 bytes");

struct RParams {
  const void* target;           // [R_t, V], 16-byte aligned rows
  int V, B;
  const int32_t* draft_tokens;  // [R_d]
  const int32_t* cu;            // [B + 1]
  const uint8_t* mode;          // [B] or NULL
  const float* uniforms;        // [R_t, 2]
  float c;                      // log2(e) / T
  int32_t* out_tokens;
  int32_t* out_len;
  float* out_probs;             // [R_t, 2] or NULL
  unsigned* status;             // SV_DATA_* bits
  unsigned long long* arrive;   // [B] rows of each request finished; 0 between calls
  RRow* rows;                   // [row_cap]
  long long row_cap;            // target rows the workspace holds
  int greedy_all;
  int nvec;                     // 16-byte vectors per row
};

// Rows of at most this many 16-byte vectors (a draw's tile sums then fit
// one per thread): 1 MiB.
constexpr int kOneHotMaxVec = 65536;

// One CTA per row the workspace holds (rows past R_t = cu[B] + B leave at
// once). dtype: 0 fp32, 1 bf16.
cudaError_t launch_onehot_verify(const RParams& P, int dtype, cudaStream_t st);

}  // namespace sv
