// sv_cluster.cuh -- launcher of the cluster verify kernel (cluster.cu), the
// path run_verify takes for batches of few rows.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// Result of one target row, left for the request's commit (16 bytes).
struct alignas(16) CRow {
  unsigned accept;  // the slot's draft token is accepted
  int y;            // greedy rows: the argmax; sampled rows that reject (or the
                    // bonus row): the drawn token; otherwise -1
  float py, qy;     // p(y), q(y) of the drawn token
};
static_assert(sizeof(CRow) == 16, "cluster row result is 16 bytes");

struct CParams {
  const void* target;           // [R_t, V], 16-byte aligned rows
  const void* draft;            // [R_d, V] or NULL (one-hot proposals)
  int V, B;
  const int32_t* draft_tokens;  // [R_d]
  const int32_t* cu;            // [B + 1]
  const uint8_t* mode;          // [B] or NULL
  const float* uniforms;        // [R_t, 2]
  float c;                      // log2(e) / T
  int32_t* out_tokens;
  int32_t* out_len;
  float* out_probs;             // [R_t, 2] or NULL
  unsigned* status;             // SV_DATA_* / SV_DEV_* bits
  unsigned long long* arrive;   // [B] rows of each request finished; 0 between calls
  CRow* rows;                   // [row_cap]
  long long row_cap;            // target rows the workspace holds
  int greedy_all;
  int nvec;                     // 16-byte vectors per row
  int vp;                       // 16-byte vectors per CTA slice
};

// CTAs per cluster: one cluster per target row.
constexpr int kCluster = 8;

// Dynamic shared memory of the cluster kernel for rows of `row_bytes` (a
// multiple of 16) with or without draft rows; 0 if they do not fit.
size_t cluster_smem_bytes(size_t row_bytes, bool has_draft);

// Launches one cluster per row the workspace holds (row_cap clusters; those
// past R_t = cu[B] + B leave at once). dtype: 0 fp32, 1 bf16.
cudaError_t launch_cluster_verify(const CParams& P, int dtype, cudaStream_t st);

}  // namespace sv
