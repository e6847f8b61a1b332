// sv_filter.cuh -- launcher of the per-row top-k / top-p threshold kernel
// (filter.cu), used by the filtered verify entry point.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// Softmax statistics of a filtered row, left by the threshold kernel when
// its buffer held every kept logit of the row (ok = 1): mc = fp32(M * c) for
// the row maximum M, and S = sum over the kept logits z of 2^(z c - mc).
// ok = 0: the verify kernel computes them from the row.
struct alignas(16) FStat {
  float mc;
  int ok;
  double S;
};
static_assert(sizeof(FStat) == 16, "filtered row statistics are 16 bytes");

struct FtParams {
  const void* target;   // [R_t, V]
  const void* draft;    // [R_d, V] or NULL (one-hot proposals: no draft rows)
  int V, B;
  int rows_t;           // target rows the caller holds (threshold writes stop there)
  const int32_t* cu;    // [B+1]
  const uint8_t* mode;  // [B] or NULL
  float c;              // log2(e) / T
  int top_k;            // 0: off
  float top_p;          // >= 1: off
  bool vec;             // rows are 16-byte aligned with V * s % 16 == 0
  float* thr_t;         // [rows_t]
  float* thr_d;         // [rows_t - B]
  FStat* fst_t;         // [rows_t] filtered statistics of the target rows, or NULL
  FStat* fst_d;         // [rows_t - B] of the draft rows, or NULL
  bool after_warp;      // the one-warp-per-row kernel ran first: skip the rows it finished
};

cudaError_t launch_thresholds(const FtParams& P, int dtype, cudaStream_t st);

}  // namespace sv
