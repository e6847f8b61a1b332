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
// nl > 0: the row's kept logits are also listed, nl entries (token, logit)
// in the row's block of the kept lists, so that a draw from the row reads
// the list instead of the row. nl = 0: no list.
struct alignas(16) FStat {
  float mc;
  int ok;
  double S;
  int nl;
  int unused[3];
};
static_assert(sizeof(FStat) == 32, "filtered row statistics are 32 bytes");

// Entries of a kept list per target row, at most; more kept logits (ties at
// the threshold) leave no list.
constexpr int kKeptListCap = 256;

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
  int2* list_t;         // [rows_t, kKeptListCap] kept (token, logit bits) of the target rows, or NULL
  bool after_warp;      // the one-warp-per-row kernel ran first: skip the rows it finished
  unsigned* rows_left;  // set to 1 by the warp kernel for a row it leaves to the CTA kernel, which
                        // leaves at once while it reads 0 (the filtered commit clears it); or NULL
};

// Launches the thresholds; *warp_ran tells whether the one-warp-per-row
// kernel ran (then the statistics and kept lists of its rows are there).
cudaError_t launch_thresholds(const FtParams& P, int dtype, cudaStream_t st, bool* warp_ran);

// The filtered step's decisions, draws and commits for the requests whose
// rows all carry their statistics (and whose stop row its kept list), one
// CTA per request, before the verify kernel (fcommit.cu). Requests it leaves
// (greedy ones, K above 31, a row without statistics or list, bad offsets)
// raise *need_slow and keep done[b] = 0; the verify kernel then runs and
// skips the requests marked done, and otherwise leaves at once.
struct FcParams {
  const void* target;           // [R_t, V], 16-byte vector rows
  const void* draft;            // [R_d, V] or NULL (one-hot proposals)
  int V, B;
  int rows_t;                   // target rows the caller holds
  const int32_t* draft_tokens;  // [R_d]
  const int32_t* cu;            // [B+1]
  const uint8_t* mode;          // [B] or NULL
  const float* uniforms;        // [R_t, 2]
  float c;                      // log2(e) / T
  const float* thr_t;           // [R_t] thresholds
  const float* thr_d;           // [R_d] or NULL
  const FStat* fst_t;           // [R_t]
  const FStat* fst_d;           // [R_d] or NULL
  const int2* list_t;           // [R_t, kKeptListCap]
  int32_t* out_tokens;
  int32_t* out_len;
  float* out_probs;             // [R_t, 2] or NULL
  unsigned* status;             // the verify workspace's SV_DATA_* word
  unsigned* need_slow;          // raised (set to 1) if a request is left
  unsigned char* done;          // [B] 1: committed here
  unsigned* rows_left;          // the threshold kernels' word, cleared here; or NULL
};

cudaError_t launch_filtered_commit(const FcParams& P, int dtype, cudaStream_t st);

}  // namespace sv
