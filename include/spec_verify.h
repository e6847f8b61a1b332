/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verify-and-commit library (libspecverify.so).
 *
 * What the library computes is the verify-and-commit step of speculative
 * decoding and the model-free proposers (n-gram and suffix), as these pages
 * define them:
 *
 *   "Draft Model（草稿模型）" (compassingai.com), §2 "接受-拒绝准则" and the
 *   box "算法：Speculative Decoding (一步)": for draft slots i = 1..K in
 *   order, accept the draft token x̂_i with probability min(1, p(x̂_i)/q(x̂_i));
 *   at the first rejection emit a token drawn from norm(max(0, p - q)) and
 *   stop; if all K are accepted emit one more token drawn from p_{K+1}.
 *   Each round emits 1..K+1 tokens.
 *
 *   "投机解码从零实现" (CSDN), §3.2 "算法的数学推导" and §4.3 "验证器实现":
 *   both logit rows are divided by the temperature before the softmax;
 *   p'(x) = max(0, p(x) - q(x)) / Z with Z = sum_x max(0, p(x) - q(x));
 *   a draft probability q(x̂) <= 0 rejects.
 *
 *   "Speculative Decoding在分布式推理中的应用", §二 "推测解码的工作流程":
 *   strict verification accepts iff the draft token equals the target's own
 *   choice (with greedy decoding: the argmax).
 *
 *   "5.2 Draft 模型与无模型方案：怎样便宜地猜得更准", §4 "N-gram" and §6
 *   "动手实验": the prompt-lookup proposer; §4.3: a copied proposal is the
 *   one-hot distribution q(y) = 1 on the proposed token; §5 "Suffix
 *   Decoding": continuations ranked by how often they follow a suffix.
 *
 * Conventions for every entry point:
 *   - Array arguments are DEVICE pointers owned by the caller. The library
 *     allocates no device memory; scratch space is the caller's workspace
 *     (spec_verify_noalloc instead uses a fixed block inside the library).
 *   - Work is enqueued asynchronously on `cuda_stream` (a cudaStream_t; NULL
 *     is the legacy default stream). Results are valid once the stream has
 *     reached that point.
 *   - Errors visible on the host (NULL where a pointer is required, bad sizes,
 *     misaligned pointers, temperature <= 0) return SV_ERR_INVALID_ARG
 *     before anything is launched. A failed launch returns SV_ERR_CUDA.
 *   - Errors that depend on device data (offsets, token ids, rows without a
 *     finite logit) are found by the kernels, which never trap: they set bits
 *     in a status word inside the workspace (SV_DATA_* below), keep every
 *     memory access in bounds, and finish. sv_check_status() reads and clears
 *     that word. Outputs of a call whose status word is non-zero (other than
 *     the informational SV_DATA_DEGENERATE_RESIDUAL bit) are unspecified.
 *   - Logits must be finite or -inf (a masked token); NaN and +inf are not
 *     supported. Each row needs at least one finite logit.
 *
 * Packed ragged layout (B requests, request b has K_b >= 0 draft tokens):
 *   cu_draft[B+1]        exclusive prefix sums of K_b; cu_draft[0] = 0.
 *   R_d = cu_draft[B]    draft rows;  R_t = R_d + B  target rows.
 *   draft slot (b, i), i < K_b:   draft row / draft token at cu_draft[b] + i.
 *   target row (b, i), i <= K_b:  at cu_draft[b] + b + i. Row i is the
 *       target's distribution for draft slot i; row K_b is the bonus slot.
 *   Logit matrices are row-major [rows, V] with row stride V elements.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,   /* rejected on the host before any launch */
  SV_ERR_CUDA = 2,          /* a CUDA runtime call or launch failed */
  SV_ERR_TIMEOUT = 3,       /* a bounded device-side wait gave up (sv_check_status) */
  SV_ERR_UNIMPLEMENTED = 4, /* reserved */
  SV_ERR_DATA = 5           /* sv_check_status found device-side data errors */
} sv_status;

typedef enum { SV_FP32 = 0, SV_BF16 = 1 } sv_dtype;

enum { SV_MODE_SAMPLE = 0, SV_MODE_GREEDY = 1 };

/* Bits of the device status word (sv_check_status). */
#define SV_DATA_BAD_OFFSETS 0x1u   /* cu_draft[0] != 0, decreasing, or R_t beyond the workspace */
#define SV_DATA_BAD_TOKEN 0x2u     /* a draft token outside [0, V) (the slot is rejected) */
#define SV_DATA_EMPTY_ROW 0x4u     /* a sampled row without any finite logit */
#define SV_DATA_BAD_MODE 0x8u      /* mode[b] not SAMPLE or GREEDY (treated as SAMPLE) */
#define SV_DATA_DEGENERATE_RESIDUAL 0x10u /* informational: residual mass 0 after a reject; drew from p */
#define SV_DEV_COPY_TIMEOUT 0x20u  /* a bounded wait for an asynchronous copy gave up (never expected);
                                      the call's outputs are invalid and the workspace must be
                                      zero-filled again before reuse */

/*
 * Bytes of workspace spec_verify / spec_verify_greedy need for B requests,
 * R_t target rows and vocabulary size V (0 if an argument is out of range).
 * The workspace holds a 64-byte header, an 8-byte progress word per request,
 * per target row a 32-byte record and the tile sums (4 bytes per 1024
 * vocabulary entries) that a row streamed alone (a bonus row, or a draft
 * slot with a one-hot proposal) leaves for a draw there, a fixed 528 KiB region
 * for rows that the kernel splits across CTAs near the end of a call, and,
 * for up to min(B, 4096) final draws it splits the same way, a descriptor and
 * the partial sums of each. It must be 16-byte aligned and zero-filled
 * before its first use; every call leaves its counters at zero again, so
 * calls in stream order with the same B and V (the layout) may reuse it
 * without clearing. A call with another B or V needs it zero-filled again:
 * the counters then sit where the last call left other data. Calls that may
 * run concurrently (other streams) need distinct workspaces.
 */
size_t spec_verify_workspace_size(int32_t B, int32_t R_t, int32_t V);

/*
 * Lossless verify-and-commit ("Draft Model（草稿模型）", §2 and the algorithm
 * box; "投机解码从零实现" §3.2/§4.3).
 *
 *   target_logits  [R_t, V] dtype.
 *   draft_logits   [R_d, V] dtype, or NULL: every proposal is one-hot
 *                  (q = e_x̂, "5.2 Draft 模型与无模型方案" §4.3); then
 *                  min(1, p/q) = p(x̂) and the residual is p without x̂.
 *   dtype          SV_FP32 or SV_BF16 for both logit matrices.
 *   1 <= V <= 262144 (fp32) or 524288 (bf16); B >= 0 (B == 0 is a no-op).
 *   draft_tokens   [R_d] int32 proposed tokens (may be NULL when R_d == 0).
 *   cu_draft       [B+1] int32 offsets (see the layout above).
 *   mode           [B] uint8 SV_MODE_* per request, or NULL (all SAMPLE).
 *                  GREEDY requests use strict verification (as
 *                  spec_verify_greedy) and ignore draft rows and uniforms.
 *   uniforms       [R_t, 2] float32 in [0, 1): per target row, u (accept
 *                  test of that row's draft slot) and u' (the draw made at
 *                  that row, if it is the request's stop row).
 *   temperature    T > 0: p = softmax(z_target / T), q = softmax(z_draft / T).
 *   out_tokens     [R_t] int32: request b's committed tokens at
 *                  cu_draft[b] + b + j, j < out_len[b]; other entries are
 *                  left untouched.
 *   out_len        [B] int32 in [1, K_b + 1].
 *   out_probs      [R_t, 2] float32 or NULL. Draft slot rows get
 *                  (p(x̂_i), q(x̂_i)) for every i < K_b (also after the stop);
 *                  the bonus-slot row K_b gets (p_s(y), q_s(y)) of the final
 *                  token y drawn at the stop row s (q_s(y) = 0 for a bonus
 *                  draw). GREEDY requests get (-1, -1).
 *   workspace      device scratch, >= spec_verify_workspace_size(B, R_t, V)
 *                  bytes, 16-byte aligned, zero-filled before first use.
 *
 * Decision rule: accept slot i iff u_i < min(1, p(x̂_i)/q(x̂_i)), with
 * q(x̂_i) = 0 rejecting. The draw at stop row s takes the smallest k with
 * sum_{x<=k} r_x > u'_s * sum_x r_x in vocabulary order, r = max(0, p - q)
 * after a rejection and r = p for the bonus draw.
 */
sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      int32_t V, int32_t B, const int32_t* draft_tokens,
                      const int32_t* cu_draft, const uint8_t* mode, const float* uniforms,
                      float temperature, int32_t* out_tokens, int32_t* out_len,
                      float* out_probs, void* workspace, size_t workspace_bytes,
                      void* cuda_stream);

/*
 * Strict (greedy) verify-and-commit ("Speculative Decoding在分布式推理中的应用",
 * §二, strict verification): accept slot i iff x̂_i equals the argmax of
 * target row i (lowest index among ties); at the first mismatch, or at the
 * bonus row, emit that row's argmax. Bit-exact; no temperature, no
 * uniforms. Arguments as for spec_verify. On 16-byte-aligned rows whose
 * byte length is a multiple of 16, one CTA per target row streams the row
 * (sixteen 16-byte loads in flight per thread) and the request's last row
 * commits it; other rows take the persistent kernel.
 */
sv_status spec_verify_greedy(const void* target_logits, sv_dtype dtype, int32_t V, int32_t B,
                             const int32_t* draft_tokens, const int32_t* cu_draft,
                             int32_t* out_tokens, int32_t* out_len, void* workspace,
                             size_t workspace_bytes, void* cuda_stream);

/*
 * Which kernel runs spec_verify. Each computes the same step (the rule
 * above); the third, for one-hot batches, is described after this one:
 *   - a persistent kernel, a fixed number of CTAs per SM, streams rows
 *     through a shared-memory ring and commits each request as soon as its
 *     stop slot is known; the default for large batches;
 *   - a cluster kernel, one thread-block cluster of 8 CTAs per target row:
 *     the row (and its paired draft row) is held in the CTAs' shared memory,
 *     the slices' statistics are exchanged through distributed shared
 *     memory, every rejecting row (and every bonus row) draws its token at
 *     once, and each request's last row to finish commits it. For batches of
 *     few rows, where the persistent kernel's time is a chain of dependent
 *     steps rather than bytes.
 * The cluster kernel runs when the workspace holds at most `rows` target
 * rows (a workspace of spec_verify_workspace_size(B, R_t, V) bytes holds
 * R_t; each further row takes 32 + 4 * ceil(V / 1024) bytes), the rows are
 * 16-byte aligned with V * element size a multiple of 16, and a row pair fits 200 KB of
 * shared memory per CTA (V * element size <= 800 KB with draft rows, 1.6 MB
 * without). The filtered and no-allocation entry points always take the
 * persistent kernel.
 * Sets the process-wide threshold (0: never) and returns the previous one;
 * the initial value is SV_CLUSTER_ROWS_DEFAULT. Negative values are ignored
 * (the call then only returns the current threshold).
 */
#define SV_CLUSTER_ROWS_DEFAULT 64
int32_t sv_set_cluster_rows(int32_t rows);

/*
 * A third kernel takes one-hot batches (draft_logits NULL, as from the n-gram
 * or suffix proposer) of short rows that the cluster kernel does not: one
 * CTA per target row streams its row with register loads, takes the row's
 * decision, and the request's last row commits it, drawing from the stop row
 * read once more (from L2 at these sizes). It runs for rows of at most
 * `bytes` bytes (V * element size, and at most 1 MiB), 16-byte aligned with
 * V * element size a multiple of 16, in spec_verify (greedy requests of
 * such a batch included); the filtered and no-allocation entry points keep
 * the persistent kernel. Sets the process-wide limit (0: never) and returns the
 * previous one; the initial value is SV_ONEHOT_ROW_BYTES_DEFAULT. Negative
 * values are ignored (the call then only returns the current limit).
 */
#define SV_ONEHOT_ROW_BYTES_DEFAULT 131072 /* 128 KiB */
int32_t sv_set_onehot_row_bytes(int32_t bytes);

/*
 * Top-k / top-p filtered verify-and-commit ("投机解码从零实现", §5.4
 * "采样策略对比": top-k and nucleus rejection sampling keep the output
 * distribution when the same filter is applied to the target and the draft
 * distributions). Before the step, each sampled target row and draft row is
 * filtered, then renormalised:
 *   top_k (1 <= top_k < V; 0 or >= V: off): keep every token whose logit is
 *     >= the row's k-th largest logit (ties at the boundary are all kept);
 *   then top_p (0 < top_p < 1; >= 1: off): over the kept tokens, walk the
 *     distinct logit values from the largest down and keep them until the
 *     cumulative mass first reaches top_p; the last value's whole tie group
 *     is kept, the rest dropped.
 * The accept test, the residual max(0, p' - q') and the bonus draw then use
 * the filtered p' and q'. The step is lossless with respect to the filtered
 * target p' when the proposals were drawn from the filtered q'. One-hot
 * proposals (draft_logits NULL) filter the target rows only. Greedy
 * requests are unaffected, since a filter never removes the argmax.
 *
 * Arguments as for spec_verify, plus:
 *   R_t        target rows the caller holds (cu_draft[B] + B); the
 *              thresholds occupy the start of the workspace.
 *   top_k, top_p  the filters (top_k >= 0, top_p > 0).
 *   workspace  >= spec_verify_filtered_workspace_size(B, R_t, V) bytes,
 *              16-byte aligned, zero-filled before first use and again
 *              before a call with another B, R_t or V (the layout).
 * Per row, the threshold step finds the row's threshold:
 *   - top-k up to 128 on 16-byte-aligned rows whose width is a multiple of
 *     16 bytes: one warp per row reads the row once, collects the logits
 *     that can be kept in shared memory and takes the k-th largest of them
 *     (top-p then cuts that set). From the same buffer it leaves the
 *     filtered row's softmax statistics and, for target rows, the list of
 *     kept (token, logit) pairs, so the verify kernel does not read those
 *     rows again: a draw from such a row reads the list and, for a
 *     residual, the draft row at the listed tokens;
 *   - other rows (and rows whose kept logits do not fit that buffer): a
 *     CTA per row by a radix select on order-preserving keys, counts for
 *     top-k and masses 2^(z c - M c) for top-p, summed exactly in 64-bit
 *     fixed point from their fp32 values. For top-k up to 256, and for
 *     top-p alone, the row is read once; rows whose candidates do not fit
 *     (long tie groups at the threshold, or flat rows under top-p) and
 *     larger k take several passes over the row.
 * The verify step then counts every logit below its row's threshold as
 * -inf. When the one-warp-per-row kernel ran, a commit kernel with one CTA
 * per request comes next: for a sampled request with K <= 31 whose rows all
 * carry their statistics and whose stop row its kept list, it decides every
 * slot from z(x̂) alone, draws from the stop row's list and commits, without
 * reading any row again. The verify kernel then runs only for the requests
 * it left (greedy ones, larger K, rows without statistics or list), and
 * returns at once when there are none. Both take the same decisions in the
 * same arithmetic, so the split changes no output. A top-p decision within
 * about 1e-6 of its boundary can differ from a float64 evaluation.
 */
size_t spec_verify_filtered_workspace_size(int32_t B, int32_t R_t, int32_t V);
sv_status spec_verify_filtered(const void* target_logits, const void* draft_logits,
                               sv_dtype dtype, int32_t V, int32_t B, int32_t R_t,
                               const int32_t* draft_tokens, const int32_t* cu_draft,
                               const uint8_t* mode, const float* uniforms, float temperature,
                               int32_t top_k, float top_p, int32_t* out_tokens,
                               int32_t* out_len, float* out_probs, void* workspace,
                               size_t workspace_bytes, void* cuda_stream);

/*
 * spec_verify without a caller workspace: the scratch memory lives in a
 * fixed block that is part of the library's device image, so the call
 * allocates nothing and takes no workspace argument. The pages have no
 * counterpart; this is a deployment convenience, not part of the method.
 *
 * Who needs it. Some callers cannot hand over a workspace:
 *   - plain C programs that have no device allocator of their own;
 *   - serving loops that reserve all device memory when they start and may
 *     not allocate or free while requests are in flight, where a cudaMalloc
 *     could fail, or stall the whole device until it completes.
 * This entry point lets them verify without any allocation, by the library
 * or by the caller.
 *
 * Limit. The fixed block holds SV_NOALLOC_SCRATCH_BYTES (4 MiB). A batch
 * fits when spec_verify_workspace_size(B, 0, V) + 32 * R_t <=
 * SV_NOALLOC_SCRATCH_BYTES (for example B = 256, K = 7, V = 151936 needs
 * about 0.9 MiB): the block keeps a 32-byte record per row and no per-row
 * tile sums, so a draw at a bonus or one-hot row reads its row again.
 *   - If B and V alone need more than the block, the call returns
 *     SV_ERR_INVALID_ARG before anything is enqueued.
 *   - R_t is known only on the device (cu_draft[B] + B). If the rows do not
 *     fit, the kernel sets SV_DATA_BAD_OFFSETS in status_out and writes no
 *     output.
 *
 * Arguments, outputs and validation are those of spec_verify, except:
 *   status_out   optional device pointer to one uint32_t. After the call it
 *                holds that call's SV_DATA_* / SV_DEV_* bits (0 = clean).
 *                NULL: the bits are dropped.
 *
 * Every call clears the part of the block that must start at zero (the
 * counters and per-request state) on the stream before the kernel runs, so
 * a call never inherits state, not even from a call that failed.
 *
 * One block per device, shared by all callers on that device:
 *   - calls on one device must not overlap. Two calls in flight at the same
 *     time (on different streams, or from different threads without
 *     ordering) race on the block and both results are undefined.
 *     Issue them on one stream, or order them yourself;
 *   - the first call on a device does one-time setup: it looks up the
 *     block's address and configures the kernel. Make that first call
 *     outside any stream capture.
 */
#define SV_NOALLOC_SCRATCH_BYTES 4194304u /* 4 MiB */
sv_status spec_verify_noalloc(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                              int32_t V, int32_t B, const int32_t* draft_tokens,
                              const int32_t* cu_draft, const uint8_t* mode,
                              const float* uniforms, float temperature, int32_t* out_tokens,
                              int32_t* out_len, float* out_probs, uint32_t* status_out,
                              void* cuda_stream);

/*
 * Vocabulary-sharded verify-and-commit: the step of spec_verify ("Draft
 * Model（草稿模型）" §2) when each rank holds only a slice of the vocabulary,
 * as a tensor-parallel LM head leaves it. The pages deploy the draft and the
 * target on separate nodes ("Speculative Decoding在分布式推理中的应用" §三)
 * but do not split the vocabulary; this form is the library's own, and the
 * only split of the step that needs an exchange between GPUs. Shard s of S
 * holds columns [v0_s, v0_s + Vs_s) of every target and draft row; the
 * shards cover [0, V) in rank order. Per call,
 * every rank runs, between two exchanges that the caller performs (the
 * Python binding's spec_verify_vsharded does them with torch.distributed):
 *
 *   sv_vshard_stats    per row of its slice: mc = fp32(max z * c), the sum
 *                      S of 2^(z c - mc) (c = log2(e)/T), the logit of the
 *                      row's proposed token if the shard holds it, and the
 *                      argmax (largest logit, lowest global index);
 *   -- all-gather of the statistics: [S, R_t] (and [S, R_d]) in rank order --
 *   sv_vshard_decide   every rank, identically: the whole-vocabulary p(x̂),
 *                      q(x̂), the accept tests (as spec_verify), the stop
 *                      slot, the accepted prefix, out_len, out_probs of the
 *                      draft slots, greedy tokens, and one draw job per
 *                      sampled request (in `jobs`, sv_vshard_jobs_bytes(B));
 *   sv_vshard_masses   this shard's mass of the draw's r (max(0, p - q), p
 *                      without the rejected one-hot proposal, or p) over its
 *                      slice, per request, in units of 2^(z c - Mc_p);
 *   -- all-gather of the masses: [S, B], an exclusive scan in shard order --
 *   sv_vshard_draw     the shard whose part of the scan holds u' * Z
 *                      (u' = uniforms[stop row, 1]) locates the token in its
 *                      slice; the others give -1 (and probabilities -1);
 *   -- element-wise max over the shards of draw_tok [B] and draw_prob [B, 2] --
 *   sv_vshard_finish   writes the drawn tokens (and (p(y), q(y)) into the
 *                      bonus rows of out_probs).
 *
 * Arguments as for spec_verify, plus: logits are the shard's [rows, ld]
 * row-major slices (ld >= Vs elements); R_t = cu_draft[B] + B; status is a
 * device uint32 that collects SV_DATA_* bits (clear it before the call).
 * All pointers are device pointers; every call is asynchronous on its
 * stream. Results equal spec_verify's up to the summation order of the
 * shards (decisions within ~1e-6 of a tie can differ).
 */
typedef struct {
  float mc;       /* fp32(max z * c) of the slice's row, 0 if it has no finite logit */
  float zx;       /* logit of the row's proposed token, if has_x */
  double S;       /* sum of 2^(z c - mc) over the slice's row */
  float amax_v;   /* largest logit of the slice's row (-inf if none) */
  int32_t amax_i; /* its lowest global index (INT32_MAX if none) */
  int32_t has_x;  /* this shard holds the proposed token */
  int32_t pad;
} sv_shard_stat;
size_t sv_vshard_jobs_bytes(int32_t B);
sv_status sv_vshard_stats(const void* logits, sv_dtype dtype, int32_t rows, int32_t Vs, int64_t ld,
                          int32_t v0, int32_t V, int32_t is_draft, int32_t B, const int32_t* cu_draft,
                          const int32_t* draft_tokens, float temperature, sv_shard_stat* out,
                          uint32_t* status, void* cuda_stream);
sv_status sv_vshard_decide(const sv_shard_stat* target_stats, const sv_shard_stat* draft_stats,
                           int32_t S, int32_t V, int32_t B, int32_t R_t, const int32_t* cu_draft,
                           const int32_t* draft_tokens, const uint8_t* mode, const float* uniforms,
                           float temperature, int32_t* out_tokens, int32_t* out_len, float* out_probs,
                           void* jobs, uint32_t* status, void* cuda_stream);
sv_status sv_vshard_masses(const void* target, const void* draft, sv_dtype dtype, int32_t Vs, int64_t ld,
                           int32_t v0, int32_t B, int32_t R_t, const int32_t* cu_draft,
                           const sv_shard_stat* target_stats, const void* jobs, float temperature,
                           double* masses, void* cuda_stream);
sv_status sv_vshard_draw(const void* target, const void* draft, sv_dtype dtype, int32_t Vs, int64_t ld,
                         int32_t v0, int32_t shard, int32_t S, int32_t B, int32_t R_t,
                         const int32_t* cu_draft, const double* masses, const sv_shard_stat* target_stats,
                         const void* jobs, const float* uniforms, float temperature, int32_t* draw_tok,
                         float* draw_prob, uint32_t* status, void* cuda_stream);
sv_status sv_vshard_finish(const void* jobs, int32_t B, int32_t R_t, const int32_t* draw_tok,
                           const float* draw_prob, int32_t* out_tokens, float* out_probs, uint32_t* status,
                           void* cuda_stream);

/*
 * N-gram / prompt-lookup proposer ("5.2 Draft 模型与无模型方案", §4.1 and §6):
 * for n = min(max_n, L) down to min_n, take the tail h[L-n, L) of the
 * history and find the most recent earlier start s, 0 <= s <= L-2n-1, with
 * h[s, s+n) equal to the tail (the match ends before the tail starts and
 * leaves a non-empty continuation); propose h[s+n, min(s+n+max_tokens, L-n)).
 * Without a match for any n: out_n = 0 and out_count = 0.
 *
 *   histories   [B, hist_stride] int32 token ids; history b holds hist_len[b]
 *               tokens (clamped to [0, hist_stride]).
 *   min_n >= 1, max_n >= min_n, max_tokens >= 0, B >= 0.
 *   out_tokens  [B, max_tokens] int32: proposal b in row b; entries past
 *               out_count[b] are set to -1.
 *   out_count   [B] int32 proposal lengths.
 *   out_n       [B] int32 matched window length (0 if none).
 * Bit-exact. No workspace.
 */
sv_status ngram_propose(const int32_t* histories, int64_t hist_stride, const int32_t* hist_len,
                        int32_t B, int32_t min_n, int32_t max_n, int32_t max_tokens,
                        int32_t* out_tokens, int32_t* out_count, int32_t* out_n,
                        void* cuda_stream);

/*
 * Frequency-ranked suffix proposer ("5.2 Draft 模型与无模型方案", §5
 * "Suffix Decoding"): §5.1 ranks the continuations seen after a suffix by
 * how often they occur, and warns that dispersed continuations make long
 * proposals unwise; §5.2 makes the configured length a ceiling, not a fixed
 * length. The page prescribes no algorithm; this is the reading:
 *   - the tail is the longest h[L-n, L), n = min(max_n, L) down to min_n,
 *     with an earlier occurrence at some start s, 0 <= s <= L-2n-1 (the
 *     starts ngram_propose admits); the max_occ occurrences with the largest
 *     s are the voters;
 *   - step j = 0, 1, ...: each voter whose continuation token h[s+n+j] lies
 *     before the tail (s+n+j < L-n) votes for it; the token with the most
 *     votes is proposed (among equal counts, the token of the voter with the
 *     largest s); for j >= 1 the proposal ends instead when the winner's
 *     votes are fewer than min_share x the votes cast (compared in double
 *     precision, min_share widened from float); only the winner's voters
 *     vote in the next step; the proposal ends at max_tokens or when no
 *     voter is left.
 * With max_occ = 1 and min_share = 0 the result is ngram_propose's.
 *
 *   histories, hist_len, B, min_n, max_n, max_tokens, out_tokens, out_count,
 *   out_n: as for ngram_propose (rows padded with -1; out_n = 0 and
 *   out_count = 0 without a match).
 *   min_share   in [0, 1]; max_occ in [1, SV_SUFFIX_MAX_OCC].
 * Bit-exact. No workspace. Histories with hist_stride <= 16384 are staged in
 * shared memory; longer ones are read from global memory.
 */
#define SV_SUFFIX_MAX_OCC 256
sv_status suffix_propose(const int32_t* histories, int64_t hist_stride, const int32_t* hist_len,
                         int32_t B, int32_t min_n, int32_t max_n, int32_t max_tokens,
                         float min_share, int32_t max_occ, int32_t* out_tokens,
                         int32_t* out_count, int32_t* out_n, void* cuda_stream);

/*
 * Glue from ngram_propose (or suffix_propose) to spec_verify: cu_draft[B+1] = exclusive prefix
 * sums of counts[B] (clamped to [0, max_tokens]), and the proposals of
 * tokens[B, max_tokens] packed to packed[cu_draft[b] + i] (capacity
 * B * max_tokens). One launch on the stream.
 */
sv_status sv_pack_drafts(const int32_t* tokens, const int32_t* counts, int32_t B,
                         int32_t max_tokens, int32_t* cu_draft, int32_t* packed,
                         void* cuda_stream);

/*
 * Multi-candidate verification ("投机解码从零实现", §5.1 "批量验证": one
 * target pass verifies several draft candidates, each returning its
 * accepted tokens and gain; the page does not say which result to keep).
 * Flatten every request's candidates into one spec_verify call, each
 * candidate its own request; request b owns candidates cu_cand[b] ..
 * cu_cand[b+1]-1 of that call. This call keeps one candidate per request:
 * best[b] is its index in the flattened call (-1 if the request had no
 * candidate) and best_len[b] its out_len (0 then). The rule is `policy`:
 *
 *   SV_SELECT_UNIFORM: candidate min(n - 1, floor(u_select[b] * n)) of the
 *     request's n candidates (a negative u picks the first). u_select [B]
 *     float32 holds one uniform in [0, 1) per request, drawn independently
 *     of the verify uniforms. The choice depends on no verification outcome,
 *     so the kept commit is distributed exactly as a single candidate's: the
 *     step stays lossless ("Draft Model（草稿模型）", §2). It does not raise
 *     the expected number of committed tokens over one candidate.
 *   SV_SELECT_LONGEST_BIASED: the longest committed length (lowest index
 *     among ties); u_select may be NULL. This raises the expected gain but
 *     looks at the outcomes: each candidate alone is lossless, the choice
 *     among them is not, and the kept tokens no longer follow the target
 *     distribution. Opt in knowingly.
 *
 * All pointers are device arrays; asynchronous on `cuda_stream`.
 * SV_ERR_INVALID_ARG for an unknown policy, a missing u_select under
 * SV_SELECT_UNIFORM, bad pointers or B < 0.
 */
enum { SV_SELECT_UNIFORM = 0, SV_SELECT_LONGEST_BIASED = 1 };
sv_status sv_select_candidates(const int32_t* cu_cand, const int32_t* out_len, int32_t B,
                               int32_t policy, const float* u_select, int32_t* best,
                               int32_t* best_len, void* cuda_stream);

/*
 * Acceptance statistics ("5.2 Draft 模型与无模型方案", §7.1 and §7.2),
 * accumulated on the device over any number of verify calls.
 *
 * sv_accumulate_metrics adds one call's rounds to *metrics (a DEVICE
 * pointer to a caller-owned, 8-byte aligned sv_metrics that the caller
 * zero-fills to start a window). It reads the call's cu_draft [B+1] and
 * out_len [B] (device) after spec_verify / spec_verify_greedy has run on the
 * same stream. Each request is one round. Its stop slot is out_len - 1
 * (clamped to [0, K_b]): slots before it were accepted, the slot itself was
 * rejected, or was the bonus slot. Asynchronous on `cuda_stream`;
 * SV_ERR_INVALID_ARG for bad pointers or B < 0. Per-slot counts cover slots
 * i < SV_METRICS_MAX_POS; the totals cover every slot.
 *
 * Quantities the pages define, from the counters:
 *   draft acceptance rate      accepted / drafted            (C / D)
 *   mean acceptance length     1 + accepted / rounds         (1 + C / R)
 *   candidate coverage         rounds_with_draft / rounds
 *   conditional rate of slot i accepted_at[i] / reached[i]   (given all before it)
 *   rate through slot i        accepted_at[i] / offered[i]   (all of 0..i accepted)
 */
#define SV_METRICS_MAX_POS 32
typedef struct {
  unsigned long long rounds;            /* R: requests verified */
  unsigned long long rounds_with_draft; /* rounds with K_b > 0 */
  unsigned long long drafted;           /* D: sum of K_b */
  unsigned long long accepted;          /* C: sum of stop slots (accepted draft tokens) */
  unsigned long long committed;         /* sum of out_len = C + R */
  unsigned long long offered[SV_METRICS_MAX_POS];     /* rounds with K_b > i */
  unsigned long long reached[SV_METRICS_MAX_POS];     /* rounds that tested slot i */
  unsigned long long accepted_at[SV_METRICS_MAX_POS]; /* rounds that accepted slots 0..i */
} sv_metrics;
sv_status sv_accumulate_metrics(const int32_t* cu_draft, const int32_t* out_len, int32_t B,
                                sv_metrics* metrics, void* cuda_stream);

/*
 * Sliding-window draft-length controller ("投机解码从零实现", §5.2
 * "动态草稿长度策略"), host code. Each round adds its accepted fraction
 * accepted_len / max(draft_len, 1) to a window of the last `window` rounds.
 * Once the window holds at least SV_ADAPT_MIN_ROUNDS rounds, every update
 * compares the window's mean m with `target`:
 *   - m > target + SV_ADAPT_BAND: the draft length grows by one, up to max_k;
 *   - m < target - SV_ADAPT_BAND: it shrinks by one, down to min_k.
 * The mean is summed oldest round first in double precision. One
 * controller per request stream; the struct is plain data (copyable, no
 * allocation). SV_ERR_INVALID_ARG for NULL, window outside
 * [1, SV_ADAPT_MAX_WINDOW], k bounds out of order, or accepted_len outside
 * [0, draft_len].
 */
#define SV_ADAPT_MAX_WINDOW 1024
#define SV_ADAPT_MIN_ROUNDS 10
#define SV_ADAPT_BAND 0.1
typedef struct {
  int32_t window, min_k, max_k, k, count, next;
  double target;
  double ratio[SV_ADAPT_MAX_WINDOW]; /* ring of accepted fractions */
} sv_adapt;
sv_status sv_adapt_init(sv_adapt* a, int32_t window, int32_t min_k, int32_t max_k, double target,
                        int32_t initial_k);
sv_status sv_adapt_update(sv_adapt* a, int32_t draft_len, int32_t accepted_len);
int32_t sv_adapt_draft_length(const sv_adapt* a);

/*
 * Synchronizes `cuda_stream`, reads the status word of `workspace` into
 * *out_bits (SV_DATA_* / SV_DEV_* bits) and clears it. Returns SV_OK when no
 * error bit is set (SV_DATA_DEGENERATE_RESIDUAL alone is informational),
 * SV_ERR_TIMEOUT if SV_DEV_COPY_TIMEOUT is set, SV_ERR_DATA for other bits,
 * or SV_ERR_CUDA / SV_ERR_INVALID_ARG.
 */
sv_status sv_check_status(void* workspace, void* cuda_stream, uint32_t* out_bits);

/* Static, human-readable name of a status code. */
const char* sv_status_string(sv_status status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
