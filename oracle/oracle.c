/*
 * oracle.c -- plain float64 CPU oracle for the verify-and-commit step of
 * speculative decoding and for the n-gram (prompt-lookup) proposer.
 *
 * TEST INFRASTRUCTURE. This file exists to check the CUDA library against
 * the method as the pages define it. Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg load it. The CUDA library never
 * links it, and it shares no code, header or table with the CUDA library.
 *
 * Everything here is deliberately slow and literal: float64 throughout,
 * one row at a time, a sequential loop over the draft positions that stops
 * at the first rejection, exactly in the order of the algorithm box.
 *
 * Sources (page title, then section):
 *   [DM-rule]  "Draft Model（草稿模型）", §2 "接受-拒绝准则":
 *              accept x̂ with probability min(1, p(x̂)/q(x̂)); on rejection
 *              sample from norm(max(0, p(x) - q(x))).
 *   [DM-alg]   same page, box "算法：Speculative Decoding (一步)", step 3:
 *              positions i = 1..K in order; the first rejection emits
 *              [x̂_1..x̂_{i-1}, x_new] and ends the round; if all K are
 *              accepted, one extra token is drawn from p_{K+1}.
 *   [SDS-3.2]  "投机解码从零实现" (CSDN), §3.2 "算法的数学推导":
 *              reject_prob = max(0, 1 - p/q); p'(x) = max(0, p-q)/Z,
 *              Z = sum_x max(0, p(x)-q(x)).
 *   [SDS-4.3]  same article, §4.3 "验证器实现": both logit rows are
 *              divided by the temperature before the softmax; a draft
 *              probability q <= 0 rejects with certainty.
 *   [DSD-2]    "Speculative Decoding在分布式推理中的应用", §二 "推测解码的
 *              工作流程": strict verification accepts iff the draft token
 *              equals the target's own choice (greedy: the argmax).
 *   [PL-4.3]   "5.2 Draft 模型与无模型方案", §4.3: a copied (deterministic)
 *              proposal is the distribution q(y)=1 on the proposed token.
 *   [PL-6]     same page, §6 "动手实验：匹配窗口与候选覆盖": the n-gram
 *              proposer (longest window first, most recent match that ends
 *              before the current tail, non-empty continuation, truncated
 *              to max_tokens).
 *
 * Readings where the pages are silent:
 *   - accept iff u < min(1, p/q) with u a supplied uniform in [0,1);
 *   - the correction/bonus draw is the inverse CDF in vocabulary order:
 *     the smallest k with C_k > u' * Z, C_k = sum_{x<=k} r_x; if rounding
 *     leaves no such k, the last index with r_x > 0;
 *   - if Z == 0 after a rejection (impossible in exact arithmetic), draw
 *     from p instead; the row is flagged;
 *   - greedy rows ignore the temperature (it does not move the argmax);
 *     ties go to the lowest index;
 *   - one-hot q ignores the temperature; its residual is p with the
 *     proposed token's mass removed.
 *
 * Parity pins: see tests/test_oracle_pins.py (worked example p=0.4,
 * q=0.6 -> reject 1/3; closed-form residuals; black-box lattice integration
 * of the emitted marginal against p; chi-square on a V=16 toy; argmax
 * semantics; the printed n-gram cases; brute force against a naive search).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_FP32 0
#define OR_BF16 1
#define OR_MODE_SAMPLE 0
#define OR_MODE_GREEDY 1

/* Decision margin below which a row is flagged (spec tolerance). */
#define OR_MARGIN_EPS 1e-6

/* ------------------------------------------------------------------ */
/* Neumaier-compensated summation.                                     */
/* ------------------------------------------------------------------ */
typedef struct {
  double sum;
  double comp;
} nsum_t;

static void nsum_add(nsum_t* s, double x) {
  double t = s->sum + x;
  if (fabs(s->sum) >= fabs(x))
    s->comp += (s->sum - t) + x;
  else
    s->comp += (x - t) + s->sum;
  s->sum = t;
}

static double nsum_value(const nsum_t* s) { return s->sum + s->comp; }

/* ------------------------------------------------------------------ */
/* Logit access: fp32 or bf16 (raw 16-bit pattern), widened exactly.   */
/* ------------------------------------------------------------------ */
static double logit_at(const void* base, int dtype, int64_t idx) {
  if (dtype == OR_FP32) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Temperature softmax of one row:
 *   p_x = exp((z_x - m)/T) / sum_y exp((z_y - m)/T),  m = max_y z_y.
 * [SDS-4.3] divides the logits by T before F.softmax; subtracting the row
 * maximum does not change the value and keeps exp() in range.
 * Returns the sum (in units of exp((z-m)/T)); 0 means the row had no
 * finite logit. */
double oracle_softmax(const void* row, int dtype, int V, double T, double* p) {
  double m = -INFINITY;
  for (int x = 0; x < V; ++x) {
    double z = logit_at(row, dtype, x);
    if (z > m) m = z;
  }
  if (!(m > -INFINITY)) {
    for (int x = 0; x < V; ++x) p[x] = 0.0;
    return 0.0;
  }
  nsum_t s = {0.0, 0.0};
  for (int x = 0; x < V; ++x) {
    double e = exp((logit_at(row, dtype, x) - m) / T);
    p[x] = e;
    nsum_add(&s, e);
  }
  double S = nsum_value(&s);
  for (int x = 0; x < V; ++x) p[x] /= S;
  return S;
}

/* Top-k / top-p filtered temperature softmax (the filters that
 * "投机解码从零实现" §5.4 lists as distribution-preserving verify
 * strategies; the same filter is applied to the target and the draft row).
 * Readings, in this order:
 *   top-k (1 <= top_k < V): keep every x whose logit is >= the k-th largest
 *     logit (ties at the boundary are all kept);
 *   top-p (0 < top_p < 1): on the renormalised top-k distribution, walk the
 *     distinct kept values from the largest down; keep the values whose
 *     cumulative mass first reaches top_p (a value's whole tie group counts
 *     together), drop the rest.
 * p receives the renormalised filtered distribution. *margin receives the
 * distance of the top-p decision from equality, min(top_p - C_before,
 * C_at - top_p) in normalised mass (+inf when top-p is off). Returns the
 * unfiltered normaliser as oracle_softmax does (0: no finite logit). */
static int cmp_desc(const void* a, const void* b) {
  double x = *(const double*)a, y = *(const double*)b;
  return x < y ? 1 : (x > y ? -1 : 0);
}

double oracle_filtered_softmax(const void* row, int dtype, int V, double T, int top_k,
                               double top_p, double* p, double* margin) {
  if (margin) *margin = INFINITY;
  const int use_k = top_k >= 1 && top_k < V;
  const int use_p = top_p > 0.0 && top_p < 1.0;
  double S_all = oracle_softmax(row, dtype, V, T, p);
  if (!(S_all > 0.0) || (!use_k && !use_p)) return S_all;
  double* z = (double*)malloc(sizeof(double) * (size_t)V);
  double* sorted = (double*)malloc(sizeof(double) * (size_t)V);
  if (!z || !sorted) {
    free(z);
    free(sorted);
    return -1.0;
  }
  for (int x = 0; x < V; ++x) z[x] = sorted[x] = logit_at(row, dtype, x);
  qsort(sorted, (size_t)V, sizeof(double), cmp_desc);
  const double m = sorted[0];
  double thr = use_k ? sorted[top_k - 1] : -INFINITY;
  if (use_p) {
    /* Mass of the top-k set, then the cumulative mass by distinct value. */
    nsum_t tot = {0.0, 0.0};
    for (int x = 0; x < V; ++x)
      if (z[x] >= thr) nsum_add(&tot, exp((z[x] - m) / T));
    const double S_k = nsum_value(&tot);
    nsum_t cum = {0.0, 0.0};
    double before = 0.0;
    int j = 0;
    while (j < V && sorted[j] >= thr) {
      const double v = sorted[j];
      int g = j;
      while (g < V && sorted[g] == v) {
        nsum_add(&cum, exp((v - m) / T));
        ++g;
      }
      const double at = nsum_value(&cum) / S_k;
      if (at >= top_p) {
        if (margin) *margin = fmin(top_p - before, at - top_p);
        if (v > thr) thr = v;
        break;
      }
      before = at;
      j = g;
    }
  }
  nsum_t s = {0.0, 0.0};
  for (int x = 0; x < V; ++x) {
    p[x] = z[x] >= thr ? exp((z[x] - m) / T) : 0.0;
    nsum_add(&s, p[x]);
  }
  const double S = nsum_value(&s);
  for (int x = 0; x < V; ++x) p[x] /= S;
  free(z);
  free(sorted);
  return S_all;
}

/* Greedy choice of the target: the first index holding the maximum
 * (torch.argmax semantics), compared on the exact logit values. */
int oracle_argmax(const void* row, int dtype, int V) {
  int best = 0;
  double bv = logit_at(row, dtype, 0);
  for (int x = 1; x < V; ++x) {
    double z = logit_at(row, dtype, x);
    if (z > bv) {
      bv = z;
      best = x;
    }
  }
  return best;
}

/* Inverse-CDF draw from the unnormalised weights r[0..V):
 * Z = sum r; the smallest k with C_k = sum_{x<=k} r_x > u * Z.
 * If rounding leaves no such k, the last index with r_x > 0.
 * *margin receives min(u - C_{k-1}/Z, C_k/Z - u): the distance from u to
 * the chosen bucket's edges in normalised units. Returns -1 if Z <= 0. */
int oracle_inverse_cdf(const double* r, int V, double u, double* margin) {
  nsum_t zs = {0.0, 0.0};
  int last_pos = -1;
  for (int x = 0; x < V; ++x) {
    nsum_add(&zs, r[x]);
    if (r[x] > 0.0) last_pos = x;
  }
  double Z = nsum_value(&zs);
  if (!(Z > 0.0)) {
    if (margin) *margin = 0.0;
    return -1;
  }
  double target = u * Z;
  nsum_t c = {0.0, 0.0};
  double prev = 0.0;
  for (int k = 0; k < V; ++k) {
    nsum_add(&c, r[k]);
    double ck = nsum_value(&c);
    if (ck > target) {
      if (margin) {
        double lo = u - prev / Z, hi = ck / Z - u;
        *margin = lo < hi ? lo : hi;
      }
      return k;
    }
    prev = ck;
  }
  if (margin) *margin = 0.0;
  return last_pos;
}

/* ------------------------------------------------------------------ */
/* Verify-and-commit for one request.                                  */
/* ------------------------------------------------------------------ */
typedef struct {
  const void* target;        /* [R_t, V] */
  const void* draft;         /* [R_d, V] or NULL (one-hot q) */
  int dtype, V, B;
  const int32_t* draft_tokens; /* [R_d] */
  const int32_t* cu_draft;     /* [B+1] */
  const uint8_t* mode;         /* [B] or NULL */
  const float* uniforms;       /* [R_t, 2] */
  double T;
  int32_t* out_tokens;         /* [R_t] */
  int32_t* out_len;            /* [B] */
  double* out_probs;           /* [R_t, 2] or NULL */
  double* out_margin;          /* [R_t] or NULL: smallest decision margin per row */
  double* out_rho;             /* [R_t] or NULL: min(1, p/q) per tested row */
  int32_t* out_stop;           /* [B] or NULL */
  int top_k;                   /* 0: off */
  double top_p;                /* >= 1: off */
} verify_args_t;

static const void* row_ptr(const void* base, int dtype, int64_t row, int V) {
  size_t es = dtype == OR_FP32 ? 4 : 2;
  return (const char*)base + (size_t)row * (size_t)V * es;
}

static void set_margin(const verify_args_t* a, int64_t t, double m) {
  if (a->out_margin && m < a->out_margin[t]) a->out_margin[t] = m;
}

/* Softmax of a target or draft row with the call's filters; the top-p
 * decision margin is charged to target row t (the row of that slot). */
static void row_softmax(const verify_args_t* a, const void* row, double* p, int64_t t) {
  double fm = INFINITY;
  oracle_filtered_softmax(row, a->dtype, a->V, a->T, a->top_k, a->top_p, p, &fm);
  set_margin(a, t, fm);
}

/* Returns 0 on success, nonzero on invalid data for this request. */
static int verify_request(const verify_args_t* a, int b, double* p, double* q,
                          double* r) {
  const int V = a->V;
  const int K = a->cu_draft[b + 1] - a->cu_draft[b];
  const int64_t t0 = (int64_t)a->cu_draft[b] + b; /* first target row */
  const int64_t d0 = a->cu_draft[b];              /* first draft row  */
  const int greedy = a->mode && a->mode[b] == OR_MODE_GREEDY;
  if (K < 0) return 1;
  for (int i = 0; i < K; ++i) {
    int x = a->draft_tokens[d0 + i];
    if (x < 0 || x >= V) return 2;
  }
  for (int i = 0; i <= K; ++i) {
    if (a->out_margin) a->out_margin[t0 + i] = INFINITY;
    if (a->out_rho) a->out_rho[t0 + i] = NAN;
  }

  /* Diagnostic row probabilities (p(x̂_i), q(x̂_i)) of every draft slot,
   * including slots after the stop; greedy rows carry -1. */
  if (a->out_probs) {
    for (int i = 0; i < K; ++i) {
      double* o = a->out_probs + 2 * (t0 + i);
      if (greedy) {
        o[0] = o[1] = -1.0;
        continue;
      }
      int x = a->draft_tokens[d0 + i];
      row_softmax(a, row_ptr(a->target, a->dtype, t0 + i, V), p, t0 + i);
      o[0] = p[x];
      if (a->draft) {
        row_softmax(a, row_ptr(a->draft, a->dtype, d0 + i, V), q, t0 + i);
        o[1] = q[x];
      } else {
        o[1] = 1.0;
      }
    }
  }

  /* [DM-alg] step 3: test positions in order, stop at the first reject. */
  int stop = K;
  for (int i = 0; i < K; ++i) {
    const int64_t t = t0 + i;
    const int x = a->draft_tokens[d0 + i];
    int accept;
    if (greedy) {
      /* [DSD-2] strict: accept iff the draft equals the target's choice. */
      accept = (x == oracle_argmax(row_ptr(a->target, a->dtype, t, V), a->dtype, V));
    } else {
      row_softmax(a, row_ptr(a->target, a->dtype, t, V), p, t);
      double ph = p[x], qh;
      if (a->draft) {
        row_softmax(a, row_ptr(a->draft, a->dtype, d0 + i, V), q, t);
        qh = q[x];
      } else {
        qh = 1.0; /* [PL-4.3] one-hot proposal */
      }
      /* [DM-rule] accept with probability min(1, p/q); [SDS-4.3] q <= 0
       * rejects. */
      double rho = qh > 0.0 ? fmin(1.0, ph / qh) : 0.0;
      double u = (double)a->uniforms[2 * t];
      accept = u < rho;
      set_margin(a, t, fabs(u - rho));
      if (a->out_rho) a->out_rho[t] = rho;
    }
    if (!accept) {
      stop = i;
      break;
    }
  }

  /* Commit: the accepted prefix [x̂_1 .. x̂_{stop}] ... */
  for (int j = 0; j < stop; ++j) a->out_tokens[t0 + j] = a->draft_tokens[d0 + j];

  /* ... then one token from row `stop`. */
  const int64_t s = t0 + stop;
  int y;
  double py = -1.0, qy = -1.0;
  if (greedy) {
    y = oracle_argmax(row_ptr(a->target, a->dtype, s, V), a->dtype, V);
  } else {
    row_softmax(a, row_ptr(a->target, a->dtype, s, V), p, s);
    int have_q = 0;
    if (stop < K) {
      const int x = a->draft_tokens[d0 + stop];
      if (a->draft) {
        /* [DM-rule], [SDS-3.2]: r = max(0, p - q). */
        row_softmax(a, row_ptr(a->draft, a->dtype, d0 + stop, V), q, s);
        for (int k = 0; k < V; ++k) r[k] = p[k] > q[k] ? p[k] - q[k] : 0.0;
        have_q = 1;
      } else {
        /* One-hot q = e_x: max(0, p - e_x) is p with x removed. */
        for (int k = 0; k < V; ++k) r[k] = p[k];
        r[x] = 0.0;
        for (int k = 0; k < V; ++k) q[k] = 0.0;
        q[x] = 1.0;
        have_q = 1;
      }
    } else {
      /* [DM-alg]: all K accepted -> extra token from p_{K+1}. */
      for (int k = 0; k < V; ++k) r[k] = p[k];
    }
    double u2 = (double)a->uniforms[2 * s + 1], margin = 0.0;
    y = oracle_inverse_cdf(r, V, u2, &margin);
    if (y < 0) {
      /* Z == 0: cannot happen in exact arithmetic after a rejection. */
      y = oracle_inverse_cdf(p, V, u2, &margin);
      margin = 0.0;
    }
    set_margin(a, s, margin);
    py = p[y];
    qy = have_q ? q[y] : 0.0;
  }
  a->out_tokens[s] = y;
  a->out_len[b] = stop + 1;
  if (a->out_stop) a->out_stop[b] = stop;
  if (a->out_probs) {
    double* o = a->out_probs + 2 * (t0 + K);
    o[0] = py;
    o[1] = qy;
  }
  return 0;
}

typedef struct {
  const verify_args_t* a;
  int begin, end;
  int status;
} verify_job_t;

static void* verify_worker(void* arg) {
  verify_job_t* job = (verify_job_t*)arg;
  const int V = job->a->V;
  double* buf = (double*)malloc(sizeof(double) * 3 * (size_t)V);
  if (!buf) {
    job->status = -1;
    return NULL;
  }
  for (int b = job->begin; b < job->end; ++b) {
    int st = verify_request(job->a, b, buf, buf + V, buf + 2 * (size_t)V);
    if (st && !job->status) job->status = st;
  }
  free(buf);
  return NULL;
}

static int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/* Number of threads the oracle would use for nthreads <= 0. */
int oracle_default_threads(void) { return resolve_threads(0); }

/*
 * Verify-and-commit for a batch of B requests, split across threads by
 * request (requests are independent). Returns 0, or the first per-request
 * error code (1: negative draft count, 2: draft token out of range,
 * -1: out of memory).
 */
int oracle_spec_verify_filtered(const void* target, const void* draft, int dtype, int V, int B,
                                const int32_t* draft_tokens, const int32_t* cu_draft,
                                const uint8_t* mode, const float* uniforms, double T,
                                int top_k, double top_p, int32_t* out_tokens, int32_t* out_len,
                                double* out_probs, double* out_margin, double* out_rho,
                                int32_t* out_stop, int nthreads) {
  verify_args_t a = {target,     draft,   dtype,     V,         B,        draft_tokens,
                     cu_draft,   mode,    uniforms,  T,         out_tokens, out_len,
                     out_probs,  out_margin, out_rho, out_stop, top_k,    top_p};
  if (B <= 0) return 0;
  int nt = resolve_threads(nthreads);
  if (nt > B) nt = B;
  verify_job_t* jobs = (verify_job_t*)calloc((size_t)nt, sizeof(verify_job_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -1;
  }
  for (int i = 0; i < nt; ++i) {
    jobs[i].a = &a;
    jobs[i].begin = (int)((int64_t)B * i / nt);
    jobs[i].end = (int)((int64_t)B * (i + 1) / nt);
  }
  for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, verify_worker, &jobs[i]);
  verify_worker(&jobs[0]);
  for (int i = 1; i < nt; ++i) pthread_join(th[i], NULL);
  int status = 0;
  for (int i = 0; i < nt && !status; ++i) status = jobs[i].status;
  free(jobs);
  free(th);
  return status;
}

/* Unfiltered form (the method as the algorithm box gives it). */
int oracle_spec_verify(const void* target, const void* draft, int dtype, int V, int B,
                       const int32_t* draft_tokens, const int32_t* cu_draft,
                       const uint8_t* mode, const float* uniforms, double T,
                       int32_t* out_tokens, int32_t* out_len, double* out_probs,
                       double* out_margin, double* out_rho, int32_t* out_stop,
                       int nthreads) {
  return oracle_spec_verify_filtered(target, draft, dtype, V, B, draft_tokens, cu_draft, mode,
                                     uniforms, T, 0, 1.0, out_tokens, out_len, out_probs,
                                     out_margin, out_rho, out_stop, nthreads);
}

/* ------------------------------------------------------------------ */
/* N-gram / prompt-lookup proposer, [PL-6].                            */
/* ------------------------------------------------------------------ */
/*
 * For n from min(max_n, L) down to min_n: the tail is h[L-n, L). Starts
 * are tried from L-2n down to 0 (most recent first); a start matches when
 * h[start, start+n) equals the tail, and it is taken when the continuation
 * h[start+n, L-n) is non-empty. The proposal is the continuation cut to
 * max_tokens. Without a match: n = 0 and no tokens.
 */
static void ngram_one(const int32_t* h, int L, int min_n, int max_n, int max_tokens,
                      int32_t* out, int32_t* count, int32_t* nout) {
  int nhi = max_n < L ? max_n : L;
  for (int n = nhi; n >= min_n; --n) {
    int tail = L - n;
    for (int start = tail - n; start >= 0; --start) {
      int equal = 1;
      for (int j = 0; j < n; ++j) {
        if (h[start + j] != h[tail + j]) {
          equal = 0;
          break;
        }
      }
      if (!equal) continue;
      int cont = tail - (start + n);
      if (cont <= 0) continue;
      int c = cont < max_tokens ? cont : max_tokens;
      for (int j = 0; j < c; ++j) out[j] = h[start + n + j];
      *count = c;
      *nout = n;
      return;
    }
  }
  *count = 0;
  *nout = 0;
}

/* Batch form: history b at histories + b*hist_stride, hist_len[b] tokens;
 * proposals at out_tokens + b*max_tokens. Returns 0, or 1 on a bad length. */
int oracle_ngram_propose(const int32_t* histories, int64_t hist_stride,
                         const int32_t* hist_len, int B, int min_n, int max_n,
                         int max_tokens, int32_t* out_tokens, int32_t* out_count,
                         int32_t* out_n) {
  for (int b = 0; b < B; ++b) {
    int L = hist_len[b];
    if (L < 0 || L > hist_stride) return 1;
    ngram_one(histories + (int64_t)b * hist_stride, L, min_n, max_n, max_tokens,
              out_tokens + (int64_t)b * max_tokens, out_count + b, out_n + b);
  }
  return 0;
}
