/*
 * rlk_oracle.c -- plain fp64 CPU oracle for the selected-token log-probability
 * operator `linear_logp` (forward, backward, vocab-shard statistics, shard merge).
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The product path (the CUDA library and
 * its Python binding) never calls it, and the two share no source, header, table
 * or helper: this file is self-contained C99.
 *
 * What it computes, and where the definition comes from:
 *
 *   z[t][v]  = sum_k h[t][k] * W[v][k]                       (an explicit dot product)
 *   lse[t]   = M + log sum_{v < V_true} exp(z[t][v] - M),    M = max_{v < V_true} z[t][v]
 *   logp[t]  = z[t][y[t]] - lse[t]
 *
 * i.e. log_softmax(hidden @ W^T)[target] over the true vocabulary range
 * ("Announcing RL-Kernel for vime", section "Key Capabilities", first bullet; the
 * operator boundary "hidden + lm_head_weight + target_ids -> selected logprob" in
 * section "Why the Fused Path Wins"; the true-vocabulary-range and target-ownership
 * items of the "Linear logprob" row in the table "Boundary Fixes in the RL-Kernel
 * Strict Path" of "vLLM RL-Kernel v0.1.0: Bitwise Train-Rollout Consistency on ROCm").
 *
 * Backward of L = sum_t g[t] * logp[t] (full gradient for hidden and weight,
 * "Announcing RL-Kernel for vime", "Key Capabilities", bullet "Full-gradient
 * support"), by the textbook softmax gradient:
 *
 *   p[t][v]  = exp(z[t][v] - lse[t])                   for v < V_true
 *   dz[t][v] = g[t] * (1[v == y[t]] - p[t][v])          for v < V_true, 0 otherwise
 *   dH[t]    = sum_v dz[t][v] * W[v]
 *   dW[v]    = sum_t dz[t][v] * h[t]                    (0 for v >= V_true)
 *
 * Vocab shards ("Why the Fused Path Wins", third reason: each rank reduces its
 * local vocab shard and only the statistics are combined): a shard covering
 * global columns [vocab_start, vocab_start + V_local) reports per token
 *   m  = max of z over its columns below V_true,
 *   s  = sum of exp(z - m) over the same columns,
 *   zt = z[y] if the shard owns y, else -inf,
 * and the merge of S such triples is lse = log sum_i s_i exp(m_i), logp = zt_owner - lse.
 *
 * Inputs arrive either as float64 or as raw bf16 bit patterns (uint16); bf16 is
 * widened exactly (bf16 -> binary32 -> binary64), so the oracle sees the same
 * rounded values the GPU receives. All arithmetic is binary64. Targets outside
 * [0, V_true) give NaN log-probabilities and zero gradient rows.
 *
 * FP8 LM head. The RL training forward may have to reproduce an FP8 inference
 * GEMM: the weights are quantized to FP8 again at every forward, both sides use
 * one quantization rounding rule and one batch-invariant GEMM for every batch
 * size, and the backward takes gradients for the BF16 master weights with the
 * quantization treated as the identity (straight-through estimator) (the AREX
 * feed article on vLLM's bitwise-consistent RL training, sections
 * "训练前向直接调用推理内核" -- the training forward calls the inference kernels --
 * and "对齐的代价：逐算子拆解" -- the cost of alignment, operator by operator).
 * The pages fix neither the FP8 format nor the scale granularity;
 * the reading used here: OCP E4M3 ("FN": no infinities, max 448) with one
 * power-of-two scale per row (per token of h, per vocab row of W), so that a
 * token's quantized values never depend on the rest of the batch and the
 * quantization is exactly reproducible:
 *
 *   e[r]     = the smallest integer with max_k |x[r][k]| <= 448 * 2^e   (0 for an all-zero row)
 *   q[r][k]  = the E4M3 code nearest to x[r][k] / 2^e[r], ties to the even code
 *   xq[r][k] = decode(q[r][k]) * 2^e[r]
 *
 * and the FP8 forward is the definition above evaluated on (hq, Wq); the STE
 * backward forms p and dz from the logits of (hq, Wq) and contracts dz with the
 * unquantized h and W.
 *
 * Built with -O2 -ffp-contract=off and without -ffast-math (see build.py). The
 * dot product keeps four running sums; in binary64 the summation order changes
 * results only at the 1e-16 relative level, far below every tolerance in use.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define RLKO_F64 0
#define RLKO_BF16 1
#define RLKO_E4M3 2 /* operand = const rlko_e4m3_rows*: codes [rows][H] and a scale per row */

typedef struct {
  const uint8_t* codes;
  const double* scale;
} rlko_e4m3_rows;

#define RLKO_OK 0
#define RLKO_EINVAL 1
#define RLKO_ENOMEM 2

/* ------------------------------------------------------------------------- */
/* element access                                                              */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double rlko_bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 holds the subnormals M * 2^-9; S.1111.111 is NaN and there
 * is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double rlko_e4m3_to_double(uint8_t c) {
  const int sign = c >> 7, E = (c >> 3) & 15, M = c & 7;
  double v;
  if (E == 15 && M == 7) return NAN;
  if (E == 0)
    v = ldexp((double)M, -9);
  else
    v = ldexp(1.0 + M / 8.0, E - 7);
  return sign ? -v : v;
}

/* rlko_e4m3_to_double of every code, filled once */
static double g_e4m3_value[256];
static pthread_once_t g_e4m3_once = PTHREAD_ONCE_INIT;
static void e4m3_table_init(void) {
  for (int c = 0; c < 256; ++c) g_e4m3_value[c] = rlko_e4m3_to_double((uint8_t)c);
}

static void load_row(int dtype, const void* base, int64_t row, int64_t H, double* out) {
  if (dtype == RLKO_F64) {
    memcpy(out, (const double*)base + row * H, (size_t)H * sizeof(double));
  } else if (dtype == RLKO_E4M3) {
    const rlko_e4m3_rows* m = (const rlko_e4m3_rows*)base;
    const uint8_t* p = m->codes + row * H;
    const double s = m->scale[row];
    pthread_once(&g_e4m3_once, e4m3_table_init);
    for (int64_t k = 0; k < H; ++k) out[k] = g_e4m3_value[p[k]] * s;
  } else {
    const uint16_t* p = (const uint16_t*)base + row * H;
    for (int64_t k = 0; k < H; ++k) out[k] = rlko_bf16_to_double(p[k]);
  }
}

static double dot(const double* a, const double* b, int64_t n) {
  double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
  int64_t k = 0;
  for (; k + 4 <= n; k += 4) {
    s0 += a[k] * b[k];
    s1 += a[k + 1] * b[k + 1];
    s2 += a[k + 2] * b[k + 2];
    s3 += a[k + 3] * b[k + 3];
  }
  for (; k < n; ++k) s0 += a[k] * b[k];
  return (s0 + s1) + (s2 + s3);
}

/* out += c * x */
static void axpy(double c, const double* x, double* out, int64_t n) {
  for (int64_t k = 0; k < n; ++k) out[k] += c * x[k];
}

static int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

int rlko_default_threads(void) { return resolve_threads(0); }

/* ------------------------------------------------------------------------- */
/* a tiny fork/join helper over an index range                                 */
/* ------------------------------------------------------------------------- */

typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end, int tid);

typedef struct {
  range_fn fn;
  void* ctx;
  int64_t begin, end;
  int tid;
} range_job;

static void* range_thread(void* arg) {
  range_job* j = (range_job*)arg;
  j->fn(j->ctx, j->begin, j->end, j->tid);
  return NULL;
}

/* Splits [0, n) into `nthreads` contiguous chunks and runs fn on each. */
static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx) {
  if (n <= 0) return;
  if (nthreads > n) nthreads = (int)n;
  if (nthreads <= 1) {
    fn(ctx, 0, n, 0);
    return;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  range_job* jobs = (range_job*)malloc(sizeof(range_job) * (size_t)nthreads);
  int* started = (int*)calloc((size_t)nthreads, sizeof(int));
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].fn = fn;
    jobs[i].ctx = ctx;
    jobs[i].begin = n * i / nthreads;
    jobs[i].end = n * (i + 1) / nthreads;
    jobs[i].tid = i;
    started[i] = pthread_create(&th[i], NULL, range_thread, &jobs[i]) == 0;
    if (!started[i]) range_thread(&jobs[i]); /* run inline if a thread cannot start */
  }
  for (int i = 0; i < nthreads; ++i)
    if (started[i]) pthread_join(th[i], NULL);
  free(started);
  free(jobs);
  free(th);
}

/* The E4M3 code nearest to y (|y| <= 448), ties to the code with the even mantissa.
 * Positive codes 0 .. 126 are increasing in value (tab[c] = their values), so a
 * binary search finds the largest code not above |y|; its successor is the only
 * other candidate. */
static uint8_t e4m3_nearest(double y, const double* tab) {
  const int neg = y < 0.0 || (y == 0.0 && signbit(y));
  const double a = fabs(y);
  int lo = 0, hi = 126;
  while (lo < hi) { /* largest c with tab[c] <= a */
    int mid = (lo + hi + 1) / 2;
    if (tab[mid] <= a) lo = mid;
    else hi = mid - 1;
  }
  int c = lo;
  if (c < 126) {
    const double d0 = a - tab[c];
    const double d1 = tab[c + 1] - a;
    if (d1 < d0 || (d1 == d0 && ((c + 1) & 1) == 0)) c = c + 1;
  }
  return (uint8_t)(neg ? (c | 0x80) : c);
}

typedef struct {
  int dtype;
  const void* x;
  int64_t cols;
  uint8_t* q;
  double* scale;
  double tab[127];
  int failed; /* 1: out of memory, 2: a non-finite input */
} quant_ctx;

static void quantize_range(void* vctx, int64_t begin, int64_t end, int tid) {
  quant_ctx* c = (quant_ctx*)vctx;
  (void)tid;
  const int64_t cols = c->cols;
  double* buf = (double*)malloc(sizeof(double) * (size_t)(cols > 0 ? cols : 1));
  if (!buf) {
    c->failed = 1;
    return;
  }
  for (int64_t r = begin; r < end; ++r) {
    double amax = 0.0;
    load_row(c->dtype, c->x, r, cols, buf);
    for (int64_t k = 0; k < cols; ++k) {
      if (!isfinite(buf[k])) {
        c->failed = 2;
        free(buf);
        return;
      }
      if (fabs(buf[k]) > amax) amax = fabs(buf[k]);
    }
    int e = 0;
    if (amax > 0.0) {
      int k2;
      frexp(amax, &k2); /* amax in [2^(k2-1), 2^k2) */
      e = k2 - 9;       /* a first guess, then the two defining inequalities */
      while (amax > ldexp(448.0, e)) ++e;
      while (amax <= ldexp(448.0, e - 1)) --e;
    }
    c->scale[r] = ldexp(1.0, e);
    for (int64_t k = 0; k < cols; ++k) c->q[r * cols + k] = e4m3_nearest(ldexp(buf[k], -e), c->tab);
  }
  free(buf);
}

/* Per-row power-of-two scale and E4M3 codes of x [rows][cols] (bf16 bits or
 * float64, see the header comment for the definition), rows split over threads.
 * Non-finite inputs are outside the definition and rejected. */
int rlko_quantize_rows_e4m3(int dtype, const void* x, int64_t rows, int64_t cols, uint8_t* q,
                            double* scale, int nthreads) {
  if (!x || !q || !scale || rows < 0 || cols < 0 || (dtype != RLKO_F64 && dtype != RLKO_BF16))
    return RLKO_EINVAL;
  quant_ctx c;
  memset(&c, 0, sizeof c);
  c.dtype = dtype; c.x = x; c.cols = cols; c.q = q; c.scale = scale;
  for (int i = 0; i < 127; ++i) c.tab[i] = rlko_e4m3_to_double((uint8_t)i);
  parallel_for(rows, resolve_threads(nthreads), quantize_range, &c);
  if (c.failed == 2) return RLKO_EINVAL;
  return c.failed ? RLKO_ENOMEM : RLKO_OK;
}

/* ------------------------------------------------------------------------- */
/* forward: z for a block of tokens, then max-shifted log-sum-exp and gather   */
/* ------------------------------------------------------------------------- */

typedef struct {
  int dtype;           /* h, W: the operands the gradients are contracted with */
  const void* h;
  const void* W;
  int zdtype;          /* zh, zW: the operands the logits are formed from (the same */
  const void* zh;      /* as h, W except in the straight-through FP8 backward)      */
  const void* zW;
  const int64_t* y;
  const double* g;     /* backward only */
  const double* lse_in; /* dW only */
  int64_t T, H, V, V_true;
  int64_t vocab_start, V_local; /* shard statistics only */
  const int64_t* rows;
  int64_t n_rows;
  int64_t block;       /* tokens per block */
  double* out0;        /* logp | m  | dH | dW */
  double* out1;        /* lse  | s  |    |    */
  double* out2;        /*      | zt |    |    */
  int failed;
} job_ctx;

static int64_t row_at(const job_ctx* c, int64_t i) { return c->rows ? c->rows[i] : i; }

static int target_valid(int64_t y, int64_t V_true) { return y >= 0 && y < V_true; }

/* z[b][v] for the tokens rows[i0 .. i0+nb) and columns v in [v0, v1). */
static void logits_block(const job_ctx* c, int64_t i0, int64_t nb, int64_t v0, int64_t v1,
                         double* hbuf, double* wbuf, double* z) {
  const int64_t H = c->H, n = v1 - v0;
  for (int64_t b = 0; b < nb; ++b) load_row(c->zdtype, c->zh, row_at(c, i0 + b), H, hbuf + b * H);
  for (int64_t v = v0; v < v1; ++v) {
    load_row(c->zdtype, c->zW, v - c->vocab_start, H, wbuf);
    for (int64_t b = 0; b < nb; ++b) z[b * n + (v - v0)] = dot(hbuf + b * H, wbuf, H);
  }
}

/* log sum_{j<n} exp(z[j]) with the maximum factored out; -inf for n == 0. */
static double logsumexp(const double* z, int64_t n) {
  if (n <= 0) return -INFINITY;
  double M = z[0];
  for (int64_t j = 1; j < n; ++j)
    if (z[j] > M) M = z[j];
  double s = 0.0;
  for (int64_t j = 0; j < n; ++j) s += exp(z[j] - M);
  return M + log(s);
}

static void forward_range(void* vctx, int64_t begin, int64_t end, int tid) {
  job_ctx* c = (job_ctx*)vctx;
  (void)tid;
  const int64_t H = c->H, Vt = c->V_true, B = c->block;
  double* hbuf = (double*)malloc(sizeof(double) * (size_t)(B * H));
  double* wbuf = (double*)malloc(sizeof(double) * (size_t)H);
  double* z = (double*)malloc(sizeof(double) * (size_t)(B * Vt));
  if (!hbuf || !wbuf || !z) {
    c->failed = 1;
    free(hbuf); free(wbuf); free(z);
    return;
  }
  for (int64_t i0 = begin; i0 < end; i0 += B) {
    int64_t nb = end - i0 < B ? end - i0 : B;
    logits_block(c, i0, nb, 0, Vt, hbuf, wbuf, z);
    for (int64_t b = 0; b < nb; ++b) {
      const double* zb = z + b * Vt;
      double lse = logsumexp(zb, Vt);
      int64_t y = c->y[row_at(c, i0 + b)];
      double logp = target_valid(y, Vt) ? zb[y] - lse : NAN;
      if (c->out0) c->out0[i0 + b] = logp;
      if (c->out1) c->out1[i0 + b] = lse;
    }
  }
  free(hbuf); free(wbuf); free(z);
}

static int64_t pick_block(int64_t n_rows, int nthreads) {
  int64_t per = (n_rows + nthreads - 1) / nthreads;
  return per < 8 ? (per < 1 ? 1 : per) : 8;
}

/*
 * logp[i], lse[i] for token rows[i] (i < n_rows), or for every token when
 * rows == NULL (then n_rows must equal T). Either output may be NULL.
 */
int rlko_forward(int dtype, const void* h, const void* W, const int64_t* y, int64_t T, int64_t H,
                 int64_t V, int64_t V_true, const int64_t* rows, int64_t n_rows, double* logp,
                 double* lse, int nthreads) {
  if (!h || !W || !y || T < 0 || H <= 0 || V_true < 1 || V_true > V) return RLKO_EINVAL;
  if (!rows) n_rows = T;
  for (int64_t i = 0; rows && i < n_rows; ++i)
    if (rows[i] < 0 || rows[i] >= T) return RLKO_EINVAL;
  int nt = resolve_threads(nthreads);
  job_ctx c;
  memset(&c, 0, sizeof c);
  c.dtype = dtype; c.h = h; c.W = W; c.y = y;
  c.zdtype = dtype; c.zh = h; c.zW = W;
  c.T = T; c.H = H; c.V = V; c.V_true = V_true;
  c.vocab_start = 0; c.V_local = V;
  c.rows = rows; c.n_rows = n_rows;
  c.block = pick_block(n_rows, nt);
  c.out0 = logp; c.out1 = lse;
  parallel_for(n_rows, nt, forward_range, &c);
  return c.failed ? RLKO_ENOMEM : RLKO_OK;
}

/* ------------------------------------------------------------------------- */
/* vocab-shard statistics (m, s, zt) and their merge                          */
/* ------------------------------------------------------------------------- */

static void shard_range(void* vctx, int64_t begin, int64_t end, int tid) {
  job_ctx* c = (job_ctx*)vctx;
  (void)tid;
  const int64_t H = c->H, B = c->block;
  int64_t v0 = c->vocab_start;
  int64_t v1 = c->vocab_start + c->V_local;
  if (v1 > c->V_true) v1 = c->V_true;
  int64_t n = v1 > v0 ? v1 - v0 : 0;
  double* hbuf = (double*)malloc(sizeof(double) * (size_t)(B * H));
  double* wbuf = (double*)malloc(sizeof(double) * (size_t)H);
  double* z = (double*)malloc(sizeof(double) * (size_t)(B * (n > 0 ? n : 1)));
  if (!hbuf || !wbuf || !z) {
    c->failed = 1;
    free(hbuf); free(wbuf); free(z);
    return;
  }
  for (int64_t i0 = begin; i0 < end; i0 += B) {
    int64_t nb = end - i0 < B ? end - i0 : B;
    if (n > 0) logits_block(c, i0, nb, v0, v1, hbuf, wbuf, z);
    for (int64_t b = 0; b < nb; ++b) {
      const double* zb = z + b * n;
      double m = -INFINITY, s = 0.0;
      for (int64_t j = 0; j < n; ++j)
        if (zb[j] > m) m = zb[j];
      for (int64_t j = 0; j < n; ++j) s += exp(zb[j] - m);
      int64_t y = c->y[row_at(c, i0 + b)];
      double zt;
      if (!target_valid(y, c->V_true)) zt = NAN;
      else if (y >= v0 && y < v1) zt = zb[y - v0];
      else zt = -INFINITY;
      c->out0[i0 + b] = m;
      c->out1[i0 + b] = s;
      c->out2[i0 + b] = zt;
    }
  }
  free(hbuf); free(wbuf); free(z);
}

/*
 * Per-token statistics of one vocab shard: W_local holds rows for global
 * columns [vocab_start, vocab_start + V_local); columns at or above V_true are
 * excluded. An empty shard yields m = -inf, s = 0, zt = -inf.
 */
int rlko_shard_stats(int dtype, const void* h, const void* W_local, const int64_t* y, int64_t T,
                     int64_t H, int64_t V_local, int64_t vocab_start, int64_t V_true,
                     const int64_t* rows, int64_t n_rows, double* m, double* s, double* zt,
                     int nthreads) {
  if (!h || !W_local || !y || !m || !s || !zt || T < 0 || H <= 0 || V_local < 0 ||
      vocab_start < 0 || V_true < 1)
    return RLKO_EINVAL;
  if (!rows) n_rows = T;
  for (int64_t i = 0; rows && i < n_rows; ++i)
    if (rows[i] < 0 || rows[i] >= T) return RLKO_EINVAL;
  int nt = resolve_threads(nthreads);
  job_ctx c;
  memset(&c, 0, sizeof c);
  c.dtype = dtype; c.h = h; c.W = W_local; c.y = y;
  c.zdtype = dtype; c.zh = h; c.zW = W_local;
  c.T = T; c.H = H; c.V = V_local; c.V_true = V_true;
  c.vocab_start = vocab_start; c.V_local = V_local;
  c.rows = rows; c.n_rows = n_rows;
  c.block = pick_block(n_rows, nt);
  c.out0 = m; c.out1 = s; c.out2 = zt;
  parallel_for(n_rows, nt, shard_range, &c);
  return c.failed ? RLKO_ENOMEM : RLKO_OK;
}

/*
 * Merge of S per-shard triples per token, arrays laid out [S][T]:
 *   lse = log sum_i s_i exp(m_i)   (max factored out; shards with s_i == 0 add nothing)
 *   logp = zt_owner - lse, where zt_owner is the largest zt (non-owners hold -inf);
 *   any NaN zt makes logp NaN.
 */
int rlko_lse_merge(const double* m, const double* s, const double* zt, int64_t S, int64_t T,
                   double* logp, double* lse) {
  if (!m || !s || !zt || !logp || !lse || S < 1 || T < 0) return RLKO_EINVAL;
  for (int64_t t = 0; t < T; ++t) {
    double M = -INFINITY, best = -INFINITY;
    int nan_target = 0;
    for (int64_t i = 0; i < S; ++i) {
      if (s[i * T + t] > 0.0 && m[i * T + t] > M) M = m[i * T + t];
      double z = zt[i * T + t];
      if (isnan(z)) nan_target = 1;
      else if (z > best) best = z;
    }
    double acc = 0.0;
    for (int64_t i = 0; i < S; ++i)
      if (s[i * T + t] > 0.0) acc += s[i * T + t] * exp(m[i * T + t] - M);
    double l = acc > 0.0 ? M + log(acc) : -INFINITY;
    lse[t] = l;
    logp[t] = nan_target ? NAN : best - l;
  }
  return RLKO_OK;
}

/* ------------------------------------------------------------------------- */
/* backward                                                                    */
/* ------------------------------------------------------------------------- */

/* dH for the tokens rows[i]: forward for the token, then dH = sum_v dz_v W_v. */
static void dh_range(void* vctx, int64_t begin, int64_t end, int tid) {
  job_ctx* c = (job_ctx*)vctx;
  (void)tid;
  const int64_t H = c->H, Vt = c->V_true, B = c->block;
  double* hbuf = (double*)malloc(sizeof(double) * (size_t)(B * H));
  double* wbuf = (double*)malloc(sizeof(double) * (size_t)H);
  double* z = (double*)malloc(sizeof(double) * (size_t)(B * Vt));
  if (!hbuf || !wbuf || !z) {
    c->failed = 1;
    free(hbuf); free(wbuf); free(z);
    return;
  }
  for (int64_t i0 = begin; i0 < end; i0 += B) {
    int64_t nb = end - i0 < B ? end - i0 : B;
    logits_block(c, i0, nb, 0, Vt, hbuf, wbuf, z);
    /* z -> dz in place */
    for (int64_t b = 0; b < nb; ++b) {
      double* zb = z + b * Vt;
      int64_t t = row_at(c, i0 + b);
      int64_t y = c->y[t];
      double g = c->g[t];
      if (!target_valid(y, Vt)) {
        for (int64_t v = 0; v < Vt; ++v) zb[v] = 0.0;
        continue;
      }
      double lse = logsumexp(zb, Vt);
      for (int64_t v = 0; v < Vt; ++v) zb[v] = g * ((v == y ? 1.0 : 0.0) - exp(zb[v] - lse));
    }
    double* dH = c->out0 + i0 * H;
    memset(dH, 0, sizeof(double) * (size_t)(nb * H));
    for (int64_t v = 0; v < Vt; ++v) {
      load_row(c->dtype, c->W, v, H, wbuf);
      for (int64_t b = 0; b < nb; ++b) axpy(z[b * Vt + v], wbuf, dH + b * H, H);
    }
  }
  free(hbuf); free(wbuf); free(z);
}

/*
 * dH[i][:] for token rows[i] (every token when rows == NULL), of
 * L = sum_t g[t] * logp[t]. dH is [n_rows][H].
 *
 * The straight-through form takes the logits (hence p and dz) from the operands
 * (zh, zW) and contracts dz with W: dH = dz W. With (zh, zW) = (h, W) it is the
 * plain gradient.
 */
int rlko_backward_dh_ste(int zdtype, const void* zh, const void* zW, int dtype, const void* h,
                         const void* W, const int64_t* y, const double* g, int64_t T, int64_t H,
                         int64_t V, int64_t V_true, const int64_t* rows, int64_t n_rows, double* dH,
                         int nthreads) {
  if (!zh || !zW || !h || !W || !y || !g || !dH || T < 0 || H <= 0 || V_true < 1 || V_true > V)
    return RLKO_EINVAL;
  if (!rows) n_rows = T;
  for (int64_t i = 0; rows && i < n_rows; ++i)
    if (rows[i] < 0 || rows[i] >= T) return RLKO_EINVAL;
  int nt = resolve_threads(nthreads);
  job_ctx c;
  memset(&c, 0, sizeof c);
  c.dtype = dtype; c.h = h; c.W = W; c.y = y; c.g = g;
  c.zdtype = zdtype; c.zh = zh; c.zW = zW;
  c.T = T; c.H = H; c.V = V; c.V_true = V_true;
  c.vocab_start = 0; c.V_local = V;
  c.rows = rows; c.n_rows = n_rows;
  c.block = pick_block(n_rows, nt);
  c.out0 = dH;
  parallel_for(n_rows, nt, dh_range, &c);
  return c.failed ? RLKO_ENOMEM : RLKO_OK;
}

int rlko_backward_dh(int dtype, const void* h, const void* W, const int64_t* y, const double* g,
                     int64_t T, int64_t H, int64_t V, int64_t V_true, const int64_t* rows,
                     int64_t n_rows, double* dH, int nthreads) {
  return rlko_backward_dh_ste(dtype, h, W, dtype, h, W, y, g, T, H, V, V_true, rows, n_rows, dH,
                              nthreads);
}

/* dW rows: dW_v = sum_t dz[t][v] h_t, using the given per-token lse. */
typedef struct {
  job_ctx* c;
  const double* hwide;  /* [T][H] widened h (the gradient operand) */
  const double* hzwide; /* [T][H] widened zh (the logit operand), or hwide */
} dw_ctx;

static void dw_range(void* vctx, int64_t begin, int64_t end, int tid) {
  dw_ctx* d = (dw_ctx*)vctx;
  job_ctx* c = d->c;
  (void)tid;
  const int64_t H = c->H, T = c->T;
  double* wbuf = (double*)malloc(sizeof(double) * (size_t)H);
  if (!wbuf) {
    c->failed = 1;
    return;
  }
  for (int64_t i = begin; i < end; ++i) {
    int64_t v = row_at(c, i);
    double* out = c->out0 + i * H;
    memset(out, 0, sizeof(double) * (size_t)H);
    if (v >= c->V_true) continue; /* padded rows take no gradient */
    load_row(c->zdtype, c->zW, v, H, wbuf); /* only the logits use W's row */
    for (int64_t t = 0; t < T; ++t) {
      double g = c->g[t];
      int64_t y = c->y[t];
      /* a zero upstream gradient or an invalid target contributes exactly nothing */
      if (g == 0.0 || !target_valid(y, c->V_true)) continue;
      double zv = dot(d->hzwide + t * H, wbuf, H);
      double dz = g * ((v == y ? 1.0 : 0.0) - exp(zv - c->lse_in[t]));
      axpy(dz, d->hwide + t * H, out, H);
    }
  }
  free(wbuf);
}

/*
 * dW[i][:] for vocab row vrows[i] (every row of W when vrows == NULL, then
 * n_vrows must equal V), given lse[t] for every token with g[t] != 0 (tokens
 * with g[t] == 0 are skipped, so their lse entry is never read).
 *
 * The straight-through form takes the logits from (zh, zW) and contracts dz with
 * h: dW = dz^T h. With (zh, zW) = (h, W) it is the plain gradient (W itself then
 * enters only through the logits).
 */
int rlko_backward_dw_ste(int zdtype, const void* zh, const void* zW, int dtype, const void* h,
                         const int64_t* y, const double* g, const double* lse, int64_t T,
                         int64_t H, int64_t V, int64_t V_true, const int64_t* vrows,
                         int64_t n_vrows, double* dW, int nthreads) {
  if (!zh || !zW || !h || !y || !g || !lse || !dW || T < 0 || H <= 0 || V_true < 1 || V_true > V)
    return RLKO_EINVAL;
  if (!vrows) n_vrows = V;
  for (int64_t i = 0; vrows && i < n_vrows; ++i)
    if (vrows[i] < 0 || vrows[i] >= V) return RLKO_EINVAL;
  const size_t n = (size_t)((T > 0 ? T : 1) * H);
  double* hwide = (double*)malloc(sizeof(double) * n);
  double* hzwide = (zh == h && zdtype == dtype) ? hwide : (double*)malloc(sizeof(double) * n);
  if (!hwide || !hzwide) {
    free(hwide);
    if (hzwide != hwide) free(hzwide);
    return RLKO_ENOMEM;
  }
  for (int64_t t = 0; t < T; ++t) load_row(dtype, h, t, H, hwide + t * H);
  if (hzwide != hwide)
    for (int64_t t = 0; t < T; ++t) load_row(zdtype, zh, t, H, hzwide + t * H);
  int nt = resolve_threads(nthreads);
  job_ctx c;
  memset(&c, 0, sizeof c);
  c.dtype = dtype; c.h = h; c.y = y; c.g = g; c.lse_in = lse;
  c.zdtype = zdtype; c.zh = zh; c.zW = zW;
  c.T = T; c.H = H; c.V = V; c.V_true = V_true;
  c.rows = vrows; c.n_rows = n_vrows;
  c.out0 = dW;
  dw_ctx d = {&c, hwide, hzwide};
  parallel_for(n_vrows, nt, dw_range, &d);
  if (hzwide != hwide) free(hzwide);
  free(hwide);
  return c.failed ? RLKO_ENOMEM : RLKO_OK;
}

int rlko_backward_dw(int dtype, const void* h, const void* W, const int64_t* y, const double* g,
                     const double* lse, int64_t T, int64_t H, int64_t V, int64_t V_true,
                     const int64_t* vrows, int64_t n_vrows, double* dW, int nthreads) {
  if (!W) return RLKO_EINVAL;
  return rlko_backward_dw_ste(dtype, h, W, dtype, h, y, g, lse, T, H, V, V_true, vrows, n_vrows,
                              dW, nthreads);
}
