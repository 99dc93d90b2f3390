/*
 * attn_res_ref.c -- scalar CPU oracle for the Kimi-K3 attention-residual
 * (AttnRes) mixture.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this; the product path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, per token row t (width H), following the implementation
 * walkthrough of "Add Kimi K3 attention residual fusion" (vllm-ascend #14840)
 * and the kernel excerpt of "SM100 Kimi-K3 AttnRes defaults to native CUDA"
 * (vllm #54261, key source excerpt of attn_res_kernel.cu):
 *
 *   1. current-layer row  c = bf16_rne(prefix + delta)   (c = prefix if no
 *      delta) -- #54261 excerpt: delta is accumulated into the prefix row,
 *      which is packed back to bf16 and stored.
 *   2. candidates: the num_blocks valid bank rows blocks[t, 0..S-1], then c as
 *      the last candidate -- #14840 walkthrough ("append prefix_sum as the
 *      final candidate stream"); bank capacity is not the valid count.
 *   3. pseudo-query q = rms_w * res_w -- #14840 walkthrough ("score each
 *      candidate with norm.weight * proj.weight"); vllm #50185 builds the same
 *      product into q_cache.
 *   4. each candidate is RMS-normalised, 1/sqrt(mean(x^2) + eps), and its
 *      logit is <x_hat, q> -- #14840 walkthrough.
 *   5. softmax across the S+1 logits -- #14840 walkthrough.
 *   6. mix the RAW candidate rows with the softmax weights -- #14840
 *      walkthrough ("form the weighted residual sum").
 *   7. optional output RMSNorm y = acc * 1/sqrt(mean(acc^2) + out_eps) * w_o
 *      on the fp32-style accumulator -- #54261 excerpt, HAS_OUTPUT_NORM branch.
 *   8. cast to bf16 (round to nearest even).
 *   9. write-backs of c: into prefix when delta is given, into
 *      blocks[t, block_write_idx] when block_write_idx >= 0 -- #54261
 *      summary (Tensor! blocks, block_write_idx, -1 = no write) and excerpt.
 *  10. the bank row of token t is t / B (B >= 1, default 1) -- the #54261
 *      excerpt addresses block_res at row tb / B.
 *
 * Every arithmetic step is done in IEEE double; bf16 <-> double conversions
 * are exact in one direction and round-to-nearest-even (written out from the
 * IEEE 754 definition) in the other.  The softmax is the plain two-pass form
 * (max, exp, sum): no online rescaling, no blocking, no reordering.
 *
 * Readings where the pages are silent (also listed in the design notes):
 *   - eps sits inside the square root with the mean over H (standard RMSNorm);
 *   - no temperature and no 1/sqrt(H) on the logit;
 *   - normalised rows and the accumulator are never rounded to bf16;
 *   - the mixed current-layer candidate is the rounded row c;
 *   - all reads of a token see the values from before the call
 *     (read-before-write when block_write_idx < num_blocks);
 *   - B (the excerpt's divisor, never defined on the pages) maps B
 *     consecutive token rows to one bank row; of the rows sharing it, the
 *     last one's c is what the slot holds after the call, and with B > 1 the
 *     written slot may not also be a source.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_OK 0
#define REF_EINVAL 1
#define REF_ENOMEM 2

/* ---- bf16 <-> double -------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32: 1 sign bit, 8 exponent bits
 * (bias 127), 7 fraction bits.  Widening is exact. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even (IEEE 754
 * roundTiesToEven).  Written from the definition: find the spacing of bf16
 * numbers at |x|'s binade (2^(E-7) for normals, 2^-133 below 2^-126), scale
 * |x| so that spacing is 1, round the scaled value to an integer with ties to
 * even, and encode.  Values at or above the midpoint between the largest
 * finite bf16 and 2^128 overflow to infinity. */
static uint16_t double_to_bf16_rne(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
  if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
  double a = fabs(x);
  if (a == 0.0) return sign;
  int e2;
  (void)frexp(a, &e2);          /* a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;               /* unbiased exponent of a */
  if (E > 127) return (uint16_t)(sign | 0x7F80u);
  int qexp = (E < -126 ? -126 : E) - 7; /* exponent of one bf16 ulp here */
  double scaled = ldexp(a, -qexp);      /* exact: power-of-two scaling */
  double fl = floor(scaled);
  double frac = scaled - fl;            /* exact */
  uint32_t n = (uint32_t)fl;
  if (frac > 0.5 || (frac == 0.5 && (n & 1u))) n += 1u;
  if (E >= -126) {
    /* normal binade: n in [128, 256]; 256 carries into the next binade */
    int biased = E + 127;
    if (n == 256u) {
      n = 128u;
      biased += 1;
    }
    if (biased >= 255) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | ((uint32_t)biased << 7) | (n - 128u));
  }
  /* subnormal range: n in [0, 128]; n == 128 encodes the smallest normal */
  return (uint16_t)(sign | n);
}

void attn_res_ref_round_bf16(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16_rne(in[i]);
}

void attn_res_ref_widen_bf16(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_double(in[i]);
}

/* ---- the mixture ------------------------------------------------------ */

typedef struct {
  uint16_t* prefix;
  const uint16_t* delta;
  uint16_t* blocks;
  int num_blocks;
  int block_write_idx;
  const uint16_t* out_norm_w;
  double eps, out_eps;
  uint16_t* out;
  int64_t H;
  int64_t prefix_row, delta_row, blocks_token, blocks_slot, out_row;
  int64_t group;       /* token rows per bank row (B) */
  int64_t T;
  double* weights_out; /* [T, N] or NULL */
  double* logits_out;  /* [T, N] or NULL */
  const double* q;     /* [H] pseudo-query, shared read-only */
  int64_t t0, t1;      /* token range of this worker */
  int status;
} ref_job;

static void ref_token(const ref_job* j, int64_t t, uint16_t* c, double* acc,
                      double* ss, double* dt, double* logit, double* w) {
  const int64_t H = j->H;
  const int S = j->num_blocks;
  const int N = S + 1;
  uint16_t* prow = j->prefix + t * j->prefix_row;
  /* bank row of this token: t / B (the excerpt's block_res row tb / B) */
  const uint16_t* bank = j->blocks ? j->blocks + (t / j->group) * j->blocks_token : NULL;

  /* step 1: current-layer row */
  for (int64_t h = 0; h < H; ++h) {
    if (j->delta) {
      const uint16_t* drow = j->delta + t * j->delta_row;
      c[h] = double_to_bf16_rne(bf16_to_double(prow[h]) +
                                bf16_to_double(drow[h]));
    } else {
      c[h] = prow[h];
    }
  }

  /* steps 2-4: per-candidate sum of squares, dot with q, logit */
  for (int i = 0; i < N; ++i) {
    const uint16_t* x =
        (i < S) ? bank + (int64_t)i * j->blocks_slot
                : c;
    double s2 = 0.0, sd = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      double v = bf16_to_double(x[h]);
      s2 += v * v;
      sd += v * j->q[h];
    }
    ss[i] = s2;
    dt[i] = sd;
    logit[i] = sd / sqrt(s2 / (double)H + j->eps);
  }

  /* step 5: softmax, two-pass */
  double m = logit[0];
  for (int i = 1; i < N; ++i)
    if (logit[i] > m) m = logit[i];
  double z = 0.0;
  for (int i = 0; i < N; ++i) {
    w[i] = exp(logit[i] - m);
    z += w[i];
  }
  for (int i = 0; i < N; ++i) w[i] /= z;

  /* step 6: mix the raw rows */
  for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
  for (int i = 0; i < N; ++i) {
    const uint16_t* x =
        (i < S) ? bank + (int64_t)i * j->blocks_slot
                : c;
    for (int64_t h = 0; h < H; ++h) acc[h] += w[i] * bf16_to_double(x[h]);
  }

  /* steps 7-8: optional output RMSNorm, then bf16 */
  uint16_t* orow = j->out + t * j->out_row;
  if (j->out_norm_w) {
    double sq = 0.0;
    for (int64_t h = 0; h < H; ++h) sq += acc[h] * acc[h];
    double r = 1.0 / sqrt(sq / (double)H + j->out_eps);
    for (int64_t h = 0; h < H; ++h)
      orow[h] = double_to_bf16_rne(acc[h] * r * bf16_to_double(j->out_norm_w[h]));
  } else {
    for (int64_t h = 0; h < H; ++h) orow[h] = double_to_bf16_rne(acc[h]);
  }

  /* step 9: write-backs, after every read of this token.  With B > 1 token
   * rows share a bank row; in token order each would overwrite the slot, so
   * it ends holding the c of the group's last row, which alone writes. */
  if (j->delta) memcpy(prow, c, (size_t)H * sizeof(uint16_t));
  if (j->block_write_idx >= 0 &&
      (t % j->group == j->group - 1 || t == j->T - 1)) {
    uint16_t* dst = j->blocks + (t / j->group) * j->blocks_token +
                    (int64_t)j->block_write_idx * j->blocks_slot;
    memcpy(dst, c, (size_t)H * sizeof(uint16_t));
  }

  if (j->weights_out)
    for (int i = 0; i < N; ++i) j->weights_out[t * N + i] = w[i];
  if (j->logits_out)
    for (int i = 0; i < N; ++i) j->logits_out[t * N + i] = logit[i];
}

static void* ref_worker(void* arg) {
  ref_job* j = (ref_job*)arg;
  const int64_t H = j->H;
  uint16_t* c = (uint16_t*)malloc((size_t)H * sizeof(uint16_t));
  double* acc = (double*)malloc((size_t)H * sizeof(double));
  double ss[9], dt[9], logit[9], w[9];
  if (!c || !acc) {
    j->status = REF_ENOMEM;
  } else {
    for (int64_t t = j->t0; t < j->t1; ++t) ref_token(j, t, c, acc, ss, dt, logit, w);
    j->status = REF_OK;
  }
  free(c);
  free(acc);
  return NULL;
}

/*
 * attn_res_ref: host arrays of bf16 bit patterns (uint16), strides in
 * elements.  Same in-place contract as the library: out is written; prefix is
 * overwritten with c when delta != NULL; blocks[t, block_write_idx] is
 * overwritten with c when block_write_idx >= 0.  weights_out / logits_out
 * ([T, num_blocks+1], optional) expose the softmax weights and logits.
 * blocks_group (B >= 1) token rows share one bank row: token t reads bank
 * row t / B, and only the last row of each group writes the slot; with
 * B > 1 the written slot may not be one of the sources.  Tokens are split
 * into contiguous ranges over n_threads POSIX threads; the per-token code is
 * the scalar loop above.  Returns 0 on success.
 */
int attn_res_ref(uint16_t* prefix, const uint16_t* delta, uint16_t* blocks,
                 int num_blocks, int block_write_idx, int blocks_capacity,
                 const uint16_t* res_w, const uint16_t* rms_w,
                 const uint16_t* out_norm_w, float eps, float out_eps,
                 uint16_t* out, int64_t T, int64_t H, int64_t prefix_row,
                 int64_t delta_row, int64_t blocks_token, int64_t blocks_slot,
                 int64_t out_row, int64_t blocks_group, double* weights_out,
                 double* logits_out, int n_threads) {
  if (blocks_group < 1) return REF_EINVAL;
  /* a shared bank row may not be both read and written within one call */
  if (blocks_group > 1 && block_write_idx >= 0 && block_write_idx < num_blocks)
    return REF_EINVAL;
  if (T < 0 || H <= 0 || num_blocks < 0 || num_blocks > 8 ||
      num_blocks > blocks_capacity || block_write_idx < -1 ||
      block_write_idx >= blocks_capacity || !prefix || !res_w || !rms_w || !out)
    return REF_EINVAL;
  if ((num_blocks > 0 || block_write_idx >= 0) && !blocks) return REF_EINVAL;
  if (T == 0) return REF_OK;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > T) n_threads = (int)T;

  double* q = (double*)malloc((size_t)H * sizeof(double));
  if (!q) return REF_ENOMEM;
  for (int64_t h = 0; h < H; ++h)
    q[h] = bf16_to_double(rms_w[h]) * bf16_to_double(res_w[h]);

  ref_job* jobs = (ref_job*)calloc((size_t)n_threads, sizeof(ref_job));
  pthread_t* th = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(q);
    free(jobs);
    free(th);
    return REF_ENOMEM;
  }
  int status = REF_OK;
  for (int k = 0; k < n_threads; ++k) {
    ref_job* j = &jobs[k];
    j->prefix = prefix;
    j->delta = delta;
    j->blocks = blocks;
    j->num_blocks = num_blocks;
    j->block_write_idx = block_write_idx;
    j->out_norm_w = out_norm_w;
    j->eps = (double)eps;
    j->out_eps = (double)out_eps;
    j->out = out;
    j->H = H;
    j->prefix_row = prefix_row;
    j->delta_row = delta_row;
    j->blocks_token = blocks_token;
    j->blocks_slot = blocks_slot;
    j->out_row = out_row;
    j->group = blocks_group;
    j->T = T;
    j->weights_out = weights_out;
    j->logits_out = logits_out;
    j->q = q;
    j->t0 = T * k / n_threads;
    j->t1 = T * (k + 1) / n_threads;
  }
  if (n_threads == 1) {
    ref_worker(&jobs[0]);
  } else {
    int started = 0;
    for (int k = 0; k < n_threads; ++k) {
      if (pthread_create(&th[k], NULL, ref_worker, &jobs[k]) != 0) break;
      ++started;
    }
    for (int k = 0; k < started; ++k) pthread_join(th[k], NULL);
    /* run any range a thread could not be started for on this thread */
    for (int k = started; k < n_threads; ++k) ref_worker(&jobs[k]);
  }
  for (int k = 0; k < n_threads; ++k)
    if (jobs[k].status != REF_OK) status = jobs[k].status;
  free(q);
  free(jobs);
  free(th);
  return status;
}
