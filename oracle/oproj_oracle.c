/*
 * Output-projection consumer epilogue, single GPU: the CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call it.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Source of the method: the vLLM API page
 *   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.oproj.consumer"
 * (class OprojConsumer: module docstring, methods poll_sum, combined_weight,
 * pre and post).  On that page one token's hidden vector is spread over a
 * cluster of CTAs and the tensor-parallel partial sums arrive in remote
 * mailboxes; here every partial is a plain array, and what is restated is the
 * arithmetic per token:
 *
 *   1. poll_sum / post: the TP partial outputs are summed in FP32 (ranks in
 *      groups, in rank order), the sum is rounded to BF16 and, with a delta
 *      (has_delta), added to the stored prefix and rounded to BF16 again.
 *      That value p is the new prefix (written back) and the residual input.
 *   2. combined_weight: w = norm * query, elementwise.
 *   3. pre: per earlier block b, logit_b = (v_b . w) * rstd(v_b . v_b, eps).
 *   4. post: the prefix takes part as one more candidate with logit
 *      (p . w) * rstd(p . p, eps); a softmax over blocks and prefix weights
 *      the mix y = sum_b e_b v_b + e_p p, and the output is
 *      bf16(out_norm * y * rstd(y . y, out_eps)) (the page keeps the mix
 *      unnormalised and folds the softmax denominator into the eps term,
 *      which is the same RMSNorm).  With no blocks the output is the RMSNorm
 *      of p.
 *
 * Reading (the page does not define rstd): rstd(s, e) = 1 / sqrt(s / hidden
 * + e), the RMSNorm reciprocal of a sum of squares over the whole hidden
 * vector, as the name and the out_norm weight suggest.
 *
 * Compiled twice from this source (KDA_OPROJ_F64):
 *   0 -> kda_oracle_oproj_f32: the page's FP32 operation order, every
 *        operation correctly rounded to FP32 (exp via double, one rounding),
 *        sums over features sequential in index order;
 *   1 -> kda_oracle_oproj_f64: the plain definition above in double, with
 *        the same BF16 rounding points (the reference the tests bound).
 * Must be built with -ffp-contract=off.
 *
 * Layouts (row-major): partials bf16 [tp, tokens, hidden]; prefix bf16
 * [tokens, hidden] in/out; blocks bf16 [tokens, nb, hidden]; norm, query,
 * out_norm bf16 [hidden]; output bf16 [tokens, hidden].
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#if KDA_OPROJ_F64
typedef double real;
#define SUFFIXED(name) name##_f64
#define R_SQRT(a) sqrt(a)
#define R_EXP(a) exp(a)
#define R_FMA(a, b, c) fma((a), (b), (c))
#else
typedef float real;
#define SUFFIXED(name) name##_f32
#define R_SQRT(a) sqrtf(a)
#define R_EXP(a) ((float)exp((double)(a)))
#define R_FMA(a, b, c) fmaf((a), (b), (c))
#endif

#define OPROJ_GROUPS 4

typedef struct {
  int32_t tp, tokens, hidden, nb, has_delta;
  const uint16_t *partials, *blocks, *norm, *query, *out_norm;
  uint16_t *prefix, *output;
  float eps, out_eps;
  /* Test hooks (optional, NULL = unused). */
  const uint16_t *prefix_in; /* [tokens, hidden]: new prefix values forced in  */
                             /* place of the oracle's own (teacher forcing)    */
  double *pre_out;           /* [tokens, hidden]: the new prefix before its    */
                             /* last BF16 rounding                             */
  double *out_pre;           /* [tokens, hidden]: the output before rounding   */
  int32_t threads;
} oproj_oracle_args;

static real bf16_to_real(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (real)f;
}

/* Round to the nearest BF16 value, ties to even; NaN stays NaN. */
static uint16_t to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
  int e;
  frexp(v, &e);
  int qexp = e - 8;
  if (qexp < -133) qexp = -133;
  double q = ldexp(1.0, qexp);
  double r = nearbyint(v / q) * q;
  float f = (float)r;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* rstd(s, e) = 1 / sqrt(s * (1 / hidden) + e), each operation rounded once. */
static real rstd(real s, real e, int hidden) {
  const real inv_n = (real)1 / (real)hidden;
  return (real)1 / R_SQRT(s * inv_n + e);
}

/* Step 1: the new prefix of feature f of one token (before and after its
 * last BF16 rounding).  FP32 mode: ranks in OPROJ_GROUPS groups of
 * S = max(4, ceil(tp / groups)); each group summed in rank order from its
 * first rank, the group sums added in group order.  Double mode: the ranks in
 * rank order (exact for BF16 inputs of ordinary range). */
static void new_prefix(const oproj_oracle_args *a, int t, int f, double *pre,
                       uint16_t *p) {
  const int64_t stride = (int64_t)a->tokens * a->hidden;
  const int64_t at = (int64_t)t * a->hidden + f;
#if KDA_OPROJ_F64
  double attn = 0.0;
  for (int r = 0; r < a->tp; ++r) attn += bf16_to_real(a->partials[r * stride + at]);
#else
  const int per = (a->tp + OPROJ_GROUPS - 1) / OPROJ_GROUPS;
  const int S = per > 4 ? per : 4;
  float attn = 0.0f;
  int first_group = 1;
  for (int g = 0; g < OPROJ_GROUPS; ++g) {
    const int lo = g * S, hi = (lo + S < a->tp) ? lo + S : a->tp;
    if (lo >= hi) continue;
    float gs = bf16_to_real(a->partials[lo * stride + at]);
    for (int r = lo + 1; r < hi; ++r) gs = gs + bf16_to_real(a->partials[r * stride + at]);
    attn = first_group ? gs : attn + gs;
    first_group = 0;
  }
#endif
  const real rounded = bf16_to_real(to_bf16((double)attn));
  real value = rounded;
  if (a->has_delta) value = bf16_to_real(a->prefix[at]) + rounded;
  *pre = (double)value;
  *p = to_bf16((double)value);
}

static void run_token(const oproj_oracle_args *a, int t) {
  const int D = a->hidden, nb = a->nb;
  const int64_t row = (int64_t)t * D;
  /* 1. the new prefix (teacher-forced on request) */
  for (int f = 0; f < D; ++f) {
    double pre;
    uint16_t p;
    new_prefix(a, t, f, &pre, &p);
    if (a->pre_out) a->pre_out[row + f] = pre;
    if (a->prefix_in) p = a->prefix_in[row + f];
    a->prefix[row + f] = p;
  }
  const uint16_t *pb = a->prefix + row;

  if (nb == 0) {
    /* RMSNorm of p (post, no blocks). */
    real pp = 0;
    for (int f = 0; f < D; ++f) {
      const real v = bf16_to_real(pb[f]);
      pp = R_FMA(v, v, pp);
    }
    const real cp = rstd(pp, (real)a->out_eps, D);
    for (int f = 0; f < D; ++f) {
      const real y = (cp * bf16_to_real(pb[f])) * bf16_to_real(a->out_norm[f]);
      if (a->out_pre) a->out_pre[row + f] = (double)y;
      a->output[row + f] = to_bf16((double)y);
    }
    return;
  }

  const uint16_t *vb = a->blocks + (int64_t)t * nb * D;
  /* 2-3. combined weight and block logits */
  real logit[8];
  for (int b = 0; b < nb; ++b) {
    real ss = 0, qk = 0;
    for (int f = 0; f < D; ++f) {
      const real v = bf16_to_real(vb[(int64_t)b * D + f]);
      const real w = bf16_to_real(a->norm[f]) * bf16_to_real(a->query[f]);
      ss = R_FMA(v, v, ss);
      qk = R_FMA(v, w, qk);
    }
    logit[b] = qk * rstd(ss, (real)a->eps, D);
  }
  /* the prefix's own logit */
  real pp = 0, pw = 0;
  for (int f = 0; f < D; ++f) {
    const real v = bf16_to_real(pb[f]);
    const real w = bf16_to_real(a->norm[f]) * bf16_to_real(a->query[f]);
    pp = R_FMA(v, v, pp);
    pw = R_FMA(v, w, pw);
  }
  const real lp = pw * rstd(pp, (real)a->eps, D);

#if KDA_OPROJ_F64
  /* 4. the definition: softmax over blocks and prefix, mix, RMSNorm. */
  double m = lp;
  for (int b = 0; b < nb; ++b) m = logit[b] > m ? logit[b] : m;
  double e[9], den = 0.0;
  for (int b = 0; b < nb; ++b) {
    e[b] = exp(logit[b] - m);
    den += e[b];
  }
  const double ep = exp(lp - m);
  den += ep;
  double ss = 0.0;
  for (int f = 0; f < D; ++f) {
    double y = ep * bf16_to_real(pb[f]);
    for (int b = 0; b < nb; ++b) y += e[b] * bf16_to_real(vb[(int64_t)b * D + f]);
    y /= den;
    ss += y * y;
  }
  const double r = 1.0 / sqrt(ss / D + (double)a->out_eps);
  for (int f = 0; f < D; ++f) {
    double y = ep * bf16_to_real(pb[f]);
    for (int b = 0; b < nb; ++b) y += e[b] * bf16_to_real(vb[(int64_t)b * D + f]);
    y = (y / den) * r * bf16_to_real(a->out_norm[f]);
    if (a->out_pre) a->out_pre[row + f] = y;
    a->output[row + f] = to_bf16(y);
  }
#else
  /* 4. the page's order: block softmax first (max, exponentials, their sum,
   * the unnormalised mix), then the prefix merged in with a rescale, the
   * mix's RMS from the expanded square, and the output coefficients. */
  float mx = logit[0];
  for (int b = 1; b < nb; ++b) mx = logit[b] > mx ? logit[b] : mx;
  float e[8], esum = 0.0f;
  for (int b = 0; b < nb; ++b) {
    e[b] = R_EXP(logit[b] - mx);
    esum = esum + e[b];
  }
  float t0 = 0, t1 = 0; /* mix . p, mix . mix */
  for (int f = 0; f < D; ++f) {
    float mix = 0.0f;
    for (int b = 0; b < nb; ++b) mix = fmaf(e[b], bf16_to_real(vb[(int64_t)b * D + f]), mix);
    t0 = fmaf(mix, bf16_to_real(pb[f]), t0);
    t1 = fmaf(mix, mix, t1);
  }
  const float m2 = lp > mx ? lp : mx;
  const float alpha = R_EXP(mx - m2);
  const float ep = R_EXP(lp - m2);
  const float den = fmaf(alpha, esum, ep);
  const float a2 = alpha * alpha;
  const float ae2 = (2.0f * alpha) * ep;
  const float quad = fmaf(a2, t1, fmaf(ae2, t0, (ep * ep) * pp));
  const float scale = rstd(quad, (a->out_eps * den) * den, D);
  const float ca = alpha * scale, cp = ep * scale;
  for (int f = 0; f < D; ++f) {
    float mix = 0.0f;
    for (int b = 0; b < nb; ++b) mix = fmaf(e[b], bf16_to_real(vb[(int64_t)b * D + f]), mix);
    float y = cp * bf16_to_real(pb[f]);
    y = fmaf(ca, mix, y);
    y = y * bf16_to_real(a->out_norm[f]);
    if (a->out_pre) a->out_pre[row + f] = (double)y;
    a->output[row + f] = to_bf16((double)y);
  }
#endif
}

int SUFFIXED(kda_oracle_oproj)(const oproj_oracle_args *a) {
  if (!a || a->tp < 1 || a->tokens < 0 || a->hidden < 1 || a->nb < 0 || a->nb > 8)
    return 1;
#ifdef _OPENMP
  const int nt = a->threads > 0 ? a->threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
  for (int t = 0; t < a->tokens; ++t) run_token(a, t);
  return 0;
}
