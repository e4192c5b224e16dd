/*
 * KDA decode / speculative-verify step: the CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * restatement of the step that the GPU library is checked against.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may build,
 * load or call it.  It shares no code, header, table or helper with the CUDA
 * path (the library under linear_attention_recurrent_kda_gb300/csrc): it has
 * its own argument struct, its own BF16 rounding and its own arithmetic.
 *
 * Source of the method: the vLLM API page
 *   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide"
 * (class KdaWide; its module docstring, the `kernel` method and the helper
 * methods `silu`, `decay`, `quad_sum`).  Each function below names the part of
 * that page it restates.  Where the page leaves a step open the reading taken
 * is stated at the step.
 *
 * Precision (module docstring of the page): FP32 arithmetic with BF16 rounding
 * of the convolution outputs, the raw gates and the recurrence outputs; only
 * the FP32 reduction order may differ between implementations.  This file is
 * compiled twice from the same source:
 *   KDA_ORACLE_F64=0  -> kda_oracle_step_f32: every elementary operation is a
 *                        correctly rounded FP32 operation (exp through double
 *                        then one rounding to float), reductions summed
 *                        sequentially in index order;
 *   KDA_ORACLE_F64=1  -> kda_oracle_step_f64: the same BF16 rounding points,
 *                        every other operation in double.
 * It must be compiled with -ffp-contract=off so that no a*b+c is silently
 * fused; every fused multiply-add below is an explicit fma call.
 *
 * Layouts (row-major, dim = heads*dk):
 *   x           bf16 [batch*tokens, 3*dim]     q | k | v column blocks
 *   conv_weight bf16 [3, 4, dim]               (part, tap, channel)
 *   conv_bias   bf16 [3*dim]                   (has_bias only)
 *   conv_state  bf16 [num_slots, 3*dim, conv_width]   in/out
 *   f_a         bf16 [batch*tokens, rank]
 *   f_b         bf16 [dim, rank]               (feature, rank)
 *   beta        bf16 [batch*tokens, heads]     raw logits
 *   a_log       f32  [heads];  dt_bias f32 [dim]
 *   gate        bf16 [batch*tokens, dim];  norm_weight bf16 [dk]
 *   slots       i32  [batch] (tokens==1) or [batch, slot_cols] (tokens>1)
 *   accepted    i32  [batch] (tokens>1)
 *   state       f32  [num_slots, heads, dk (value row i), dk (key j)]   in/out
 *   output      bf16 [batch*tokens, dim]
 *   rec_u       f32  [batch, heads, tokens, dk]       (record only)
 *   rec_kg      bf16 [batch, heads, tokens, 2*dk]     (record only)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#if KDA_ORACLE_F64
typedef double real;
#define SUFFIXED(name) name##_f64
#define R_FMA(a, b, c) fma((a), (b), (c))
#define R_SQRT(a) sqrt(a)
#define R_EXP(a) exp(a)
#else
typedef float real;
#define SUFFIXED(name) name##_f32
#define R_FMA(a, b, c) fmaf((a), (b), (c))
#define R_SQRT(a) sqrtf(a)
/* exp correctly rounded to FP32: evaluate in double, round once. */
#define R_EXP(a) ((float)exp((double)(a)))
#endif

/* Device-style error flags (same meaning as the library's error word). */
#define ORACLE_ERR_SLOT 1
#define ORACLE_ERR_ACCEPTED 2

typedef struct {
  int32_t batch, heads, tokens, dk, rank;
  int32_t num_slots, conv_width, slot_cols;
  int32_t gate_mode, has_bias, record;
  const uint16_t *x, *conv_weight, *conv_bias, *f_a, *f_b, *beta, *gate,
      *norm_weight;
  const float *a_log, *dt_bias;
  const int32_t *slots, *accepted;
  uint16_t *conv_state;
  float *state;
  uint16_t *output;
  float *rec_u;
  uint16_t *rec_kg;
  float lower_bound, scale, eps;
  /* Test hooks (all optional, NULL = unused). */
  const int32_t *items;      /* item list (r*heads + h); NULL = every item   */
  int32_t n_items;
  uint16_t *inter_out;       /* bf16 [batch,heads,tokens,4,dk]: q,k,v,raw_g   */
  double *pre_out;           /* same shape: the values before BF16 rounding  */
  const uint16_t *inter_in;  /* same shape: BF16 values forced in place of   */
                             /* the oracle's own q,k,v,raw_g (teacher force) */
  double *o_out;             /* [batch,heads,tokens,dk]: o before rounding   */
  int32_t *err;              /* OR of ORACLE_ERR_* over items                */
  int32_t threads;           /* OpenMP threads (<=0: library default)        */
  /* FP32 conv state (the page's conv_type is the pool's own element type):
   * when conv_f32 != 0, conv_state_f32 [num_slots, 3*dim, W] replaces
   * conv_state; taps are read as stored and the window is written as FP32. */
  int32_t conv_f32;
  float *conv_state_f32;
  /* Test hook: double [batch,heads,tokens,3,dk], the SiLU argument (the
   * convolution's FP32 sum) of q, k, v; the parity checks bound the error of
   * an approximate SiLU by it.  NULL = unused. */
  double *silu_in_out;
} kda_oracle_args;

/* ---- BF16 <-> binary floating point -------------------------------------- */

static real bf16_to_real(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (real)f;
}

/* Round to the nearest BF16 value, ties to even; NaN stays NaN. */
#if KDA_ORACLE_F64
static uint16_t real_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
  /* BF16 keeps 8 significant bits; its smallest quantum is 2^-133. */
  int e;
  frexp(v, &e); /* |v| = m * 2^e, 0.5 <= m < 1 */
  int qexp = e - 8;
  if (qexp < -133) qexp = -133;
  double q = ldexp(1.0, qexp);
  double r = nearbyint(v / q) * q; /* default rounding mode: ties to even */
  float f = (float)r;              /* exact, or +-inf past the BF16 range  */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}
#else
static uint16_t real_to_bf16(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}
#endif

static real round_bf16(real v) { return bf16_to_real(real_to_bf16(v)); }

/* ---- elementary functions as the page names them --------------------------
 * KdaWide.silu: x / (1 + exp(-x)), stored BF16 (the rounding is done by the
 * caller).  triton_sigmoid (used for beta, the decay and the output gate):
 * 1 / (1 + exp(-z)).  Reading: both are the mathematical functions, each
 * operation rounded once in the working precision. */
static real sigmoid(real z) {
  real e = R_EXP(-z);
  real den = (real)1 + e;
  return (real)1 / den;
}

static real silu_unrounded(real a) {
  real e = R_EXP(-a);
  real den = (real)1 + e;
  return a / den;
}

/* KdaWide.decay: exp(lower_bound * sigmoid(exp(A_log) * (raw_g + dt_bias))). */
static real decay_of(real a_log, real raw_g, real dt, real lower_bound) {
  real ea = R_EXP(a_log);
  real z = ea * (raw_g + dt);
  real s = sigmoid(z);
  real g = lower_bound * s;
  return R_EXP(g);
}

/* ---- one (request, head) item ---------------------------------------------- */

static void pad_item(const kda_oracle_args *a, int r, int h) {
  /* KdaWide.kernel, `if slot <= 0`: BF16 zeros for every token of the item;
   * nothing else is written. */
  const long dim = (long)a->heads * a->dk;
  for (int t = 0; t < a->tokens; ++t)
    for (int c = 0; c < a->dk; ++c)
      a->output[((long)r * a->tokens + t) * dim + (long)h * a->dk + c] = 0;
}

/* Returns the error flags raised by this item (0 when none). */
static int run_item(const kda_oracle_args *a, int r, int h) {
  const int T = a->tokens, D = a->dk, R = a->rank, H = a->heads;
  const int W = a->conv_width;
  const long dim = (long)H * D;

  /* Slot resolution (KdaWide.kernel, first block): decode reads slot = conv
   * slot = slots[r] at window offset 0; verify reads the state of the last
   * accepted token, slots[r, accepted-1], and the conv rows of slots[r, 0] at
   * window offset accepted-1.  Indices the page leaves unchecked are checked
   * here: a bad one makes the item an error item, handled like padding. */
  int s, cs, off;
  if (T == 1) {
    s = a->slots[r];
    cs = s;
    off = 0;
  } else {
    int acc = a->accepted[r];
    if (acc < 1 || acc > T) {
      pad_item(a, r, h);
      return ORACLE_ERR_ACCEPTED;
    }
    off = acc - 1;
    s = a->slots[(long)r * a->slot_cols + off];
    cs = a->slots[(long)r * a->slot_cols];
  }
  if (s <= 0) {
    pad_item(a, r, h);
    return 0;
  }
  if (s >= a->num_slots || cs <= 0 || cs >= a->num_slots) {
    pad_item(a, r, h);
    return ORACLE_ERR_SLOT;
  }
  if (T > 1 && !a->record) {
    for (int t = 0; t < T; ++t)
      if (a->slots[(long)r * a->slot_cols + t] >= a->num_slots) {
        pad_item(a, r, h);
        return ORACLE_ERR_SLOT;
      }
  }

  const long item = (long)r * H + h;
  real *q = malloc(sizeof(real) * T * D), *k = malloc(sizeof(real) * T * D);
  real *v = malloc(sizeof(real) * T * D), *graw = malloc(sizeof(real) * T * D);
  real *dec = malloc(sizeof(real) * T * D), *qn = malloc(sizeof(real) * T * D);
  real *kn = malloc(sizeof(real) * T * D), *ob = malloc(sizeof(real) * T * D);
  real *P = malloc(sizeof(real) * D * D), *u = malloc(sizeof(real) * D);
  real beta_t[8];
  real *old_taps = malloc(sizeof(real) * 3 * D * 3);
  real *parts[3] = {q, k, v};

  /* Short causal depthwise convolution + SiLU (KdaWide.kernel, "The
   * convolution (stock tap order) and SiLU, BF16-rounded"): window = the three
   * cached taps at columns off..off+2 followed by the T new inputs; token t
   * starts from the bias (or 0) and adds tap i of the window at t+i with a
   * fused multiply-add, i = 0..3 in order. */
  for (int p = 0; p < 3; ++p) {
    for (int c = 0; c < D; ++c) {
      const long ch = (long)p * dim + (long)h * D + c;
      const long rowix = ((long)cs * 3 * dim + ch) * W;
      real win[3 + 8];
      for (int i = 0; i < 3; ++i) {
        win[i] = a->conv_f32 ? (real)a->conv_state_f32[rowix + off + i]
                             : bf16_to_real(a->conv_state[rowix + off + i]);
        old_taps[(p * D + c) * 3 + i] = win[i];
      }
      for (int t = 0; t < T; ++t)
        win[3 + t] = bf16_to_real(a->x[((long)r * T + t) * 3 * dim + ch]);
      real wt[4];
      for (int i = 0; i < 4; ++i)
        wt[i] = bf16_to_real(a->conv_weight[(long)(p * 4 + i) * dim + (long)h * D + c]);
      for (int t = 0; t < T; ++t) {
        real acc = a->has_bias ? bf16_to_real(a->conv_bias[ch]) : (real)0;
        for (int i = 0; i < 4; ++i) acc = R_FMA(win[t + i], wt[i], acc);
        real y = silu_unrounded(acc);
        const long ix = ((item * T + t) * 4 + p) * D + c;
        if (a->silu_in_out) a->silu_in_out[((item * T + t) * 3 + p) * D + c] = (double)acc;
        if (a->pre_out) a->pre_out[ix] = (double)y;
        uint16_t yb = real_to_bf16(y);
        if (a->inter_out) a->inter_out[ix] = yb;
        if (a->inter_in) yb = a->inter_in[ix];
        parts[p][t * D + c] = bf16_to_real(yb);
      }
    }
  }

  /* Low-rank gate projection (KdaWide.kernel, "Gate projection"): raw_g[t,f]
   * = BF16( sum_k f_b[h*D+f, k] * f_a[r*T+t, k] ).  The BF16 products are exact
   * in FP32.  gate_mode 0: one chain over k in order; gate_mode 1: four chains
   * over consecutive quarters of k, combined as 0 + (((c0 + c1) + c2) + c3). */
  for (int t = 0; t < T; ++t) {
    const uint16_t *fa = a->f_a + ((long)r * T + t) * R;
    for (int f = 0; f < D; ++f) {
      const uint16_t *fb = a->f_b + ((long)h * D + f) * R;
      real acc;
      if (a->gate_mode == 0) {
        acc = 0;
        for (int kk = 0; kk < R; ++kk)
          acc = R_FMA(bf16_to_real(fb[kk]), bf16_to_real(fa[kk]), acc);
      } else {
        real chain[4];
        const int quarter = R / 4;
        for (int m = 0; m < 4; ++m) {
          chain[m] = 0;
          for (int kk = m * quarter; kk < (m + 1) * quarter; ++kk)
            chain[m] = R_FMA(bf16_to_real(fb[kk]), bf16_to_real(fa[kk]), chain[m]);
        }
        acc = (real)0 + (((chain[0] + chain[1]) + chain[2]) + chain[3]);
      }
      const long ix = ((item * T + t) * 4 + 3) * D + f;
      if (a->pre_out) a->pre_out[ix] = (double)acc;
      uint16_t gb = real_to_bf16(acc);
      if (a->inter_out) a->inter_out[ix] = gb;
      if (a->inter_in) gb = a->inter_in[ix];
      graw[t * D + f] = bf16_to_real(gb);
      /* KdaWide.decay on the BF16 raw gate. */
      dec[t * D + f] = decay_of((real)a->a_log[h], graw[t * D + f],
                                (real)a->dt_bias[(long)h * D + f],
                                (real)a->lower_bound);
    }
  }

  /* beta: sigmoid of the raw logit beta[r*T+t, h]. */
  for (int t = 0; t < T; ++t)
    beta_t[t] = sigmoid(bf16_to_real(a->beta[((long)r * T + t) * H + h]));

  /* L2 normalisation ("Normalized q (with the 1/sqrt(K) scale) and k"):
   * squares summed, + 1e-6, reciprocal of the square root; q is then scaled,
   * each product rounded on its own (no fused operations). */
  for (int t = 0; t < T; ++t) {
    real sq = 0, sk = 0;
    for (int c = 0; c < D; ++c) {
      real pq = q[t * D + c] * q[t * D + c];
      real pk = k[t * D + c] * k[t * D + c];
      sq = sq + pq;
      sk = sk + pk;
    }
    real fq = (real)1 / R_SQRT(sq + (real)1.0e-6);
    real fk = (real)1 / R_SQRT(sk + (real)1.0e-6);
    for (int c = 0; c < D; ++c) {
      real t1 = q[t * D + c] * fq;
      qn[t * D + c] = t1 * (real)a->scale;
      kn[t * D + c] = k[t * D + c] * fk;
    }
  }

  /* The recurrence ("The recurrence"): the page P = state[s, h] is read once,
   * indexed [value row i][key j].  Per token: decay every key column; the
   * row's dot with k; u = (v - dot) * beta; P += k u (fused, k first); o = the
   * row's dot with q, rounded to BF16.  Then the per-token write: record mode
   * writes the records, otherwise the page goes to slot (decode) or
   * slots[r, t] (verify) when that target is > 0. */
  const float *page = a->state + ((long)s * H + h) * (long)D * D;
  for (long e = 0; e < (long)D * D; ++e) P[e] = (real)page[e];
  for (int t = 0; t < T; ++t) {
    const real *dt_ = dec + t * D, *kt = kn + t * D, *qt = qn + t * D;
    for (int i = 0; i < D; ++i)
      for (int j = 0; j < D; ++j) P[i * D + j] = P[i * D + j] * dt_[j];
    for (int i = 0; i < D; ++i) {
      real dot = 0;
      for (int j = 0; j < D; ++j) dot = R_FMA(P[i * D + j], kt[j], dot);
      real diff = v[t * D + i] - dot;
      u[i] = diff * beta_t[t];
    }
    for (int i = 0; i < D; ++i)
      for (int j = 0; j < D; ++j) P[i * D + j] = R_FMA(kt[j], u[i], P[i * D + j]);
    for (int i = 0; i < D; ++i) {
      real o = 0;
      for (int j = 0; j < D; ++j) o = R_FMA(P[i * D + j], qt[j], o);
      if (a->o_out) a->o_out[(item * T + t) * D + i] = (double)o;
      ob[t * D + i] = round_bf16(o);
    }
    if (a->record) {
      /* Records: BF16 k before the L2 norm, BF16 raw gate, FP32 u.  Reading:
       * the page's record_row(args, request) is the request index. */
      uint16_t *kg = a->rec_kg + (item * T + t) * 2 * D;
      for (int c = 0; c < D; ++c) {
        kg[c] = real_to_bf16(k[t * D + c]);
        kg[D + c] = real_to_bf16(graw[t * D + c]);
      }
      for (int i = 0; i < D; ++i) a->rec_u[(item * T + t) * D + i] = (float)u[i];
    } else {
      int tgt = (T == 1) ? s : a->slots[(long)r * a->slot_cols + t];
      if (tgt > 0) {
        float *dst = a->state + ((long)tgt * H + h) * (long)D * D;
        for (long e = 0; e < (long)D * D; ++e) dst[e] = (float)P[e];
      }
    }
  }

  /* Gated output RMSNorm ("Gated RMSNorm"): var = (sum_c o_c^2) * (1/D) + eps;
   * out = BF16(((o * rstd) * norm_weight) * sigmoid(gate)). */
  for (int t = 0; t < T; ++t) {
    real ss = 0;
    for (int c = 0; c < D; ++c) {
      real sq = ob[t * D + c] * ob[t * D + c];
      ss = ss + sq;
    }
    real var = ss * ((real)1 / (real)D) + (real)a->eps;
    real rstd = (real)1 / R_SQRT(var);
    for (int c = 0; c < D; ++c) {
      const long col = (long)h * D + c;
      real sg = sigmoid(bf16_to_real(a->gate[((long)r * T + t) * dim + col]));
      real y = ((ob[t * D + c] * rstd) * bf16_to_real(a->norm_weight[c])) * sg;
      a->output[((long)r * T + t) * dim + col] = real_to_bf16(y);
    }
  }

  /* Convolution window write: columns [tap1, tap2, x_0 .. x_{T-1}] of the
   * conv slot, raw copies of the stored values. */
  for (int p = 0; p < 3; ++p)
    for (int c = 0; c < D; ++c) {
      const long ch = (long)p * dim + (long)h * D + c;
      const long rowix = ((long)cs * 3 * dim + ch) * W;
      if (a->conv_f32) {
        float *row = a->conv_state_f32 + rowix;
        row[0] = (float)old_taps[(p * D + c) * 3 + 1];
        row[1] = (float)old_taps[(p * D + c) * 3 + 2];
        for (int t = 0; t < T; ++t)
          row[2 + t] = (float)bf16_to_real(a->x[((long)r * T + t) * 3 * dim + ch]);
      } else {
        uint16_t *row = a->conv_state + rowix;
        row[0] = real_to_bf16(old_taps[(p * D + c) * 3 + 1]);
        row[1] = real_to_bf16(old_taps[(p * D + c) * 3 + 2]);
        for (int t = 0; t < T; ++t) row[2 + t] = a->x[((long)r * T + t) * 3 * dim + ch];
      }
    }

  free(q); free(k); free(v); free(graw); free(dec); free(qn); free(kn);
  free(ob); free(P); free(u); free(old_taps);
  return 0;
}

/* Runs the step over every item (or the listed ones).  Returns 0, or -1 when
 * the static arguments are outside what the page allows (tokens 1..8,
 * gate_mode 0|1, record only with tokens > 1) or the shapes are inconsistent. */
int SUFFIXED(kda_oracle_step)(const kda_oracle_args *a) {
  if (a->tokens < 1 || a->tokens > 8) return -1;
  if (a->gate_mode != 0 && a->gate_mode != 1) return -1;
  if (a->record && a->tokens == 1) return -1;
  if (a->conv_width < a->tokens + 2) return -1;
  if (a->tokens > 1 && a->slot_cols < a->tokens) return -1;
  if (a->rank % 4 != 0 || a->dk < 1) return -1;
  const long n = a->items ? a->n_items : (long)a->batch * a->heads;
  int flags = 0;
#ifdef _OPENMP
  int nt = a->threads > 0 ? a->threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nt) reduction(| : flags)
#endif
  for (long e = 0; e < n; ++e) {
    long it = a->items ? a->items[e] : e;
    flags |= run_item(a, (int)(it / a->heads), (int)(it % a->heads));
  }
  if (a->err) *a->err |= flags;
  return 0;
}

/* ---- record replay ---------------------------------------------------------
 * The page's record mode ("RecoverSSM verify": checkpoint slot, records out)
 * writes no state; it leaves per token the BF16 k before the L2 norm, the BF16
 * raw gate and the FP32 u of every value row.  The replay the page refers to
 * (RecoverSSM) is not shown; reading taken: for the first `accepted[r]` tokens
 * of request r, starting from the checkpoint page, apply the recurrence's own
 * state update with those records -- decay every key column by the decay of
 * the recorded raw gate, then P += k_hat u (fused, k first) with k_hat the L2
 * normalised recorded k -- and write the result to dst_slots[r].  This
 * reproduces the state a non-record step writes after token accepted-1. */
typedef struct {
  int32_t batch, heads, tokens, dk, num_slots;
  const int32_t *src_slots, *dst_slots, *accepted;
  const float *rec_u;       /* [batch, heads, tokens, dk] */
  const uint16_t *rec_kg;   /* bf16 [batch, heads, tokens, 2*dk] */
  const float *a_log, *dt_bias;
  float lower_bound;
  float *state;             /* [num_slots, heads, dk, dk] in/out */
  int32_t *err;
  int32_t threads;
} kda_oracle_recover_args;

static int recover_item(const kda_oracle_recover_args *a, int r, int h) {
  const int T = a->tokens, D = a->dk, H = a->heads;
  const int src = a->src_slots[r], dst = a->dst_slots[r], acc = a->accepted[r];
  if (src <= 0 || dst <= 0) return 0; /* padding: nothing written */
  if (src >= a->num_slots || dst >= a->num_slots) return ORACLE_ERR_SLOT;
  if (acc < 0 || acc > T) return ORACLE_ERR_ACCEPTED;
  real *P = malloc(sizeof(real) * D * D), *kh = malloc(sizeof(real) * D);
  real *dec = malloc(sizeof(real) * D);
  const float *page = a->state + ((long)src * H + h) * (long)D * D;
  for (long e = 0; e < (long)D * D; ++e) P[e] = (real)page[e];
  const long item = (long)r * H + h;
  for (int t = 0; t < acc; ++t) {
    const uint16_t *kg = a->rec_kg + (item * T + t) * 2 * D;
    const float *u = a->rec_u + (item * T + t) * D;
    real sk = 0;
    for (int c = 0; c < D; ++c) {
      real kc = bf16_to_real(kg[c]);
      real pk = kc * kc;
      sk = sk + pk;
    }
    real fk = (real)1 / R_SQRT(sk + (real)1.0e-6);
    for (int c = 0; c < D; ++c) kh[c] = bf16_to_real(kg[c]) * fk;
    for (int f = 0; f < D; ++f)
      dec[f] = decay_of((real)a->a_log[h], bf16_to_real(kg[D + f]),
                        (real)a->dt_bias[(long)h * D + f], (real)a->lower_bound);
    for (int i = 0; i < D; ++i)
      for (int j = 0; j < D; ++j) P[i * D + j] = P[i * D + j] * dec[j];
    for (int i = 0; i < D; ++i)
      for (int j = 0; j < D; ++j) P[i * D + j] = R_FMA(kh[j], (real)u[i], P[i * D + j]);
  }
  float *out = a->state + ((long)dst * H + h) * (long)D * D;
  for (long e = 0; e < (long)D * D; ++e) out[e] = (float)P[e];
  free(P); free(kh); free(dec);
  return 0;
}

/* Replays every item; src and dst pages of different requests must be
 * distinct, and an item's dst may equal its src. */
int SUFFIXED(kda_oracle_recover)(const kda_oracle_recover_args *a) {
  if (a->tokens < 1 || a->tokens > 8) return -1;
  const long n = (long)a->batch * a->heads;
  int flags = 0;
#ifdef _OPENMP
  int nt = a->threads > 0 ? a->threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nt) reduction(| : flags)
#endif
  for (long e = 0; e < n; ++e)
    flags |= recover_item(a, (int)(e / a->heads), (int)(e % a->heads));
  if (a->err) *a->err |= flags;
  return 0;
}

/* Threads an OpenMP build will use by default (1 without OpenMP). */
int SUFFIXED(kda_oracle_max_threads)(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
