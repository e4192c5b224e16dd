/*
 * kda.h -- C ABI of the GB300 (sm_103a) KDA decode / speculative-verify step,
 * its record replay (kda_recover) and the output-projection consumer epilogue
 * that follows the attention layer (kda_oproj, declared at the end).
 *
 * The operation is the one defined by the vLLM API page
 *   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide"
 * (class KdaWide: the constructor's validation, `kernel`, and the helpers
 * `silu`, `decay`, `quad_sum`).  For every (request r, head h) item one call:
 *
 *   1. resolves the item's slots (decode: slot = conv slot = slots[r], window
 *      offset 0; verify: slot = slots[r, accepted[r]-1], conv slot =
 *      slots[r, 0], window offset accepted[r]-1); slot <= 0 marks padding:
 *      the item's output rows are BF16 zeros and nothing else is written;
 *   2. runs the 4-tap causal depthwise convolution over the three cached taps
 *      and the new inputs (plus optional bias), SiLU, BF16 rounding (q, k, v);
 *   3. computes the low-rank gate raw_g = BF16(f_b[h] . f_a[row]) and the decay
 *      exp(lower_bound * sigmoid(exp(A_log[h]) * (raw_g + dt_bias)));
 *   4. beta = sigmoid(beta_raw); L2-normalises q (times scale) and k;
 *   5. applies the per-key-decayed delta rule to the 128x128 FP32 state page
 *      [value row i][key j]:  S *= d (per key);  u = (v - S k) * beta;
 *      S += u k^T;  o = BF16(S q);  and writes the page after every token to
 *      slot (decode) or slots[r, t] when > 0 (verify), or, in record mode,
 *      writes the records instead of any state;
 *   6. writes the new conv window [tap1, tap2, x_0 .. x_{T-1}];
 *   7. out = BF16(((o * rsqrt(mean(o^2) + eps)) * norm_weight) * sigmoid(gate)).
 *
 * Sizes fixed by the method: dk = dv = 128 and gate rank 128, conv kernel 4.
 * Arithmetic: FP32 with BF16 rounding of q, k, v, raw_g and o; exp is
 * 2^(x*log2 e) on the hardware's approximate exp2, division / square root /
 * reciprocal are the hardware's approximate (full-range) instructions, the
 * gate projection runs on tensor cores with FP32 accumulation.  Only FP32
 * reduction order differs from a sequential evaluation.
 *
 * Ownership and threading: the caller owns every buffer; every pointer is a
 * DEVICE pointer of the current device.  The library allocates nothing,
 * never synchronises, and enqueues exactly one kernel on `stream` per call.
 * Calls are reentrant and may come from several host threads at once (the
 * first call on a device reads its attributes and configures the kernel
 * under a lock); two calls that write the same pool regions must be ordered
 * by the caller (same stream or events).
 *
 * Aliasing contract: within one call, the state pages and conv rows touched
 * by different requests must be distinct (distinct slots per request).  An
 * item may write the page it read (same slot): its read completes first.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 7
#define KDA_DK 128
#define KDA_MAX_TOKENS 8

/* Host-side return codes (nothing is launched unless KDA_SUCCESS). */
enum {
  KDA_SUCCESS = 0,
  KDA_ERR_NULL_ARGS = 1,      /* args == NULL                                  */
  KDA_ERR_TOKENS = 2,         /* tokens outside 1..8 (KdaWide.__init__), or    */
                              /* kda_decode with tokens != 1, kda_verify == 1  */
  KDA_ERR_GATE_MODE = 3,      /* gate_mode not 0|1 (KdaWide.__init__)          */
  KDA_ERR_RECORD = 4,         /* record with tokens == 1 (KdaWide.__init__)    */
  KDA_ERR_NULL_POINTER = 5,   /* a required pointer is NULL                    */
  KDA_ERR_CONV_WIDTH = 6,     /* conv_width < tokens + 2, or too wide to stage */
  KDA_ERR_ALIGNMENT = 7,      /* a pointer breaks its alignment rule (below)   */
  KDA_ERR_SHAPE = 8,          /* negative sizes, num_slots < 1, slot_cols <    */
                              /* tokens, or an item count beyond 2^31-1        */
  KDA_ERR_DEVICE = 9,         /* no usable device, or not an sm_103 device     */
  KDA_ERR_LAUNCH = 10,        /* the kernel launch failed (CUDA error)         */
  KDA_ERR_PATH = 11           /* path outside 0..2                             */
};

/* Device-side error flags, OR-ed into *err when err != NULL.  An item that
 * raises one is handled like padding (zero output rows, nothing written). */
enum {
  KDA_DEVERR_SLOT = 1,        /* slot, conv slot or a write target >= num_slots,
                                 or a conv slot <= 0 on a live verify item     */
  KDA_DEVERR_ACCEPTED = 2,    /* accepted[r] outside 1..tokens                 */
  KDA_DEVERR_TIMEOUT = 4      /* an on-chip copy wait ran out (the kernel      */
                              /* stopped early; outputs are incomplete)        */
};

/* Arguments of one step.  Layouts are row-major; dim = heads * 128.
 * Alignment: state, f_a, f_b, x, gate and conv_state 16 bytes; the other BF16
 * arrays 2 bytes, FP32/int32 arrays 4 bytes. */
typedef struct kda_args {
  int32_t batch;       /* B requests (0 is a no-op)                          */
  int32_t heads;       /* H heads (0 is a no-op)                             */
  int32_t tokens;      /* T: 1 = decode, 2..8 = verify                       */
  int32_t num_slots;   /* slots in both pools; slot 0 is the null slot       */
  int32_t conv_width;  /* W columns per conv channel row, >= T + 2           */
  int32_t slot_cols;   /* row stride of `slots` in verify, >= T (decode: 1)  */
  int32_t gate_mode;   /* 0: one FP32 chain over the rank; 1: four chains    */
                       /* over rank quarters, then 0 + (((c0+c1)+c2)+c3)     */
  int32_t has_bias;    /* conv bias present                                  */
  int32_t record;      /* record ("RecoverSSM verify") mode, T > 1 only      */
  int32_t use_pdl;     /* launch with programmatic dependent launch (the     */
                       /* page's griddepcontrol ordering): the kernel may    */
                       /* start before the preceding kernel on the stream    */
                       /* ends.  It reads the state pages, slots and         */
                       /* accepted BEFORE waiting for that kernel; every     */
                       /* other input (x, gate, f_a, beta, the conv pool,    */
                       /* the weights) and all of its writes come after.  So */
                       /* the preceding kernel must not write the state      */
                       /* pool, slots or accepted: two steps chained with    */
                       /* PDL must use disjoint state pages.  Ignored by the */
                       /* cluster-split path (path 2).                       */

  const void *x;            /* bf16 [B*T, 3*dim]  q | k | v column blocks    */
  const void *conv_weight;  /* bf16 [3, 4, dim]   (part, tap, channel)       */
  const void *conv_bias;    /* bf16 [3*dim] (has_bias) else ignored          */
  const void *f_a;          /* bf16 [B*T, 128]                               */
  const void *f_b;          /* bf16 [dim, 128]    (feature, rank)            */
  const void *beta;         /* bf16 [B*T, H]      raw logits                 */
  const void *gate;         /* bf16 [B*T, dim]    output gate logits         */
  const void *norm_weight;  /* bf16 [128]         shared by all heads        */
  const float *a_log;       /* f32  [H]                                      */
  const float *dt_bias;     /* f32  [dim]                                    */
  const int32_t *slots;     /* i32  [B] (decode) or [B, slot_cols] (verify)  */
  const int32_t *accepted;  /* i32  [B] (verify), ignored by decode          */

  void *conv_state;         /* bf16 (or f32, conv_f32) [num_slots, 3*dim, W] */
  float *state;             /* f32  [num_slots, H, 128, 128]     in/out      */
  void *output;             /* bf16 [B*T, dim]                   out         */
  float *rec_u;             /* f32  [B, H, T, 128]  record only, else NULL   */
  void *rec_kg;             /* bf16 [B, H, T, 256]  record only: k | raw_g   */

  float lower_bound;        /* decay lower bound (e.g. -5)                   */
  float scale;              /* q scale (e.g. 128^-0.5)                       */
  float eps;                /* RMSNorm epsilon (the L2 norms use 1e-6)       */

  int32_t *err;             /* optional device word for KDA_DEVERR_* flags   */
  void *dbg;                /* optional bf16 [B, H, T, 4, 128]: q, k, v      */
                            /* (after SiLU, before the norm) and raw_g, as   */
                            /* this call rounded them; for parity checks     */
  int32_t path;             /* kernel: 0 = automatic; 1 = persistent, one    */
                            /* CTA per SM walking a range of items (for many */
                            /* items); 2 = one item per cluster of 4 CTAs,   */
                            /* each owning 32 value rows (for few items;     */
                            /* ignores use_pdl).  Both give the same bits.   */
  int32_t conv_f32;         /* conv_state holds FP32 instead of BF16: taps   */
                            /* are read as stored and the new window is      */
                            /* written as FP32 (the page's conv_type is the  */
                            /* pool's element type)                          */
  int32_t *sched;           /* optional i32 [2] device scheduler words, zero */
                            /* before first use; the kernel leaves them zero */
                            /* when it ends.  With them the persistent path  */
                            /* hands the items past the CTAs' contiguous     */
                            /* ranges out one at a time to whichever CTA is  */
                            /* free (an eighth of the items for decode with  */
                            /* >= 32 items per SM and for record steps, else */
                            /* the remainder of an even split; same bits as  */
                            /* without); NULL = fixed contiguous ranges.     */
                            /* Launches that may run at the same time (other */
                            /* streams, other threads) need separate words;  */
                            /* launches in order on one stream, PDL-chained  */
                            /* or captured in a graph, may share them.       */
                            /* Ignored by the cluster-split path (path 2).   */
} kda_args;

/* One decode step (tokens == 1) on `stream` (a cudaStream_t; NULL = the
 * legacy default stream).  Returns KDA_SUCCESS or a KDA_ERR_* code. */
int kda_decode(const kda_args *args, void *stream);

/* One speculative-verify step (tokens 2..8, record optional) on `stream`. */
int kda_verify(const kda_args *args, void *stream);

/* kda_decode (tokens == 1) or kda_verify (tokens > 1) with no caller
 * allocation: args->sched is ignored and the library's own scheduler words
 * (a static, zero-initialised device array per GPU, left zero by every
 * launch) are used instead.  Every launch through this entry on one GPU
 * shares those words, so such launches must not run at the same time: issue
 * them in order on one stream (PDL chaining and graph capture are fine);
 * concurrent streams or threads pass their own words to kda_decode /
 * kda_verify.  Same return codes and bits as those calls. */
int kda_step_noalloc(const kda_args *args, void *stream);

/* Arguments of one record replay (kda_recover). */
typedef struct kda_recover_args {
  int32_t batch;            /* B requests (0 is a no-op)                       */
  int32_t heads;            /* H heads (0 is a no-op)                          */
  int32_t tokens;           /* T of the records, 1..8                          */
  int32_t num_slots;        /* slots in the state pool                         */
  const int32_t *src_slots; /* i32 [B]: checkpoint page; <= 0 = padding        */
  const int32_t *dst_slots; /* i32 [B]: page to write; <= 0 = padding; may     */
                            /* equal src_slots[r]                              */
  const int32_t *accepted;  /* i32 [B]: tokens to replay, 0..T (0 = copy)      */
  const float *rec_u;       /* f32 [B, H, T, 128] from a record-mode verify    */
  const void *rec_kg;       /* bf16 [B, H, T, 256]: k (pre-norm) | raw_g       */
  const float *a_log;       /* f32 [H]                                         */
  const float *dt_bias;     /* f32 [H*128]                                     */
  float lower_bound;        /* as in the step that wrote the records           */
  float *state;             /* f32 [num_slots, H, 128, 128]       in/out       */
  int32_t *err;             /* optional device word for KDA_DEVERR_* flags     */
  int32_t *sched;           /* optional i32 [2] scheduler words, as in         */
                            /* kda_args (zero before first use, left zero;     */
                            /* concurrent launches need their own); NULL =     */
                            /* contiguous item ranges only.  Same bits.        */
} kda_recover_args;

/* Record replay ("RecoverSSM" on the page, referenced but not shown there).
 * A record-mode kda_verify writes no state; it leaves per token the BF16 k
 * before the L2 norm, the BF16 raw gate and the FP32 u of every value row.
 * For each (request r, head h): start from state[src_slots[r], h], for the
 * first accepted[r] tokens decay every key column by the decay of the
 * recorded raw gate and add k_hat u^T (k_hat: L2-normalised recorded k), and
 * write the page to state[dst_slots[r], h].  The arithmetic is the step's, so
 * replaying the records of a record-mode verify reproduces bit for bit the
 * page a non-record verify writes after token accepted[r]-1.
 * Pointers are device pointers; state, rec_u and rec_kg need 16-byte
 * alignment.  Slot >= num_slots or accepted outside 0..T raise
 * KDA_DEVERR_SLOT / KDA_DEVERR_ACCEPTED and the item writes nothing.  Pages
 * of different requests must be distinct.  One kernel on `stream`. */
int kda_recover(const kda_recover_args *args, void *stream);

/* Arguments of one output-projection consumer epilogue (kda_oproj). */
typedef struct kda_oproj_args {
  int32_t tp;               /* partial outputs per token (TP ranks), 1..64     */
  int32_t tokens;           /* rows (0 is a no-op)                             */
  int32_t hidden;           /* features per row: a multiple of 256, <= 7168    */
  int32_t nb;               /* earlier block outputs per token, 0..8           */
  int32_t has_delta;        /* nonzero: new prefix = BF16(prefix + BF16(sum)); */
                            /* zero: new prefix = BF16(sum)                    */
  const void *partials;     /* bf16 [tp, tokens, hidden]: the partial sums     */
  const void *blocks;       /* bf16 [tokens, nb, hidden]; NULL when nb == 0    */
  const void *norm;         /* bf16 [hidden] (nb > 0): block RMSNorm weight    */
  const void *query;        /* bf16 [hidden] (nb > 0): block query             */
  const void *out_norm;     /* bf16 [hidden]: output RMSNorm weight            */
  void *prefix;             /* bf16 [tokens, hidden], in/out: the residual     */
                            /* stream, replaced by the new prefix              */
  void *output;             /* bf16 [tokens, hidden], out                      */
  float eps;                /* epsilon of the block (and prefix) RMS           */
  float out_eps;            /* epsilon of the output RMSNorm                   */
} kda_oproj_args;

/* Output-projection consumer epilogue on one GPU: the per-token arithmetic
 * of class OprojConsumer on the vLLM API page
 *   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.oproj.consumer"
 * (poll_sum, combined_weight, pre, post), with the tensor-parallel partial
 * outputs read from `partials` instead of remote mailboxes and the whole
 * hidden vector of a token in one CTA instead of a cluster.  Per token:
 *   1. sum = the tp partials, summed in FP32 in four rank groups of
 *      S = max(4, ceil(tp/4)) (each in rank order, then the groups in order);
 *      p = BF16(sum), or BF16(prefix + BF16(sum)) with has_delta; p is
 *      written back to `prefix`;
 *   2. with nb > 0: w = norm * query; logit_b = (v_b . w) * rstd(v_b . v_b,
 *      eps) for every block and likewise for p; a softmax over the blocks and
 *      p weights y = sum_b e_b v_b + e_p p;
 *   3. output = BF16(out_norm * y * rstd(y . y, out_eps)) (y = p when nb == 0),
 * where rstd(s, e) = 1 / sqrt(s / hidden + e) (a reading: the page uses rstd
 * without defining it).  FP32 arithmetic; exp and the reciprocal square root
 * on the hardware's approximate instructions; only the FP32 reduction order
 * over features differs from a sequential evaluation.  The MoE "latent"
 * copies and hints of the page's publish step are multi-GPU plumbing and are
 * not produced.  All pointers are device pointers of the current device with
 * 16-byte alignment; partials, blocks and prefix must not overlap output.
 * Errors: KDA_ERR_NULL_ARGS, KDA_ERR_NULL_POINTER, KDA_ERR_SHAPE (sizes
 * outside the ranges above), KDA_ERR_ALIGNMENT, KDA_ERR_DEVICE,
 * KDA_ERR_LAUNCH; nothing is launched on error.  One kernel on `stream`. */
int kda_oproj(const kda_oproj_args *args, void *stream);

/* Self-test of the bounded on-chip waits that every kernel above uses: one
 * CTA waits on an mbarrier that nothing completes; the wait gives up after
 * its wall-clock limit (2 s), KDA_DEVERR_TIMEOUT is OR-ed into *err (a
 * device word, 4-byte aligned) and the kernel returns -- no trap, no fault,
 * the context stays usable.  For failure-detection tests.  Returns
 * KDA_ERR_NULL_POINTER / KDA_ERR_ALIGNMENT / KDA_ERR_LAUNCH or KDA_SUCCESS;
 * one kernel on `stream`. */
int kda_selftest_wait_timeout(int32_t *err, void *stream);

/* Static description of a return code (never NULL). */
const char *kda_strerror(int code);

/* KDA_ABI_VERSION of the loaded library. */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
