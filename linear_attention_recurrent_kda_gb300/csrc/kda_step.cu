// KDA decode / speculative-verify step for GB300 (sm_103a).
//
// Method: vLLM API page
//   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide"
// (class KdaWide: `kernel`, `silu`, `decay`, `quad_sum`); the C ABI and the
// step it runs are described in include/kda.h.
//
// Design (GB300-first; the page's one-CTA-per-item kernel is prior art):
//   * Persistent kernel, one CTA of four warpgroups per SM.  Each CTA owns a
//     contiguous range of items in head-major order (item = h * batch + r), so
//     the per-head f_b tensor-core fragments stay in registers across its
//     items; with scheduler words the items past the ranges then go one at a
//     time to whichever CTA's producer asks first (an atomic counter the last
//     CTA zeroes), so CTAs on slower SMs or with slower pages take fewer and
//     the CTAs finish together.
//   * Three warp roles work on consecutive items at the same time:
//       producer   (warpgroup 3, one thread): picks the next item (its
//                  range, then shared items, then an end marker), resolves the slots,
//                  loads beta and the write targets into an item descriptor and
//                  stages the 64 KiB FP32 state page plus the item's conv rows,
//                  x, gate and f_a rows into a 2-3 stage shared-memory ring
//                  with TMA bulk copies completing on an mbarrier; it runs 2-3
//                  items ahead;
//       front      (warpgroup 2): item j's conv + SiLU, gate projection on
//                  tensor cores (mma.sync m16n8k16 BF16, FP32 accumulate),
//                  decay, beta, L2 norms -> a double-buffered hand-off slot;
//                  before that, the gated RMSNorm of the item the recurrence
//                  last finished in that slot (o and gate are there);
//       recurrence (warpgroups 0-1): item j-1's delta rule with the page in
//                  registers: thread (g = tid/8, l = tid%8) holds keys
//                  {32c + 4l + e} of value rows g, g+32, g+64, g+96 (64
//                  floats), packed FP32 (f32x2) multiplies/FMAs, row sums by an
//                  8-lane reduce-scatter; o goes back into the slot.
//                  Updated pages leave shared memory through TMA bulk stores,
//                  so no per-thread global stores queue in L1TEX:
//                  decode: the page goes, one 16 KiB quarter (32 rows) at a
//                  time, into a ring of quarter buffers served by
//       store      (warpgroup 3, one thread), which bulk-stores each quarter
//                  and frees its buffer once the copy has read it; the stage
//                  is refilled as soon as the page is in registers;
//                  verify: after each written token the page goes back into
//                  its stage buffer and the recurrence leader bulk-stores it;
//                  the stage is released once the last store has read it.
//                  Verify and record steps
//                  also send the new conv windows back from the staged rows
//                  with bulk stores (decode's 3-element windows go direct).
//     The time per item is max(front, recurrence), not their sum.
//   * setmaxnreg moves registers from the producer warpgroup (40 a thread) to
//     the recurrence (160) and front (144) warpgroups; launch gives 128.
//   * Every wait is bounded (wall clock); a timeout raises a shared abort flag
//     that stops every role, and KDA_DEVERR_TIMEOUT is reported.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_device.cuh"
#include "kda_host.h"

namespace kda {

// The cluster-split kernel (kda_split.cu) for few items.
int launch_split(const kda_args *a, cudaStream_t stream);

constexpr int kDk = 128;                          // dk = dv = gate rank
constexpr int kRecThreads = 256;                  // warpgroups 0-1
constexpr int kFrontThreads = 128;                // warpgroup 2
constexpr int kProducer = kRecThreads + kFrontThreads;  // warpgroup 3, thread 0
constexpr int kStorer = kProducer + 32;                 // warpgroup 3, warp 1 lane 0
constexpr int kThreads = kProducer + 128;
constexpr int kRecRegs = 160;                     // setmaxnreg split (launch: 128)
constexpr int kFrontRegs = 144;
constexpr int kProducerRegs = 40;
constexpr uint32_t kPageBytes = kDk * kDk * 4;
constexpr int kMaxStages = 3;
constexpr int kSlots = 2;                         // front -> recurrence hand-off
constexpr int kMaxQuarterBufs = 4;                // 16 KiB quarter-page store ring
constexpr uint32_t kQuarterBytes = kPageBytes / 4;
constexpr int kLive = 0, kPad = 1, kError = 2, kEnd = 3;  // kEnd: no more items

static_assert(kRecThreads * kRecRegs + kFrontThreads * kFrontRegs + 128 * kProducerRegs <=
                  kThreads * 128,
              "register split exceeds the launch allocation");

struct __align__(16) ItemDesc {
  int32_t item;  // n = h * batch + r
  int32_t status;
  int32_t slot;
  int32_t conv_slot;
  int32_t offset;
  int32_t target[KDA_MAX_TOKENS];
  uint16_t beta_bits[KDA_MAX_TOKENS];
};

struct Params {
  int32_t batch, heads, num_slots, conv_width, slot_cols, gate_mode, has_bias;
  int32_t conv_f32;  // conv pool element: FP32 (1) or BF16 (0)
  int32_t items, stages;
  // Item schedule: CTA b owns items [b*q, b*q + q) (q = dyn0 / grid); with a
  // scheduler word pair, items dyn0 .. items-1 then go one at a time to the
  // CTA whose producer asks first (sched[0] counts them out, sched[1] counts
  // finished CTAs; the last CTA zeroes both).  Without one, the items are
  // split into contiguous ranges only.
  int32_t *sched;
  int32_t dyn0;
  uint32_t stage_bytes, conv_off, x_off, gate_off, fa_off;
  uint32_t bar_off, desc_off, slot_off, slot_bytes, scratch_off, rscratch_off;
  uint32_t qbuf_off;
  int32_t nqbuf;
  const __nv_bfloat16 *x, *conv_weight, *conv_bias, *f_a, *f_b, *beta, *gate,
      *norm_weight;
  const float *a_log, *dt_bias;
  const int32_t *slots, *accepted;
  __nv_bfloat16 *conv_state;
  float *state;
  __nv_bfloat16 *output;
  float *rec_u;
  __nv_bfloat16 *rec_kg;
  float lower_bound, scale, eps;
  int32_t *err;
  __nv_bfloat16 *dbg;
};

// Shared-memory control block (barriers, abort flag), at p.bar_off.
struct Ctrl {
  uint64_t full[kMaxStages];   // producer -> front + recurrence (bytes landed)
  uint64_t empty[kMaxStages];  // front + recurrence -> producer (stage free)
  uint64_t fready[kSlots];     // front -> recurrence (slot inputs written)
  uint64_t sfree[kSlots];      // recurrence -> front (slot consumed)
  uint64_t qready[kMaxQuarterBufs];  // recurrence -> store (quarter written)
  uint64_t qfree[kMaxQuarterBufs];   // store -> recurrence (quarter read out)
  float *qdst[kMaxQuarterBufs];      // HBM destination of each quarter, or null
                                     // to end the store thread's loop
  uint32_t abort;
};

// Hand-off slot between the front and the recurrence (one per live item in
// flight): FP32 [T][128] q_hat, k_hat, decay; BF16 [T][128] v, gate, o (all
// three are BF16 values, so the bits move unchanged); beta, targets, item.
template <int T>
struct SlotView {
  float *q, *k, *d, *beta;
  uint16_t *v, *gate, *o;
  int32_t *tgt, *meta;
  __device__ __forceinline__ explicit SlotView(uint8_t *base) {
    float *f = reinterpret_cast<float *>(base);
    q = f;
    k = q + T * kDk;
    d = k + T * kDk;
    beta = d + T * kDk;
    tgt = reinterpret_cast<int32_t *>(beta + KDA_MAX_TOKENS);
    meta = tgt + KDA_MAX_TOKENS;
    v = reinterpret_cast<uint16_t *>(meta + 4);
    gate = v + T * kDk;
    o = gate + T * kDk;
  }
};

// ----------------------------------------------------------------- producer

template <int T, bool RECORD>
__device__ __forceinline__ int resolve_item(const Params &p, int n, ItemDesc &d) {
  const int h = n / p.batch;
  const int r = n - h * p.batch;
  (void)h;
  int s, cs, off;
  int flags = 0;
  if (T == 1) {
    s = __ldg(p.slots + r);
    cs = s;
    off = 0;
  } else {
    const int a = __ldg(p.accepted + r);
    if (a < 1 || a > T) {
      d.status = kError;
      return KDA_DEVERR_ACCEPTED;
    }
    off = a - 1;
    s = __ldg(p.slots + static_cast<int64_t>(r) * p.slot_cols + off);
    cs = __ldg(p.slots + static_cast<int64_t>(r) * p.slot_cols);
  }
  d.slot = s;
  d.conv_slot = cs;
  d.offset = off;
  if (s <= 0) {
    d.status = kPad;
    return 0;
  }
  if (s >= p.num_slots || cs <= 0 || cs >= p.num_slots) flags |= KDA_DEVERR_SLOT;
  if (T > 1 && !RECORD) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int tg = __ldg(p.slots + static_cast<int64_t>(r) * p.slot_cols + t);
      d.target[t] = tg;
      if (tg >= p.num_slots) flags |= KDA_DEVERR_SLOT;
    }
  }
  d.status = flags ? kError : kLive;
  return flags;
}

template <int T>
__device__ __forceinline__ uint32_t small_bytes(const Params &p) {
  return 3u * (p.conv_f32 ? 512u : 256u) * p.conv_width + 3u * T * 256u + 2u * T * 256u;
}

__device__ __forceinline__ void issue_page(const Params &p, uint8_t *stage, int n,
                                           const ItemDesc &d, uint64_t *bar,
                                           uint64_t pol) {
  const int h = n / p.batch;
  const float *src = p.state + (static_cast<int64_t>(d.slot) * p.heads + h) *
                                   static_cast<int64_t>(kDk * kDk);
  bulk_g2s_hint(stage, src, kPageBytes, bar, pol);
}

template <int T>
__device__ __forceinline__ void issue_small(const Params &p, uint8_t *stage, int n,
                                            const ItemDesc &d, uint64_t *bar) {
  const int h = n / p.batch;
  const int r = n - h * p.batch;
  const int64_t dim = static_cast<int64_t>(p.heads) * kDk;
  const uint32_t elem = p.conv_f32 ? 4u : 2u;
  const uint32_t row_bytes = 128u * elem * p.conv_width;  // 128 channels x W
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    const uint8_t *src =
        reinterpret_cast<const uint8_t *>(p.conv_state) +
        (static_cast<int64_t>(d.conv_slot) * 3 * dim + part * dim +
         static_cast<int64_t>(h) * kDk) *
            p.conv_width * elem;
    bulk_g2s(stage + p.conv_off + part * row_bytes, src, row_bytes, bar);
  }
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const int64_t row = static_cast<int64_t>(r) * T + t;
#pragma unroll
    for (int part = 0; part < 3; ++part)
      bulk_g2s(stage + p.x_off + (t * 3 + part) * 256,
               p.x + row * 3 * dim + part * dim + static_cast<int64_t>(h) * kDk, 256,
               bar);
    bulk_g2s(stage + p.gate_off + t * 256,
             p.gate + row * dim + static_cast<int64_t>(h) * kDk, 256, bar);
  }
  bulk_g2s(stage + p.fa_off, p.f_a + static_cast<int64_t>(r) * T * kDk, T * 256u, bar);
}

template <int T>
__device__ __forceinline__ void load_beta(const Params &p, int n, ItemDesc &d) {
  const int h = n / p.batch;
  const int r = n - h * p.batch;
#pragma unroll
  for (int t = 0; t < T; ++t)
    d.beta_bits[t] = __ldg(reinterpret_cast<const uint16_t *>(p.beta) +
                           (static_cast<int64_t>(r) * T + t) * p.heads + h);
}

template <int T, bool RECORD>
__device__ void producer_role(const Params &p, uint8_t *smem, Ctrl *ctl,
                              ItemDesc *desc, int n0, int n1) {
  const int S = p.stages;
  const uint64_t pol = policy_evict_first();
  const int pro = (n1 - n0) < S ? (n1 - n0) : S;
  int issued = 0;
  bool aborted = false;
  bool drained = p.sched == nullptr;  // no shared items left to ask for
  // The CTA's k-th item: its own range first, then shared items (after the
  // wait on the preceding kernel); -1 once none is left.
  auto item_at = [&](int k) -> int {
    if (n0 + k < n1) return n0 + k;
    if (drained) return -1;
    // 64-bit, the counter read unsigned: no wrap however many items there are.
    const int64_t n = p.dyn0 + static_cast<int64_t>(static_cast<uint32_t>(atomicAdd(p.sched, 1)));
    if (n < p.items) return static_cast<int>(n);
    drained = true;
    return -1;
  };

  // Prologue: the first pages go out before waiting on the preceding kernel
  // (the state pool, slots and accepted must not be its outputs); nothing is
  // written and no other input is read before the wait.
  int pro_flags = 0;
  for (int k = 0; k < pro; ++k) {
    ItemDesc &d = desc[k];
    d.item = n0 + k;
    pro_flags |= resolve_item<T, RECORD>(p, n0 + k, d);
    if (d.status == kLive) {
      mbar_expect_tx(&ctl->full[k], kPageBytes);
      issue_page(p, smem + static_cast<size_t>(k) * p.stage_bytes, n0 + k, d,
                 &ctl->full[k], pol);
    }
  }
  griddep_wait();
  if (pro_flags && p.err) atomicOr(p.err, pro_flags);
  for (int k = 0; k < pro; ++k) {
    ItemDesc &d = desc[k];
    load_beta<T>(p, n0 + k, d);
    if (d.status == kLive) {
      mbar_arrive_expect_tx(&ctl->full[k], small_bytes<T>(p));
      issue_small<T>(p, smem + static_cast<size_t>(k) * p.stage_bytes, n0 + k, d,
                     &ctl->full[k]);
    } else {
      mbar_arrive(&ctl->full[k]);
    }
    ++issued;
  }
  for (int k = pro;; ++k) {
    const int stage = k % S;
    const uint32_t round = static_cast<uint32_t>(k / S);
    const int n = item_at(k);
    // Verify items resolve their slots (dependent global loads) while the
    // stage is still busy; decode items after the wait (measured faster).
    ItemDesc nd;
    int flags = 0;
    if (T > 1 && n >= 0) {
      flags = resolve_item<T, RECORD>(p, n, nd);
      load_beta<T>(p, n, nd);
    }
    if (round > 0 && !mbar_wait(&ctl->empty[stage], (round - 1u) & 1u, &ctl->abort)) {
      aborted = true;
      break;
    }
    ItemDesc &d = desc[stage];
    if (n < 0) {
      // End of the stream for the front and the recurrence.
      d.item = -1;
      d.status = kEnd;
      mbar_arrive(&ctl->full[stage]);
      break;
    }
    if (T > 1) {
      d = nd;
    } else {
      flags = resolve_item<T, RECORD>(p, n, d);
      load_beta<T>(p, n, d);
    }
    d.item = n;
    if (flags && p.err) atomicOr(p.err, flags);
    uint8_t *st = smem + static_cast<size_t>(stage) * p.stage_bytes;
    if (d.status == kLive) {
      mbar_arrive_expect_tx(&ctl->full[stage], kPageBytes + small_bytes<T>(p));
      issue_page(p, st, n, d, &ctl->full[stage], pol);
      issue_small<T>(p, st, n, d, &ctl->full[stage]);
    } else {
      mbar_arrive(&ctl->full[stage]);
    }
    ++issued;
  }
  griddep_launch_dependents();
  if (p.sched) {
    // This CTA asks for no more shared items; the last CTA to get here zeroes
    // the scheduler words for the next launch (every request of this launch
    // precedes its CTA's count).
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
  }
  if (aborted || ctl->abort) {
    if (p.err) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
    // Drain: every copy issued into a stage must land before the CTA exits.
    uint32_t keep_waiting = 0;
    for (int k = (issued > S ? issued - S : 0); k < issued; ++k)
      (void)mbar_wait(&ctl->full[k % S], static_cast<uint32_t>(k / S) & 1u,
                      &keep_waiting);
  }
}

// ----------------------------------------------------------------- front

// Per-head constants kept in registers across a CTA's items of one head: the
// f_b fragments of this warp's 32 features, the conv taps and bias of this
// thread's channel, dt_bias of its MMA features and exp(A_log).
struct FrontConst {
  uint32_t wa[2][8][4];  // f_b A fragments: [tile][k chunk][a0..a3]
  float wt[3][4];        // conv taps of channel c, parts q, k, v
  float bias[3];
  float dt[2][2];        // dt_bias of features 32w + 16m + g + 8i
  float ea;              // exp(A_log[h])
};

__device__ __forceinline__ void load_front_const(const Params &p, int h, int c,
                                                 FrontConst &fc) {
  const int fw = c >> 5, lane = c & 31;
  const int g = lane >> 2, q = lane & 3;
  const int64_t dim = static_cast<int64_t>(p.heads) * kDk;
  const uint2 *fb = reinterpret_cast<const uint2 *>(p.f_b);
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int fA = h * kDk + 32 * fw + 16 * m + g;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      // Rank columns 16kc + 4q + {0,1,2,3} play the fragment's k positions
      // {2q, 2q+1, 2q+8, 2q+9}; f_a uses the same permutation (sum unchanged).
      const uint2 lo =
          __ldg(fb + (static_cast<int64_t>(fA) * kDk + 16 * kc + 4 * q) / 4);
      const uint2 hi =
          __ldg(fb + (static_cast<int64_t>(fA + 8) * kDk + 16 * kc + 4 * q) / 4);
      fc.wa[m][kc][0] = lo.x;
      fc.wa[m][kc][2] = lo.y;
      fc.wa[m][kc][1] = hi.x;
      fc.wa[m][kc][3] = hi.y;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
      fc.dt[m][i] = __ldg(p.dt_bias + h * kDk + 32 * fw + 16 * m + g + 8 * i);
  }
  const uint16_t *cw = reinterpret_cast<const uint16_t *>(p.conv_weight);
  const uint16_t *cb = reinterpret_cast<const uint16_t *>(p.conv_bias);
#pragma unroll
  for (int part = 0; part < 3; ++part) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      fc.wt[part][i] = bf16_bits_to_float(
          __ldg(cw + (static_cast<int64_t>(part) * 4 + i) * dim + h * kDk + c));
    fc.bias[part] = p.has_bias
                        ? bf16_bits_to_float(__ldg(cb + part * dim + h * kDk + c))
                        : 0.0f;
  }
  fc.ea = exp_approx(__ldg(p.a_log + h));
}

// Front of one live item: conv + SiLU + BF16, gate projection + decay, beta,
// L2 norms, written to slot `sv`.  Conv windows: decode stores each channel's
// new window (T + 2 elements) directly and releases the stage as soon as its
// reads are done; verify and record steps (longer windows) write them over
// the staged conv rows, which leave through three TMA bulk stores issued by
// channel 0, and release the stage once those stores have read it.
template <int T, bool RECORD>
__device__ __forceinline__ void front_item(const Params &p, uint8_t *st,
                                           const ItemDesc &dsc, int n,
                                           const SlotView<T> &sv, float *ssum,
                                           const FrontConst &fc, int c,
                                           uint64_t *empty_bar) {
  const int fw = c >> 5, lane = c & 31;
  const int h = n / p.batch;
  const int r = n - h * p.batch;
  const int64_t dim = static_cast<int64_t>(p.heads) * kDk;
  const int64_t item = static_cast<int64_t>(r) * p.heads + h;
  const int cs = dsc.conv_slot, off = dsc.offset;
  uint16_t *conv_s = reinterpret_cast<uint16_t *>(st + p.conv_off);
  const uint16_t *x_s = reinterpret_cast<const uint16_t *>(st + p.x_off);
  const uint16_t *gate_s = reinterpret_cast<const uint16_t *>(st + p.gate_off);
  const uint16_t *fa_s = reinterpret_cast<const uint16_t *>(st + p.fa_off);

  // --- convolution + SiLU + BF16 (KdaWide.kernel, "The convolution (stock
  // tap order) and SiLU"): this thread owns channel c of q, k and v.  Loads,
  // window writes, arithmetic and stores are separate phases so that the
  // independent per-(part, token) chains overlap.
  uint16_t xb[3][T];
  float tap[3][3];
#pragma unroll
  for (int part = 0; part < 3; ++part)
#pragma unroll
    for (int t = 0; t < T; ++t) xb[part][t] = x_s[(t * 3 + part) * kDk + c];
  // Taps of this channel, as the pool stores them (the page's conv_type), and
  // its new window [tap1, tap2, x_0 .. x_{T-1}]: to the pool (decode) or over
  // its staged row (columns past T + 1 keep their loaded values).
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    const int64_t rix = (static_cast<int64_t>(cs) * 3 * dim + part * dim + h * kDk + c) *
                        p.conv_width;
    if (p.conv_f32) {
      float *row = reinterpret_cast<float *>(conv_s) + (part * kDk + c) * p.conv_width;
#pragma unroll
      for (int i = 0; i < 3; ++i) tap[part][i] = row[off + i];
      float *dst = (T == 1) ? reinterpret_cast<float *>(p.conv_state) + rix : row;
      dst[0] = tap[part][1];
      dst[1] = tap[part][2];
#pragma unroll
      for (int t = 0; t < T; ++t) dst[2 + t] = bf16_bits_to_float(xb[part][t]);
    } else {
      uint16_t *row = conv_s + (part * kDk + c) * p.conv_width;
      uint16_t tb[3];
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        tb[i] = row[off + i];
        tap[part][i] = bf16_bits_to_float(tb[i]);
      }
      uint16_t *dst = (T == 1) ? reinterpret_cast<uint16_t *>(p.conv_state) + rix : row;
      dst[0] = tb[1];
      dst[1] = tb[2];
#pragma unroll
      for (int t = 0; t < T; ++t) dst[2 + t] = xb[part][t];
    }
  }
  float y[3][T];
#pragma unroll
  for (int part = 0; part < 3; ++part) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float acc = fc.bias[part];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float w = (t + i < 3) ? tap[part][t + i] : bf16_bits_to_float(xb[part][t + i - 3]);
        acc = __fmaf_rn(w, fc.wt[part][i], acc);
      }
      y[part][t] = bf16_round(silu_approx(acc));
    }
  }
  constexpr int NS = NextPow2<2 * T>::value;  // square sums, padded with zeros
  float sq[NS];
#pragma unroll
  for (int i = 2 * T; i < NS; ++i) sq[i] = 0.0f;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    sv.q[t * kDk + c] = y[0][t];
    sv.k[t * kDk + c] = y[1][t];
    sv.v[t * kDk + c] = __bfloat16_as_ushort(__float2bfloat16_rn(y[2][t]));
    if (RECORD) p.rec_kg[(item * T + t) * 2 * kDk + c] = __float2bfloat16_rn(y[1][t]);
    sq[2 * t] = __fmul_rn(y[0][t], y[0][t]);
    sq[2 * t + 1] = __fmul_rn(y[1][t], y[1][t]);
  }
  if (p.dbg) {
#pragma unroll
    for (int part = 0; part < 3; ++part)
#pragma unroll
      for (int t = 0; t < T; ++t)
        p.dbg[((item * T + t) * 4 + part) * kDk + c] = __float2bfloat16_rn(y[part][t]);
  }
  {
    // Each lane ends with one warp total (the same tree as a butterfly).
    const float tot = warp_reduce_scatter<NS>(sq, lane);
    const int idx = (lane / (32 / NS)) % NS;
    if (idx < 2 * T && lane % (32 / NS) == 0) ssum[idx * 4 + fw] = tot;
  }
  // The rewritten conv rows are read next by the async proxy (bulk stores).
  if (T > 1) fence_proxy_async_smem();
#pragma unroll
  for (int t = 0; t < T; ++t) sv.gate[t * kDk + c] = gate_s[t * kDk + c];
  if (c < T) {
    sv.beta[c] = sigmoid_approx(bf16_bits_to_float(dsc.beta_bits[c]));
    sv.tgt[c] = (T == 1) ? dsc.slot : (RECORD ? 0 : dsc.target[c]);
  }
  if (c == 0) sv.meta[0] = n;

  // --- gate projection on tensor cores (KdaWide.kernel, "Gate projection"):
  // D[feature, token] over 8 rank chunks of 16; token column n = lane/4;
  // warp fw owns features 32fw .. 32fw+31 (two m16 tiles).
  {
    const int g = lane >> 2, q = lane & 3;
    uint32_t fb0[8], fb1[8];
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      if (g < T) {
        const uint2 v =
            *reinterpret_cast<const uint2 *>(fa_s + g * kDk + 16 * kc + 4 * q);
        fb0[kc] = v.x;
        fb1[kc] = v.y;
      } else {
        fb0[kc] = 0u;
        fb1[kc] = 0u;
      }
    }
    // Decode: all reads of the stage (and its descriptor) are done.
    if (T == 1) mbar_arrive(empty_bar);
    // gate_mode 0: one chain per tile, the two tiles interleaved; gate_mode
    // 1: four chains of two MMAs per tile, 0 + (((c0 + c1) + c2) + c3).
    float gv[2][4];
    if (p.gate_mode == 0) {
      float acc[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[m][e] = 0.0f;
#pragma unroll
      for (int kc = 0; kc < 8; ++kc)
#pragma unroll
        for (int m = 0; m < 2; ++m) mma_bf16(acc[m], fc.wa[m][kc], fb0[kc], fb1[kc]);
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) gv[m][e] = acc[m][e];
    } else {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        float acc[4][4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[ch][e] = 0.0f;
#pragma unroll
        for (int kc = 0; kc < 8; ++kc)
          mma_bf16(acc[kc >> 1], fc.wa[m][kc], fb0[kc], fb1[kc]);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          gv[m][e] = __fadd_rn(
              0.0f, __fadd_rn(__fadd_rn(__fadd_rn(acc[0][e], acc[1][e]), acc[2][e]),
                              acc[3][e]));
      }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = 2 * q + (e & 1);
        const int f = 32 * fw + 16 * m + g + 8 * (e >> 1);
        if (t < T) {
          const __nv_bfloat16 gb = __float2bfloat16_rn(gv[m][e]);
          const float raw = __bfloat162float(gb);
          // KdaWide.decay
          const float z = __fmul_rn(fc.ea, __fadd_rn(raw, fc.dt[m][e >> 1]));
          sv.d[t * kDk + f] = exp_approx(__fmul_rn(p.lower_bound, sigmoid_approx(z)));
          if (p.dbg) p.dbg[((item * T + t) * 4 + 3) * kDk + f] = gb;
          if (RECORD) p.rec_kg[(item * T + t) * 2 * kDk + kDk + f] = gb;
        }
      }
    }
  }
  front_sync();
  if (T > 1 && c == 0) {
    // Every channel's new window is in the staged rows: store them back.
    const uint32_t elem = p.conv_f32 ? 4u : 2u;
    const uint32_t row_bytes = 128u * elem * p.conv_width;
    const uint64_t pol = policy_evict_first();
    const int64_t hd = static_cast<int64_t>(p.heads) * kDk;
    const int64_t row0 = static_cast<int64_t>(dsc.conv_slot) * 3 * hd +
                         static_cast<int64_t>(n / p.batch) * kDk;
#pragma unroll
    for (int part = 0; part < 3; ++part)
      bulk_s2g(reinterpret_cast<uint8_t *>(p.conv_state) +
                   (row0 + part * hd) * p.conv_width * elem,
               st + p.conv_off + part * row_bytes, row_bytes, pol);
    bulk_commit();
  }

  // --- L2 norms ("Normalized q (with the 1/sqrt(K) scale) and k"), partial
  // sums combined as KdaWide.quad_sum does.
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const float4 sq4 = *reinterpret_cast<const float4 *>(ssum + t * 8);
    const float4 sk4 = *reinterpret_cast<const float4 *>(ssum + t * 8 + 4);
    const float qn =
        __fadd_rn(__fadd_rn(__fadd_rn(sq4.x, sq4.z), __fadd_rn(sq4.y, sq4.w)), 1.0e-6f);
    const float kn =
        __fadd_rn(__fadd_rn(__fadd_rn(sk4.x, sk4.z), __fadd_rn(sk4.y, sk4.w)), 1.0e-6f);
    const float fq = rcp_approx(sqrt_approx(qn));
    const float fk = rcp_approx(sqrt_approx(kn));
    sv.q[t * kDk + c] = __fmul_rn(__fmul_rn(sv.q[t * kDk + c], fq), p.scale);
    sv.k[t * kDk + c] = __fmul_rn(sv.k[t * kDk + c], fk);
  }
  if (T > 1) {
    // All reads of the stage (and its descriptor) are done; channel 0 also
    // waits until its conv-row stores have read the stage.
    if (c == 0) bulk_wait_read(0);
    mbar_arrive(empty_bar);
  }
}

// Gated RMSNorm ("Gated RMSNorm") of the item whose o the recurrence left in
// slot `sv`: thread = channel c; the four warps' partial sums of a token are
// combined as KdaWide.quad_sum does.  `osum` ([T][4]) is free on entry.
template <int T>
__device__ __forceinline__ void front_epilogue(const Params &p, const SlotView<T> &sv,
                                               float *osum, float nw, int c) {
  const int lane = c & 31, fw = c >> 5;
  const int n = sv.meta[0];
  const int h = n / p.batch;
  const int r = n - h * p.batch;
  const int64_t dim = static_cast<int64_t>(p.heads) * kDk;
  constexpr int NE = NextPow2<T>::value;
  float ov[T], gv[T], sq[NE];
#pragma unroll
  for (int t = T; t < NE; ++t) sq[t] = 0.0f;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    ov[t] = bf16_bits_to_float(sv.o[t * kDk + c]);
    gv[t] = bf16_bits_to_float(sv.gate[t * kDk + c]);
    sq[t] = __fmul_rn(ov[t], ov[t]);
  }
  {
    const float tot = warp_reduce_scatter<NE>(sq, lane);
    const int idx = (lane / (32 / NE)) % NE;
    if (idx < T && lane % (32 / NE) == 0) osum[idx * 4 + fw] = tot;
  }
  front_sync();
  float y[T];
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const float4 o4 = *reinterpret_cast<const float4 *>(osum + t * 4);
    const float sumsq = __fadd_rn(__fadd_rn(o4.x, o4.z), __fadd_rn(o4.y, o4.w));
    const float var = __fadd_rn(__fmul_rn(sumsq, 1.0f / 128.0f), p.eps);
    const float rstd = rcp_approx(sqrt_approx(var));
    y[t] = __fmul_rn(__fmul_rn(__fmul_rn(ov[t], rstd), nw), sigmoid_approx(gv[t]));
  }
#pragma unroll
  for (int t = 0; t < T; ++t)
    p.output[(static_cast<int64_t>(r) * T + t) * dim + h * kDk + c] =
        __float2bfloat16_rn(y[t]);
}

template <int T, bool RECORD>
__device__ void front_role(const Params &p, uint8_t *smem, Ctrl *ctl,
                           const ItemDesc *desc) {
  const int c = threadIdx.x - kRecThreads;  // channel 0..127
  const int S = p.stages;
  const int64_t dim = static_cast<int64_t>(p.heads) * kDk;
  float *ssum = reinterpret_cast<float *>(smem + p.scratch_off);   // [T][2][4]
  float *osum = reinterpret_cast<float *>(smem + p.rscratch_off);  // [T][4]
  float nw = 0.0f;  // norm weight of channel c, read after the first stage lands
  bool aborted = false;
  FrontConst fc;
  int cur_head = -1;
  int j = 0;  // live items seen
  for (int k = 0;; ++k) {
    const int stage = k % S;
    const uint32_t round = static_cast<uint32_t>(k / S);
    const bool ok = mbar_wait(&ctl->full[stage], round & 1u, &ctl->abort);
    if (front_sync_or(!ok)) {
      aborted = true;
      break;
    }
    const ItemDesc &dsc = desc[stage];
    if (dsc.status == kEnd) break;
    // A landed stage means the producer has passed its wait on the preceding
    // kernel (programmatic dependent launch): inputs other than the state
    // pool, slots and accepted may be read from here on.
    if (k == 0)
      nw = bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.norm_weight) + c));
    const int n = dsc.item;
    const int h = n / p.batch;
    if (dsc.status != kLive) {
      const int r = n - h * p.batch;
      mbar_arrive(&ctl->empty[stage]);
#pragma unroll
      for (int t = 0; t < T; ++t)
        p.output[(static_cast<int64_t>(r) * T + t) * dim + h * kDk + c] =
            __float2bfloat16_rn(0.0f);
      continue;
    }
    const int s = j & 1;
    SlotView<T> sv(smem + p.slot_off + s * p.slot_bytes);
    if (j >= 2) {
      // The recurrence is done with live item j-2: its outputs, then the slot
      // takes item j.
      const bool okr = mbar_wait(&ctl->sfree[s], ((j - 2) >> 1) & 1, &ctl->abort);
      if (front_sync_or(!okr)) {
        aborted = true;
        break;
      }
      front_epilogue<T>(p, sv, osum, nw, c);
    }
    if (h != cur_head) {
      load_front_const(p, h, c, fc);
      cur_head = h;
    }
    front_item<T, RECORD>(p, smem + static_cast<size_t>(stage) * p.stage_bytes, dsc,
                          n, sv, ssum, fc, c, &ctl->empty[stage]);
    mbar_arrive(&ctl->fready[s]);
    ++j;
  }
  // Outputs of the last (up to two) live items.
  for (int i = (j >= 2 ? j - 2 : 0); i < j && !aborted; ++i) {
    const bool okr = mbar_wait(&ctl->sfree[i & 1], (i >> 1) & 1, &ctl->abort);
    if (front_sync_or(!okr)) break;
    front_epilogue<T>(p, SlotView<T>(smem + p.slot_off + (i & 1) * p.slot_bytes), osum,
                      nw, c);
  }
  // The conv-row stores are complete before the thread that issued them exits.
  if (T > 1 && c == 0) bulk_wait_all();
}

// ----------------------------------------------------------------- recurrence

// Passes of the delta rule over the page held in registers (thread (g8, l8):
// rows g8 + 32m, keys 32cc + 4l8 .. +3).  Each returns, per row m, this
// thread's partial dot product (x and y halves of the packed accumulator
// added last); a row's total is the 8-lane reduce_scatter8 of them.  The k vector
// travels in registers (kr): loaded once per token by the pass that first
// needs it and reused by the next, which saves a quarter of the vector loads
// from shared memory (the recurrence's shared-memory wavefronts, not its
// FMAs, are what the record step's token loop competes for).

// S *= d; partial rows of S k.
__device__ __forceinline__ void pass_decay_dot(float4 (&S4)[4][4], const float *d,
                                               const float *k, int l8, float (&part)[4],
                                               float4 (&kr)[4]) {
  float2 acc[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) acc[m] = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int key = 32 * cc + 4 * l8;
    const float4 d4 = *reinterpret_cast<const float4 *>(d + key);
    const float4 k4 = *reinterpret_cast<const float4 *>(k + key);
    kr[cc] = k4;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 lo = __fmul2_rn(make_float2(S4[m][cc].x, S4[m][cc].y),
                                   make_float2(d4.x, d4.y));
      const float2 hi = __fmul2_rn(make_float2(S4[m][cc].z, S4[m][cc].w),
                                   make_float2(d4.z, d4.w));
      S4[m][cc] = make_float4(lo.x, lo.y, hi.x, hi.y);
      acc[m] = __ffma2_rn(lo, make_float2(k4.x, k4.y), acc[m]);
      acc[m] = __ffma2_rn(hi, make_float2(k4.z, k4.w), acc[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) part[m] = __fadd_rn(acc[m].x, acc[m].y);
}

// S += k u (u of row m in U[m]); partial rows of S q.
__device__ __forceinline__ void pass_update_dot(float4 (&S4)[4][4], const float4 (&kr)[4],
                                                const float *q, const float (&U)[4],
                                                int l8, float (&part)[4]) {
  float2 acc[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) acc[m] = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int key = 32 * cc + 4 * l8;
    const float4 k4 = kr[cc];
    const float4 q4 = *reinterpret_cast<const float4 *>(q + key);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 uu = make_float2(U[m], U[m]);
      const float2 lo = __ffma2_rn(make_float2(k4.x, k4.y), uu,
                                   make_float2(S4[m][cc].x, S4[m][cc].y));
      const float2 hi = __ffma2_rn(make_float2(k4.z, k4.w), uu,
                                   make_float2(S4[m][cc].z, S4[m][cc].w));
      S4[m][cc] = make_float4(lo.x, lo.y, hi.x, hi.y);
      acc[m] = __ffma2_rn(lo, make_float2(q4.x, q4.y), acc[m]);
      acc[m] = __ffma2_rn(hi, make_float2(q4.z, q4.w), acc[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) part[m] = __fadd_rn(acc[m].x, acc[m].y);
}

// Token t's update and output dot fused with token t+1's decay and k dot in
// one sweep over the page: S += k u -> partial rows of S q (opart); S *= dn ->
// partial rows of S kn (dpart).  Every element and accumulator sees the same
// operations in the same order as pass_update_dot then pass_decay_dot, so the
// results are identical; the two row reductions that follow are independent.
__device__ __forceinline__ void pass_update_dot_decay_dot(
    float4 (&S4)[4][4], float4 (&kr)[4], const float *q, const float (&U)[4],
    const float *dn, const float *kn, int l8, float (&opart)[4], float (&dpart)[4]) {
  float2 oacc[4], dacc[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    oacc[m] = make_float2(0.0f, 0.0f);
    dacc[m] = make_float2(0.0f, 0.0f);
  }
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int key = 32 * cc + 4 * l8;
    const float4 k4 = kr[cc];
    const float4 q4 = *reinterpret_cast<const float4 *>(q + key);
    const float4 d4 = *reinterpret_cast<const float4 *>(dn + key);
    const float4 n4 = *reinterpret_cast<const float4 *>(kn + key);
    kr[cc] = n4;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 uu = make_float2(U[m], U[m]);
      const float2 lo = __ffma2_rn(make_float2(k4.x, k4.y), uu,
                                   make_float2(S4[m][cc].x, S4[m][cc].y));
      const float2 hi = __ffma2_rn(make_float2(k4.z, k4.w), uu,
                                   make_float2(S4[m][cc].z, S4[m][cc].w));
      oacc[m] = __ffma2_rn(lo, make_float2(q4.x, q4.y), oacc[m]);
      oacc[m] = __ffma2_rn(hi, make_float2(q4.z, q4.w), oacc[m]);
      const float2 lo2 = __fmul2_rn(lo, make_float2(d4.x, d4.y));
      const float2 hi2 = __fmul2_rn(hi, make_float2(d4.z, d4.w));
      S4[m][cc] = make_float4(lo2.x, lo2.y, hi2.x, hi2.y);
      dacc[m] = __ffma2_rn(lo2, make_float2(n4.x, n4.y), dacc[m]);
      dacc[m] = __ffma2_rn(hi2, make_float2(n4.z, n4.w), dacc[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    opart[m] = __fadd_rn(oacc[m].x, oacc[m].y);
    dpart[m] = __fadd_rn(dacc[m].x, dacc[m].y);
  }
}


template <int T, bool RECORD>
__device__ void recurrence_role(const Params &p, uint8_t *smem, Ctrl *ctl,
                                const ItemDesc *desc) {
  const int tid = threadIdx.x;  // 0..255
  const int lane = tid & 31;
  const int g8 = tid >> 3, l8 = tid & 7;
  const int my_row = g8 + 32 * ((l8 >> 1) & 3);
  const int S = p.stages;
  const uint64_t pol = policy_evict_first();
  int j = 0;
  uint32_t wq = 0;  // decode: quarters handed to the store thread so far
  for (int k = 0;; ++k) {
    const int stage = k % S;
    const uint32_t round = static_cast<uint32_t>(k / S);
    bool ok = mbar_wait(&ctl->full[stage], round & 1u, &ctl->abort);
    // Every thread reads the item's status BEFORE the barrier: thread 0 frees
    // a non-live item's stage right after it, and the producer then rewrites
    // the descriptor; a read after that could see the next item's status and
    // split the recurrence warps between two barrier sequences.
    const int status = ok ? desc[stage].status : kError;
    const int n = ok ? desc[stage].item : 0;
    if (rec_sync_or(!ok)) {
      if (T > 1 && !RECORD && tid == 0) bulk_wait_all();
      return;
    }
    if (status == kEnd) break;
    if (status != kLive) {
      if (tid == 0) mbar_arrive(&ctl->empty[stage]);
      continue;
    }
    const int h = n / p.batch;
    const int r = n - h * p.batch;
    const int64_t item = static_cast<int64_t>(r) * p.heads + h;

    // The page (rows g8 + 32m, keys 32cc + 4l8 .. +3) into registers.
    float *page_s =
        reinterpret_cast<float *>(smem + static_cast<size_t>(stage) * p.stage_bytes);
    float4 S4[4][4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        S4[m][cc] = *reinterpret_cast<const float4 *>(page_s + (g8 + 32 * m) * kDk +
                                                      32 * cc + 4 * l8);
    rec_sync();
    // Page loaded: decode and record steps free the stage now; verify steps
    // reuse it as the store buffer of the written pages.
    if ((T == 1 || RECORD) && tid == 0) mbar_arrive(&ctl->empty[stage]);
    bool stored = false;

    const int s = j & 1;
    ok = mbar_wait(&ctl->fready[s], (j >> 1) & 1, &ctl->abort);
    if (rec_sync_or(!ok)) {
      if (T > 1 && !RECORD && tid == 0) bulk_wait_all();
      return;
    }
    SlotView<T> sv(smem + p.slot_off + s * p.slot_bytes);

    // The recurrence ("The recurrence").
    if (RECORD) {
      // No state is written between tokens: token t's update and output sweep
      // is fused with token t+1's decay and k-dot sweep (same arithmetic).
      float part[4];
      float4 kr[4];
      pass_decay_dot(S4, sv.d, sv.k, l8, part, kr);
      float u = __fmul_rn(
          __fsub_rn(bf16_bits_to_float(sv.v[my_row]), reduce_scatter8(part, l8)),
          sv.beta[0]);
#pragma unroll 1
      for (int t = 0; t < T; ++t) {
        if ((l8 & 1) == 0) p.rec_u[(item * T + t) * kDk + my_row] = u;
        float U[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
          U[m] = __shfl_sync(0xffffffffu, u, (lane & ~7) | (2 * m));
        const float *qt = sv.q + t * kDk;
        float opart[4];
        if (t + 1 < T) {
          float dpart[4];
          pass_update_dot_decay_dot(S4, kr, qt, U, sv.d + (t + 1) * kDk,
                                    sv.k + (t + 1) * kDk, l8, opart, dpart);
          const float o = reduce_scatter8(opart, l8);
          const float dot = reduce_scatter8(dpart, l8);
          if ((l8 & 1) == 0)
            sv.o[t * kDk + my_row] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
          u = __fmul_rn(__fsub_rn(bf16_bits_to_float(sv.v[(t + 1) * kDk + my_row]), dot),
                        sv.beta[t + 1]);
        } else {
          pass_update_dot(S4, kr, qt, U, l8, opart);
          const float o = reduce_scatter8(opart, l8);
          if ((l8 & 1) == 0)
            sv.o[t * kDk + my_row] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
        }
      }
    } else {
#pragma unroll 1
      for (int t = 0; t < T; ++t) {
        const float *kt = sv.k + t * kDk, *qt = sv.q + t * kDk;
        float part[4];
        float4 kr[4];
        pass_decay_dot(S4, sv.d + t * kDk, kt, l8, part, kr);
        const float dot = reduce_scatter8(part, l8);
        const float u = __fmul_rn(
            __fsub_rn(bf16_bits_to_float(sv.v[t * kDk + my_row]), dot), sv.beta[t]);
        float U[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
          U[m] = __shfl_sync(0xffffffffu, u, (lane & ~7) | (2 * m));
        pass_update_dot(S4, kr, qt, U, l8, part);
        const float o = reduce_scatter8(part, l8);
        if ((l8 & 1) == 0)
          sv.o[t * kDk + my_row] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
        const int tgt = sv.tgt[t];
        if (tgt > 0) {
          float *page_g = p.state + (static_cast<int64_t>(tgt) * p.heads + h) *
                                        static_cast<int64_t>(kDk * kDk);
          if (T == 1) {
            // Quarter m = value rows 32m .. 32m+31 = this thread's row g8 + 32m.
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int b = static_cast<int>(wq % static_cast<uint32_t>(p.nqbuf));
              const uint32_t use = wq / static_cast<uint32_t>(p.nqbuf);
              if (use > 0) {
                ok = mbar_wait(&ctl->qfree[b], (use - 1u) & 1u, &ctl->abort);
                if (rec_sync_or(!ok)) return;
              }
              float *qb =
                  reinterpret_cast<float *>(smem + p.qbuf_off + b * kQuarterBytes);
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<float4 *>(qb + g8 * kDk + 32 * cc + 4 * l8) =
                    S4[m][cc];
              fence_proxy_async_smem();
              rec_sync();
              if (tid == 0) {
                ctl->qdst[b] = page_g + m * (kQuarterBytes / 4);
                mbar_arrive(&ctl->qready[b]);
              }
              ++wq;
            }
          } else {
            // The stage buffer may still be read by the previous token's store.
            if (stored) {
              if (tid == 0) bulk_wait_read(0);
              rec_sync();
            }
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<float4 *>(page_s + (g8 + 32 * m) * kDk + 32 * cc +
                                            4 * l8) = S4[m][cc];
            fence_proxy_async_smem();
            rec_sync();
            if (tid == 0) {
              bulk_s2g(page_g, page_s, kPageBytes, pol);
              bulk_commit();
            }
            stored = true;
          }
        }
      }
    }
    // o of every token is in the slot; the front applies the gated RMSNorm.
    mbar_arrive(&ctl->sfree[s]);
    if (T > 1 && !RECORD && tid == 0) {
      bulk_wait_read(0);
      mbar_arrive(&ctl->empty[stage]);
    }
    ++j;
  }
  if (T > 1 && !RECORD && tid == 0) bulk_wait_all();
  if (T == 1) {
    // End of stream for the store thread.
    const int b = static_cast<int>(wq % static_cast<uint32_t>(p.nqbuf));
    const uint32_t use = wq / static_cast<uint32_t>(p.nqbuf);
    if (use > 0) {
      const bool ok = mbar_wait(&ctl->qfree[b], (use - 1u) & 1u, &ctl->abort);
      if (rec_sync_or(!ok)) return;
    }
    if (tid == 0) {
      ctl->qdst[b] = nullptr;
      mbar_arrive(&ctl->qready[b]);
    }
  }
}

// ----------------------------------------------------------------- store

// Serves the quarter ring in order.  Quarter #q sits in buffer q % n.  The
// loop issues the next quarter as soon as the recurrence has written it;
// otherwise it retires the oldest store in flight (waits until that copy has
// read shared memory) and frees its buffer; with nothing in flight it sleeps
// until the next quarter.  A null destination ends the stream.
__device__ void store_role(const Params &p, uint8_t *smem, Ctrl *ctl) {
  const uint64_t pol = policy_evict_first();
  const uint32_t n = static_cast<uint32_t>(p.nqbuf);
  uint32_t issued = 0, freed = 0;
  for (;;) {
    const int b = static_cast<int>(issued % n);
    const uint32_t par = (issued / n) & 1u;
    if (mbar_test_wait(&ctl->qready[b], par)) {
      float *dst = ctl->qdst[b];
      if (dst == nullptr) break;
      bulk_s2g(dst, smem + p.qbuf_off + b * kQuarterBytes, kQuarterBytes, pol);
      bulk_commit();
      ++issued;
    } else if (issued > freed) {
      const uint32_t pending = issued - freed;
      bulk_wait_read(static_cast<int>(pending > 4u ? 3u : pending - 1u));
      mbar_arrive(&ctl->qfree[freed % n]);
      ++freed;
    } else if (!mbar_wait(&ctl->qready[b], par, &ctl->abort)) {
      break;
    }
  }
  bulk_wait_all();
}

template <int T, bool RECORD>
__global__ void __launch_bounds__(kThreads, 1) kda_step_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  Ctrl *ctl = reinterpret_cast<Ctrl *>(smem + p.bar_off);
  ItemDesc *desc = reinterpret_cast<ItemDesc *>(smem + p.desc_off);
  const int G = gridDim.x;
  int n0, n1;
  if (p.sched) {
    const int q = p.dyn0 / G;
    n0 = q * static_cast<int>(blockIdx.x);
    n1 = n0 + q;
  } else {
    n0 = static_cast<int>((static_cast<int64_t>(p.items) * blockIdx.x) / G);
    n1 = static_cast<int>((static_cast<int64_t>(p.items) * (blockIdx.x + 1)) / G);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1 + kFrontThreads);  // front, recurrence
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&ctl->fready[s], kFrontThreads);
      mbar_init(&ctl->sfree[s], kRecThreads);
    }
    for (int b = 0; b < kMaxQuarterBufs; ++b) {
      mbar_init(&ctl->qready[b], 1);
      mbar_init(&ctl->qfree[b], 1);
    }
    ctl->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x < kRecThreads) {
    regs_inc<kRecRegs>();
    recurrence_role<T, RECORD>(p, smem, ctl, desc);
  } else if (threadIdx.x < kProducer) {
    regs_inc<kFrontRegs>();
    front_role<T, RECORD>(p, smem, ctl, desc);
  } else {
    regs_dec<kProducerRegs>();
    if (threadIdx.x == kProducer) producer_role<T, RECORD>(p, smem, ctl, desc, n0, n1);
    if (T == 1 && threadIdx.x == kStorer) store_role(p, smem, ctl);
  }
}

// ------------------------------------------------------------------ host side

struct Layout {
  uint32_t stage_bytes, conv_off, x_off, gate_off, fa_off;
  uint32_t bar_off, desc_off, slot_off, slot_bytes, scratch_off, rscratch_off;
  uint32_t qbuf_off, total;
  int stages, nqbuf;
};

static uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Stage: page | conv rows (3 x 128 x W bf16) | x (T x 3 x 128) | gate | f_a.
// Then the quarter-page store ring, the control block, item descriptors, two
// hand-off slots and the partial-sum scratch.  Decode uses two stages and as
// many 16 KiB quarter buffers (up to 4) as fit; verify and record steps take
// three stages when they fit, else two.
static bool make_layout(int T, int W, bool record, bool conv_f32, int max_smem,
                        Layout &L) {
  L.conv_off = kPageBytes;
  L.x_off = align_up(L.conv_off + 3u * (conv_f32 ? 512u : 256u) * W, 128);
  L.gate_off = L.x_off + 3u * T * 256u;
  L.fa_off = L.gate_off + T * 256u;
  L.stage_bytes = align_up(L.fa_off + T * 256u, 128);
  L.slot_bytes = align_up((3u * T * kDk + 2u * KDA_MAX_TOKENS + 4u) * 4u +
                              3u * T * kDk * 2u,
                          128);
  const uint32_t ctrl = align_up(sizeof(Ctrl), 128);
  const uint32_t descs = align_up(kMaxStages * sizeof(ItemDesc), 128);
  const uint32_t scratch = align_up(T * 8u * 4u, 128);   // front q/k square sums
  const uint32_t rscratch = align_up(T * 4u * 4u, 128);  // front: o square sums
  const uint32_t fixed = ctrl + descs + kSlots * L.slot_bytes + scratch + rscratch;
  const bool ring = T == 1 && !record;
  const int s_max = ring ? 2 : kMaxStages;
  for (int s = s_max; s >= 2; --s) {
    for (int nq = ring ? kMaxQuarterBufs : 0; nq >= (ring ? 1 : 0); --nq) {
      const uint32_t total = s * L.stage_bytes + fixed + nq * kQuarterBytes;
      if (total > static_cast<uint32_t>(max_smem)) continue;
      L.stages = s;
      L.nqbuf = nq;
      L.qbuf_off = s * L.stage_bytes;
      L.bar_off = L.qbuf_off + nq * kQuarterBytes;
      L.desc_off = L.bar_off + ctrl;
      L.slot_off = L.desc_off + descs;
      L.scratch_off = L.slot_off + kSlots * L.slot_bytes;
      L.rscratch_off = L.scratch_off + scratch;
      L.total = total;
      return true;
    }
  }
  return false;
}

template <int T, bool RECORD>
static int launch_t(const Params &prm, const Layout &L, int dev, const DeviceFacts &df,
                    int grid, int use_pdl, cudaStream_t stream) {
  auto kern = kda_step_kernel<T, RECORD>;
  static std::atomic<bool> configured[kMaxDevices];
  if (!set_smem_limit_once(configured, dev, reinterpret_cast<const void *>(kern),
                           df.max_smem))
    return KDA_ERR_LAUNCH;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (use_pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) return KDA_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? KDA_SUCCESS : KDA_ERR_LAUNCH;
}

// The library's own scheduler words (kda_step_noalloc): a static device
// array, zero at module load and left zero by every launch; its address on
// the current GPU.
static __device__ __align__(256) int32_t g_sched_words[64];

static bool library_sched_words(int32_t **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_sched_words) != cudaSuccess) return false;
  *out = static_cast<int32_t *>(p);
  return true;
}

static bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// own_sched: the library's scheduler words replace a->sched
// (kda_step_noalloc; decode or verify by the token count).
static int run_step(const kda_args *a, cudaStream_t stream, bool verify,
                    bool own_sched = false) {
  if (!a) return KDA_ERR_NULL_ARGS;
  const int T = a->tokens;
  if (T < 1 || T > KDA_MAX_TOKENS) return KDA_ERR_TOKENS;
  if (own_sched) verify = T > 1;
  if (verify ? T == 1 : T != 1) return KDA_ERR_TOKENS;
  if (a->gate_mode != 0 && a->gate_mode != 1) return KDA_ERR_GATE_MODE;
  if (a->record && T == 1) return KDA_ERR_RECORD;
  if (a->path < 0 || a->path > 2) return KDA_ERR_PATH;
  if (a->batch < 0 || a->heads < 0) return KDA_ERR_SHAPE;
  if (a->batch == 0 || a->heads == 0) return KDA_SUCCESS;
  if (a->num_slots < 1) return KDA_ERR_SHAPE;
  if (T > 1 && a->slot_cols < T) return KDA_ERR_SHAPE;
  if (static_cast<int64_t>(a->batch) * a->heads > 0x7fffffffLL) return KDA_ERR_SHAPE;
  if (static_cast<int64_t>(a->heads) * kDk * 3 > 0x7fffffffLL) return KDA_ERR_SHAPE;
  if (a->conv_width < T + 2) return KDA_ERR_CONV_WIDTH;
  if (!a->x || !a->conv_weight || !a->f_a || !a->f_b || !a->beta || !a->gate ||
      !a->norm_weight || !a->a_log || !a->dt_bias || !a->slots || !a->conv_state ||
      !a->state || !a->output)
    return KDA_ERR_NULL_POINTER;
  if (a->has_bias && !a->conv_bias) return KDA_ERR_NULL_POINTER;
  if (T > 1 && !a->accepted) return KDA_ERR_NULL_POINTER;
  if (a->record && (!a->rec_u || !a->rec_kg)) return KDA_ERR_NULL_POINTER;
  if (!aligned(a->state, 16) || !aligned(a->f_a, 16) || !aligned(a->f_b, 16) ||
      !aligned(a->x, 16) || !aligned(a->gate, 16) || !aligned(a->conv_state, 16) ||
      !aligned(a->conv_weight, 2) || !aligned(a->beta, 2) ||
      !aligned(a->norm_weight, 2) || !aligned(a->output, 2) ||
      !aligned(a->a_log, 4) || !aligned(a->dt_bias, 4) || !aligned(a->slots, 4) ||
      (a->accepted && !aligned(a->accepted, 4)) ||
      (a->has_bias && !aligned(a->conv_bias, 2)) ||
      (a->rec_u && !aligned(a->rec_u, 4)) || (a->rec_kg && !aligned(a->rec_kg, 2)) ||
      (a->err && !aligned(a->err, 4)) || (a->dbg && !aligned(a->dbg, 2)) ||
      (!own_sched && a->sched && !aligned(a->sched, 4)))
    return KDA_ERR_ALIGNMENT;

  int dev = 0;
  DeviceFacts df;
  if (!current_device(&dev, &df)) return KDA_ERR_DEVICE;
  Layout L;
  if (!make_layout(T, a->conv_width, a->record != 0, a->conv_f32 != 0, df.max_smem, L))
    return KDA_ERR_CONV_WIDTH;

  Params prm;
  prm.batch = a->batch;
  prm.heads = a->heads;
  prm.num_slots = a->num_slots;
  prm.conv_width = a->conv_width;
  prm.slot_cols = T > 1 ? a->slot_cols : 1;
  prm.gate_mode = a->gate_mode;
  prm.has_bias = a->has_bias ? 1 : 0;
  prm.items = a->batch * a->heads;
  prm.stages = L.stages;
  prm.sched = a->sched;
  if (own_sched && !library_sched_words(&prm.sched)) return KDA_ERR_DEVICE;
  prm.stage_bytes = L.stage_bytes;
  prm.conv_off = L.conv_off;
  prm.x_off = L.x_off;
  prm.gate_off = L.gate_off;
  prm.fa_off = L.fa_off;
  prm.bar_off = L.bar_off;
  prm.desc_off = L.desc_off;
  prm.slot_off = L.slot_off;
  prm.slot_bytes = L.slot_bytes;
  prm.scratch_off = L.scratch_off;
  prm.rscratch_off = L.rscratch_off;
  prm.qbuf_off = L.qbuf_off;
  prm.nqbuf = L.nqbuf;
  prm.x = static_cast<const __nv_bfloat16 *>(a->x);
  prm.conv_weight = static_cast<const __nv_bfloat16 *>(a->conv_weight);
  prm.conv_bias = static_cast<const __nv_bfloat16 *>(a->has_bias ? a->conv_bias : a->conv_weight);
  prm.f_a = static_cast<const __nv_bfloat16 *>(a->f_a);
  prm.f_b = static_cast<const __nv_bfloat16 *>(a->f_b);
  prm.beta = static_cast<const __nv_bfloat16 *>(a->beta);
  prm.gate = static_cast<const __nv_bfloat16 *>(a->gate);
  prm.norm_weight = static_cast<const __nv_bfloat16 *>(a->norm_weight);
  prm.a_log = a->a_log;
  prm.dt_bias = a->dt_bias;
  prm.slots = a->slots;
  prm.accepted = a->accepted;
  prm.conv_state = static_cast<__nv_bfloat16 *>(a->conv_state);
  prm.conv_f32 = a->conv_f32 ? 1 : 0;
  prm.state = a->state;
  prm.output = static_cast<__nv_bfloat16 *>(a->output);
  prm.rec_u = a->rec_u;
  prm.rec_kg = static_cast<__nv_bfloat16 *>(a->rec_kg);
  prm.lower_bound = a->lower_bound;
  prm.scale = a->scale;
  prm.eps = a->eps;
  prm.err = a->err;
  prm.dbg = static_cast<__nv_bfloat16 *>(a->dbg);

  // Few items: one item per cluster of four CTAs (latency); many items: the
  // persistent kernel (bandwidth).
  const bool split = a->path == 2 || (a->path == 0 && 4 * prm.items <= 2 * df.sms);
  if (split) return launch_split(a, stream);
  const int grid = prm.items < df.sms ? prm.items : df.sms;
  // With a scheduler word pair, each CTA keeps a contiguous range (per-head
  // constants stay in registers, the first pages can go out before the wait
  // on the preceding kernel) and the items past the ranges are handed out one
  // at a time, so CTAs on slower SMs or with slower pages take fewer.  A
  // shared item usually changes the CTA's head (its constants are reloaded),
  // so the ranges cover 7/8 of the items where the CTAs' finishing times
  // spread most (decode with 32 or more items a CTA, record steps) and all
  // but the remainder of an even split elsewhere (measured on the GB300).
  const bool wide = (T == 1 && prm.items >= 32 * grid) || a->record;
  const int64_t ranged = static_cast<int64_t>(prm.items) * (wide ? 7 : 8) / 8;
  prm.dyn0 = prm.sched ? static_cast<int>(ranged / grid) * grid : prm.items;
  const int pdl = a->use_pdl ? 1 : 0;
  const bool rec = a->record != 0;
  switch (T) {
    case 1: return launch_t<1, false>(prm, L, dev, df, grid, pdl, stream);
    case 2: return rec ? launch_t<2, true>(prm, L, dev, df, grid, pdl, stream)
                       : launch_t<2, false>(prm, L, dev, df, grid, pdl, stream);
    case 3: return rec ? launch_t<3, true>(prm, L, dev, df, grid, pdl, stream)
                       : launch_t<3, false>(prm, L, dev, df, grid, pdl, stream);
    case 4: return rec ? launch_t<4, true>(prm, L, dev, df, grid, pdl, stream)
                       : launch_t<4, false>(prm, L, dev, df, grid, pdl, stream);
    case 5: return rec ? launch_t<5, true>(prm, L, dev, df, grid, pdl, stream)
                       : launch_t<5, false>(prm, L, dev, df, grid, pdl, stream);
    case 6: return rec ? launch_t<6, true>(prm, L, dev, df, grid, pdl, stream)
                       : launch_t<6, false>(prm, L, dev, df, grid, pdl, stream);
    case 7: return rec ? launch_t<7, true>(prm, L, dev, df, grid, pdl, stream)
                       : launch_t<7, false>(prm, L, dev, df, grid, pdl, stream);
    default: return rec ? launch_t<8, true>(prm, L, dev, df, grid, pdl, stream)
                        : launch_t<8, false>(prm, L, dev, df, grid, pdl, stream);
  }
}

}  // namespace kda

extern "C" {

int kda_decode(const kda_args *args, void *stream) {
  return kda::run_step(args, static_cast<cudaStream_t>(stream), false);
}

int kda_verify(const kda_args *args, void *stream) {
  return kda::run_step(args, static_cast<cudaStream_t>(stream), true);
}

int kda_step_noalloc(const kda_args *args, void *stream) {
  return kda::run_step(args, static_cast<cudaStream_t>(stream), false, true);
}

const char *kda_strerror(int code) {
  switch (code) {
    case KDA_SUCCESS: return "success";
    case KDA_ERR_NULL_ARGS: return "args is NULL";
    case KDA_ERR_TOKENS: return "tokens outside 1..8 or wrong entry point for tokens";
    case KDA_ERR_GATE_MODE: return "gate_mode must be 0 or 1";
    case KDA_ERR_RECORD: return "record mode needs tokens > 1";
    case KDA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case KDA_ERR_CONV_WIDTH: return "conv_width < tokens + 2, or too wide to stage";
    case KDA_ERR_ALIGNMENT: return "a pointer is not aligned as required";
    case KDA_ERR_SHAPE: return "invalid sizes";
    case KDA_ERR_DEVICE: return "no usable sm_103 device";
    case KDA_ERR_LAUNCH: return "kernel launch failed";
    case KDA_ERR_PATH: return "path must be 0, 1 or 2";
    default: return "unknown error code";
  }
}

int kda_abi_version(void) { return KDA_ABI_VERSION; }

}  // extern "C"
