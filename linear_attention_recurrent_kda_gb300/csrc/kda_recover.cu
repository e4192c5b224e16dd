// Record replay for GB300 (sm_103a): rebuild the accepted state from a
// checkpoint page and the records a record-mode verify step wrote.
//
// Method: vLLM API page
//   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide"
// (KdaWide's record mode, "RecoverSSM verify: checkpoint slot, records out").
// The replay itself (RecoverSSM) is not shown on the page; this kernel applies
// the recurrence's own state update with the records: for the first
// accepted[r] tokens, decay every key column by the decay of the recorded raw
// gate, then S += k_hat u (fused, k first) with k_hat the L2-normalised
// recorded k.  The arithmetic, including the order of the partial sums of the
// k norm, is the step kernel's, so replaying a record step reproduces the page
// a non-record step writes after token accepted-1 bit for bit.
//
// Design: persistent, one CTA per SM, items (request, head) in head-major
// contiguous ranges (with scheduler words, the items past the ranges then go
// one at a time to whichever CTA's producer asks first, as in the step).
// Warp 8 lane 0 (producer) stages each item's checkpoint
// page and the records of its accepted tokens into a 3-stage shared-memory
// ring with TMA bulk copies and, once the compute warps have written the
// replayed page back into the stage, stores it with one TMA bulk store and
// reuses the stage after the copy has read it.  Warps 0-7 first form k_hat
// and the decay of every accepted token (two barriers per item), then hold
// the page in registers (thread (g, l): keys {32c + 4l + e} of value rows
// g + 32m) and sweep the tokens with no barrier between them.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_device.cuh"
#include "kda_host.h"

namespace kda {
namespace recover {

constexpr int kDk = 128;
constexpr int kCompute = 256;
constexpr int kThreads = kCompute + 32;
constexpr int kStages = 3;
constexpr uint32_t kPageBytes = kDk * kDk * 4;
constexpr int kLive = 0, kSkip = 1, kEnd = 2;  // kEnd: no more items

struct Params {
  int32_t batch, heads, tokens, num_slots, items;
  int32_t *sched;  // scheduler words or null (contiguous ranges only)
  int32_t dyn0;    // first shared item; CTA b owns [b*q, b*q + q), q = dyn0 / grid
  uint32_t stage_bytes, kg_off, u_off, bar_off, desc_off, vec_off;
  const int32_t *src_slots, *dst_slots, *accepted;
  const float *rec_u;
  const __nv_bfloat16 *rec_kg;
  const float *a_log, *dt_bias;
  float lower_bound;
  float *state;
  int32_t *err;
};

struct __align__(16) Desc {
  int32_t status;   // kLive / kSkip / kEnd
  int32_t src, dst, accepted;
  int32_t load;     // the stage holds the page (and records)
  int32_t store;    // the replayed page goes to dst
  int32_t item;     // n = h * batch + r
  int32_t pad;
};

struct Ctrl {
  uint64_t full[kStages];  // producer -> compute (bytes landed)
  uint64_t done[kStages];  // compute -> producer (page written back / skipped)
  uint32_t abort;
};

__device__ __forceinline__ bool compute_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void compute_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ int resolve(const Params &p, int n, Desc &d) {
  const int h = n / p.batch;
  const int r = n - h * p.batch;
  (void)h;
  d.src = __ldg(p.src_slots + r);
  d.dst = __ldg(p.dst_slots + r);
  d.accepted = __ldg(p.accepted + r);
  d.load = d.store = 0;
  d.status = kSkip;
  if (d.src <= 0 || d.dst <= 0) return 0;  // padding
  if (d.src >= p.num_slots || d.dst >= p.num_slots) return KDA_DEVERR_SLOT;
  if (d.accepted < 0 || d.accepted > p.tokens) return KDA_DEVERR_ACCEPTED;
  // Nothing to replay onto the same page: no traffic at all.
  if (d.accepted == 0 && d.dst == d.src) return 0;
  d.status = kLive;
  d.load = d.store = 1;
  return 0;
}

__device__ void producer(const Params &p, uint8_t *smem, Ctrl *ctl, Desc *desc,
                         int n0, int n1) {
  const uint64_t pol = policy_evict_first();
  const int64_t page_elems = static_cast<int64_t>(kDk) * kDk;
  bool ok = true;
  bool drained = p.sched == nullptr;
  int end_k = -1;  // index of the end marker once sent
  int issued = 0;
  for (int k = 0; ok; ++k) {
    const int stage = k % kStages;
    uint8_t *st = smem + static_cast<size_t>(stage) * p.stage_bytes;
    // Retire item k - kStages of this stage: store its replayed page.
    if (k >= kStages && (end_k < 0 || k - kStages < end_k)) {
      const int kk = k - kStages;
      ok = mbar_wait(&ctl->done[stage], static_cast<uint32_t>(kk / kStages) & 1u,
                     &ctl->abort);
      if (!ok) break;
      const Desc &od = desc[stage];
      if (od.store) {
        const int h = od.item / p.batch;
        bulk_s2g(p.state + (static_cast<int64_t>(od.dst) * p.heads + h) * page_elems,
                 st, kPageBytes, pol);
        bulk_commit();
        bulk_wait_read(0);
      }
    }
    if (end_k >= 0) {
      if (k - kStages + 1 >= end_k) break;  // every item before the marker retired
      continue;
    }
    // The CTA's k-th item: its own range, then shared items.
    int n = n0 + k < n1 ? n0 + k : -1;
    if (n < 0 && !drained) {
      // 64-bit, the counter read unsigned: no wrap however many items there are.
      const int64_t m =
          p.dyn0 + static_cast<int64_t>(static_cast<uint32_t>(atomicAdd(p.sched, 1)));
      if (m >= p.items) {
        drained = true;
      } else {
        n = static_cast<int>(m);
      }
    }
    Desc &d = desc[stage];
    if (n < 0) {
      d.status = kEnd;
      d.load = d.store = 0;
      mbar_arrive(&ctl->full[stage]);
      end_k = k;
      if (k - kStages + 1 >= end_k) break;  // nothing left to retire
      continue;
    }
    const int flags = resolve(p, n, d);
    d.item = n;
    if (flags && p.err) atomicOr(p.err, flags);
    if (d.load) {
      const int h = n / p.batch;
      const int r = n - h * p.batch;
      const int64_t item = static_cast<int64_t>(r) * p.heads + h;
      const uint32_t rec_bytes = static_cast<uint32_t>(d.accepted) * kDk * 4u;
      mbar_arrive_expect_tx(&ctl->full[stage], kPageBytes + 2u * rec_bytes);
      bulk_g2s_hint(st, p.state + (static_cast<int64_t>(d.src) * p.heads + h) * page_elems,
                    kPageBytes, &ctl->full[stage], pol);
      if (rec_bytes > 0) {
        bulk_g2s(st + p.kg_off, p.rec_kg + item * p.tokens * 2 * kDk, rec_bytes,
                 &ctl->full[stage]);
        bulk_g2s(st + p.u_off, p.rec_u + item * p.tokens * kDk, rec_bytes,
                 &ctl->full[stage]);
      }
    } else {
      mbar_arrive(&ctl->full[stage]);
    }
    ++issued;
  }
  if (!ok && p.err) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
  bulk_wait_all();
  if (p.sched) {
    // The last CTA to get here zeroes the scheduler words for the next launch.
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
  }
  if (!ok) {
    // Every copy issued into a stage must land before the CTA exits.
    uint32_t keep_waiting = 0;
    for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
      (void)mbar_wait(&ctl->full[k % kStages], static_cast<uint32_t>(k / kStages) & 1u,
                      &keep_waiting);
  }
}

__device__ void compute(const Params &p, uint8_t *smem, Ctrl *ctl, const Desc *desc) {
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g8 = tid >> 3, l8 = tid & 7;
  float *kh = reinterpret_cast<float *>(smem + p.vec_off);  // [T][128] k_hat
  float *dd = kh + KDA_MAX_TOKENS * kDk;                      // [T][128] decay
  float *ks = dd + KDA_MAX_TOKENS * kDk;                      // [T][4] k square sums
  int cur_head = -1;
  float ea = 0.0f, dtb = 0.0f;
  for (int k = 0;; ++k) {
    const int stage = k % kStages;
    const bool ok = mbar_wait(&ctl->full[stage], static_cast<uint32_t>(k / kStages) & 1u,
                              &ctl->abort);
    if (compute_sync_or(!ok)) return;
    const Desc &d = desc[stage];
    if (d.status == kEnd) break;
    if (!d.load) {
      mbar_arrive(&ctl->done[stage]);
      continue;
    }
    const int n = d.item;
    const int h = n / p.batch;
    if (h != cur_head) {
      ea = exp_approx(__ldg(p.a_log + h));
      if (tid >= 128) dtb = __ldg(p.dt_bias + h * kDk + (tid - 128));
      cur_head = h;
    }
    uint8_t *st = smem + static_cast<size_t>(stage) * p.stage_bytes;
    float *page_s = reinterpret_cast<float *>(st);
    const uint16_t *kg = reinterpret_cast<const uint16_t *>(st + p.kg_off);
    const float *us = reinterpret_cast<const float *>(st + p.u_off);
    const int acc = d.accepted;
    if (acc > 0) {
      float4 S4[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          S4[m][cc] = *reinterpret_cast<const float4 *>(page_s + (g8 + 32 * m) * kDk +
                                                        32 * cc + 4 * l8);
      // k_hat (threads 0-127, channel c) and decay (threads 128-255, feature
      // f) of every accepted token first, computed as the step kernel's front
      // computes them (the k square sums by the same warp tree); then the
      // token sweeps need no barrier (each thread's rows are its own).
      float kv[KDA_MAX_TOKENS];
      if (tid < 128) {
        float sq[KDA_MAX_TOKENS];
#pragma unroll
        for (int t = 0; t < KDA_MAX_TOKENS; ++t) {
          kv[t] = t < acc ? bf16_bits_to_float(kg[t * 2 * kDk + tid]) : 0.0f;
          sq[t] = __fmul_rn(kv[t], kv[t]);
        }
        const float tot = warp_reduce_scatter<KDA_MAX_TOKENS>(sq, lane);
        const int idx = lane >> 2;
        if ((lane & 3) == 0 && idx < acc) ks[idx * 4 + warp] = tot;
      } else {
        const int f = tid - 128;
#pragma unroll 1
        for (int t = 0; t < acc; ++t) {
          const float raw = bf16_bits_to_float(kg[t * 2 * kDk + kDk + f]);
          const float z = __fmul_rn(ea, __fadd_rn(raw, dtb));
          dd[t * kDk + f] = exp_approx(__fmul_rn(p.lower_bound, sigmoid_approx(z)));
        }
      }
      compute_sync();
      if (tid < 128) {
#pragma unroll
        for (int t = 0; t < KDA_MAX_TOKENS; ++t) {
          if (t < acc) {
            const float *k4s = ks + t * 4;
            const float kn = __fadd_rn(
                __fadd_rn(__fadd_rn(k4s[0], k4s[2]), __fadd_rn(k4s[1], k4s[3])), 1.0e-6f);
            kh[t * kDk + tid] = __fmul_rn(kv[t], rcp_approx(sqrt_approx(kn)));
          }
        }
      }
      compute_sync();
#pragma unroll 1
      for (int t = 0; t < acc; ++t) {
        float U[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) U[m] = us[t * kDk + g8 + 32 * m];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int key = 32 * cc + 4 * l8;
          const float4 d4 = *reinterpret_cast<const float4 *>(dd + t * kDk + key);
          const float4 k4 = *reinterpret_cast<const float4 *>(kh + t * kDk + key);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float2 lo = __fmul2_rn(make_float2(S4[m][cc].x, S4[m][cc].y),
                                   make_float2(d4.x, d4.y));
            float2 hi = __fmul2_rn(make_float2(S4[m][cc].z, S4[m][cc].w),
                                   make_float2(d4.z, d4.w));
            const float2 uu = make_float2(U[m], U[m]);
            lo = __ffma2_rn(make_float2(k4.x, k4.y), uu, lo);
            hi = __ffma2_rn(make_float2(k4.z, k4.w), uu, hi);
            S4[m][cc] = make_float4(lo.x, lo.y, hi.x, hi.y);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          *reinterpret_cast<float4 *>(page_s + (g8 + 32 * m) * kDk + 32 * cc + 4 * l8) =
              S4[m][cc];
      fence_proxy_async_smem();
    }
    mbar_arrive(&ctl->done[stage]);
  }
}

__global__ void __launch_bounds__(kThreads, 1) kda_recover_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  Ctrl *ctl = reinterpret_cast<Ctrl *>(smem + p.bar_off);
  Desc *desc = reinterpret_cast<Desc *>(smem + p.desc_off);
  const int G = gridDim.x;
  int n0, n1;
  if (p.sched) {
    n0 = (p.dyn0 / G) * static_cast<int>(blockIdx.x);
    n1 = n0 + p.dyn0 / G;
  } else {
    n0 = static_cast<int>((static_cast<int64_t>(p.items) * blockIdx.x) / G);
    n1 = static_cast<int>((static_cast<int64_t>(p.items) * (blockIdx.x + 1)) / G);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->done[s], kCompute);
    }
    ctl->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x < kCompute) {
    compute(p, smem, ctl, desc);
  } else if (threadIdx.x == kCompute) {
    producer(p, smem, ctl, desc, n0, n1);
  }
}

static uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

static int run(const kda_recover_args *a, cudaStream_t stream) {
  if (!a) return KDA_ERR_NULL_ARGS;
  if (a->tokens < 1 || a->tokens > KDA_MAX_TOKENS) return KDA_ERR_TOKENS;
  if (a->batch < 0 || a->heads < 0) return KDA_ERR_SHAPE;
  if (a->batch == 0 || a->heads == 0) return KDA_SUCCESS;
  if (a->num_slots < 1) return KDA_ERR_SHAPE;
  if (static_cast<int64_t>(a->batch) * a->heads > 0x7fffffffLL) return KDA_ERR_SHAPE;
  if (!a->src_slots || !a->dst_slots || !a->accepted || !a->rec_u || !a->rec_kg ||
      !a->a_log || !a->dt_bias || !a->state)
    return KDA_ERR_NULL_POINTER;
  auto al = [](const void *q, uintptr_t n) {
    return (reinterpret_cast<uintptr_t>(q) & (n - 1)) == 0;
  };
  if (!al(a->state, 16) || !al(a->rec_u, 16) || !al(a->rec_kg, 16) ||
      !al(a->src_slots, 4) || !al(a->dst_slots, 4) || !al(a->accepted, 4) ||
      !al(a->a_log, 4) || !al(a->dt_bias, 4) || (a->err && !al(a->err, 4)) ||
      (a->sched && !al(a->sched, 4)))
    return KDA_ERR_ALIGNMENT;
  int dev = 0;
  DeviceFacts df;
  if (!current_device(&dev, &df)) return KDA_ERR_DEVICE;
  const int T = a->tokens;
  Params prm;
  prm.batch = a->batch;
  prm.heads = a->heads;
  prm.tokens = T;
  prm.num_slots = a->num_slots;
  prm.items = a->batch * a->heads;
  prm.kg_off = kPageBytes;
  prm.u_off = prm.kg_off + T * kDk * 4u;
  prm.stage_bytes = align_up(prm.u_off + T * kDk * 4u, 128);
  prm.bar_off = kStages * prm.stage_bytes;
  prm.desc_off = prm.bar_off + align_up(sizeof(Ctrl), 128);
  prm.vec_off = prm.desc_off + align_up(kStages * sizeof(Desc), 128);
  const uint32_t total = prm.vec_off + (2 * KDA_MAX_TOKENS * kDk + 4 * KDA_MAX_TOKENS) * 4;
  if (total > static_cast<uint32_t>(df.max_smem)) return KDA_ERR_SHAPE;
  prm.src_slots = a->src_slots;
  prm.dst_slots = a->dst_slots;
  prm.accepted = a->accepted;
  prm.rec_u = a->rec_u;
  prm.rec_kg = static_cast<const __nv_bfloat16 *>(a->rec_kg);
  prm.a_log = a->a_log;
  prm.dt_bias = a->dt_bias;
  prm.lower_bound = a->lower_bound;
  prm.state = a->state;
  prm.err = a->err;
  static std::atomic<bool> configured[kMaxDevices];
  if (!set_smem_limit_once(configured, dev, reinterpret_cast<const void *>(kda_recover_kernel),
                           df.max_smem))
    return KDA_ERR_LAUNCH;
  const int grid = prm.items < df.sms ? prm.items : df.sms;
  // With scheduler words the CTAs' ranges cover half of the items and the
  // rest is shared: an item's cost varies with its accepted tokens, and a
  // shared item costs no more than a ranged one here (the per-head constants
  // are two loads).  Measured on the GB300: 7/8 in ranges 83.8 us, 1/2 83.3,
  // ranges only 85.5 (record q8 replay).
  prm.sched = a->sched;
  prm.dyn0 = a->sched ? static_cast<int>(static_cast<int64_t>(prm.items) / 2 / grid) * grid
                      : prm.items;
  kda_recover_kernel<<<grid, kThreads, total, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? KDA_SUCCESS : KDA_ERR_LAUNCH;
}

}  // namespace recover
}  // namespace kda

extern "C" int kda_recover(const kda_recover_args *args, void *stream) {
  return kda::recover::run(args, static_cast<cudaStream_t>(stream));
}
