// KDA decode / verify step for few items: one item over a cluster of 4 CTAs.
//
// Method: vLLM API page
//   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide"
// (KdaWide.kernel and its helpers; the page's module docstring names KdaSplit,
// which "splits a head over a cluster to spread a few requests over the GPU";
// its source is not shown, so this split is designed here).
//
// The delta-rule recurrence is independent per value row once q_hat, k_hat,
// the decay and beta are known, so CTA p of the cluster owns value rows,
// channels and gate features [32p, 32p + 32):
//   * warps 0-2: conv + SiLU + BF16 of channel 32p + lane of q, k, v (and the
//     conv-window write of those channels); per-token sums of squares of its
//     32 q and 32 k values;
//   * warps 3-4: the gate projection of features 32p .. 32p+31 (one m16 tile
//     each, mma.sync BF16 -> FP32) and their decay;
//   * the q, k, decay slices and the square sums are all-gathered through
//     distributed shared memory (cluster barrier), then every CTA forms q_hat
//     and k_hat;
//   * all 8 warps run the recurrence on the CTA's 32 rows (thread (g, l): row
//     32p + g, keys {32c + 4l + e}), write the rows of every target page, and
//     the RMS partial sums of o are all-gathered the same way.
// Every partial sum is formed over the same 32-element groups and in the same
// order as in the one-CTA-per-SM kernel (kda_step.cu), so both paths give the
// same bits.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_device.cuh"

namespace kda {
namespace split {

constexpr int kDk = 128;
constexpr int kParts = 4;     // CTAs per item (cluster size)
constexpr int kRows = 32;     // value rows / channels / features per CTA
constexpr int kThreads = 256;
constexpr int kLive = 0, kPad = 1, kError = 2;

struct Params {
  int32_t batch, heads, num_slots, conv_width, slot_cols, gate_mode, has_bias;
  int32_t conv_f32;  // conv pool element: FP32 (1) or BF16 (0)
  const __nv_bfloat16 *x, *conv_weight, *conv_bias, *f_a, *f_b, *beta, *gate;
  const __nv_bfloat16 *norm_weight;
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

template <int T>
struct Smem {
  float q[T][kDk];        // all-gathered q (then q_hat)
  float k[T][kDk];        // all-gathered k (then k_hat)
  float d[T][kDk];        // all-gathered decay
  float ssum[T][2][4];    // q, k square sums of each 32-channel group
  float osum[T][4];       // o square sums of each 32-channel group
  float v[T][kRows];      // this CTA's v
  float o[T][kRows];      // this CTA's o (BF16 values)
  float beta[KDA_MAX_TOKENS];
  int32_t tgt[KDA_MAX_TOKENS];
};

// Stores `v` at `local` in the shared memory of every CTA of the cluster.
__device__ __forceinline__ void all_gather(const float *local, float v) {
#pragma unroll
  for (uint32_t rk = 0; rk < kParts; ++rk) st_cluster_f32(cluster_map(local, rk), v);
}

// Butterfly sum over the 8 lanes of a row group (pairs l^4, l^2, l^1: the
// same pairing as the other kernel's reduce-scatter uses for every row).
__device__ __forceinline__ float row_sum8(float v) {
  v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return v;
}

template <int T, bool RECORD>
__global__ void __launch_bounds__(kThreads) kda_split_kernel(const __grid_constant__ Params p) {
  __shared__ __align__(16) Smem<T> sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int part = static_cast<int>(cluster_ctarank());
  const int n = blockIdx.x / kParts;
  const int h = n % p.heads;
  const int r = n / p.heads;
  const int64_t dim = static_cast<int64_t>(p.heads) * kDk;
  const int64_t item = static_cast<int64_t>(r) * p.heads + h;
  const int row0 = kRows * part;

  // --- slots (every thread resolves the same item; uniform over the cluster)
  int s, cs, off, status = kLive, flags = 0;
  if (T == 1) {
    s = __ldg(p.slots + r);
    cs = s;
    off = 0;
  } else {
    const int a = __ldg(p.accepted + r);
    if (a < 1 || a > T) {
      status = kError;
      flags = KDA_DEVERR_ACCEPTED;
      s = cs = off = 0;
    } else {
      off = a - 1;
      s = __ldg(p.slots + static_cast<int64_t>(r) * p.slot_cols + off);
      cs = __ldg(p.slots + static_cast<int64_t>(r) * p.slot_cols);
    }
  }
  if (status == kLive) {
    if (s <= 0) {
      status = kPad;
    } else {
      if (s >= p.num_slots || cs <= 0 || cs >= p.num_slots) flags |= KDA_DEVERR_SLOT;
      if (T > 1 && !RECORD)
        for (int t = 0; t < T; ++t)
          if (__ldg(p.slots + static_cast<int64_t>(r) * p.slot_cols + t) >= p.num_slots)
            flags |= KDA_DEVERR_SLOT;
      if (flags) status = kError;
    }
  }
  if (status != kLive) {
    if (flags && p.err && part == 0 && tid == 0) atomicOr(p.err, flags);
    if (tid < kRows) {
#pragma unroll
      for (int t = 0; t < T; ++t)
        p.output[(static_cast<int64_t>(r) * T + t) * dim + h * kDk + row0 + tid] =
            __float2bfloat16_rn(0.0f);
    }
    return;  // the whole cluster takes this branch
  }

  // Peers write into this CTA's shared memory only after the whole cluster
  // has started.
  cluster_sync_all();

  // --- the CTA's 32 page rows into registers: row row0 + g8, keys 32c + 4l8
  const int g8 = tid >> 3, l8 = tid & 7;
  const float *page = p.state + (static_cast<int64_t>(s) * p.heads + h) *
                                    static_cast<int64_t>(kDk * kDk);
  float4 S4[4];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
    S4[cc] = __ldg(reinterpret_cast<const float4 *>(page + (row0 + g8) * kDk + 32 * cc +
                                                    4 * l8));

  if (warp < 3) {
    // --- convolution + SiLU + BF16 (KdaWide.kernel, "The convolution (stock
    // tap order) and SiLU"): warp = part (q, k, v), channel row0 + lane.
    const int pt = warp;
    const int c = row0 + lane;
    const int64_t ch = pt * dim + h * kDk + c;
    const uint16_t *cw = reinterpret_cast<const uint16_t *>(p.conv_weight);
    const uint16_t *cb = reinterpret_cast<const uint16_t *>(p.conv_bias);
    const int64_t rix = (static_cast<int64_t>(cs) * 3 * dim + ch) * p.conv_width;
    float win[3 + T];
    uint16_t xb[T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      xb[t] = __ldg(reinterpret_cast<const uint16_t *>(p.x) +
                    (static_cast<int64_t>(r) * T + t) * 3 * dim + ch);
      win[3 + t] = bf16_bits_to_float(xb[t]);
    }
    float wt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      wt[i] = bf16_bits_to_float(
          __ldg(cw + (static_cast<int64_t>(pt) * 4 + i) * dim + h * kDk + c));
    const float bias = p.has_bias ? bf16_bits_to_float(__ldg(cb + ch)) : 0.0f;
    // Taps as the pool stores them (the page's conv_type); new window
    // [tap1, tap2, x_0 .. x_{T-1}] of this channel.
    if (p.conv_f32) {
      float *crow = reinterpret_cast<float *>(p.conv_state) + rix;
      win[0] = crow[off];
      win[1] = crow[off + 1];
      win[2] = crow[off + 2];
      crow[0] = win[1];
      crow[1] = win[2];
#pragma unroll
      for (int t = 0; t < T; ++t) crow[2 + t] = win[3 + t];
    } else {
      uint16_t *crow = reinterpret_cast<uint16_t *>(p.conv_state) + rix;
      const uint16_t tap0 = crow[off], tap1 = crow[off + 1], tap2 = crow[off + 2];
      win[0] = bf16_bits_to_float(tap0);
      win[1] = bf16_bits_to_float(tap1);
      win[2] = bf16_bits_to_float(tap2);
      crow[0] = tap1;
      crow[1] = tap2;
#pragma unroll
      for (int t = 0; t < T; ++t) crow[2 + t] = xb[t];
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float acc = bias;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc = __fmaf_rn(win[t + i], wt[i], acc);
      const float y = bf16_round(silu_approx(acc));
      if (p.dbg) p.dbg[((item * T + t) * 4 + pt) * kDk + c] = __float2bfloat16_rn(y);
      if (pt == 2) {
        sm.v[t][lane] = y;
      } else {
        if (RECORD && pt == 1)
          p.rec_kg[(item * T + t) * 2 * kDk + c] = __float2bfloat16_rn(y);
        all_gather(pt == 0 ? &sm.q[t][c] : &sm.k[t][c], y);
        const float sq = warp_sum(__fmul_rn(y, y));
        if (lane == 0) all_gather(&sm.ssum[t][pt][part], sq);
      }
    }
  } else if (warp < 5) {
    // --- gate projection on tensor cores (KdaWide.kernel, "Gate projection"):
    // one m16 tile of features row0 + 16m + g (+8), token column n = lane/4.
    const int m = warp - 3;
    const int g = lane >> 2, q = lane & 3;
    const uint2 *fb = reinterpret_cast<const uint2 *>(p.f_b);
    const int fA = h * kDk + row0 + 16 * m + g;
    uint32_t wa[8][4], fb0[8], fb1[8];
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      // Rank columns 16kc + 4q + {0..3} play the fragment's k positions
      // {2q, 2q+1, 2q+8, 2q+9} on both operands (the sum is unchanged).
      const uint2 lo = __ldg(fb + (static_cast<int64_t>(fA) * kDk + 16 * kc + 4 * q) / 4);
      const uint2 hi =
          __ldg(fb + (static_cast<int64_t>(fA + 8) * kDk + 16 * kc + 4 * q) / 4);
      wa[kc][0] = lo.x;
      wa[kc][2] = lo.y;
      wa[kc][1] = hi.x;
      wa[kc][3] = hi.y;
      if (g < T) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p.f_a) +
                              ((static_cast<int64_t>(r) * T + g) * kDk + 16 * kc + 4 * q) / 4);
        fb0[kc] = v.x;
        fb1[kc] = v.y;
      } else {
        fb0[kc] = fb1[kc] = 0u;
      }
    }
    float gv[4];
    if (p.gate_mode == 0) {
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) mma_bf16(acc, wa[kc], fb0[kc], fb1[kc]);
#pragma unroll
      for (int e = 0; e < 4; ++e) gv[e] = acc[e];
    } else {
      float acc[4][4];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[ch][e] = 0.0f;
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) mma_bf16(acc[kc >> 1], wa[kc], fb0[kc], fb1[kc]);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        gv[e] = __fadd_rn(
            0.0f, __fadd_rn(__fadd_rn(__fadd_rn(acc[0][e], acc[1][e]), acc[2][e]),
                            acc[3][e]));
    }
    const float ea = exp_approx(__ldg(p.a_log + h));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = 2 * q + (e & 1);
      const int f = row0 + 16 * m + g + 8 * (e >> 1);
      if (t < T) {
        const __nv_bfloat16 gb = __float2bfloat16_rn(gv[e]);
        const float raw = __bfloat162float(gb);
        // KdaWide.decay
        const float z = __fmul_rn(ea, __fadd_rn(raw, __ldg(p.dt_bias + h * kDk + f)));
        all_gather(&sm.d[t][f], exp_approx(__fmul_rn(p.lower_bound, sigmoid_approx(z))));
        if (p.dbg) p.dbg[((item * T + t) * 4 + 3) * kDk + f] = gb;
        if (RECORD) p.rec_kg[(item * T + t) * 2 * kDk + kDk + f] = gb;
      }
    }
  } else if (warp == 5 && lane < T) {
    sm.beta[lane] = sigmoid_approx(bf16_bits_to_float(__ldg(
        reinterpret_cast<const uint16_t *>(p.beta) + (static_cast<int64_t>(r) * T + lane) *
                                                         p.heads + h)));
    sm.tgt[lane] = (T == 1) ? s
                            : (RECORD ? 0
                                      : __ldg(p.slots + static_cast<int64_t>(r) * p.slot_cols +
                                              lane));
  }
  cluster_sync_all();

  // --- L2 norms ("Normalized q (with the 1/sqrt(K) scale) and k"), group
  // sums combined as KdaWide.quad_sum does.
  if (tid < kDk) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const float *q4 = sm.ssum[t][0], *k4 = sm.ssum[t][1];
      const float qn =
          __fadd_rn(__fadd_rn(__fadd_rn(q4[0], q4[2]), __fadd_rn(q4[1], q4[3])), 1.0e-6f);
      const float kn =
          __fadd_rn(__fadd_rn(__fadd_rn(k4[0], k4[2]), __fadd_rn(k4[1], k4[3])), 1.0e-6f);
      const float fq = rcp_approx(sqrt_approx(qn));
      const float fk = rcp_approx(sqrt_approx(kn));
      sm.q[t][tid] = __fmul_rn(__fmul_rn(sm.q[t][tid], fq), p.scale);
      sm.k[t][tid] = __fmul_rn(sm.k[t][tid], fk);
    }
  }
  __syncthreads();

  // --- the recurrence ("The recurrence") on rows row0 + g8.
#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int key = 32 * cc + 4 * l8;
      const float4 d4 = *reinterpret_cast<const float4 *>(&sm.d[t][key]);
      const float4 k4 = *reinterpret_cast<const float4 *>(&sm.k[t][key]);
      const float2 lo = __fmul2_rn(make_float2(S4[cc].x, S4[cc].y), make_float2(d4.x, d4.y));
      const float2 hi = __fmul2_rn(make_float2(S4[cc].z, S4[cc].w), make_float2(d4.z, d4.w));
      S4[cc] = make_float4(lo.x, lo.y, hi.x, hi.y);
      acc = __ffma2_rn(lo, make_float2(k4.x, k4.y), acc);
      acc = __ffma2_rn(hi, make_float2(k4.z, k4.w), acc);
    }
    const float dot = row_sum8(__fadd_rn(acc.x, acc.y));
    const float u = __fmul_rn(__fsub_rn(sm.v[t][g8], dot), sm.beta[t]);
    if (RECORD && l8 == 0) p.rec_u[(item * T + t) * kDk + row0 + g8] = u;
    acc = make_float2(0.0f, 0.0f);
    const float2 uu = make_float2(u, u);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int key = 32 * cc + 4 * l8;
      const float4 k4 = *reinterpret_cast<const float4 *>(&sm.k[t][key]);
      const float4 q4 = *reinterpret_cast<const float4 *>(&sm.q[t][key]);
      const float2 lo = __ffma2_rn(make_float2(k4.x, k4.y), uu, make_float2(S4[cc].x, S4[cc].y));
      const float2 hi = __ffma2_rn(make_float2(k4.z, k4.w), uu, make_float2(S4[cc].z, S4[cc].w));
      S4[cc] = make_float4(lo.x, lo.y, hi.x, hi.y);
      acc = __ffma2_rn(lo, make_float2(q4.x, q4.y), acc);
      acc = __ffma2_rn(hi, make_float2(q4.z, q4.w), acc);
    }
    const float o = row_sum8(__fadd_rn(acc.x, acc.y));
    if (l8 == 0) sm.o[t][g8] = bf16_round(o);
    if (!RECORD) {
      const int tgt = sm.tgt[t];
      if (tgt > 0) {
        float *dst = p.state + (static_cast<int64_t>(tgt) * p.heads + h) *
                                   static_cast<int64_t>(kDk * kDk) +
                     (row0 + g8) * kDk;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          __stcs(reinterpret_cast<float4 *>(dst + 32 * cc + 4 * l8), S4[cc]);
      }
    }
  }
  __syncthreads();

  // --- gated RMSNorm ("Gated RMSNorm"): warp 0, channel row0 + lane.
  float ov[T];
  if (warp == 0) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      ov[t] = sm.o[t][lane];
      const float tot = warp_sum(__fmul_rn(ov[t], ov[t]));
      if (lane == 0) all_gather(&sm.osum[t][part], tot);
    }
  }
  cluster_sync_all();
  if (warp == 0) {
    const int c = row0 + lane;
    const float nw =
        bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.norm_weight) + c));
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const float *o4 = sm.osum[t];
      const float sumsq = __fadd_rn(__fadd_rn(o4[0], o4[2]), __fadd_rn(o4[1], o4[3]));
      const float var = __fadd_rn(__fmul_rn(sumsq, 1.0f / 128.0f), p.eps);
      const float rstd = rcp_approx(sqrt_approx(var));
      const float sg = sigmoid_approx(bf16_bits_to_float(__ldg(
          reinterpret_cast<const uint16_t *>(p.gate) + (static_cast<int64_t>(r) * T + t) * dim +
          h * kDk + c)));
      const float y = __fmul_rn(__fmul_rn(__fmul_rn(ov[t], rstd), nw), sg);
      p.output[(static_cast<int64_t>(r) * T + t) * dim + h * kDk + c] = __float2bfloat16_rn(y);
    }
  }
}

template <int T, bool RECORD>
static int launch_t(const Params &prm, int items, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items * kParts);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kParts;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kda_split_kernel<T, RECORD>, prm) != cudaSuccess)
    return KDA_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? KDA_SUCCESS : KDA_ERR_LAUNCH;
}

}  // namespace split

// Launches the cluster-split step; the arguments were validated by the caller.
int launch_split(const kda_args *a, cudaStream_t stream) {
  using namespace split;
  Params prm;
  prm.batch = a->batch;
  prm.heads = a->heads;
  prm.num_slots = a->num_slots;
  prm.conv_width = a->conv_width;
  prm.slot_cols = a->tokens > 1 ? a->slot_cols : 1;
  prm.gate_mode = a->gate_mode;
  prm.has_bias = a->has_bias ? 1 : 0;
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
  const int items = a->batch * a->heads;
  const bool rec = a->record != 0;
  switch (a->tokens) {
    case 1: return launch_t<1, false>(prm, items, stream);
    case 2: return rec ? launch_t<2, true>(prm, items, stream) : launch_t<2, false>(prm, items, stream);
    case 3: return rec ? launch_t<3, true>(prm, items, stream) : launch_t<3, false>(prm, items, stream);
    case 4: return rec ? launch_t<4, true>(prm, items, stream) : launch_t<4, false>(prm, items, stream);
    case 5: return rec ? launch_t<5, true>(prm, items, stream) : launch_t<5, false>(prm, items, stream);
    case 6: return rec ? launch_t<6, true>(prm, items, stream) : launch_t<6, false>(prm, items, stream);
    case 7: return rec ? launch_t<7, true>(prm, items, stream) : launch_t<7, false>(prm, items, stream);
    default: return rec ? launch_t<8, true>(prm, items, stream) : launch_t<8, false>(prm, items, stream);
  }
}

}  // namespace kda
