// Output-projection consumer epilogue on one GPU (sm_103a).
//
// Method: vLLM API page
//   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.oproj.consumer"
// (class OprojConsumer: poll_sum, combined_weight, pre, post).  The page
// spreads one token's hidden vector over a cluster of CTAs and receives the
// tensor-parallel partial outputs in remote mailboxes; on one GPU every
// partial is a plain array, so one CTA holds a whole token: thread i owns
// features 8i .. 8i+7 (one 16-byte vector of each BF16 row).
//
// Per token (the operation is stated in include/kda.h):
//   1. the partials are streamed in rank groups (up to four 16-byte loads in
//      flight per thread), summed in the page's order, rounded to BF16,
//      optionally added to the prefix and rounded again; the new prefix is
//      stored;
//   2. nb > 0: one block-wide sum gives every block's and the prefix's
//      squares and projections on w = norm * query; the softmax weights and
//      the unnormalised mix follow per thread (the blocks are re-read, from
//      L1); a second block-wide sum gives mix.p and mix.mix;
//   3. the output coefficients as the page forms them (the prefix merged into
//      the block softmax with a rescale, the mix's squared norm expanded), the
//      output row is stored.
// Block-wide sums: a butterfly inside each warp, the warps' partials added in
// warp order.  HBM-bound: (tp + nb + 2 + has_delta) rows of 2*hidden bytes
// per token, the weights L2-resident.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_device.cuh"
#include "kda_host.h"

namespace kda {
namespace oproj {

constexpr int kGroups = 4;      // rank groups of the partial sum
constexpr int kMaxBlocks = 8;
constexpr int kMaxTp = 64;
constexpr int kMaxHidden = 7168;  // the page's hidden size
constexpr int kThreads = 448;     // a CTA: two 8-feature chunks a thread at hidden 7168

struct Params {
  int tp, tokens, vec, nb, has_delta;  // vec = hidden / 8
  const uint4 *partials, *blocks, *norm, *query, *out_norm;
  uint4 *prefix, *output;
  float eps, out_eps, inv_hidden;
};

__device__ __forceinline__ void unpack8(const uint4 &u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    w[j] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * j]))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * j + 1])))
            << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// rstd(s, e) = 1 / sqrt(s / hidden + e) on the approximate instructions.
__device__ __forceinline__ float rstd(float s, float e, float inv_hidden) {
  return rcp_approx(sqrt_approx(__fadd_rn(__fmul_rn(s, inv_hidden), e)));
}

// Block-wide sums of N per-thread values; every thread gets the totals.
// `red` holds 32 * N floats, `tot` N floats.
template <int N>
__device__ __forceinline__ void block_sum(float (&v)[N], float *red, float *tot) {
  warp_sum_n(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) red[warp * N + i] = v[i];
  }
  __syncthreads();
  if (threadIdx.x < N) {
    float s = red[threadIdx.x];
    for (int w = 1; w < nw; ++w) s = __fadd_rn(s, red[w * N + threadIdx.x]);
    tot[threadIdx.x] = s;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = tot[i];
}

// Rank-group sum of the tp partials of one 8-feature chunk (poll_sum / post:
// the groups in order, each summed in rank order from its first rank; up to
// four 16-byte loads in flight), the new prefix p = BF16(sum) or BF16(prefix
// + BF16(sum)), written back.
__device__ __forceinline__ void prefix_chunk(const Params &p, int64_t row, int64_t rank_stride,
                                             float (&pv)[8]) {
  const int per = (p.tp + kGroups - 1) / kGroups;
  const int S = per > 4 ? per : 4;
  float attn[8];
  for (int g = 0; g < kGroups; ++g) {
    const int lo = g * S;
    const int hi = lo + S < p.tp ? lo + S : p.tp;
    if (lo >= hi) break;
    float gs[8];
    for (int r0 = lo; r0 < hi; r0 += 4) {
      const int n = hi - r0 < 4 ? hi - r0 : 4;
      uint4 u[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < n) u[j] = __ldcs(p.partials + (r0 + j) * rank_stride + row);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < n) {
          float v[8];
          unpack8(u[j], v);
          if (r0 + j == lo) {
#pragma unroll
            for (int k = 0; k < 8; ++k) gs[k] = v[k];
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) gs[k] = __fadd_rn(gs[k], v[k]);
          }
        }
      }
    }
    if (g == 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) attn[k] = gs[k];
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) attn[k] = __fadd_rn(attn[k], gs[k]);
    }
  }
  float old[8];
  if (p.has_delta) unpack8(p.prefix[row], old);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float v = bf16_round(attn[k]);
    if (p.has_delta) v = bf16_round(__fadd_rn(old[k], v));
    pv[k] = v;
  }
  p.prefix[row] = pack8(pv);
}

// One CTA of kThreads threads per token row; thread i owns the 8-feature
// chunks i and i + kThreads (one 16-byte vector of each BF16 row), so that two
// CTAs fit on an SM (registers) and every row of a 256-row batch starts at
// once; the new prefix and the mix wait in shared memory between the
// CTA-wide sums.
template <int NB>
__global__ void __launch_bounds__(kThreads, 2) oproj_kernel(const __grid_constant__ Params p) {
  constexpr int NR = NB > 0 ? 2 * NB + 2 : 1;
  __shared__ float red[32 * NR];
  __shared__ float tot[NR];
  extern __shared__ __align__(16) float chunk_smem[];  // pv | mix: [2][vec][8]
  const int t = blockIdx.x;
  const int i = threadIdx.x;
  const int nthr = blockDim.x;
  const int64_t rank_stride = static_cast<int64_t>(p.tokens) * p.vec;
  float *pvs = chunk_smem;                    // [vec][8] new prefix
  float *mxs = chunk_smem + 8 * p.vec;        // [vec][8] unnormalised mix

  // --- 1. the new prefix of every chunk this thread owns.
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    const int c = i + ch * nthr;
    if (c >= p.vec) break;
    float pv[8];
    prefix_chunk(p, static_cast<int64_t>(t) * p.vec + c, rank_stride, pv);
#pragma unroll
    for (int k = 0; k < 8; ++k) pvs[c * 8 + k] = pv[k];
  }

  if constexpr (NB == 0) {
    // RMSNorm of the prefix.
    float s[1] = {0.0f};
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int c = i + ch * nthr;
      if (c >= p.vec) break;
#pragma unroll
      for (int k = 0; k < 8; ++k) s[0] = __fmaf_rn(pvs[c * 8 + k], pvs[c * 8 + k], s[0]);
    }
    block_sum<1>(s, red, tot);
    const float cp = rstd(s[0], p.out_eps, p.inv_hidden);
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int c = i + ch * nthr;
      if (c >= p.vec) break;
      float on[8], y[8];
      unpack8(__ldg(p.out_norm + c), on);
#pragma unroll
      for (int k = 0; k < 8; ++k) y[k] = __fmul_rn(__fmul_rn(cp, pvs[c * 8 + k]), on[k]);
      p.output[static_cast<int64_t>(t) * p.vec + c] = pack8(y);
    }
  } else {
    // --- 2. combined weight, block and prefix logits (pre / post).
    float acc[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r] = 0.0f;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int c = i + ch * nthr;
      if (c >= p.vec) break;
      float w[8];
      {
        float nq[8], qq[8];
        unpack8(__ldg(p.norm + c), nq);
        unpack8(__ldg(p.query + c), qq);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = __fmul_rn(nq[k], qq[k]);
      }
      const uint4 *vb = p.blocks + static_cast<int64_t>(t) * NB * p.vec + c;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float v[8];
        unpack8(__ldg(vb + b * p.vec), v);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          acc[2 * b] = __fmaf_rn(v[k], v[k], acc[2 * b]);
          acc[2 * b + 1] = __fmaf_rn(v[k], w[k], acc[2 * b + 1]);
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float pk = pvs[c * 8 + k];
        acc[2 * NB] = __fmaf_rn(pk, pk, acc[2 * NB]);
        acc[2 * NB + 1] = __fmaf_rn(pk, w[k], acc[2 * NB + 1]);
      }
    }
    block_sum<NR>(acc, red, tot);
    float logit[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b)
      logit[b] = __fmul_rn(acc[2 * b + 1], rstd(acc[2 * b], p.eps, p.inv_hidden));
    const float lp = __fmul_rn(acc[2 * NB + 1], rstd(acc[2 * NB], p.eps, p.inv_hidden));
    float mx = logit[0];
#pragma unroll
    for (int b = 1; b < NB; ++b) mx = fmaxf(mx, logit[b]);
    float e[NB], esum = 0.0f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      e[b] = exp_approx(__fsub_rn(logit[b], mx));
      esum = __fadd_rn(esum, e[b]);
    }
    // The unnormalised block mix (blocks again, now from L1/L2), mix . p and
    // mix . mix.
    float m2[2] = {0.0f, 0.0f};
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int c = i + ch * nthr;
      if (c >= p.vec) break;
      const uint4 *vb = p.blocks + static_cast<int64_t>(t) * NB * p.vec + c;
      float mix[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mix[k] = 0.0f;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float v[8];
        unpack8(__ldg(vb + b * p.vec), v);
#pragma unroll
        for (int k = 0; k < 8; ++k) mix[k] = __fmaf_rn(e[b], v[k], mix[k]);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        m2[0] = __fmaf_rn(mix[k], pvs[c * 8 + k], m2[0]);
        m2[1] = __fmaf_rn(mix[k], mix[k], m2[1]);
        mxs[c * 8 + k] = mix[k];
      }
    }
    block_sum<2>(m2, red, tot);
    // --- 3. the prefix merged into the softmax, the output coefficients.
    const float top = fmaxf(mx, lp);
    const float alpha = exp_approx(__fsub_rn(mx, top));
    const float ep = exp_approx(__fsub_rn(lp, top));
    const float den = __fmaf_rn(alpha, esum, ep);
    const float a2 = __fmul_rn(alpha, alpha);
    const float ae2 = __fmul_rn(__fmul_rn(2.0f, alpha), ep);
    const float quad =
        __fmaf_rn(a2, m2[1], __fmaf_rn(ae2, m2[0], __fmul_rn(__fmul_rn(ep, ep), acc[2 * NB])));
    const float scale =
        rstd(quad, __fmul_rn(__fmul_rn(p.out_eps, den), den), p.inv_hidden);
    const float ca = __fmul_rn(alpha, scale), cp = __fmul_rn(ep, scale);
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int c = i + ch * nthr;
      if (c >= p.vec) break;
      float on[8], y[8];
      unpack8(__ldg(p.out_norm + c), on);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        y[k] = __fmul_rn(__fmaf_rn(ca, mxs[c * 8 + k], __fmul_rn(cp, pvs[c * 8 + k])), on[k]);
      p.output[static_cast<int64_t>(t) * p.vec + c] = pack8(y);
    }
  }
}

template <int NB>
static int launch(const Params &prm, int dev, int threads, cudaStream_t stream) {
  // the new prefix and the mix of every chunk: 2 x hidden floats
  const int smem = prm.vec * 8 * 2 * static_cast<int>(sizeof(float));
  static std::atomic<bool> configured[kMaxDevices];
  if (!set_smem_limit_once(configured, dev, reinterpret_cast<const void *>(oproj_kernel<NB>),
                           kMaxHidden * 2 * static_cast<int>(sizeof(float))))
    return KDA_ERR_LAUNCH;
  oproj_kernel<NB><<<prm.tokens, threads, smem, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? KDA_SUCCESS : KDA_ERR_LAUNCH;
}

static bool aligned16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

static int run(const kda_oproj_args *a, cudaStream_t stream) {
  if (!a) return KDA_ERR_NULL_ARGS;
  if (a->tp < 1 || a->tp > kMaxTp || a->tokens < 0 || a->nb < 0 || a->nb > kMaxBlocks ||
      a->hidden < 256 || a->hidden > kMaxHidden || a->hidden % 256 != 0)
    return KDA_ERR_SHAPE;
  if (a->tokens == 0) return KDA_SUCCESS;
  if (static_cast<int64_t>(a->tp) * a->tokens * a->hidden > (int64_t(1) << 40))
    return KDA_ERR_SHAPE;
  if (!a->partials || !a->out_norm || !a->prefix || !a->output) return KDA_ERR_NULL_POINTER;
  if (a->nb > 0 && (!a->blocks || !a->norm || !a->query)) return KDA_ERR_NULL_POINTER;
  if (!aligned16(a->partials) || !aligned16(a->out_norm) || !aligned16(a->prefix) ||
      !aligned16(a->output) ||
      (a->nb > 0 && (!aligned16(a->blocks) || !aligned16(a->norm) || !aligned16(a->query))))
    return KDA_ERR_ALIGNMENT;
  int dev = 0;
  DeviceFacts df;
  if (!current_device(&dev, &df)) return KDA_ERR_DEVICE;

  Params prm;
  prm.tp = a->tp;
  prm.tokens = a->tokens;
  prm.vec = a->hidden / 8;
  prm.nb = a->nb;
  prm.has_delta = a->has_delta ? 1 : 0;
  prm.partials = static_cast<const uint4 *>(a->partials);
  prm.blocks = static_cast<const uint4 *>(a->blocks);
  prm.norm = static_cast<const uint4 *>(a->norm);
  prm.query = static_cast<const uint4 *>(a->query);
  prm.out_norm = static_cast<const uint4 *>(a->out_norm);
  prm.prefix = static_cast<uint4 *>(a->prefix);
  prm.output = static_cast<uint4 *>(a->output);
  prm.eps = a->eps;
  prm.out_eps = a->out_eps;
  prm.inv_hidden = 1.0f / static_cast<float>(a->hidden);
  // two chunks a thread: ceil(vec / 2) threads rounded up to whole warps
  const int threads = ((prm.vec + 1) / 2 + 31) / 32 * 32;
  switch (a->nb) {
    case 0: return launch<0>(prm, dev, threads, stream);
    case 1: return launch<1>(prm, dev, threads, stream);
    case 2: return launch<2>(prm, dev, threads, stream);
    case 3: return launch<3>(prm, dev, threads, stream);
    case 4: return launch<4>(prm, dev, threads, stream);
    case 5: return launch<5>(prm, dev, threads, stream);
    case 6: return launch<6>(prm, dev, threads, stream);
    case 7: return launch<7>(prm, dev, threads, stream);
    default: return launch<8>(prm, dev, threads, stream);
  }
}

}  // namespace oproj
}  // namespace kda

extern "C" int kda_oproj(const kda_oproj_args *args, void *stream) {
  return kda::oproj::run(args, static_cast<cudaStream_t>(stream));
}
