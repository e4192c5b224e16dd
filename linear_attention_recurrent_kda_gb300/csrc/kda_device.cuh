// Device helpers shared by the KDA kernels (sm_103a): mbarrier, TMA bulk
// copies, named barriers, the tensor-core MMA, and the approximate math of the
// vLLM page "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.wide"
// (KdaWide: exp as 2^(x log2 e) on the approximate exp2, the full-range
// approximate divide, square root and reciprocal; KdaWide.silu).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits: 2 s

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase of `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about `hint_ns` pass, instead of spinning on issue slots that
// the other roles' warps on the same SM sub-partition need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `parity` to complete.  Returns false, and raises the
// CTA's abort flag, after kWaitLimitNs of wall clock (or 2^24 sleeps); returns
// false early when another thread raised the flag.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          volatile uint32_t *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) break;
  }
  *abort_flag = 1u;
  return false;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// TMA bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src,
                                              uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// TMA bulk copy of this CTA's shared memory -> global, tracked as a bulk
// group of the issuing thread.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
          dst),
      "r"(smem_addr(src)), "r"(bytes), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most `pending` committed bulk stores are still reading
// shared memory (0..3).
__device__ __forceinline__ void bulk_wait_read(int pending) {
  switch (pending) {
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
  }
}
// Waits until every committed bulk store is complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier 1 over the 256 recurrence threads.
__device__ __forceinline__ void rec_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// Named barrier 1 over the 256 recurrence threads that also ORs a predicate.
__device__ __forceinline__ bool rec_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

// Named barrier 2 over the 128 front threads.
__device__ __forceinline__ void front_sync() {
  asm volatile("bar.sync 2, 128;" ::: "memory");
}

// Named barrier 2 over the 128 front threads that also ORs a predicate.
__device__ __forceinline__ bool front_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 2, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// m16n8k16 BF16 tensor-core MMA, FP32 accumulate in place.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------- clusters / distributed smem

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of `p` (this CTA's shared memory) in cluster CTA `rank`'s window.
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(a)
               : "r"(smem_addr(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Full cluster barrier: every thread of every CTA of the cluster; orders the
// distributed shared-memory stores before it with the loads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------- the page's approximate math
// exp(x) = 2^(x log2 e) on the approximate exp2 instruction; division, square
// root and reciprocal on the approximate full-range instructions.

__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float exp_approx(float x) {
  return exp2_approx(__fmul_rn(x, 1.4426950408889634f));
}
__device__ __forceinline__ float div_full(float a, float b) {
  float y;
  asm("div.full.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_approx(float z) {
  return div_full(1.0f, __fadd_rn(1.0f, exp_approx(-z)));
}
// KdaWide.silu before its BF16 rounding.
__device__ __forceinline__ float silu_approx(float a) {
  return div_full(a, __fadd_rn(1.0f, exp_approx(-a)));
}
__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, s));
  return v;
}

// warp_sum of N independent values, reduced level by level so that the N
// shuffle chains overlap; each value sees the same additions as warp_sum.
template <int N>
__device__ __forceinline__ void warp_sum_n(float (&v)[N]) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1)
#pragma unroll
    for (int i = 0; i < N; ++i)
      v[i] = __fadd_rn(v[i], __shfl_xor_sync(0xffffffffu, v[i], s));
}

// Warp sums of N values (N a power of two <= 32), scattered: lane L ends up
// with the total of value (L / (32 / N)) % N.  Each level halves the values a
// lane keeps and adds its partner's copy of the same values (xor distance 16,
// 8, ... ), then the remaining levels add the partner's single value; every
// total is the same pairwise tree as warp_sum's, so the bits are identical.
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(const float (&v)[N], int lane) {
  static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
  float cur[N];
#pragma unroll
  for (int j = 0; j < N; ++j) cur[j] = v[j];
  int n = N;
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    if (n > 1) {
      const int h = n >> 1;
      const bool hi = (lane & s) != 0;
#pragma unroll
      for (int j = 0; j < N / 2; ++j) {
        if (j < h) {
          const float keep = hi ? cur[j + h] : cur[j];
          const float send = hi ? cur[j] : cur[j + h];
          cur[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, s));
        }
      }
      n = h;
    } else {
      cur[0] = __fadd_rn(cur[0], __shfl_xor_sync(0xffffffffu, cur[0], s));
    }
  }
  return cur[0];
}

template <int X>
struct NextPow2 {
  static constexpr int value = X <= 1 ? 1 : 2 * NextPow2<(X + 1) / 2>::value;
};
template <>
struct NextPow2<1> {
  static constexpr int value = 1;
};

// Sum over the 8 lanes of a row group of four partial sums (one per value row
// m = 0..3); returns the total of row (lane >> 1) & 3.
__device__ __forceinline__ float reduce_scatter8(const float (&x)[4], int l) {
  const bool hi2 = (l >> 2) & 1;
  float keep0 = hi2 ? x[2] : x[0], keep1 = hi2 ? x[3] : x[1];
  const float send0 = hi2 ? x[0] : x[2], send1 = hi2 ? x[1] : x[3];
  keep0 = __fadd_rn(keep0, __shfl_xor_sync(0xffffffffu, send0, 4));
  keep1 = __fadd_rn(keep1, __shfl_xor_sync(0xffffffffu, send1, 4));
  const bool hi1 = (l >> 1) & 1;
  float keep = hi1 ? keep1 : keep0;
  const float send = hi1 ? keep0 : keep1;
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, keep, 1));
  return keep;
}

}  // namespace kda
