// Measurement probe: the HBM access pattern of the decode / verify step
// without its arithmetic (sm_103a).
//
// Per (request, head) item, the 64 KiB FP32 state page the step reads is
// read by one TMA bulk copy into a shared-memory stage and written by bulk
// stores to every page the step writes (decode: back in place; verify: the
// slots of the T tokens): the bytes and the order of the step (persistent
// CTAs, one per SM, over contiguous item ranges and, with scheduler words,
// the step's shared items; a ring of `stages` pages per CTA), with no conv,
// gate, recurrence or epilogue.  Its bandwidth is the
// ceiling that the step's own page traffic can reach on this memory system.
// One thread per CTA issues everything.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda_probe.h"
#include "kda_device.cuh"
#include "kda_host.h"

namespace kda {
namespace probe {

constexpr uint32_t kPage = 128u * 128u * 4u;

// An item's pages: the one it reads (src) and the ones it writes (dst; T of
// them, the slots of its tokens, <= 0 skipped).  Live unless padded or out of
// range (then flagged and skipped, as the step does).
struct ProbeItem {
  int src;
  int dst[KDA_MAX_TOKENS];
};

__device__ __forceinline__ bool probe_resolve(const kda_probe_args &a, int n, ProbeItem &it) {
  const int h = n / a.batch, r = n - h * a.batch;
  (void)h;
  const int T = a.tokens;
  const int32_t *row = a.slots + static_cast<int64_t>(r) * a.slot_cols;
  int off = 0;
  if (T > 1) {
    const int acc = __ldg(a.accepted + r);
    if (acc < 1 || acc > T) {
      if (a.err) atomicOr(a.err, KDA_DEVERR_ACCEPTED);
      return false;
    }
    off = acc - 1;
  }
  it.src = __ldg(row + off);
  if (it.src <= 0) return false;
  bool bad = it.src >= a.num_slots;
#pragma unroll
  for (int t = 0; t < KDA_MAX_TOKENS; ++t) {
    it.dst[t] = t < T ? (T > 1 ? __ldg(row + t) : it.src) : 0;
    bad |= it.dst[t] >= a.num_slots;
  }
  if (bad && a.err) atomicOr(a.err, KDA_DEVERR_SLOT);
  return !bad;
}

// Items dyn0 .. items-1 go one at a time to the CTA that asks first when the
// scheduler words are given (the step's schedule, same rule for dyn0).
template <int S>
__global__ void __launch_bounds__(32) page_copy_kernel(const __grid_constant__ kda_probe_args a,
                                                       int dyn0) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[S];
  __shared__ uint32_t abort_flag;
  if (threadIdx.x != 0) return;
  const int items = a.batch * a.heads, G = gridDim.x;
  int n0, n1;
  if (a.sched) {
    n0 = (dyn0 / G) * static_cast<int>(blockIdx.x);
    n1 = n0 + dyn0 / G;
  } else {
    n0 = static_cast<int>(static_cast<int64_t>(items) * blockIdx.x / G);
    n1 = static_cast<int>(static_cast<int64_t>(items) * (blockIdx.x + 1) / G);
  }
  abort_flag = 0u;
  for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  auto page = [&](int n, int slot) -> float * {
    const int h = n / a.batch;
    return a.state + (static_cast<int64_t>(slot) * a.heads + h) * (kPage / 4);
  };
  // The CTA's next live item after its cursor n (its range, then shared
  // items), resolved into `it`; -1 when none is left.
  bool drained = a.sched == nullptr;
  auto next_live = [&](int &n, ProbeItem &it) -> int {
    for (; n < n1; ++n)
      if (probe_resolve(a, n, it)) return n++;
    while (!drained) {
      // 64-bit, the counter read unsigned: no wrap however many items there are.
      const int64_t m = dyn0 + static_cast<int64_t>(static_cast<uint32_t>(atomicAdd(a.sched, 1)));
      if (m >= items) {
        drained = true;
        break;
      }
      if (probe_resolve(a, static_cast<int>(m), it)) return static_cast<int>(m);
    }
    return -1;
  };
  const uint64_t pol = policy_evict_first();
  // The j-th live item of the range goes through stage j % S.
  int item[S];
  ProbeItem res[S];
  int loaded = 0, n = n0;
  for (int s = 0; s < S; ++s) {
    const int m = next_live(n, res[s]);
    if (m < 0) break;
    item[s] = m;
    mbar_arrive_expect_tx(&full[s], kPage);
    bulk_g2s(smem + s * kPage, page(item[s], res[s].src), kPage, &full[s]);
    ++loaded;
  }
  for (int i = 0; i < loaded; ++i) {
    const int st = i % S;
    if (!mbar_wait(&full[st], static_cast<uint32_t>(i / S) & 1u, &abort_flag)) {
      if (a.err) atomicOr(a.err, KDA_DEVERR_TIMEOUT);
      uint32_t z = 0;  // bounded drain of the loads still in flight
      for (int q = i + 1; q < loaded; ++q)
        (void)mbar_wait(&full[q % S], static_cast<uint32_t>(q / S) & 1u, &z);
      break;
    }
    // Every write of the item leaves from the staged page (one bulk group).
    for (int t = 0; t < a.tokens; ++t)
      if (res[st].dst[t] > 0)
        bulk_s2g(page(item[st], res[st].dst[t]), smem + st * kPage, kPage, pol);
    bulk_commit();
    if (i >= 1) {
      // Refill the stage of item i-1 once its stores have read it.
      bulk_wait_read(1);
      const int ps = (i - 1) % S;
      const int m = next_live(n, res[ps]);
      if (m >= 0) {
        item[ps] = m;
        mbar_arrive_expect_tx(&full[ps], kPage);
        bulk_g2s(smem + ps * kPage, page(item[ps], res[ps].src), kPage, &full[ps]);
        ++loaded;
      }
    }
  }
  bulk_wait_all();
  if (a.sched) {
    // The last CTA zeroes the scheduler words for the next launch.
    __threadfence();
    if (atomicAdd(a.sched + 1, 1) == G - 1) {
      atomicExch(a.sched, 0);
      atomicExch(a.sched + 1, 0);
    }
  }
}

template <int S>
static int launch(const kda_probe_args *a, int dev, int grid, int dyn0, cudaStream_t stream) {
  static std::atomic<bool> configured[kMaxDevices];
  if (!set_smem_limit_once(configured, dev, reinterpret_cast<const void *>(page_copy_kernel<S>),
                           S * kPage))
    return KDA_ERR_LAUNCH;
  page_copy_kernel<S><<<grid, 32, S * kPage, stream>>>(*a, dyn0);
  return cudaGetLastError() == cudaSuccess ? KDA_SUCCESS : KDA_ERR_LAUNCH;
}

static int run(const kda_probe_args *a, cudaStream_t stream) {
  if (!a) return KDA_ERR_NULL_ARGS;
  if (a->batch < 0 || a->heads < 0 || a->num_slots < 1 || a->stages < 2 || a->stages > 3)
    return KDA_ERR_SHAPE;
  if (a->tokens < 1 || a->tokens > KDA_MAX_TOKENS) return KDA_ERR_TOKENS;
  if (a->slot_cols < (a->tokens > 1 ? a->tokens : 1)) return KDA_ERR_SHAPE;
  if (static_cast<int64_t>(a->batch) * a->heads > (int64_t(1) << 30)) return KDA_ERR_SHAPE;
  if (a->batch == 0 || a->heads == 0) return KDA_SUCCESS;
  if (!a->state || !a->slots || (a->tokens > 1 && !a->accepted)) return KDA_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(a->state) & 15u) || (reinterpret_cast<uintptr_t>(a->slots) & 3u) ||
      (a->err && (reinterpret_cast<uintptr_t>(a->err) & 3u)) ||
      (a->tokens > 1 && (reinterpret_cast<uintptr_t>(a->accepted) & 3u)) ||
      (reinterpret_cast<uintptr_t>(a->sched) & 3u))
    return KDA_ERR_ALIGNMENT;
  int dev = 0;
  DeviceFacts df;
  if (!current_device(&dev, &df)) return KDA_ERR_DEVICE;
  const int64_t items = static_cast<int64_t>(a->batch) * a->heads;
  const int grid = static_cast<int>(items < df.sms ? items : df.sms);
  // The step's split between contiguous ranges and shared items.
  const bool wide = a->tokens == 1 && items >= 32 * static_cast<int64_t>(grid);
  const int dyn0 = a->sched ? static_cast<int>(items * (wide ? 7 : 8) / 8 / grid) * grid
                            : static_cast<int>(items);
  return a->stages == 2 ? launch<2>(a, dev, grid, dyn0, stream)
                        : launch<3>(a, dev, grid, dyn0, stream);
}

}  // namespace probe
}  // namespace kda

extern "C" int kda_probe_page_copy(const kda_probe_args *args, void *stream) {
  return kda::probe::run(args, static_cast<cudaStream_t>(stream));
}
