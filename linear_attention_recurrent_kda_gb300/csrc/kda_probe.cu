// Measurement probe: the HBM access pattern of the decode step without its
// arithmetic (sm_103a).
//
// Per (request, head) item, the 64 KiB FP32 state page at
// state[slots[r], h] is read by one TMA bulk copy into a shared-memory stage
// and written back to the same place by one bulk store: the bytes and the
// order of the decode step (persistent CTAs, one per SM, over contiguous
// item ranges, a ring of `stages` pages per CTA), with no conv, gate,
// recurrence or epilogue.  Its bandwidth is the ceiling that the decode
// step's own page traffic can reach on this memory system; the state pool is
// unchanged by it.  One thread per CTA issues everything.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_device.cuh"

namespace kda {
namespace probe {

constexpr uint32_t kPage = 128u * 128u * 4u;

template <int S>
__global__ void __launch_bounds__(32) page_copy_kernel(float *state, const int32_t *slots,
                                                       int batch, int heads, int num_slots,
                                                       int32_t *err) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[S];
  __shared__ uint32_t abort_flag;
  if (threadIdx.x != 0) return;
  const int items = batch * heads, G = gridDim.x;
  const int n0 = static_cast<int>(static_cast<int64_t>(items) * blockIdx.x / G);
  const int n1 = static_cast<int>(static_cast<int64_t>(items) * (blockIdx.x + 1) / G);
  abort_flag = 0u;
  for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  // Live items of the range, in order (slot <= 0: padding; slot beyond the
  // pool: error flag, skipped).
  auto next_live = [&](int n) -> int {
    for (; n < n1; ++n) {
      const int s = __ldg(slots + (n - (n / batch) * batch));
      if (s >= num_slots) {
        if (err) atomicOr(err, KDA_DEVERR_SLOT);
      } else if (s > 0) {
        break;
      }
    }
    return n;
  };
  auto page = [&](int n) -> float * {
    const int h = n / batch, r = n - h * batch;
    return state + (static_cast<int64_t>(__ldg(slots + r)) * heads + h) * (kPage / 4);
  };
  const uint64_t pol = policy_evict_first();
  // The j-th live item of the range goes through stage j % S.
  int item[S];
  int loaded = 0, n = n0;
  for (int s = 0; s < S; ++s) {
    n = next_live(n);
    if (n >= n1) break;
    item[s] = n++;
    mbar_arrive_expect_tx(&full[s], kPage);
    bulk_g2s(smem + s * kPage, page(item[s]), kPage, &full[s]);
    ++loaded;
  }
  for (int i = 0; i < loaded; ++i) {
    const int st = i % S;
    if (!mbar_wait(&full[st], static_cast<uint32_t>(i / S) & 1u, &abort_flag)) {
      if (err) atomicOr(err, KDA_DEVERR_TIMEOUT);
      uint32_t z = 0;  // bounded drain of the loads still in flight
      for (int q = i + 1; q < loaded; ++q)
        (void)mbar_wait(&full[q % S], static_cast<uint32_t>(q / S) & 1u, &z);
      break;
    }
    bulk_s2g(page(item[st]), smem + st * kPage, kPage, pol);
    bulk_commit();
    if (i >= 1) {
      // Refill the stage of item i-1 once its store has read it.
      bulk_wait_read(1);
      n = next_live(n);
      if (n < n1) {
        const int ps = (i - 1) % S;
        item[ps] = n++;
        mbar_arrive_expect_tx(&full[ps], kPage);
        bulk_g2s(smem + ps * kPage, page(item[ps]), kPage, &full[ps]);
        ++loaded;
      }
    }
  }
  bulk_wait_all();
}

template <int S>
static int launch(const kda_probe_args *a, int grid, cudaStream_t stream) {
  if (cudaFuncSetAttribute(page_copy_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           S * kPage) != cudaSuccess)
    return KDA_ERR_LAUNCH;
  page_copy_kernel<S><<<grid, 32, S * kPage, stream>>>(
      a->state, a->slots, a->batch, a->heads, a->num_slots, a->err);
  return cudaGetLastError() == cudaSuccess ? KDA_SUCCESS : KDA_ERR_LAUNCH;
}

static int run(const kda_probe_args *a, cudaStream_t stream) {
  if (!a) return KDA_ERR_NULL_ARGS;
  if (a->batch < 0 || a->heads < 0 || a->num_slots < 1 || a->stages < 2 || a->stages > 3)
    return KDA_ERR_SHAPE;
  if (static_cast<int64_t>(a->batch) * a->heads > (int64_t(1) << 30)) return KDA_ERR_SHAPE;
  if (a->batch == 0 || a->heads == 0) return KDA_SUCCESS;
  if (!a->state || !a->slots) return KDA_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(a->state) & 15u) || (reinterpret_cast<uintptr_t>(a->slots) & 3u) ||
      (a->err && (reinterpret_cast<uintptr_t>(a->err) & 3u)))
    return KDA_ERR_ALIGNMENT;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KDA_ERR_DEVICE;
  if (major != 10 || minor != 3) return KDA_ERR_DEVICE;
  const int64_t items = static_cast<int64_t>(a->batch) * a->heads;
  const int grid = static_cast<int>(items < sms ? items : sms);
  return a->stages == 2 ? launch<2>(a, grid, stream) : launch<3>(a, grid, stream);
}

}  // namespace probe
}  // namespace kda

extern "C" int kda_probe_page_copy(const kda_probe_args *args, void *stream) {
  return kda::probe::run(args, static_cast<cudaStream_t>(stream));
}
