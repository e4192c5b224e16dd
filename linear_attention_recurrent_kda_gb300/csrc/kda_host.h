// Host-side helpers shared by the launchers of the KDA library: the facts of
// the current device, read once per device, and a kernel's shared-memory
// limit, raised once per device.  Both are safe to call from several host
// threads at once (the first call on a device does the work under a lock or
// std::call_once; later calls only read).
#pragma once
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace kda {

constexpr int kMaxDevices = 64;

struct DeviceFacts {
  int sms = 0;       // streaming multiprocessors
  int max_smem = 0;  // opt-in dynamic shared memory per block (bytes)
};

// The current device, when it is an sm_103 part, and its facts.  Returns
// false (nothing usable) otherwise.  Thread-safe.
inline bool current_device(int *dev_out, DeviceFacts *facts) {
  struct Entry {
    std::once_flag once;
    DeviceFacts facts;
    bool ok = false;
  };
  static Entry entries[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  Entry &e = entries[dev];
  std::call_once(e.once, [&] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&e.facts.sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&e.facts.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               dev) != cudaSuccess)
      return;
    e.ok = major == 10 && minor == 3;
  });
  if (!e.ok) return false;
  *dev_out = dev;
  *facts = e.facts;
  return true;
}

inline std::mutex &config_mutex() {
  static std::mutex m;
  return m;
}

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on device `dev`
// the first time it is asked for there (the attribute belongs to the device's
// context).  `done` is the caller's per-kernel flag array.  Thread-safe.
inline bool set_smem_limit_once(std::atomic<bool> (&done)[kMaxDevices], int dev,
                                const void *kernel, int bytes) {
  if (done[dev].load(std::memory_order_acquire)) return true;
  std::lock_guard<std::mutex> lock(config_mutex());
  if (done[dev].load(std::memory_order_relaxed)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  done[dev].store(true, std::memory_order_release);
  return true;
}

}  // namespace kda
