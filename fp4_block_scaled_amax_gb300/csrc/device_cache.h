// Per-device, thread-safe memo of launch facts that are fixed for a device
// (SM count, an occupancy result, a kernel attribute already set), so that a
// process driving several GPUs, or several host threads, gets each device's
// own value.  A device index beyond the table is recomputed on every call.
#pragma once

#include <atomic>
#include <cuda_runtime.h>

namespace fp4lib {

constexpr int MAX_CACHED_DEVICES = 64;

// One int per device; 0 means "not known yet".  compute() must return the
// value (> 0) or a value <= 0 on failure, which is returned and not cached.
// Two threads may both compute a missing value; both store the same number.
struct DeviceInts {
  std::atomic<int> v[MAX_CACHED_DEVICES];
  DeviceInts() {
    for (auto& x : v) x.store(0, std::memory_order_relaxed);
  }
  template <class F>
  int get(F compute) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_CACHED_DEVICES) return compute();
    int x = v[dev].load(std::memory_order_acquire);
    if (x > 0) return x;
    x = compute();
    if (x > 0) v[dev].store(x, std::memory_order_release);
    return x;
  }
};

inline int current_sm_count() {
  static DeviceInts cache;
  return cache.get([] {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    return n;
  });
}

}  // namespace fp4lib
