// Per-device, thread-safe one-time set-up.
//
// Some CUDA settings are recorded per device, not per process: a kernel's
// opt-in to more than 48 KB of dynamic shared memory
// (cudaFuncAttributeMaxDynamicSharedMemorySize) is one.  A process that drives
// several GPUs must make the call once on each of them, with that device
// current, and host threads may launch concurrently.  PerDeviceOnce runs a
// set-up function at most once per device id that succeeds; a failed set-up
// is retried on the next launch.  Plain host C++ (no CUDA types), so the
// bookkeeping can be tested on a machine without a GPU.
#pragma once

#include <atomic>
#include <mutex>

namespace ulysses {

template <int kMaxDevices = 64>
class PerDeviceOnce {
 public:
  // Runs `setup()` (returning 0 on success, an error code otherwise) unless
  // it already succeeded for `dev`.  Returns 0, setup()'s error code, or
  // `out_of_range` when dev is outside [0, kMaxDevices).
  template <class F>
  int run(int dev, F&& setup, int out_of_range) {
    if (dev < 0 || dev >= kMaxDevices) return out_of_range;
    if (done_[dev].load(std::memory_order_acquire)) return 0;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return 0;
    const int rc = setup();
    if (rc == 0) done_[dev].store(true, std::memory_order_release);
    return rc;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

}  // namespace ulysses
