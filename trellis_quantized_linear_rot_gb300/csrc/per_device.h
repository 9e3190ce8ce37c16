// Once-per-device set-up for host code (plain C++, no CUDA types).
//
// A kernel attribute such as its dynamic shared-memory limit belongs to the
// device that is current when it is set, so a process that drives several
// GPUs must set it once on each. PerDeviceOnce runs a set-up function the
// first time it is asked for a device and returns that first result (a CUDA
// error code as an int, 0 = success) on every later call for the same
// device; a failed set-up is retried on the next call. Calls may come from
// several host threads.
#pragma once

#include <atomic>
#include <mutex>

namespace tfx {

template <int kMaxDevices>
class PerDeviceOnce {
 public:
  // Returns f()'s result for `device` (run at most once while it succeeds),
  // or `bad_device` when the index is out of range.
  template <typename F>
  int run(int device, int bad_device, F&& f) {
    if (device < 0 || device >= kMaxDevices) return bad_device;
    if (done_[device].load(std::memory_order_acquire)) return 0;
    std::lock_guard<std::mutex> lock(mutex_);
    if (done_[device].load(std::memory_order_relaxed)) return 0;
    const int err = f();
    if (err == 0) done_[device].store(true, std::memory_order_release);
    return err;
  }

 private:
  std::mutex mutex_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

}  // namespace tfx
