// devcache.h -- one-time host set-up per CUDA device.
//
// Kernel function attributes (cudaFuncSetAttribute) and occupancy figures
// belong to a device: a process that drives several GPUs must set and read
// them once per device, not once per process.  PerDevice<T> keeps one value
// per device ordinal, computed by the first call made with that device
// current; later calls read it without taking a lock.  Plain C++ (no CUDA
// headers), so the cache logic is testable on the host.
#pragma once
#include <atomic>
#include <mutex>

namespace trellis {

constexpr int kMaxDevices = 64;

template <typename T>
class PerDevice {
 public:
  // The value for device `dev` (0 <= dev < kMaxDevices): make() runs once per
  // device, under a lock, and its result is kept for every later call.
  // Returns `fallback` for an ordinal outside the table.
  template <typename F>
  T get(int dev, F make, T fallback) {
    if (dev < 0 || dev >= kMaxDevices) return fallback;
    if (ready_[dev].load(std::memory_order_acquire)) return value_[dev];
    std::lock_guard<std::mutex> lock(mu_);
    if (!ready_[dev].load(std::memory_order_relaxed)) {
      value_[dev] = make();
      ready_[dev].store(true, std::memory_order_release);
    }
    return value_[dev];
  }

 private:
  std::mutex mu_;
  std::atomic<bool> ready_[kMaxDevices] = {};
  T value_[kMaxDevices] = {};
};

}  // namespace trellis
