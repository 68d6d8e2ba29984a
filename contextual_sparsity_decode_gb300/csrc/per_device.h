// A value computed once per CUDA device.
//
// Function attributes (the dynamic shared-memory limit, non-portable cluster
// sizes), occupancy answers and symbol addresses belong to one device, so a
// process that drives several GPUs needs one slot per device id rather than
// one process-wide flag.  Slots are atomics: two threads racing on the first
// call may both compute the value, which is harmless for every use here
// (setting an attribute twice, asking the same occupancy question twice).
//
// Plain C++ (no CUDA header), so the host-side logic can be tested on its own.
#pragma once

#include <atomic>
#include <climits>

namespace dv {

constexpr int kMaxDevices = 64;

class PerDevice {
 public:
  static constexpr int kUnset = INT_MIN;

  PerDevice() {
    for (auto& s : slot_) s.store(kUnset, std::memory_order_relaxed);
  }

  // The value for device `dev`, computing it with `compute()` on the first
  // request from that device.  Device ids outside [0, kMaxDevices) are not
  // cached: the value is computed on every call.
  template <typename F>
  int get(int dev, F&& compute) {
    if (dev < 0 || dev >= kMaxDevices) return compute();
    int v = slot_[dev].load(std::memory_order_acquire);
    if (v == kUnset) {
      v = compute();
      slot_[dev].store(v, std::memory_order_release);
    }
    return v;
  }

  // Whether device `dev` already has a value (for tests).
  bool known(int dev) const {
    return dev >= 0 && dev < kMaxDevices && slot_[dev].load(std::memory_order_acquire) != kUnset;
  }

 private:
  std::atomic<int> slot_[kMaxDevices];
};

}  // namespace dv
