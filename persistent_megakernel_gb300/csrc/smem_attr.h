// Per-device record of the dynamic shared-memory size a kernel has been allowed.
//
// cudaFuncSetAttribute(cudaFuncAttributeMaxDynamicSharedMemorySize) applies to the device that is
// current when it is called, so a process that launches on several devices must raise the limit
// on each of them; host threads that launch at once must not race on the record. Plain C++ (no
// CUDA types), so that a host-only test can drive it with a fake setter.
#pragma once

#include <cstddef>
#include <mutex>

namespace decimpl {

class SmemAttrCache {
 public:
  static constexpr int kMaxDevices = 64;

  // Make sure `bytes` of dynamic shared memory are allowed on device `dev`: calls set(bytes)
  // unless that device has already been given at least as much, and records the size when
  // set returns 0 (success). Devices outside [0, kMaxDevices) are set on every call. Returns
  // set's error code, or 0 when no call was needed.
  template <class SetFn>
  int ensure(int dev, size_t bytes, SetFn set) {
    std::lock_guard<std::mutex> lock(mu_);
    const bool tracked = dev >= 0 && dev < kMaxDevices;
    if (tracked && bytes <= allowed_[dev]) return 0;
    const int e = set(bytes);
    if (e == 0 && tracked) allowed_[dev] = bytes;
    return e;
  }

  size_t allowed(int dev) {
    std::lock_guard<std::mutex> lock(mu_);
    return dev >= 0 && dev < kMaxDevices ? allowed_[dev] : 0;
  }

 private:
  std::mutex mu_;
  size_t allowed_[kMaxDevices] = {};
};

}  // namespace decimpl
