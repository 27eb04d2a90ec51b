// Scratch for the allocation-free LM-head entry point (dec_lm_head_noalloc in api.cpp).
//
// The kernel's cross-CTA scratch for that call (step state, status word, argmax ticket, per-CTA
// argmax partials, the op descriptor) lives in this file-scope device array instead of a
// caller-allocated workspace. Every GPU that loads the library holds it until the process exits.
// In host code `g_noalloc_scratch` names a host-side stand-in, not device memory: the device
// address is looked up once per device with cudaGetSymbolAddress and only that address is handed
// to the kernel.
#include <cuda_runtime.h>

#include <mutex>

#include "dec_internal.h"

namespace decimpl {

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
}  // namespace

// Device address of the scratch array on the current device; the first call on a device looks it
// up (that device must be current, which it is: this runs on the caller's current device).
cudaError_t noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = a;
  }
  *ptr = g_addr[dev];
  return cudaSuccess;
}

}  // namespace decimpl
