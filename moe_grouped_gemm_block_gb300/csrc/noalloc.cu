// noalloc.cu -- the fixed device scratch of fp8_gemm_nt_noalloc, in a translation unit of its own:
// with lazy module loading (the CUDA default) a device's copy of this module, and with it the
// array, is only created when the address lookup below first touches it, so callers of the other
// entry points do not pay for it.

#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace fp8g {
namespace {

// The stream-K slots of up to kNoAllocSlots SMs, then the flags.  Part of this module's device
// image, so using it allocates nothing.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kNoAllocDevices] = {};

}  // namespace

// Device address of the fixed scratch on device `dev` (the current device).  A successful lookup
// is kept; a failed one (for example while the caller's stream is being captured) is retried on
// the next call instead of being remembered.
void* noalloc_scratch(int dev) {
  if (dev < 0 || dev >= kNoAllocDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess) g_noalloc_addr[dev] = p;
    else cudaGetLastError();
  }
  return g_noalloc_addr[dev];
}

}  // namespace fp8g
