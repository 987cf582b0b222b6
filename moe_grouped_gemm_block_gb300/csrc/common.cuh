// common.cuh -- internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8gemm.h"

namespace fp8g {

// Per-device facts the launchers need, looked up once per device.
struct DeviceInfo {
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  unsigned int* status = nullptr;  // device address of this device's status word
  bool ok = false;
};

// Look up (and cache) the current device.  Returns FP8G_OK, FP8G_ERR_CUDA or
// FP8G_ERR_UNSUPPORTED_DEVICE (not sm_103).
int current_device(DeviceInfo** out);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
int encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                CUtensorMapSwizzle swizzle);

// Cycle budget of every device-side wait (clock64 ticks).  FP8G_WAIT_BUDGET_CYCLES overrides.
long long wait_budget_cycles();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Stream-K workspace: one FP32 partial-tile slot per SM (128 rows x 256 columns at most) and one
// flag per SM.  fp8_gemm_nt_noalloc uses a fixed scratch holding kNoAllocSlots slots and
// kNoAllocFlagBytes of flags (noalloc.cu); noalloc_scratch() returns its device address on `dev`
// (the current device), or null if the lookup failed.
constexpr size_t kSkSlotBytes = static_cast<size_t>(128) * 256 * 4;
constexpr int kNoAllocSlots = 160;
constexpr size_t kNoAllocFlagBytes = 1024;
constexpr size_t kNoAllocBytes = kSkSlotBytes * kNoAllocSlots + kNoAllocFlagBytes;
void* noalloc_scratch(int dev);

// Device-side: record the first error code in the status word.
__device__ __forceinline__ void record_status(unsigned int* status, unsigned int code) {
  atomicCAS(status, 0u, code);
}

}  // namespace fp8g
