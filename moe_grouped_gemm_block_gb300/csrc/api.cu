// api.cu -- device lookup, the per-device status word, tensor-map encoding and the
// status entry points of the C ABI.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace fp8g {

// One status word per device (each device that loads the library has its own copy).
__device__ unsigned int g_status_word;

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::once_flag g_device_once[kMaxDevices];
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

void init_device(int dev) {
  DeviceInfo& d = g_devices[dev];
  if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  d.status = static_cast<unsigned int*>(p);
  d.ok = true;
}
}  // namespace

int current_device(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FP8G_ERR_CUDA;
  }
  std::call_once(g_device_once[dev], init_device, dev);
  DeviceInfo& d = g_devices[dev];
  if (!d.ok) return FP8G_ERR_CUDA;
  if (d.cc_major != 10 || d.cc_minor != 3) return FP8G_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return FP8G_OK;
}

int encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  if (!g_encode) return FP8G_ERR_CUDA;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (uint32_t i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
  }
  for (uint32_t i = 0; i + 1 < rank; ++i) gstride[i] = strides_bytes[i];
  CUresult r = g_encode(map, dtype, rank, const_cast<void*>(base), gdim, gstride, bdim, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8G_OK : FP8G_ERR_CUDA;
}

long long wait_budget_cycles() {
  static const long long budget = [] {
    const char* e = std::getenv("FP8G_WAIT_BUDGET_CYCLES");
    long long v = e ? std::atoll(e) : 0;
    return v > 0 ? v : (2LL << 30);  // about one second at the SM clock
  }();
  return budget;
}

}  // namespace fp8g

extern "C" int fp8g_get_status(void* stream) {
  fp8g::DeviceInfo* d = nullptr;
  int st = fp8g::current_device(&d);
  if (st != FP8G_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  const unsigned int zero = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyAsync(&host, d->status, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return FP8G_ERR_CUDA;
  }
  return static_cast<int>(host);
}

extern "C" const char* fp8g_status_string(int code) {
  switch (code) {
    case FP8G_OK: return "FP8G_OK";
    case FP8G_ERR_INVALID_ARG: return "FP8G_ERR_INVALID_ARG";
    case FP8G_ERR_ALIGNMENT: return "FP8G_ERR_ALIGNMENT";
    case FP8G_ERR_UNSUPPORTED_DEVICE: return "FP8G_ERR_UNSUPPORTED_DEVICE";
    case FP8G_ERR_CUDA: return "FP8G_ERR_CUDA";
    case FP8G_ERR_TIMEOUT: return "FP8G_ERR_TIMEOUT";
    case FP8G_ERR_DEVICE_ASSERT: return "FP8G_ERR_DEVICE_ASSERT";
    default: return "FP8G_UNKNOWN_STATUS";
  }
}
