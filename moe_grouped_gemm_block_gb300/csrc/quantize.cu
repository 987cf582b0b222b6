// quantize.cu -- bf16 -> e4m3 block quantisation with fp32 scales s = amax / 448.
//
// "DeepGEMM explainer" sec. 3.1: a block's scale is its amax divided by the largest FP8
// value; quantising divides by the scale.  "DeepGEMM FP8 walk-through" sec. 5.2: the
// scale can be max_val / 448.  Activations get one scale per row and 128-wide K block,
// weights one per 128x128 block (explainer sec. 5.1).
//
// Both kernels are HBM-bound (2 bytes read + 1 byte written per element): 16-byte
// coalesced loads, 8-byte coalesced stores, IEEE division (__fdiv_rn) and the
// round-to-nearest-even saturating e4m3 conversion.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8g {
namespace {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float amax8(const float (&f)[8]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

// 8 values / s -> 8 e4m3 bytes (little-endian: value 0 in the lowest byte).
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s) {
  if (s == 0.0f) return make_uint2(0u, 0u);
  uint32_t w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint16_t lo = cvt_e4m3x2(__fdiv_rn(f[4 * i + 1], s), __fdiv_rn(f[4 * i + 0], s));
    const uint16_t hi = cvt_e4m3x2(__fdiv_rn(f[4 * i + 3], s), __fdiv_rn(f[4 * i + 2], s));
    w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint2(w[0], w[1]);
}

// One half-warp (16 lanes x 8 values) per (row, 128-wide K block).  Each thread keeps
// UNROLL items in flight to cover HBM latency.
constexpr int kQThreads = 256;
constexpr int kQUnroll = 2;

__global__ void __launch_bounds__(kQThreads) quantize_1x128_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t M, int64_t KB, int64_t ldx,
    uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ sA, int64_t ld_sa) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;
  const int64_t half_id = (static_cast<int64_t>(blockIdx.x) * kQThreads + threadIdx.x) >> 4;
  const int64_t n_halves = static_cast<int64_t>(gridDim.x) * (kQThreads >> 4);
  const int64_t total = M * KB;
  for (int64_t base = half_id; base - half_id < total; base += n_halves * kQUnroll) {
    uint4 raw[kQUnroll];
    int64_t item[kQUnroll];
#pragma unroll
    for (int u = 0; u < kQUnroll; ++u) {
      item[u] = base + static_cast<int64_t>(u) * n_halves;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (item[u] < total) {
        const int64_t m = item[u] / KB, kb = item[u] - m * KB;
        raw[u] = __ldg(reinterpret_cast<const uint4*>(x + m * ldx + kb * 128 + sub * 8));
      }
    }
#pragma unroll
    for (int u = 0; u < kQUnroll; ++u) {
      float f[8];
      unpack8(raw[u], f);
      float a = amax8(f);
      // reduce over the 16 lanes of this half-warp (xor offsets < 16 stay inside it)
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
      const float s = __fdiv_rn(a, kE4M3Max);
      if (item[u] < total) {
        const int64_t m = item[u] / KB, kb = item[u] - m * KB;
        *reinterpret_cast<uint2*>(q + m * ldq + kb * 128 + sub * 8) = quant8(f, s);
        if (sub == 0) sA[kb * ld_sa + m] = s;
      }
    }
  }
}

// One CTA per (expert, 128-row block, 128-wide K block).  Thread t covers rows
// t/16 + 16*i (i = 0..7) and columns 8*(t%16) .. +7 of the block.
__global__ void __launch_bounds__(256) quantize_128x128_kernel(
    const __nv_bfloat16* __restrict__ w, int64_t N, int64_t K, uint8_t* __restrict__ q,
    float* __restrict__ sB) {
  const int64_t KB = K / 128, NB = (N + 127) / 128;
  const int64_t kb = blockIdx.x, nb = blockIdx.y, e = blockIdx.z;
  const int t = threadIdx.x;
  const int r0 = t >> 4, c = (t & 15) * 8;
  const __nv_bfloat16* wb = w + (e * N + nb * 128) * K + kb * 128 + c;
  uint8_t* qb = q + (e * N + nb * 128) * K + kb * 128 + c;
  const int rows = N - nb * 128 < 128 ? static_cast<int>(N - nb * 128) : 128;
  uint4 raw[8];
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + 16 * i;
    raw[i] = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) raw[i] = __ldg(reinterpret_cast<const uint4*>(wb + static_cast<int64_t>(r) * K));
    float f[8];
    unpack8(raw[i], f);
    a = fmaxf(a, amax8(f));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  __shared__ float red[8];
  if ((t & 31) == 0) red[t >> 5] = a;
  __syncthreads();
  float amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = __fdiv_rn(amax, kE4M3Max);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + 16 * i;
    if (r < rows) {
      float f[8];
      unpack8(raw[i], f);
      *reinterpret_cast<uint2*>(qb + static_cast<int64_t>(r) * K) = quant8(f, s);
    }
  }
  if (t == 0) sB[(e * NB + nb) * KB + kb] = s;
}

}  // namespace
}  // namespace fp8g

using namespace fp8g;

extern "C" int fp8_quantize_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, void* q,
                                  int64_t ldq, float* sA, int64_t ld_sa, void* stream) {
  if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq < K || ld_sa < M)
    return FP8G_ERR_INVALID_ARG;
  if (!x || !q || !sA) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sA) || ldx % 8 != 0 || ldq % 16 != 0 ||
      ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  if (M == 0) return FP8G_OK;
  const int64_t items = M * (K / 128);
  const int64_t per_block = (kQThreads / 16) * kQUnroll;
  int64_t blocks = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(dev->sm_count) * (2048 / kQThreads);
  if (blocks > cap) blocks = cap;
  quantize_1x128_kernel<<<static_cast<unsigned>(blocks), kQThreads, 0,
                          static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), M, K / 128, ldx, static_cast<uint8_t*>(q), ldq, sA,
      ld_sa);
  return cudaGetLastError() == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

extern "C" int fp8_quantize_128x128(const void* w, int64_t E, int64_t N, int64_t K, void* q,
                                    float* sB, void* stream) {
  if (E < 1 || N < 1 || K <= 0 || K % 128 != 0 || !w || !q || !sB) return FP8G_ERR_INVALID_ARG;
  if (E > 65535 || (N + 127) / 128 > 65535 || K / 128 > 0x7FFFFFFF) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q) || !aligned16(sB)) return FP8G_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>((N + 127) / 128),
            static_cast<unsigned>(E));
  quantize_128x128_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(w), N, K, static_cast<uint8_t*>(q), sB);
  return cudaGetLastError() == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}
