// quant_math.cuh -- the arithmetic of 1x128 block quantisation, shared by the quantisers and by
// the GEMM's fused quantise-and-multiply form (both must give the same codes and scales).
//
// "DeepGEMM explainer" sec. 3.1: a block's scale is its amax divided by the largest FP8 value;
// quantising divides by the scale.  "DeepGEMM FP8 walk-through" sec. 5.2: the scale can be
// max_val / 448.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp8g {
namespace {

constexpr float kE4M3Max = 448.0f;
constexpr float kE5M2Max = 57344.0f;

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

// The e4m3 codes of the IEEE quotients x / s, without a division for almost every element.
//
// With r = RN(1/s), the products y_lo = RN(x * RN(r (1 - 2^-20))) and y_hi = RN(x * RN(r (1 + 2^-20)))
// differ from the exact quotient q by a relative factor 1 -+ 2^-20 up to rounding errors below
// 3 * 2^-24, so RN(q) lies strictly between them.  Rounding to e4m3 (nearest-even, saturating)
// is monotone, so when y_lo and y_hi give the same code, that is the code of RN(q).  When any
// element of a group disagrees (an e4m3 decision point within 2^-20 of its quotient, about one
// element in 2^16), the whole group takes the IEEE division; so does every element when s is
// not a normal number (r would be inexact).
// Four values -> four e4m3 codes packed in one word (value 0 in the lowest byte).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a0, float a1, float a2, float a3) {
  uint32_t w;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(w)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return w;
}
// The same for e5m2 (gradients: 1-5-2 bits, largest finite value 57344).
__device__ __forceinline__ uint32_t cvt_e5m2x4(float a0, float a1, float a2, float a3) {
  uint32_t w;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 l, %2, %1;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 h, %4, %3;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(w)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return w;
}
enum CodeFormat : int { kE4M3 = 0, kE5M2 = 1 };
template <int FMT>
__device__ __forceinline__ uint32_t cvt_x4(float a0, float a1, float a2, float a3) {
  return FMT == kE5M2 ? cvt_e5m2x4(a0, a1, a2, a3) : cvt_e4m3x4(a0, a1, a2, a3);
}

// Direct path.  For most blocks a single product y = RN(x * r) with a fixed multiplier r already
// has the code of RN(x / s) for every bf16 x with |x| <= amax, and no bracket is needed.  Whether a
// given r works depends only on amax's 8-bit bf16 significand A (with s normal, s, 1/s, the
// products and the codes all scale exactly with a power-of-two change of amax and x, and so does r
// moved by whole ulps), so an exhaustive enumeration over A and every x settles it.  The kDirectMode
// words hold 2 bits per A (bits 2 (i % 16) of word i / 16, i = A - 128): 1 = r is RN(1/s) (102 of
// the 128 significands), 2 = RN(1/s) one ulp up (15), 3 = one ulp down (4), 0 = no single multiplier
// works (7): keep the bracket.  gen_quant_tables.py, next to this package, produces the table.
constexpr uint32_t kDirectMode0 = 0x55755655u, kDirectMode1 = 0x555B5555u,  // A = 128..143, 144..159
                   kDirectMode2 = 0x656585D5u, kDirectMode3 = 0x95544569u,  // A = 160..175, 176..191
                   kDirectMode4 = 0x58556495u, kDirectMode5 = 0x55555944u,  // A = 192..207, 208..223
                   kDirectMode6 = 0x55D55555u, kDirectMode7 = 0x55A65555u;  // A = 224..239, 240..255

// The block's direct-path mode (amax as a float holding a bf16 value; s its scale): 0 when the
// bracket is needed (or s is not normal).
__device__ __forceinline__ uint32_t direct_mode(float amax, float s) {
  const uint32_t a7 = (__float_as_uint(amax) >> 16) & 0x7Fu;  // amax's stored mantissa bits
  const uint32_t g = a7 >> 4;
  const uint32_t word = g < 4u ? (g < 2u ? (g == 0u ? kDirectMode0 : kDirectMode1)
                                         : (g == 2u ? kDirectMode2 : kDirectMode3))
                               : (g < 6u ? (g == 4u ? kDirectMode4 : kDirectMode5)
                                         : (g == 6u ? kDirectMode6 : kDirectMode7));
  return s >= 1.17549435e-38f ? (word >> (2u * (a7 & 15u))) & 3u : 0u;
}

// FMT e5m2: the bracket argument holds for any monotone round-to-nearest conversion; the direct
// path's table is e4m3's, so e5m2 callers pass mode 0.
template <int N, int FMT = kE4M3>
__device__ __forceinline__ void quant_n(const float (&f)[N], float s, uint32_t direct, uint32_t (&w)[N / 4]) {
  static_assert(N % 4 == 0, "N");
  if (s == 0.0f) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) w[i] = 0u;
    return;
  }
  bool exact = !(s >= 1.17549435e-38f);  // subnormal s: divide every element
  if (!exact && direct) {
    // RN(1/s), moved one ulp up (mode 2) or down (mode 3); r is a normal float here
    const float r = __uint_as_float(__float_as_uint(__frcp_rn(s)) + (direct == 2u) - (direct == 3u));
    const float2 r2 = make_float2(r, r);
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const float2 y01 = __fmul2_rn(make_float2(f[4 * i], f[4 * i + 1]), r2);
      const float2 y23 = __fmul2_rn(make_float2(f[4 * i + 2], f[4 * i + 3]), r2);
      w[i] = cvt_x4<FMT>(y01.x, y01.y, y23.x, y23.y);
    }
    return;
  }
  if (!exact) {
    const float r = __frcp_rn(s);
    const float lo_f = __fmul_rn(r, 1.0f - 0x1p-20f), hi_f = __fmul_rn(r, 1.0f + 0x1p-20f);
    const float2 rlo = make_float2(lo_f, lo_f), rhi = make_float2(hi_f, hi_f);
    uint32_t diff = 0;
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const float2 x01 = make_float2(f[4 * i], f[4 * i + 1]), x23 = make_float2(f[4 * i + 2], f[4 * i + 3]);
      const float2 l01 = __fmul2_rn(x01, rlo), l23 = __fmul2_rn(x23, rlo);
      const float2 h01 = __fmul2_rn(x01, rhi), h23 = __fmul2_rn(x23, rhi);
      w[i] = cvt_x4<FMT>(l01.x, l01.y, l23.x, l23.y);
      diff |= w[i] ^ cvt_x4<FMT>(h01.x, h01.y, h23.x, h23.y);
    }
    exact = diff != 0u;  // rare: some element sits within 2^-20 of a decision point
  }
  if (exact) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i)
      w[i] = cvt_x4<FMT>(__fdiv_rn(f[4 * i], s), __fdiv_rn(f[4 * i + 1], s), __fdiv_rn(f[4 * i + 2], s),
                        __fdiv_rn(f[4 * i + 3], s));
  }
}

__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s, uint32_t direct) {
  uint32_t w[2];
  quant_n<8>(f, s, direct, w);
  return make_uint2(w[0], w[1]);
}

// s = RN(amax / c) for c = 7 * 2^k (448, 57344) without a division: q = RN(amax * RN(1/c)) is
// within about one ulp of the quotient, so the nearest of q and its two neighbours is RN(amax / c).
// Their residuals amax - c * q' are exact in one FMA (amax has 8 significant bits and c * q' lies
// within a few ulps of it), and no quotient of a bf16 value by 7 * 2^k lies halfway between two
// floats (it is either exact or has a non-terminating binary expansion), so the smallest residual
// decides without ties.  Results below the normal range (amax < c * 2^-126) take the division.
// (An exhaustive check over every bf16 significand and exponent is in the tests.)
template <int FMT>
__device__ __forceinline__ float block_scale(float amax) {
  constexpr float c = FMT == kE5M2 ? kE5M2Max : kE4M3Max;
  constexpr float r = 1.0f / c;  // RN(1/c), folded by the compiler
  if (!(amax >= c * 1.17549435e-38f)) return __fdiv_rn(amax, c);  // zero, subnormal results
  const float q = __fmul_rn(amax, r);
  const float qd = __uint_as_float(__float_as_uint(q) - 1u), qu = __uint_as_float(__float_as_uint(q) + 1u);
  const float e = fabsf(__fmaf_rn(-c, q, amax)), ed = fabsf(__fmaf_rn(-c, qd, amax)),
              eu = fabsf(__fmaf_rn(-c, qu, amax));
  float best = q, eb = e;
  if (ed < eb) { best = qd; eb = ed; }
  if (eu < eb) best = qu;
  return best;
}

}  // namespace
}  // namespace fp8g
