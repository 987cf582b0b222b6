// quantize.cu -- bf16 -> e4m3 block quantisation with fp32 scales s = amax / 448.
//
// "DeepGEMM explainer" sec. 3.1: a block's scale is its amax divided by the largest FP8
// value; quantising divides by the scale.  "DeepGEMM FP8 walk-through" sec. 5.2: the
// scale can be max_val / 448.  Activations get one scale per row and 128-wide K block,
// weights one per 128x128 block (explainer sec. 5.1).
//
// Also here: the 1x128 quantiser's gathering form (rows taken through a row -> token map, built
// on the device from routed tokens by the layout kernels below), its masked-layout form (only each
// expert's valid rows) and its e5m2 form for gradients (s = amax / 57344); per-row and per-tensor
// scales (walk-through sec. 2.2).
//
// The quantisers are HBM-bound (2 bytes read + 1 byte written per element): 16-byte
// coalesced loads, 8-byte coalesced stores, the e4m3 code of the IEEE fp32 quotient x / s
// (a multiplication by 1/s, with the division kept for the rare elements where the two
// could round differently) and the round-to-nearest-even saturating e4m3 conversion.

#include <cuda_bf16.h>
#include <algorithm>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

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

// Eight lanes per (row, 128-wide K block); lane i of the group holds values 8i..8i+7 and
// 64+8i..64+8i+7, so each 16-byte load instruction of a warp reads four whole 128-byte lines
// (four lanes per block, each reading 64 contiguous bytes, measured twice as slow: every load
// instruction then touches sixteen half-used lines).  Each group keeps UNR blocks in flight: two in
// general, one for small inputs (the decode activations, 64 x 7168: 8.8 -> 6.8 us, spreading the
// few blocks over more threads); four measured slower on the MoE activations (43.6 against 41.6
// us, masked rows 33.4 against 29.3).
// The (row, K block) of an item advances by fixed steps: no integer division in the loop.
constexpr int kQThreads = 128;
constexpr int kQUnroll = 2;        // blocks in flight per group (UNR), in general
constexpr int64_t kQSmallItems = 16384;  // up to this many blocks: one in flight per group
constexpr int kQLanes = 8;  // lanes per block
constexpr int kQGroupsPerBlock = kQThreads / kQLanes;
// Grids of the 1x128 quantiser are capped at the blocks that are resident at once (the occupancy
// of the instantiation, looked up once per device): a grid larger than one wave would leave a
// partial last wave, measured 5-20% slower on the bench activations.

// (row, K block) of item i = row * KB + kb
struct RowKb {
  uint32_t m, kb;
};
__device__ __forceinline__ void advance(RowKb& p, uint32_t dm, uint32_t dkb, uint32_t KB) {
  p.m += dm;
  p.kb += dkb;
  if (p.kb >= KB) {
    p.kb -= KB;
    ++p.m;
  }
}

// SCATTER (route-gather-quantize): the M input rows are tokens; token m's codes and scales go to
// the output rows row_src[m * topk + j], j < topk (none where -1), so a token chosen by several
// experts is read and quantised once.  Afterwards every output row r < rows_out with
// zero_src[r] < 0 (group padding, rows past the last group) is written as a zero row: codes 0,
// scale 0.
// FMT: e4m3 (s = amax / 448) or e5m2 (gradients, s = amax / 57344).
// MASKED: rows are experts x cap and only rows r < row_src[e] of expert e (its count, clamped to
// [0, cap]) are quantised; the others are left as they are.  Grid row blockIdx.y is expert e,
// striding over that expert's valid (row, K block) items only.
template <bool SCATTER, int FMT = kE4M3, bool MASKED = false, int UNR = kQUnroll>
__global__ void __launch_bounds__(kQThreads) quantize_1x128_kernel(
    const __nv_bfloat16* __restrict__ x, uint32_t M, uint32_t KB, int64_t ldx,
    uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ sA, int64_t ld_sa,
    const int32_t* __restrict__ row_src, uint32_t cap = 0, uint32_t topk = 1,
    const int32_t* __restrict__ zero_src = nullptr, uint32_t rows_out = 0) {
  griddep_launch_dependents();  // a GEMM launched after this may start its prologue
  const int sub = threadIdx.x & (kQLanes - 1);
  const uint32_t group = (blockIdx.x * kQThreads + threadIdx.x) / kQLanes;
  const uint32_t n_groups = gridDim.x * kQGroupsPerBlock;
  uint32_t total = M * KB;  // the host guarantees M * KB < 2^31
  uint32_t row0 = 0;        // MASKED: the expert's first row
  if (MASKED) {
    const int32_t cnt = __ldg(row_src + blockIdx.y);
    total = static_cast<uint32_t>(min(max(cnt, 0), static_cast<int32_t>(cap))) * KB;
    row0 = blockIdx.y * cap;
  }
  // steps between this group's items: n_groups within a pass, n_groups * UNR between passes
  const uint32_t step_m = n_groups / KB, step_kb = n_groups - step_m * KB;
  const uint32_t pass = n_groups * UNR;
  const uint32_t pass_m = pass / KB, pass_kb = pass - pass_m * KB;
  RowKb p{group / KB, group - (group / KB) * KB};
  for (uint32_t base = group; base < total; base += pass, advance(p, pass_m, pass_kb, KB)) {
    uint4 raw[UNR][2];
    RowKb it[UNR];
    bool live[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      it[u] = p;
      if (u > 0) {
        it[u] = it[u - 1];
        advance(it[u], step_m, step_kb, KB);
      }
      live[u] = base + u * n_groups < total;
      raw[u][0] = raw[u][1] = make_uint4(0u, 0u, 0u, 0u);
      const int64_t src_row = it[u].m + row0;
      if (live[u]) {
        const __nv_bfloat16* src = x + src_row * ldx + it[u].kb * 128 + sub * 8;
        raw[u][0] = __ldg(reinterpret_cast<const uint4*>(src));
        raw[u][1] = __ldg(reinterpret_cast<const uint4*>(src + 64));
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float f[16], lo[8], hi[8];
      unpack8(raw[u][0], lo);
      unpack8(raw[u][1], hi);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        f[i] = lo[i];
        f[8 + i] = hi[i];
      }
      float a = fmaxf(amax8(lo), amax8(hi));
      // reduce over the 8 lanes of this group (xor offsets < 8 stay inside it)
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
      const float s = block_scale<FMT>(a);
      if (live[u]) {
        uint32_t c[4];
        quant_n<16, FMT>(f, s, FMT == kE4M3 ? direct_mode(a, s) : 0u, c);
        const uint32_t m = it[u].m + row0;
        if constexpr (SCATTER) {
          griddep_wait();  // the layout kernel's rows (at once after the first time)
          for (uint32_t j = 0; j < topk; ++j) {
            const int32_t r = __ldg(row_src + static_cast<int64_t>(m) * topk + j);
            if (r < 0) continue;
            uint8_t* dst = q + static_cast<int64_t>(r) * ldq + it[u].kb * 128 + sub * 8;
            *reinterpret_cast<uint2*>(dst) = make_uint2(c[0], c[1]);
            *reinterpret_cast<uint2*>(dst + 64) = make_uint2(c[2], c[3]);
            if (sub == 0) sA[static_cast<int64_t>(it[u].kb) * ld_sa + r] = s;
          }
        } else {
          uint8_t* dst = q + static_cast<int64_t>(m) * ldq + it[u].kb * 128 + sub * 8;
          *reinterpret_cast<uint2*>(dst) = make_uint2(c[0], c[1]);
          *reinterpret_cast<uint2*>(dst + 64) = make_uint2(c[2], c[3]);
          if (sub == 0) sA[static_cast<int64_t>(it[u].kb) * ld_sa + m] = s;
        }
      }
    }
  }
  if constexpr (SCATTER) {
    // zero rows, a warp per row (the rows written above are all mapped, so none is written twice)
    griddep_wait();
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t gwarp = (blockIdx.x * kQThreads + threadIdx.x) >> 5, nwarps = gridDim.x * (kQThreads / 32);
    for (uint32_t r = gwarp; r < rows_out; r += nwarps) {
      if (__ldg(zero_src + r) >= 0) continue;
      uint4* qr = reinterpret_cast<uint4*>(q + static_cast<int64_t>(r) * ldq);
      for (uint32_t v = lane; v < KB * 8u; v += 32u) qr[v] = make_uint4(0u, 0u, 0u, 0u);
      for (uint32_t kb = lane; kb < KB; kb += 32u) sA[static_cast<int64_t>(kb) * ld_sa + r] = 0.0f;
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
  const uint32_t direct = direct_mode(amax, s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + 16 * i;
    if (r < rows) {
      float f[8];
      unpack8(raw[i], f);
      *reinterpret_cast<uint2*>(qb + static_cast<int64_t>(r) * K) = quant8(f, s, direct);
    }
  }
  if (t == 0) sB[(e * NB + nb) * KB + kb] = s;
}

// ---------------------------------------------------------------- routing layout
// One CTA builds the contiguous grouped layout from the expert choices ids[T*k] (token-major):
// group_offsets[E+1] (each group's row count rounded up to 128), row_token[M_cap] (the token of
// each row; -1 for padding rows and for rows past the last group) and entry_row[T*k] (the row of
// each entry, its inverse; -1 for a dropped entry).  Inside a group the rows follow the entries'
// order, i.e. ascending tokens.  Ids outside [0, E) are dropped and flag FP8G_ERR_DEVICE_ASSERT;
// if the padded rows would not fit into M_cap, the layout is left empty (all offsets 0, every
// entry dropped) and the same status is raised.
// ---- per-token / per-channel (one scale per row over the whole K) and per-tensor scales
// ("DeepGEMM FP8 walk-through" sec. 2.2); same scale and code rules as the block forms.

// One CTA per row.  The row's 16-byte pieces are held in registers (rows of up to
// kRowThreads * kRowVec * 8 = 8192 values) between the amax reduction and the quantisation; longer
// rows read the rest again (from L1 / L2).  128 threads a row: with ~80 registers a thread, six
// rows (96 KB at K = 8192) are in flight per SM, against three rows of half the loads a thread
// with 256 threads a row (4096 x 8192: 32.7 us).
constexpr int kRowThreads = 128;
constexpr int kRowVec = 8;

__device__ __forceinline__ float block_amax(float a, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = a;
  __syncthreads();
  float m = 0.0f;
  for (int i = 0; i < nw; ++i) m = fmaxf(m, red[i]);
  return m;
}

__global__ void __launch_bounds__(kRowThreads) quantize_rows_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t K, int64_t ldx, uint8_t* __restrict__ q, int64_t ldq,
    float* __restrict__ s_out) {
  __shared__ float red[kRowThreads / 32];
  const int64_t m = blockIdx.x;
  const int t = threadIdx.x;
  const int64_t nvec = K / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(x + m * ldx);
  uint2* qr = reinterpret_cast<uint2*>(q + m * ldq);
  uint4 raw[kRowVec];
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < kRowVec; ++i) {
    const int64_t v = t + static_cast<int64_t>(i) * kRowThreads;
    raw[i] = v < nvec ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < kRowVec; ++i) {
    float f[8];
    unpack8(raw[i], f);
    a = fmaxf(a, amax8(f));
  }
  for (int64_t v = t + kRowVec * kRowThreads; v < nvec; v += kRowThreads) {
    float f[8];
    unpack8(__ldg(xr + v), f);
    a = fmaxf(a, amax8(f));
  }
  const float amax = block_amax(a, red);
  const float s = __fdiv_rn(amax, kE4M3Max);
  const uint32_t direct = direct_mode(amax, s);
#pragma unroll
  for (int i = 0; i < kRowVec; ++i) {
    const int64_t v = t + static_cast<int64_t>(i) * kRowThreads;
    if (v < nvec) {
      float f[8];
      unpack8(raw[i], f);
      qr[v] = quant8(f, s, direct);
    }
  }
  for (int64_t v = t + kRowVec * kRowThreads; v < nvec; v += kRowThreads) {
    float f[8];
    unpack8(__ldg(xr + v), f);
    qr[v] = quant8(f, s, direct);
  }
  if (t == 0) s_out[m] = s;
}

// Per-tensor, pass 1: tensor e = blockIdx.y (rows e*M .. e*M+M-1).  Each CTA raises s[e] to
// RN(amax_cta / 448) with an integer max on the bits: for non-negative floats the bit order is
// the value order, and RN(a / 448) is non-decreasing in a, so the largest of the CTAs' values is
// RN(amax / 448) of the whole tensor.  s[e] starts at +0.
constexpr int kTensorThreads = 256;
constexpr int kTensorUnroll = 8;  // independent 16-byte loads in flight per thread

// A thread's pieces (8 values) of tensor e: p, p + S, p + 2S, ... of the tensor's M x kvec pieces
// (row-major), as (row, piece) pairs stepped without a division per piece.
struct PieceWalk {
  uint32_t r, v, sr, sv;
  __device__ __forceinline__ PieceWalk(uint32_t p, uint32_t S, uint32_t kvec)
      : r(p / kvec), v(p - (p / kvec) * kvec), sr(S / kvec), sv(S - (S / kvec) * kvec) {}
  __device__ __forceinline__ void step(uint32_t kvec) {
    r += sr;
    v += sv;
    if (v >= kvec) {
      v -= kvec;
      ++r;
    }
  }
};

__global__ void __launch_bounds__(kTensorThreads) tensor_scale_kernel(
    const __nv_bfloat16* __restrict__ x, uint32_t M, uint32_t kvec, int64_t ldx, float* __restrict__ s) {
  __shared__ float red[kTensorThreads / 32];
  griddep_launch_dependents();  // pass 2 may start loading its pieces (it waits before reading s)
  const uint32_t e = blockIdx.y;
  const __nv_bfloat16* xe = x + static_cast<int64_t>(e) * M * ldx;
  float a = 0.0f;
  PieceWalk w(blockIdx.x * kTensorThreads + threadIdx.x, gridDim.x * kTensorThreads, kvec);
  while (w.r < M) {
    uint4 raw[kTensorUnroll];
#pragma unroll
    for (int u = 0; u < kTensorUnroll; ++u) {
      raw[u] = w.r < M ? __ldg(reinterpret_cast<const uint4*>(xe + static_cast<int64_t>(w.r) * ldx) + w.v)
                       : make_uint4(0u, 0u, 0u, 0u);
      w.step(kvec);
    }
#pragma unroll
    for (int u = 0; u < kTensorUnroll; ++u) {
      float f[8];
      unpack8(raw[u], f);
      a = fmaxf(a, amax8(f));
    }
  }
  const float amax = block_amax(a, red);
  if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(s) + e, __float_as_uint(__fdiv_rn(amax, kE4M3Max)));
}

// Per-tensor, pass 2: the codes with the tensor's scale.  The direct-product test needs amax's
// bf16 significand, recovered from s: for s normal, s * 448 is within 2^-23 (relative) of amax,
// far inside half a bf16 step, so rounding it to bf16 gives amax back.  (For s subnormal or zero
// the test is not used.)
//
// Launched as a programmatic dependent of pass 1: its CTAs may start while pass 1 runs and load
// their first pieces (the input is not pass 1's output), then wait for pass 1 before reading s.
__global__ void __launch_bounds__(kTensorThreads) quantize_tensor_kernel(
    const __nv_bfloat16* __restrict__ x, uint32_t M, uint32_t kvec, int64_t ldx, uint8_t* __restrict__ q,
    int64_t ldq, const float* __restrict__ s_in) {
  const uint32_t e = blockIdx.y;
  const __nv_bfloat16* xe = x + static_cast<int64_t>(e) * M * ldx;
  uint8_t* qe = q + static_cast<int64_t>(e) * M * ldq;
  PieceWalk w(blockIdx.x * kTensorThreads + threadIdx.x, gridDim.x * kTensorThreads, kvec);
  bool first = true;
  float s = 0.0f;
  uint32_t direct = 0;
  while (w.r < M) {
    uint4 raw[kTensorUnroll];
    uint32_t rr[kTensorUnroll], vv[kTensorUnroll];
#pragma unroll
    for (int u = 0; u < kTensorUnroll; ++u) {
      rr[u] = w.r;
      vv[u] = w.v;
      raw[u] = w.r < M ? __ldg(reinterpret_cast<const uint4*>(xe + static_cast<int64_t>(w.r) * ldx) + w.v)
                       : make_uint4(0u, 0u, 0u, 0u);
      w.step(kvec);
    }
    if (first) {  // pass 1's scale, once its grid has finished
      first = false;
      griddep_wait();
      s = __ldcg(s_in + e);  // (written by pass 1 while this grid may already run: not the read-only path)
      const float amax = __bfloat162float(__float2bfloat16_rn(__fmul_rn(s, kE4M3Max)));
      direct = direct_mode(amax, s);
    }
#pragma unroll
    for (int u = 0; u < kTensorUnroll; ++u) {
      if (rr[u] < M) {
        float f[8];
        unpack8(raw[u], f);
        reinterpret_cast<uint2*>(qe + static_cast<int64_t>(rr[u]) * ldq)[vv[u]] = quant8(f, s, direct);
      }
    }
  }
}

constexpr int kRouteThreads = 1024;
constexpr int kRouteMaxExperts = 2048;
constexpr int kRouteChunk = 4096;  // entries staged in shared memory per pass of the assigning warp

__global__ void __launch_bounds__(kRouteThreads) route_layout_kernel(
    const int32_t* __restrict__ ids, int32_t n, int32_t topk, int32_t E, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_token, int32_t* __restrict__ entry_row, int64_t M_cap, unsigned int* status) {
  __shared__ int32_t s_count[kRouteMaxExperts];     // per-expert counts, then running ranks
  __shared__ int32_t s_off[kRouteMaxExperts + 1];   // padded prefix
  __shared__ int32_t s_chunk[kRouteChunk];
  __shared__ int32_t s_warp[kRouteThreads / 32];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_launch_dependents();  // the quantiser may start loading tokens (it waits before its stores)
  for (int e = tid; e < E; e += kRouteThreads) s_count[e] = 0;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int32_t i = tid; i < n; i += kRouteThreads) {
    const int32_t e = __ldg(ids + i);
    if (e >= 0 && e < E) atomicAdd(&s_count[e], 1);
    else s_bad = 1;
  }
  __syncthreads();
  // exclusive scan of the padded counts: thread tid covers experts [tid*per, tid*per + per)
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  int32_t local = 0;
  for (int j = 0; j < per; ++j) {
    const int e = tid * per + j;
    if (e < E) local += (s_count[e] + 127) / 128 * 128;
  }
  int32_t incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += v;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int32_t run = (warp > 0 ? s_warp[warp - 1] : 0) + incl - local;  // exclusive start of this thread
  for (int j = 0; j < per; ++j) {
    const int e = tid * per + j;
    if (e < E) {
      s_off[e] = run;
      run += (s_count[e] + 127) / 128 * 128;
    }
  }
  if (tid == kRouteThreads - 1) s_off[E] = s_warp[31];
  __syncthreads();
  const bool fits = static_cast<int64_t>(s_off[E]) <= M_cap;
  for (int e = tid; e <= E; e += kRouteThreads) offsets[e] = fits ? s_off[e] : 0;
  for (int64_t r = tid; r < M_cap; r += kRouteThreads) row_token[r] = -1;
  if (!fits)
    for (int32_t i = tid; i < n; i += kRouteThreads) entry_row[i] = -1;
  for (int e = tid; e < E; e += kRouteThreads) s_count[e] = 0;  // now: rows handed out per expert
  __syncthreads();
  // rows in entry order: one warp walks the entries 32 at a time; lanes choosing the same expert
  // take consecutive rows in lane order (match_any), the last of them advances the expert's count
  for (int32_t c0 = 0; fits && c0 < n; c0 += kRouteChunk) {
    const int32_t cn = n - c0 < kRouteChunk ? n - c0 : kRouteChunk;
    for (int32_t i = tid; i < cn; i += kRouteThreads) s_chunk[i] = __ldg(ids + c0 + i);
    __syncthreads();
    if (warp == 0) {
      for (int32_t b = 0; b < cn; b += 32) {
        const int32_t i = b + lane;
        int32_t e = i < cn ? s_chunk[i] : -1;
        if (e < 0 || e >= E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0) {
          const int32_t r = s_off[e] + s_count[e] + rank;
          row_token[r] = (c0 + i) / topk;
          entry_row[c0 + i] = r;
        } else if (i < cn) {
          entry_row[c0 + i] = -1;
        }
        __syncwarp();
        if (e >= 0 && (peers >> lane) == 1u) s_count[e] += __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
  }
  if (tid == 0 && (s_bad || !fits)) record_status(status, FP8G_ERR_DEVICE_ASSERT);
}

// The same layout for E <= 256 with all 32 warps assigning rows: warp w takes the contiguous
// entry range [w*L, (w+1)*L) and keeps its own per-expert counts; an exclusive scan over the
// warps gives each warp its first row per expert, so rows still follow the entries' order.
constexpr int kRouteSmallExperts = 256;

__global__ void __launch_bounds__(kRouteThreads) route_layout_small_kernel(
    const int32_t* __restrict__ ids, int32_t n, int32_t topk, int32_t E, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_token, int32_t* __restrict__ entry_row, int64_t M_cap, unsigned int* status) {
  constexpr int W = kRouteThreads / 32;
  __shared__ int32_t s_wcnt[W][kRouteSmallExperts];  // counts, then each warp's first rank
  __shared__ int32_t s_off[kRouteSmallExperts + 1];
  __shared__ int32_t s_tot[kRouteSmallExperts];       // entries per expert
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_launch_dependents();  // the quantiser may start loading tokens (it waits before its stores)
  for (int i = tid; i < W * E; i += kRouteThreads) s_wcnt[i / E][i % E] = 0;  // the counters in use
  if (tid == 0) s_bad = 0;
  __syncthreads();
  const int32_t L = (n + W - 1) / W;
  const int32_t lo = warp * L, hi = min(n, lo + L);
  // the first kIdCache * 32 entries of the warp's range are loaded once, all at the same time, and
  // kept in registers for the row assignment below (a warp's range of 8192 top-2 entries is 256)
  constexpr int kIdCache = 16;
  int32_t idc[kIdCache];
#pragma unroll
  for (int j = 0; j < kIdCache; ++j) {
    const int32_t i = lo + lane + 32 * j;
    idc[j] = i < hi ? __ldg(ids + i) : 0;
  }
#pragma unroll
  for (int j = 0; j < kIdCache; ++j) {
    if (lo + lane + 32 * j < hi) {
      if (idc[j] >= 0 && idc[j] < E) atomicAdd(&s_wcnt[warp][idc[j]], 1);
      else s_bad = 1;
    }
  }
  for (int32_t i = lo + lane + 32 * kIdCache; i < hi; i += 32) {
    const int32_t e = __ldg(ids + i);
    if (e >= 0 && e < E) atomicAdd(&s_wcnt[warp][e], 1);
    else s_bad = 1;
  }
  __syncthreads();
  static_assert(W == 32, "one lane per warp in the scan below");
  for (int e = warp; e < E; e += W) {  // per expert (a warp each): exclusive scan over the warps
    const int32_t c = s_wcnt[lane][e];
    int32_t incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    s_wcnt[lane][e] = incl - c;
    if (lane == 31) s_tot[e] = incl;
  }
  __syncthreads();
  if (warp == 0) {  // padded counts -> exclusive prefix (8 experts per lane)
    int32_t v[kRouteSmallExperts / 32];
    int32_t local = 0;
#pragma unroll
    for (int j = 0; j < kRouteSmallExperts / 32; ++j) {
      const int e = lane * (kRouteSmallExperts / 32) + j;
      v[j] = e < E ? (s_tot[e] + 127) / 128 * 128 : 0;
      local += v[j];
    }
    int32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += u;
    }
    int32_t run = incl - local;
    const int32_t total = __shfl_sync(0xffffffffu, incl, 31);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kRouteSmallExperts / 32; ++j) {
      const int e = lane * (kRouteSmallExperts / 32) + j;
      if (e < E) s_off[e] = run;
      run += v[j];
    }
    if (lane == 0) s_off[E] = total;
  }
  __syncthreads();
  const bool fits = static_cast<int64_t>(s_off[E]) <= M_cap;
  for (int e = tid; e <= E; e += kRouteThreads) offsets[e] = fits ? s_off[e] : 0;
  // token -1 for the padding rows only (every other row is written below): each group's rows past
  // its entries, and the rows past the last group
  if (fits) {
    for (int e = 0; e < E; ++e)
      for (int32_t r = s_off[e] + s_tot[e] + tid; r < s_off[e + 1]; r += kRouteThreads) row_token[r] = -1;
    for (int64_t r = s_off[E] + tid; r < M_cap; r += kRouteThreads) row_token[r] = -1;
  } else {
    for (int64_t r = tid; r < M_cap; r += kRouteThreads) row_token[r] = -1;
    for (int32_t i = tid; i < n; i += kRouteThreads) entry_row[i] = -1;
  }
  if (fits) {
    // 32 entries at a time (warp-uniform): lanes choosing the same expert take consecutive rows in
    // lane order (match_any); the last of them advances the warp's count for that expert.  The
    // match_any of the cached chunks are independent and issued first; only the count updates run
    // chunk after chunk.
    auto assign = [&](int32_t b, int32_t e, unsigned peers) {
      const int32_t i = b + lane;
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (e >= 0) {
        const int32_t r = s_off[e] + s_wcnt[warp][e] + rank;
        row_token[r] = i / topk;
        entry_row[i] = r;
      } else if (i < hi) {
        entry_row[i] = -1;
      }
      __syncwarp();
      if (e >= 0 && (peers >> lane) == 1u) s_wcnt[warp][e] += __popc(peers);
      __syncwarp();
    };
    unsigned pe[kIdCache];
#pragma unroll
    for (int j = 0; j < kIdCache; ++j) {
      const int32_t i = lo + 32 * j + lane;
      if (i >= hi || idc[j] < 0 || idc[j] >= E) idc[j] = -1;
      pe[j] = lo + 32 * j < hi ? __match_any_sync(0xffffffffu, idc[j]) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kIdCache; ++j) {
      if (lo + 32 * j >= hi) break;
      assign(lo + 32 * j, idc[j], pe[j]);
    }
    for (int32_t b = lo + 32 * kIdCache; b < hi; b += 32) {
      int32_t e = b + lane < hi ? __ldg(ids + b + lane) : -1;
      if (e < 0 || e >= E) e = -1;
      assign(b, e, __match_any_sync(0xffffffffu, e));
    }
  }
  if (tid == 0 && (s_bad || !fits)) record_status(status, FP8G_ERR_DEVICE_ASSERT);
}

// Resident blocks of `kern` (kQThreads threads, no dynamic shared memory) across the device.
template <typename Kernel>
int64_t resident_blocks(Kernel kern, const DeviceInfo* dev) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kQThreads, 0) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  return static_cast<int64_t>(per_sm) * dev->sm_count;
}

}  // namespace
}  // namespace fp8g

using namespace fp8g;

extern "C" int fp8_quantize_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, void* q,
                                  int64_t ldq, float* sA, int64_t ld_sa, void* stream) {
  if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq < K || ld_sa < M)
    return FP8G_ERR_INVALID_ARG;
  if (M == 0) return FP8G_OK;  // nothing to do; the pointers of empty tensors may be null
  if (!x || !q || !sA) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sA) || ldx % 8 != 0 || ldq % 16 != 0 ||
      ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  const int64_t items = M * (K / 128);
  if (items >= (int64_t{1} << 31) || M > 0x7FFFFFFF) return FP8G_ERR_INVALID_ARG;
  if (items <= kQSmallItems) {
    const int64_t blocks = (items + kQGroupsPerBlock - 1) / kQGroupsPerBlock;
    quantize_1x128_kernel<false, kE4M3, false, 1><<<static_cast<unsigned>(blocks), kQThreads, 0,
                                                    static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<uint32_t>(M), static_cast<uint32_t>(K / 128), ldx,
        static_cast<uint8_t*>(q), ldq, sA, ld_sa, nullptr);
    return cudaGetLastError() == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
  }
  const int64_t per_block = kQGroupsPerBlock * kQUnroll;
  int64_t blocks = (items + per_block - 1) / per_block;
  static const int64_t cap = resident_blocks(quantize_1x128_kernel<false>, dev);
  if (blocks > cap) blocks = cap;
  quantize_1x128_kernel<false><<<static_cast<unsigned>(blocks), kQThreads, 0,
                                 static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<uint32_t>(M), static_cast<uint32_t>(K / 128), ldx,
      static_cast<uint8_t*>(q), ldq, sA, ld_sa, nullptr);
  return cudaGetLastError() == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

extern "C" int fp8_quantize_1x128_masked(const void* x, int32_t E, int64_t cap, int64_t K,
                                         const int32_t* masked_m, void* q, float* sA, int64_t ld_sa,
                                         void* stream) {
  if (E < 1 || cap < 0 || K <= 0 || K % 128 != 0 || static_cast<int64_t>(E) * cap > 0x7FFFFFFF ||
      ld_sa < static_cast<int64_t>(E) * cap)
    return FP8G_ERR_INVALID_ARG;
  if (cap == 0) return FP8G_OK;
  if (!x || !q || !sA || !masked_m) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sA) || ld_sa % 4 != 0 ||
      (reinterpret_cast<uintptr_t>(masked_m) & 3u))
    return FP8G_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  const int64_t M = static_cast<int64_t>(E) * cap;
  const int64_t items = M * (K / 128);
  if (items >= (int64_t{1} << 31) || E > 65535) return FP8G_ERR_INVALID_ARG;
  // one grid row per expert, sized for a full expert; CTAs past an expert's count exit at once.
  // Capped at twice the resident blocks over all experts: the counts differ between experts, so
  // one wave's worth (each expert's blocks striding over its rows) leaves the fullest experts
  // last (MoE masked activations, 32 experts x 256 rows x 7168: 37.5 us at one wave, 33.4 us at
  // two or uncapped).
  const int64_t per_block = kQGroupsPerBlock * kQUnroll;
  int64_t bx = (cap * (K / 128) + per_block - 1) / per_block;
  static const int64_t resident = resident_blocks(quantize_1x128_kernel<false, kE4M3, true>, dev);
  const int64_t limit = std::max<int64_t>(1, 2 * resident / E);
  if (bx > limit) bx = limit;
  const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(E));
  quantize_1x128_kernel<false, kE4M3, true><<<grid, kQThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<uint32_t>(M), static_cast<uint32_t>(K / 128), K,
      static_cast<uint8_t*>(q), K, sA, ld_sa, masked_m, static_cast<uint32_t>(cap));
  return cudaGetLastError() == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

extern "C" int fp8_quantize_1x128_e5m2(const void* x, int64_t M, int64_t K, int64_t ldx, void* q,
                                       int64_t ldq, float* sA, int64_t ld_sa, void* stream) {
  if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq < K || ld_sa < M)
    return FP8G_ERR_INVALID_ARG;
  if (M == 0) return FP8G_OK;
  if (!x || !q || !sA) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sA) || ldx % 8 != 0 || ldq % 16 != 0 ||
      ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  const int64_t items = M * (K / 128);
  if (items >= (int64_t{1} << 31) || M > 0x7FFFFFFF) return FP8G_ERR_INVALID_ARG;
  const int64_t per_block = kQGroupsPerBlock * kQUnroll;
  int64_t blocks = (items + per_block - 1) / per_block;
  static const int64_t cap = resident_blocks(quantize_1x128_kernel<false, kE5M2>, dev);
  if (blocks > cap) blocks = cap;
  quantize_1x128_kernel<false, kE5M2><<<static_cast<unsigned>(blocks), kQThreads, 0,
                                        static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<uint32_t>(M), static_cast<uint32_t>(K / 128), ldx,
      static_cast<uint8_t*>(q), ldq, sA, ld_sa, nullptr);
  return cudaGetLastError() == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

// The same layout computed by several CTAs (at most 32 experts, the routing of a batch of
// tokens).  Entry i of expert e goes to row offsets[e] + (entries of e before i), exactly as in
// the one-CTA kernels above; CTA c assigns the entries [c C, (c+1) C) only.  Every CTA counts all
// entries (n ids, from L2): the totals give the same padded offsets in each CTA, and the counts
// before its range its rows' base.  Then its 32 warps take one slice of its range each.  The
// one-CTA kernel's row assignment walked 256 entries a warp for 8192 entries; here a warp walks
// n / (32 G).  8192 entries of 8 experts: 7.1 us against 11.6 (ncu), and the call with its
// quantiser 35.5 against 36.9 us.  (The quantiser waits for the layout before its first store,
// so only the layout's own time comes off.)
constexpr int kRouteChunkExperts = 32;
constexpr int kRouteChunkCtas = 8;
constexpr int32_t kRouteChunkMinEntries = 2048;  // smaller layouts keep the one-CTA kernel

__global__ void __launch_bounds__(kRouteThreads) route_layout_chunked_kernel(
    const int32_t* __restrict__ ids, int32_t n, int32_t topk, int32_t E, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_token, int32_t* __restrict__ entry_row, int64_t M_cap, unsigned int* status) {
  constexpr int W = kRouteThreads / 32;
  constexpr int XE = kRouteChunkExperts;
  __shared__ int32_t s_all[W][XE];   // per warp: entries of each expert (all of them)
  __shared__ int32_t s_pre[W][XE];   // per warp: entries of each expert before this CTA's range
  __shared__ int32_t s_wcnt[W][XE];  // this CTA's warps: counts in their slices, then their first ranks
  __shared__ int32_t s_tot[XE], s_base[XE], s_off[XE + 1];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_launch_dependents();  // the quantiser may start loading tokens (it waits before its stores)
  const int32_t C = (n + static_cast<int32_t>(gridDim.x) - 1) / static_cast<int32_t>(gridDim.x);
  const int32_t clo = min(n, static_cast<int32_t>(blockIdx.x) * C), chi = min(n, clo + C);
  for (int i = tid; i < W * XE; i += kRouteThreads) {
    (&s_all[0][0])[i] = 0;
    (&s_pre[0][0])[i] = 0;
    (&s_wcnt[0][0])[i] = 0;
  }
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // eight ids a thread loaded at once, then counted (one load latency per pass, not eight)
  constexpr int kIdBatch = 8;
  for (int32_t b0 = 0; b0 < n; b0 += kIdBatch * kRouteThreads) {
    int32_t ev[kIdBatch];
#pragma unroll
    for (int j = 0; j < kIdBatch; ++j) {
      const int32_t i = b0 + j * kRouteThreads + tid;
      ev[j] = i < n ? __ldg(ids + i) : 0;
    }
#pragma unroll
    for (int j = 0; j < kIdBatch; ++j) {
      const int32_t i = b0 + j * kRouteThreads + tid;
      if (i >= n) continue;
      if (ev[j] >= 0 && ev[j] < E) {
        atomicAdd(&s_all[warp][ev[j]], 1);
        if (i < clo) atomicAdd(&s_pre[warp][ev[j]], 1);
      } else {
        s_bad = 1;
      }
    }
  }
  // this CTA's range: warp w takes the slice [lo, hi); its first kIdCache * 32 ids stay in registers
  // for the row assignment
  const int32_t L = (chi - clo + W - 1) / W;
  const int32_t lo = min(chi, clo + warp * L), hi = min(chi, lo + L);
  constexpr int kIdCache = 4;
  int32_t idc[kIdCache];
#pragma unroll
  for (int j = 0; j < kIdCache; ++j) {
    const int32_t i = lo + 32 * j + lane;
    idc[j] = i < hi ? __ldg(ids + i) : -1;
    if (idc[j] < 0 || idc[j] >= E) idc[j] = -1;
  }
#pragma unroll
  for (int j = 0; j < kIdCache; ++j)
    if (idc[j] >= 0) atomicAdd(&s_wcnt[warp][idc[j]], 1);
  for (int32_t i = lo + 32 * kIdCache + lane; i < hi; i += 32) {
    const int32_t e = __ldg(ids + i);
    if (e >= 0 && e < E) atomicAdd(&s_wcnt[warp][e], 1);
  }
  __syncthreads();
  static_assert(W == 32 && XE <= 32, "one lane per warp and per expert below");
  for (int e = warp; e < E; e += W) {  // per expert (a warp each): sums and the scan over the warps
    const int32_t c = s_wcnt[lane][e];
    int32_t incl = c, all = s_all[lane][e], pre = s_pre[lane][e];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      all += __shfl_xor_sync(0xffffffffu, all, off);
      pre += __shfl_xor_sync(0xffffffffu, pre, off);
    }
    s_wcnt[lane][e] = incl - c;
    if (lane == 0) {
      s_tot[e] = all;
      s_base[e] = pre;
    }
  }
  __syncthreads();
  if (warp == 0) {  // padded counts -> exclusive prefix, one expert a lane
    const int32_t v = lane < E ? (s_tot[lane] + 127) / 128 * 128 : 0;
    int32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += u;
    }
    if (lane < E) s_off[lane] = incl - v;
    if (lane == 31) s_off[E] = incl;
  }
  __syncthreads();
  const bool fits = static_cast<int64_t>(s_off[E]) <= M_cap;
  if (blockIdx.x == 0) {
    for (int e = tid; e <= E; e += kRouteThreads) offsets[e] = fits ? s_off[e] : 0;
    if (fits) {  // token -1 for the padding rows only (every other row is written below)
      for (int e = 0; e < E; ++e)
        for (int32_t r = s_off[e] + s_tot[e] + tid; r < s_off[e + 1]; r += kRouteThreads) row_token[r] = -1;
      for (int64_t r = s_off[E] + tid; r < M_cap; r += kRouteThreads) row_token[r] = -1;
    }
    if (tid == 0 && (s_bad || !fits)) record_status(status, FP8G_ERR_DEVICE_ASSERT);
  }
  if (!fits) {  // an empty layout: every row padding, every entry dropped
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kRouteThreads;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kRouteThreads + tid; r < M_cap; r += stride) row_token[r] = -1;
    for (int32_t i = clo + tid; i < chi; i += kRouteThreads) entry_row[i] = -1;
    return;
  }
  // 32 entries at a time: lanes choosing the same expert take consecutive rows in lane order
  for (int32_t b = lo, j = 0; b < hi; b += 32, ++j) {
    const int32_t i = b + lane;
    int32_t e = -1;
    if (j < kIdCache) {
#pragma unroll
      for (int u = 0; u < kIdCache; ++u)
        if (u == j) e = idc[u];
    } else {
      e = i < hi ? __ldg(ids + i) : -1;
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0) {
      const int32_t r = s_off[e] + s_base[e] + s_wcnt[warp][e] + rank;
      row_token[r] = i / topk;
      entry_row[i] = r;
    } else if (i < hi) {
      entry_row[i] = -1;
    }
    __syncwarp();
    if (e >= 0 && (peers >> lane) == 1u) s_wcnt[warp][e] += __popc(peers);
    __syncwarp();
  }
}

extern "C" int fp8_route_gather_quantize_1x128(const void* x, int64_t T, int64_t K, int64_t ldx,
                                               const int32_t* topk_ids, int32_t topk, int32_t E,
                                               void* q, int64_t ldq, float* sA, int64_t ld_sa,
                                               int32_t* group_offsets, int32_t* row_token,
                                               int32_t* entry_row, int64_t M_cap, void* stream) {
  if (T < 0 || T > 0x7FFFFFFF || K <= 0 || K % 128 != 0 || topk < 1 || E < 1 ||
      E > kRouteMaxExperts || ldx < K || ldq < K)
    return FP8G_ERR_INVALID_ARG;
  const int64_t n = T * topk;
  if (n > 0x7FFFFFFF || M_cap % 128 != 0 || M_cap < n + int64_t{127} * E || ld_sa < M_cap ||
      M_cap * (K / 128) >= (int64_t{1} << 31))
    return FP8G_ERR_INVALID_ARG;
  if (!q || !sA || !group_offsets || !row_token || (n > 0 && (!x || !topk_ids || !entry_row)))
    return FP8G_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || !aligned16(q) || !aligned16(sA) || ldx % 8 != 0 || ldq % 16 != 0 ||
      ld_sa % 4 != 0 || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(group_offsets) & 3u) || (reinterpret_cast<uintptr_t>(row_token) & 3u) ||
      (reinterpret_cast<uintptr_t>(entry_row) & 3u))
    return FP8G_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (E <= kRouteChunkExperts && n >= kRouteChunkMinEntries) {
    const int64_t layout_ctas = std::min<int64_t>(kRouteChunkCtas, (n + 1023) / 1024);
    route_layout_chunked_kernel<<<static_cast<unsigned>(layout_ctas), kRouteThreads, 0, s>>>(
        topk_ids, static_cast<int32_t>(n), topk, E, group_offsets, row_token, entry_row, M_cap, dev->status);
  } else if (E <= kRouteSmallExperts)
    route_layout_small_kernel<<<1, kRouteThreads, 0, s>>>(topk_ids, static_cast<int32_t>(n), topk, E,
                                                          group_offsets, row_token, entry_row, M_cap,
                                                          dev->status);
  else
    route_layout_kernel<<<1, kRouteThreads, 0, s>>>(topk_ids, static_cast<int32_t>(n), topk, E, group_offsets,
                                                    row_token, entry_row, M_cap, dev->status);
  if (cudaGetLastError() != cudaSuccess) return FP8G_ERR_CUDA;
  // each token read and quantised once, stored to its rows; then the zero rows (a warp per row)
  const int64_t items = T * (K / 128);
  const int64_t per_block = kQGroupsPerBlock * kQUnroll;
  int64_t blocks = std::max<int64_t>((items + per_block - 1) / per_block, (M_cap + 31) / 32);
  static const int64_t cap = resident_blocks(quantize_1x128_kernel<true>, dev);
  if (blocks > cap) blocks = cap;
  // launched as a programmatic dependent of the layout kernel: its CTAs start while the layout
  // runs, load and quantise their first tokens, and wait for the layout before storing
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, quantize_1x128_kernel<true>, static_cast<const __nv_bfloat16*>(x),
                         static_cast<uint32_t>(T), static_cast<uint32_t>(K / 128), ldx, static_cast<uint8_t*>(q), ldq,
                         sA, ld_sa, static_cast<const int32_t*>(entry_row), 0u, static_cast<uint32_t>(topk),
                         static_cast<const int32_t*>(row_token), static_cast<uint32_t>(M_cap)) != cudaSuccess) {
    cudaGetLastError();
    return FP8G_ERR_CUDA;
  }
  return FP8G_OK;
}

extern "C" int fp8_quantize_per_row(const void* x, int64_t M, int64_t K, int64_t ldx, void* q,
                                    int64_t ldq, float* s, void* stream) {
  if (M < 0 || M > 0x7FFFFFFF || K <= 0 || K % 128 != 0 || ldx < K || ldq < K) return FP8G_ERR_INVALID_ARG;
  if (M == 0) return FP8G_OK;
  if (!x || !q || !s) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(s) & 3u) || ldx % 8 != 0 || ldq % 16 != 0)
    return FP8G_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  quantize_rows_kernel<<<static_cast<unsigned>(M), kRowThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), K, ldx, static_cast<uint8_t*>(q), ldq, s);
  return cudaGetLastError() == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

extern "C" int fp8_quantize_per_tensor(const void* x, int64_t E, int64_t M, int64_t K, int64_t ldx, void* q,
                                       int64_t ldq, float* s, void* stream) {
  if (E < 1 || E > 65535 || M < 0 || K <= 0 || K % 128 != 0 || ldx < K || ldq < K) return FP8G_ERR_INVALID_ARG;
  if (M * (K / 8) >= (int64_t{1} << 31)) return FP8G_ERR_INVALID_ARG;
  if (!s) return FP8G_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(s) & 3u)) return FP8G_ERR_ALIGNMENT;
  if (M > 0) {
    if (!x || !q) return FP8G_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || ldx % 8 != 0 || ldq % 16 != 0) return FP8G_ERR_ALIGNMENT;
  }
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // s starts at +0, the scale of an empty or all-zero tensor
  if (cudaMemsetAsync(s, 0, static_cast<size_t>(E) * 4, cs) != cudaSuccess) {
    cudaGetLastError();
    return FP8G_ERR_CUDA;
  }
  if (M == 0) return FP8G_OK;
  const uint32_t kvec = static_cast<uint32_t>(K / 8);
  const int64_t pieces = M * (K / 8);
  int64_t bx = (pieces + kTensorThreads - 1) / kTensorThreads;
  // enough CTAs per tensor to fill the GPU across all E tensors
  const int64_t cap = std::max<int64_t>(1, static_cast<int64_t>(dev->sm_count) * (2048 / kTensorThreads) / E);
  if (bx > cap) bx = cap;
  const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(E));
  tensor_scale_kernel<<<grid, kTensorThreads, 0, cs>>>(static_cast<const __nv_bfloat16*>(x),
                                                       static_cast<uint32_t>(M), kvec, ldx, s);
  if (cudaGetLastError() != cudaSuccess) return FP8G_ERR_CUDA;
  // pass 2 as a programmatic dependent of pass 1 (it waits for pass 1 before reading s)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTensorThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, quantize_tensor_kernel, static_cast<const __nv_bfloat16*>(x),
                         static_cast<uint32_t>(M), kvec, ldx, static_cast<uint8_t*>(q), ldq,
                         static_cast<const float*>(s)) != cudaSuccess) {
    cudaGetLastError();
    return FP8G_ERR_CUDA;
  }
  return FP8G_OK;
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
