// Device helpers shared by the libgift kernels (sm_103a).
//
// Number formats follow the GIFT reading notes (zhongzhuzhou.org), prerequisites,
// "What FP8 is" (E4M3 largest finite 448, E5M2 largest finite 57344) and the GIFT
// abstract (shd-paper.top), which names NVFP4.  Encoding uses the hardware
// round-to-nearest-even, saturate-to-finite conversions; decoding builds the IEEE
// single-precision bit pattern of each code exactly.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "gift.h"

namespace gift {

constexpr float kE4M3Max = 448.0f;
constexpr float kE5M2Max = 57344.0f;
constexpr float kNvfp4TensorDiv = 2688.0f;   // 448 * 6: E4M3 block-scale range x E2M1 range
constexpr float kF32Max = 3.402823466e38f;
constexpr int kBlock = 128;                  // edge of a BLOCK128 scale tile
constexpr int kBlock1d = 512;                // elements of a BLOCK512 scale group
constexpr int kNvGroup = 16;                 // elements per NVFP4 block scale
constexpr int kMaxRank = 32;
constexpr int kMaxReplicas = 64;

enum Fmt8 { FMT_E4M3 = 0, FMT_E5M2 = 1 };

// ------------------------------------------------------------------------------------
// status word: the first device-detected error wins
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int *st, int code) {
  if (st) atomicCAS(st, 0, code);
}

// ------------------------------------------------------------------------------------
// FP32 -> FP8 / FP4 (round to nearest even, satfinite, sign of zero kept)
// ------------------------------------------------------------------------------------
// Packs four values into four bytes, element 0 in the lowest byte.
template <int F>
__device__ __forceinline__ uint32_t pack4_fp8(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  if (F == FMT_E4M3) {
    // cvt ... d, a, b puts a in the upper half of d and b in the lower half
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  }
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

template <int F>
__device__ __forceinline__ uint8_t pack1_fp8(float x) {
  return (uint8_t)(pack4_fp8<F>(x, 0.f, 0.f, 0.f) & 0xFFu);
}

// Eight values -> eight E2M1 nibbles in a 32-bit word, element 0 in the lowest nibble.
__device__ __forceinline__ uint32_t pack8_e2m1(const float *x) {
  uint32_t r;
  asm("{\n\t"
      ".reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t"
      "}"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return r;
}

// Four values -> four nibbles in the low 16 bits.
__device__ __forceinline__ uint32_t pack4_e2m1(float x0, float x1, float x2, float x3) {
  float v[8] = {x0, x1, x2, x3, 0.f, 0.f, 0.f, 0.f};
  return pack8_e2m1(v) & 0xFFFFu;
}

// ------------------------------------------------------------------------------------
// FP8 / FP4 -> FP32, exact.  The code's magnitude bits are placed in the FP32 exponent
// and mantissa fields, which gives a single whose value is the code's value times a known
// power of two (FP32 denormals cover the code's subnormals); one exact multiplication by
// the inverse power of two restores the value.  Needs denormals preserved (no -ftz).
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float dec_e4m3(uint32_t c) {
  const uint32_t bits = ((c & 0x7Fu) << 20) | ((c & 0x80u) << 24);   // bias 127 vs 7
  return __fmul_rn(__uint_as_float(bits), 0x1p120f);
}
__device__ __forceinline__ float dec_e5m2(uint32_t c) {
  const uint32_t bits = ((c & 0x7Fu) << 21) | ((c & 0x80u) << 24);   // bias 127 vs 15
  return __fmul_rn(__uint_as_float(bits), 0x1p112f);
}
__device__ __forceinline__ float dec_e2m1(uint32_t c) {
  const uint32_t bits = ((c & 0x7u) << 22) | ((c & 0x8u) << 28);     // bias 127 vs 1
  return __fmul_rn(__uint_as_float(bits), 0x1p126f);
}
template <int F>
__device__ __forceinline__ float dec_fp8(uint32_t c) {
  return F == FMT_E4M3 ? dec_e4m3(c) : dec_e5m2(c);
}

// ------------------------------------------------------------------------------------
// scale rule: s = amax / FMAX (stored), m = FMAX / amax (multiplier), single roundings
// ------------------------------------------------------------------------------------
struct ScalePair {
  float s, m;
};
__device__ __forceinline__ ScalePair scale_pair(float amax, float fmax) {
  ScalePair p;
  if (amax == 0.0f) {
    p.s = 0.0f;
    p.m = 0.0f;
  } else {
    p.s = __fdiv_rn(amax, fmax);
    p.m = __fdiv_rn(fmax, amax);
    if (isinf(p.m)) p.m = kF32Max;
  }
  return p;
}

template <int F>
__device__ __forceinline__ float fmax_of() {
  return F == FMT_E4M3 ? kE4M3Max : kE5M2Max;
}
template <int F>
__device__ __forceinline__ uint32_t maxcode_of() {
  return F == FMT_E4M3 ? 0x7Eu : 0x7Bu;
}

// NVFP4 per-group multiplier: e = E4M3(amax_g / fl(6 s_t)), eff = fl(e * s_t), r = 1 / eff.
struct Nv4Group {
  uint8_t e_code;
  float eff;   // value(e) * s_t, the group's effective scale
  float r;     // multiplier applied to the elements
};
__device__ __forceinline__ Nv4Group nvfp4_group(float amax_g, float s_t) {
  Nv4Group g;
  float ratio = 0.0f;
  if (s_t != 0.0f) ratio = __fdiv_rn(amax_g, __fmul_rn(6.0f, s_t));
  g.e_code = pack1_fp8<FMT_E4M3>(ratio);
  const float ev = dec_e4m3(g.e_code);
  g.eff = __fmul_rn(ev, s_t);
  if (g.eff == 0.0f) {
    g.r = 0.0f;
  } else {
    g.r = __fdiv_rn(1.0f, g.eff);
    if (isinf(g.r)) g.r = kF32Max;
  }
  return g;
}
// NVFP4 dequantisation: fl(fl(value(code) * value(e)) * s_t)
__device__ __forceinline__ float nvfp4_deq(uint32_t code, float e_val, float s_t) {
  return __fmul_rn(__fmul_rn(dec_e2m1(code), e_val), s_t);
}

// ------------------------------------------------------------------------------------
// reductions
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) { return __reduce_max_sync(0xFFFFFFFFu, v); }
__device__ __forceinline__ uint32_t warp_add_u32(uint32_t v) { return __reduce_add_sync(0xFFFFFFFFu, v); }

// Block-wide max of a non-negative bit pattern; every thread gets the result.
template <int NT>
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *smem /* >= NT/32 */) {
  v = warp_max_u32(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) smem[w] = v;
  __syncthreads();
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) r = max(r, smem[i]);
  return r;
}

__host__ __device__ __forceinline__ bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace gift
