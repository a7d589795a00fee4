// Element arithmetic of the fine-grained E4M3 quantizers (DeepSeek-V3
// report excerpt, "Fine-Grained Quantization"): the scale of a tile from its
// amax, the correctly rounded quotient x / s, E4M3 and BF16 conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "common.cuh"

namespace fp8fg {

// Scale of a tile from its amax: fl32(amax / 448) (IEEE division, correctly
// rounded); 1 when that is zero; optionally raised to the next power of two.
// The division is the two-correction FMA sequence of quot_fma with the
// constant reciprocal RN(1/448) (exact for 2^-100 <= amax <= FLT_MAX, where
// the quotient and residuals are normal and finite); other amax values
// (tiny, infinite, NaN) take the IEEE division.
__device__ __forceinline__ float quot_fma(float x, float s, float r);

__device__ __forceinline__ float tile_scale(float amax, bool pow2) {
  float s;
  if (amax >= 0x1p-100f && amax <= 3.4028234663852886e38f)
    s = quot_fma(amax, 448.0f, 1.0f / 448.0f);
  else
    s = __fdiv_rn(amax, 448.0f);
  if (!(s > 0.0f)) s = 1.0f;
  if (pow2) {
    uint32_t b = __float_as_uint(s);
    uint32_t e = b >> 23;          // sign is 0: s > 0
    uint32_t m = b & 0x7FFFFFu;
    if (e != 0) {
      if (m != 0) b = (e + 1) << 23;
    } else {
      // subnormal: value m * 2^-149; next power of two of the integer m
      uint32_t p = 1u << (31 - __clz(m));
      if (p != m) p <<= 1;
      b = p;  // 2^23 lands on the smallest normal, 0x00800000
    }
    s = __uint_as_float(b);
  }
  return s;
}

// Correctly rounded x / s for a tile scale s, without a division per element.
//
// kQuotMul: s is a normal power of two, so r = 1/s is exact and RN(x * r)
//   is RN(x / s) (one rounding of the same real number).
// kQuotFma: r = RN(1/s) once per tile; per element q0 = RN(x*r), then two
//   residual corrections q <- RN(q - RN(s*q - x)*r), the residual exact by
//   FMA. After the first correction q is within one ulp of x/s, and
//   Markstein's theorem (a correctly rounded reciprocal plus a quotient
//   within one ulp gives a correctly rounded corrected quotient) makes the
//   second one RN(x/s). With the residual taken as s*q - x and subtracted,
//   a zero quotient keeps the sign of x, as IEEE division does.
//   The residuals stay exact while |x| >= 2^-103.
// kQuotDiv: a scale below 2^-80 can come with such x and a non-negligible
//   quotient, so those tiles take the IEEE division.
// The mode is uniform per tile.
enum : int { kQuotMul = 0, kQuotFma = 1, kQuotDiv = 2 };

struct TileDiv {
  float s, r;
  int mode;
};

__device__ __forceinline__ int make_tile_div_mode(float s) {
  const uint32_t b = __float_as_uint(s);
  const uint32_t e = b >> 23;
  if ((b & 0x7FFFFFu) == 0 && e >= 1 && e <= 254) return kQuotMul;
  return s < 0x1p-80f ? kQuotDiv : kQuotFma;
}

__device__ __forceinline__ float quot_fma(float x, float s, float r) {
  float q = __fmul_rn(x, r);
  float e = __fmaf_rn(s, q, -x);
  q = __fmaf_rn(-e, r, q);
  e = __fmaf_rn(s, q, -x);
  return __fmaf_rn(-e, r, q);
}

__device__ __forceinline__ float tile_quot(float x, const TileDiv& d) {
  if (d.mode == kQuotMul) return __fmul_rn(x, d.r);
  if (d.mode == kQuotDiv) return __fdiv_rn(x, d.s);
  return quot_fma(x, d.s, d.r);
}

// The quotient path for a set of tiles whose scales lanes hold: kQuotMul if
// every scale is a normal power of two, else kQuotFma if every scale allows
// it, else kQuotDiv (per-element tile_quot). Uniform across the warp.
__device__ __forceinline__ int warp_quot_mode(int my_mode) {
  if (__all_sync(0xffffffffu, my_mode == kQuotMul)) return kQuotMul;
  if (__all_sync(0xffffffffu, my_mode != kQuotDiv)) return kQuotFma;
  return kQuotDiv;
}

// ---------------------------------------------------------------- packed
// (pk2, unpk2, mul2, fma2: the f32x2 helpers in common.cuh)

// RN(x/s) for a pair given nx = -x, s2 = (s, s) and nr2 = (-r, -r) with
// r = RN(1/s): the quot_fma sequence on negated operands. q0 = RN(nx*nr) =
// RN(x*r); e = RN(s*q - x) exact; q <- RN(q - e*r). A zero quotient keeps
// the sign of x, as in quot_fma.
__device__ __forceinline__ uint64_t quot2_fma(uint64_t nx, uint64_t s2, uint64_t nr2) {
  uint64_t q = mul2(nx, nr2);
  uint64_t e = fma2(s2, q, nx);
  q = fma2(e, nr2, q);
  e = fma2(s2, q, nx);
  return fma2(e, nr2, q);
}

// Four quotients (two pairs) -> four E4M3 bytes (RNE, satfinite), the low
// element of q01 in the low byte.
__device__ __forceinline__ uint32_t e4m3x4_pk(uint64_t q01, uint64_t q23) {
  uint32_t d;
  asm("{\n\t.reg .f32 a0, a1, a2, a3;\n\t.reg .b16 c0, c1;\n\t"
      "mov.b64 {a0, a1}, %1;\n\tmov.b64 {a2, a3}, %2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c0, a1, a0;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c1, a3, a2;\n\t"
      "mov.b32 %0, {c0, c1};\n\t}"
      : "=r"(d)
      : "l"(q01), "l"(q23));
  return d;
}

// N pairs of negated values -> quotients along a path chosen by
// warp_quot_mode: kQuotFma is exact for any scale that is not kQuotDiv (a
// power of two included); kQuotDiv falls back to the per-tile choice.
template <int N>
__device__ __forceinline__ void quot2_n(uint64_t (&v)[N], int path, float s, float r) {
  if (path == kQuotMul) {
    const uint64_t nr2 = pk2(-r, -r);
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = mul2(v[i], nr2);
  } else if (path == kQuotFma) {
    const uint64_t s2 = pk2(s, s), nr2 = pk2(-r, -r);
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = quot2_fma(v[i], s2, nr2);
  } else {
    TileDiv d;
    d.s = s;
    d.r = r;
    d.mode = make_tile_div_mode(s);
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float2 f = unpk2(v[i]);
      v[i] = pk2(tile_quot(-f.x, d), tile_quot(-f.y, d));
    }
  }
}

// BF16 pair in a 32-bit word -> the negated values as an f32 pair:
// -lo = (w << 16) + 2^31 (mod 2^32) flips the sign bit, -hi likewise.
__device__ __forceinline__ uint64_t neg_bf16x2(uint32_t w) {
  return pk2(__uint_as_float(w * 65536u + 0x80000000u), __uint_as_float((w & 0xFFFF0000u) ^ 0x80000000u));
}

// Four floats -> four E4M3 bytes (RNE, satfinite), a in the low byte.
__device__ __forceinline__ uint32_t e4m3x4_f(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// The E4M3 pair in the low (lo_pk) or high (hi_pk) half of w -> the two
// values (exact) as an f32 pair, the lower byte first.
__device__ __forceinline__ uint64_t e4m3x2_lo_pk(uint32_t w) {
  uint64_t r;
  asm("{\n\t.reg .b16 l, h;\n\t.reg .b32 p;\n\t.reg .f32 a, b;\n\t"
      "mov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 p, l;\n\tmov.b32 {l, h}, p;\n\t"
      "cvt.f32.f16 a, l;\n\tcvt.f32.f16 b, h;\n\tmov.b64 %0, {a, b};\n\t}"
      : "=l"(r)
      : "r"(w));
  return r;
}

__device__ __forceinline__ uint64_t e4m3x2_hi_pk(uint32_t w) {
  uint64_t r;
  asm("{\n\t.reg .b16 l, h;\n\t.reg .b32 p;\n\t.reg .f32 a, b;\n\t"
      "mov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 p, h;\n\tmov.b32 {l, h}, p;\n\t"
      "cvt.f32.f16 a, l;\n\tcvt.f32.f16 b, h;\n\tmov.b64 %0, {a, b};\n\t}"
      : "=l"(r)
      : "r"(w));
  return r;
}

}  // namespace fp8fg
