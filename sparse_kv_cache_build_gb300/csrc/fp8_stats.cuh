// FP8 (E4M3) page statistics with outward rounding: the next-step row "compressed page
// statistics", motivated by "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM
// Decoding" (a selector's key cache quantised to few bits). The score of "EntmaxKV:
// Support-Aware Decoding for Entmax Attention" (abstract) stays an upper bound of q.k only if
// the stored [min, max] box contains the exact one, so the minimum is rounded down and the
// maximum up.
//
// Format: each (physical page, KV head) row of 2*D statistics is 2*D E4M3 bytes (the min row
// then the max row, as the bf16/fp32 layout) plus one int8 exponent e: byte c stands for
// value(c) * 2^e, where e is the smallest integer >= -126 with max|x| <= 448 * 2^e over the row
// (0 for an all-zero row). E4M3 here is the OCP "FN" byte: sign, 4 exponent bits with bias 7,
// 3 mantissa bits, exponent field 0 for subnormals m/8 * 2^-6, no infinity, 0x7F/0xFF NaN
// (never produced), largest magnitude 448. Zero is always the +0 byte.
//
// For a magnitude a >= 0 the byte values increase with the byte, and between 2^-9 and 448 the
// ladder is linear in the byte across the subnormal/normal boundary (byte 8 = 2^-6), so the
// outward bytes are a floor or a ceiling of the position on that ladder, computed exactly in
// fp32 (a power-of-two rescale of an fp32 value is exact while the result is normal, and
// every magnitude below 2^-9 maps to byte 0 or 1 whatever its low bits).
#pragma once

#include "kv_internal.cuh"

namespace skv {
namespace fp8 {

constexpr int kMinExponent = -126;

// 2^k as a float, k in [-126, 127].
__device__ __forceinline__ float pow2(int k) { return __int_as_float((k + 127) << 23); }

// Row exponent: smallest e >= -126 with m <= 448 * 2^e (m = max |x| >= 0); 0 when m == 0.
__device__ __forceinline__ int row_exponent(float m) {
  if (!(m > 0.f)) return 0;
  int ex = 0;
  const float fr = frexpf(m, &ex);            // m = fr * 2^ex, fr in [0.5, 1)
  // m = (2 fr) * 2^(ex-1) and 448 = 1.75 * 2^8
  int e = (ex - 1) - 8 + (2.f * fr > 1.75f ? 1 : 0);
  return e < kMinExponent ? kMinExponent : e;
}

// Byte magnitude (0..126) of the largest ladder value <= a, for 0 <= a <= 448.
__device__ __forceinline__ uint32_t mag_floor(float a) {
  if (a < 0x1p-9f) return 0u;
  if (a < 0x1p-6f) return (uint32_t)floorf(a * 512.f);          // subnormal: m * 2^-9
  const int E = (int)((__float_as_uint(a) >> 23) & 0xffu) - 127;   // a normal: 2^E <= a
  const float f = a * pow2(-E);                                    // [1, 2), exact
  return ((uint32_t)(E + 7) << 3) + (uint32_t)floorf((f - 1.f) * 8.f);
}

// Byte magnitude of the smallest ladder value >= a, for 0 <= a <= 448; nonzero: a stands
// for a value that is not zero (a may have underflowed to 0 in the rescale).
__device__ __forceinline__ uint32_t mag_ceil(float a, bool nonzero) {
  if (!nonzero) return 0u;
  if (a < 0x1p-9f) return 1u;
  if (a < 0x1p-6f) return (uint32_t)ceilf(a * 512.f);           // 8 is byte 0x08 = 2^-6
  const int E = (int)((__float_as_uint(a) >> 23) & 0xffu) - 127;
  const float f = a * pow2(-E);
  return ((uint32_t)(E + 7) << 3) + (uint32_t)ceilf((f - 1.f) * 8.f);   // a carry is exact
}

// Byte of the largest value v with v * 2^e <= x (inv_scale = 2^-e).
__device__ __forceinline__ uint32_t quantize_down(float x, float inv_scale) {
  const float a = fabsf(x) * inv_scale;
  if (!(x < 0.f)) return mag_floor(a);
  const uint32_t c = mag_ceil(a, true);
  return c ? (0x80u | c) : 0u;
}

// Byte of the smallest value v with v * 2^e >= x.
__device__ __forceinline__ uint32_t quantize_up(float x, float inv_scale) {
  const float a = fabsf(x) * inv_scale;
  if (x > 0.f) return mag_ceil(a, true);
  const uint32_t c = mag_floor(a);
  return c ? (0x80u | c) : 0u;
}

}  // namespace fp8
}  // namespace skv
