// E4M3 codes with a per-token power-of-two scale: the device side of the FP8
// latent cache.
//
// Format (OCP 8-bit floating point, E4M3): sign, 4 exponent bits (bias 7),
// 3 mantissa bits; exponent 0 holds the subnormals m * 2^-9; no infinities;
// largest finite 448.  Each token's 512 latent values share a scale 2^k, k
// the smallest integer with max|c| <= 448 * 2^k, so c * 2^-k is exact and
// its rounding to E4M3 is fixed whatever the working precision.
//
// Dequantisation is exact: an E4M3 value is a normal f16, the hardware
// converts a code pair to an f16 pair exactly, the f16 bits shifted right by
// three are a bf16 pattern equal to the value times 2^-112, and one bf16
// multiply by 2^(112+k) (two when 112+k leaves bf16's normal range) scales
// it without rounding.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace mla {
namespace dev {

constexpr int kFp8RowBytes = 640;   // 512 codes + 64 bf16 RoPE values per token
constexpr int kFp8Latent = 512;

// k with s = 2^k, for s a power of two (normal or subnormal fp32).
__device__ __forceinline__ int pow2_exponent(float s) {
  const uint32_t b = __float_as_uint(s);
  const int e = (int)((b >> 23) & 0xFFu);
  return e ? e - 127 : (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
}

// Smallest k with amax <= 448 * 2^k (k = 0 for amax == 0); amax >= 0 finite.
// amax = f * 2^e with f in [0.5, 1): k = e - 9 if f <= 0.875, else e - 8.
__device__ __forceinline__ int fp8_scale_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const uint32_t e = (b >> 23) & 0xFFu, m = b & 0x7FFFFFu;
  if (e) return (int)e - 135 + (m > 0x600000u ? 1 : 0);
  if (!m) return 0;
  const int p = 31 - __clz((int)m);  // subnormal: amax = m * 2^-149, top bit p
  const uint32_t thr = p >= 2 ? (7u << (p - 2)) : 0xFFFFFFFFu;
  return (p - 148) - 9 + (m > thr ? 1 : 0);
}

// 2^n as fp32 for n in [-126, 127].
__device__ __forceinline__ float exp2_int(int n) { return __uint_as_float((uint32_t)(n + 127) << 23); }

// x * 2^n exactly, for n in [-120, 142] and |x * 2^n| <= 448 (the quantiser's range).
__device__ __forceinline__ float scale_pow2(float x, int n) {
  return n > 126 ? (x * 0x1p64f) * exp2_int(n - 64) : x * exp2_int(n);
}

// Two fp32 values to an E4M3 pair, round to nearest even; lo lands in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (low byte first) to an f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(h) : "r"(two));
  return h;
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The bf16x2 factors that turn a row's shifted f16 patterns into code * 2^k.
struct Fp8Scale {
  uint32_t f1, f2;
  bool two;
};

__device__ __forceinline__ Fp8Scale fp8_row_scale(float s) {
  const int k = pow2_exponent(s);
  Fp8Scale r;
  if (k <= 15) {
    const uint32_t f = (uint32_t)(239 + k) << 7;  // bf16 2^(112+k)
    r.f1 = f | (f << 16);
    r.f2 = 0x3F803F80u;
    r.two = false;
  } else {
    r.f1 = (239u << 7) | (239u << 23);            // 2^112
    const uint32_t f = (uint32_t)(127 + k) << 7;  // 2^k
    r.f2 = f | (f << 16);
    r.two = true;
  }
  return r;
}

// The decode over the FP8 cache runs its tensor-core operands in f16: an
// E4M3 value is an exact f16, and code * 2^k stays exact in f16 while
// 2^-15 <= s = 2^k <= 2^7 (the smallest code 2^-9 * 2^-15 = 2^-24 is f16's
// smallest subnormal; 448 * 2^7 = 57344 < 65504).  fp8_f16_factor returns
// the f16x2 splat of s clamped to that range and whether s was inside it.
__device__ __forceinline__ uint32_t fp8_f16_factor(float s, bool& in_range) {
  const int e = (int)((__float_as_uint(s) >> 23) & 0xFFu) - 127;  // s = 2^e (normal s)
  in_range = e >= -15 && e <= 7 && (__float_as_uint(s) & 0x7FFFFFu) == 0u;
  const int k = e < -15 ? -15 : (e > 7 ? 7 : e);
  const uint32_t f = k >= -14 ? (uint32_t)(k + 15) << 10 : 0x0200u;  // 2^-15 is the subnormal 0x0200
  return f | (f << 16);
}

// A bf16 pair to an f16 pair (nearest even, saturating at 65504).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(__uint_as_float(u << 16)), "f"(__uint_as_float(u & 0xFFFF0000u)));
  return r;
}

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two codes to two bf16 (one word, low element first), exact.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t two, const Fp8Scale& sc) {
  const uint32_t h = e4m3x2_to_f16x2(two);
  const uint32_t w = ((h >> 3) & 0x0FFF0FFFu) | (h & 0x80008000u);
  const uint32_t y = mul_bf16x2(w, sc.f1);
  return sc.two ? mul_bf16x2(y, sc.f2) : y;
}

// Eight codes (a uint2, lowest address first) to eight bf16 (a uint4).
__device__ __forceinline__ uint4 dequant8(uint2 c, const Fp8Scale& sc) {
  uint4 o;
  o.x = dequant_pair(c.x & 0xFFFFu, sc);
  o.y = dequant_pair(c.x >> 16, sc);
  o.z = dequant_pair(c.y & 0xFFFFu, sc);
  o.w = dequant_pair(c.y >> 16, sc);
  return o;
}

}  // namespace dev
}  // namespace mla
