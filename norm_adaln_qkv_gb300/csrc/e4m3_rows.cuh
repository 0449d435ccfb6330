// e4m3_rows.cuh -- per-token E4M3 quantisation of bf16 rows, shared by the
// FP8 MLP block's first kernel (the activation a) and its y quantiser
// (flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, formula block):
//
//   s    = RN(amax_row(|v|) / 448)                FP32 division
//   code = e4m3(v / s)                            one rounding of the exact
//                                                 quotient: nearest even,
//                                                 saturating at +-448, sign
//                                                 kept (-0 for small negatives)
//
// A row whose amax is 0 has s = 0 and codes +0.
//
// One rounding in FP32.  With r_lo = RD(1/s) and r_hi = RU(1/s), the products
// RD(|v| r_lo) <= |v| / s <= RU(|v| r_hi) bracket the exact quotient;
// rounding is monotonic, so when both round to the same code, that is the
// code of |v| / s.  Otherwise the bracket holds the midpoint m of the two
// adjacent codes, and the sign of |v| - m s decides: m s is split exactly into
// hi + lo by one FMA, |v| - hi is exact (the two are within a factor of 2),
// and (|v| - hi) - lo has the sign of the exact difference.  On the midpoint
// itself the even code wins.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace mh3 {
namespace e4m3r {

constexpr float kMax = 448.0f;

struct RowScale {
  float s;     // RN(amax / 448)
  float r_lo;  // RD(1 / s)
  float r_hi;  // RU(1 / s)
};

__device__ __forceinline__ RowScale make_row_scale(float amax) {
  RowScale r;
  r.s = __fdiv_rn(amax, kMax);
  r.r_lo = r.s > 0.0f ? __frcp_rd(r.s) : 0.0f;
  r.r_hi = r.s > 0.0f ? __frcp_ru(r.s) : 0.0f;
  return r;
}

// Value of an E4M3 magnitude code (0..126), exact.
__device__ __forceinline__ float magnitude_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  return e == 0 ? __uint2float_rn(m) * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Codes of the magnitudes of two bf16 values (one word, element 0 low) from
// one side of the bracket: byte 0 = element 0.
__device__ __forceinline__ uint32_t codes2(uint32_t w, float r, bool up) {
  const float lo = __uint_as_float((w & 0x7FFFu) << 16);
  const float hi = __uint_as_float(w & 0x7FFF0000u);
  const float a = up ? __fmul_ru(lo, r) : __fmul_rd(lo, r);
  const float b = up ? __fmul_ru(hi, r) : __fmul_rd(hi, r);
  return e4m3x2_satfinite(a, b);  // non-negative: nearest even, <= 448
}

// The element whose two bracketing codes a < b differ: decide at their
// midpoint with the exact sign of |v| - m s.
__device__ __forceinline__ uint32_t decide(float mag, float s, uint32_t a, uint32_t b) {
  const float m = __fmul_rn(__fadd_rn(magnitude_value(a), magnitude_value(b)), 0.5f);  // exact
  const float hi = __fmul_rn(m, s);
  const float lo = __fmaf_rn(m, s, -hi);
  const float d = __fsub_rn(__fsub_rn(mag, hi), lo);
  if (d > 0.0f) return b;
  if (d < 0.0f) return a;
  return (a & 1u) ? b : a;
}

// Eight bf16 values (uint4, element 0 in the low half of x) -> eight codes
// (uint2, element 0 in byte 0 of x).
__device__ __forceinline__ uint2 quantize8(const uint4& w, const RowScale& r) {
  if (r.s == 0.0f) return make_uint2(0u, 0u);  // an all-zero row
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t lo[2], hi[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lo[i] = codes2(ws[2 * i], r.r_lo, false) | (codes2(ws[2 * i + 1], r.r_lo, false) << 16);
    hi[i] = codes2(ws[2 * i], r.r_hi, true) | (codes2(ws[2 * i + 1], r.r_hi, true) << 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t diff = lo[i] ^ hi[i];
    while (diff != 0u) {
      const int j = (__ffs(static_cast<int>(diff)) - 1) >> 3;  // byte with differing codes
      diff &= ~(0xFFu << (8 * j));
      const uint32_t a = (lo[i] >> (8 * j)) & 0xFFu, b = (hi[i] >> (8 * j)) & 0xFFu;
      const uint32_t word = (j >> 1) ? ws[2 * i + 1] : ws[2 * i];
      const uint32_t h = (j & 1) ? (word >> 16) : word;
      const float mag = __uint_as_float((h & 0x7FFFu) << 16);
      const uint32_t pick = decide(mag, r.s, a, b);
      lo[i] = (lo[i] & ~(0xFFu << (8 * j))) | (pick << (8 * j));
    }
  }
  // the signs: bit 15 of each bf16 value to bit 7 of its code byte
  uint32_t sg[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w0 = ws[2 * i], w1 = ws[2 * i + 1];
    sg[i] = ((w0 >> 8) & 0x80u) | ((w0 >> 16) & 0x8000u) | ((w1 << 8) & 0x800000u) |
            (w1 & 0x80000000u);
  }
  return make_uint2(lo[0] | sg[0], lo[1] | sg[1]);
}

// max |v| of eight bf16 values (exact).
__device__ __forceinline__ float amax8(const uint4& w) {
  uint32_t m;
  asm("{\n\t.reg .b32 t0, t1;\n\t"
      "max.xorsign.abs.bf16x2 t0, %1, %2;\n\t"
      "max.xorsign.abs.bf16x2 t1, %3, %4;\n\t"
      "max.xorsign.abs.bf16x2 %0, t0, t1;\n\t}"
      : "=r"(m)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w));
  m &= 0x7FFF7FFFu;
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

}  // namespace e4m3r
}  // namespace mh3
