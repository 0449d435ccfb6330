// e4m3.cuh -- per-tensor e4m3 quantisation of bf16 values, shared by the
// stage's e4m3 epilogue and the standalone quantiser:
//
//   code = e4m3_sat(RN32(v / descale))
//
// (flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention, Parameters:
// out_mode "e4m3", q/k/v_descale: per-tensor dequantisation scales, so a
// value is recovered as code * descale; the quotient is the IEEE FP32
// division, rounded to nearest even e4m3 and saturated to +-448.)
//
// An IEEE division per element costs more than the rest of the epilogue, so
// the quotient is formed by Markstein's method (P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Develop. 34(1), 1990): with r = RN(1/d) and q = RN(v r), the remainder
// v - q d is exact under one FMA and q' = RN(q + (v - q d) r) = RN(v / d).
// It is used only where no intermediate can leave the normal range:
// |d| in [2^-60, 2^60] (else a true division, warp-uniform) and |q| in
// [2^-20, 1024).  Outside that band q itself gives the same code: below
// 2^-20 every quotient rounds to a signed e4m3 zero with the sign of q, and
// at or above 1024 every quotient saturates to +-448.  For bf16 v the
// method was checked exhaustively against the IEEE quotient (all 2^7
// significands of v times all 2^23 significands of d; exponents only scale
// every step inside the band).
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace mh3 {
namespace e4m3q {

struct Divisor {
  float d;     // descale
  float r;     // RN(1/d)
  bool fast;   // |d| in [2^-60, 2^60]: Markstein quotient
};

__device__ __forceinline__ Divisor make_divisor(float d) {
  Divisor v;
  v.d = d;
  v.r = __frcp_rn(d);
  const float a = fabsf(d);
  v.fast = a >= 0x1p-60f && a <= 0x1p60f;
  return v;
}

// RN32(v / d) on the fast path (see the header comment for the band).
__device__ __forceinline__ float quotient_fast(float v, const Divisor& dv) {
  const float q = __fmul_rn(v, dv.r);
  const float a = fabsf(q);
  const float q2 = __fmaf_rn(__fmaf_rn(-q, dv.d, v), dv.r, q);
  return (a >= 0x1p-20f && a < 1024.0f) ? q2 : q;
}

// Two bf16 values (one 32-bit word, element 0 in the low half) -> two codes
// in the low 16 bits (element 0 in bits 0-7).
template <bool kFast>
__device__ __forceinline__ uint32_t quantize_word(uint32_t w, const Divisor& dv) {
  const float lo = bf16_lo(w), hi = bf16_hi(w);
  if (kFast) return e4m3x2_satfinite(quotient_fast(lo, dv), quotient_fast(hi, dv));
  return e4m3x2_satfinite(__fdiv_rn(lo, dv.d), __fdiv_rn(hi, dv.d));
}

// Eight bf16 values (uint4) -> eight codes (uint2).
template <bool kFast>
__device__ __forceinline__ uint2 quantize8(const uint4& b, const Divisor& dv) {
  return make_uint2(quantize_word<kFast>(b.x, dv) | (quantize_word<kFast>(b.y, dv) << 16),
                    quantize_word<kFast>(b.z, dv) | (quantize_word<kFast>(b.w, dv) << 16));
}

}  // namespace e4m3q
}  // namespace mh3
