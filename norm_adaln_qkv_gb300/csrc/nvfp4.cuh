// nvfp4.cuh -- NVFP4 block quantisation (E2M1 elements, one UE4M3 scale per
// 16 elements, an FP32 global scale), shared by the NVFP4 stage's first
// kernel and the standalone quantiser
// (flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention, summary:
// fp4_quantize(a, act_global_scale, sf_vec_size=16)):
//
//   s    = ue4m3(RN(RN(amax / 6) * gs))       amax = max |v| over the block
//   enc  = s == 0 ? 0 : RN(gs / s)            (a 128-entry table per block)
//   code = e2m1(RN(v * enc))                  nearest even, saturating at 6
//
// Codes are packed two per byte, element 2j in the low nibble.  Scales are
// stored either row-major ([rows, cols/16]) or in the tiled form the
// block-scaled MMA consumes: 512-byte atoms of 128 rows x 4 scales (one
// 64-element K step), row r of the atom at byte (r % 32) * 16 + (r / 32) * 4,
// atoms ordered [row / 128][k / 64].
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace mh3 {
namespace fp4 {

constexpr int kBlock = 16;
constexpr int kAtomRows = 128;
constexpr int kAtomBytes = 512;

// UE4M3 code (0..126) -> its value (exact).
__device__ __forceinline__ float ue4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  return e == 0 ? __uint2float_rn(m) * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// RN(v / 6) for v >= 0: Markstein's quotient with the constant r = RN(1/6)
// (one multiply, two FMAs), exact whenever no step leaves the normal range,
// i.e. for v in [2^-100, 2^127) (checked for every bf16 value there); outside
// that range (tiny, huge, infinite or NaN) a true division.
__device__ __forceinline__ float div6_rn(float v) {
  if (!(v >= 0x1p-100f && v < 0x1p127f)) return __fdiv_rn(v, 6.0f);
  const float r = 0x1.555556p-3f;  // RN(1/6)
  const float q = __fmul_rn(v, r);
  return __fmaf_rn(__fmaf_rn(-q, 6.0f, v), r, q);
}

// enc[c] = RN(gs / s_c) for every UE4M3 code c (0 for c = 0): the per-block
// division of the encode multiplier, done once per code.  Fill with all
// threads of the block, then synchronise.
constexpr int kEncLut = 128;
__device__ __forceinline__ void init_enc_lut(float* lut, float gs, int tid, int nthreads) {
  for (int c = tid; c < kEncLut; c += nthreads) {
    const float s = c < 127 ? ue4m3_value(static_cast<uint32_t>(c)) : 0.0f;
    lut[c] = s == 0.0f ? 0.0f : __fdiv_rn(gs, s);
  }
}

struct BlockScale {
  uint32_t code;  // UE4M3 scale code
  float enc;      // multiplier that maps the block onto the E2M1 range
};

__device__ __forceinline__ BlockScale block_scale(float amax, float gs, const float* enc_lut) {
  const float t = __fmul_rn(div6_rn(amax), gs);
  BlockScale b;
  b.code = e4m3x2_satfinite(t, 0.0f) & 0xFFu;  // t >= 0: nearest even, <= 448
  b.enc = enc_lut[b.code];
  return b;
}

// Eight FP32 values -> eight E2M1 codes in one word (element 0 in bits 0-3).
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Eight bf16 values (uint4) and the block's encode multiplier -> 8 codes;
// the products are packed two-lane FP32 multiplies (each lane one IEEE
// round-to-nearest multiply).
__device__ __forceinline__ uint32_t encode8(const uint4& w, float enc) {
  const uint64_t e2 = f2_pack(enc, enc);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(f2_from_bf16x2(ws[i]), e2), v[2 * i], v[2 * i + 1]);
  return e2m1x8(v);
}

// max |v| of eight bf16 values (exact): packed magnitude maxima
// (max.xorsign.abs keeps the larger magnitude), then the sign bits cleared.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float amax8(const uint4& w) {
  const uint32_t m = bf16x2_absmax(bf16x2_absmax(w.x, w.y), bf16x2_absmax(w.z, w.w)) & 0x7FFF7FFFu;
  return fmaxf(bf16_lo(m), bf16_hi(m));
}

// Byte offset of the 4 scales of (row, 64-element K step `kstep`).
__device__ __forceinline__ int64_t scale_offset(int64_t row, int kstep, int ksteps, bool tiled) {
  if (!tiled) return row * (ksteps * 4) + kstep * 4;
  return ((row >> 7) * ksteps + kstep) * kAtomBytes + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

}  // namespace fp4
}  // namespace mh3
