// nvfp4.cuh -- NVFP4 block quantisation (E2M1 elements, one UE4M3 scale per
// 16 elements, an FP32 global scale gs), shared by the NVFP4 stage's first
// kernel and the standalone quantiser.  The convention is the FlashInfer
// block-16 one that flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj
// prints in its summary (and that minimax_h3_nvfp4_pre_attention applies to
// its activation):
//
//   sf   = UE4M3(amax * gs / 6)      amax = max |v| over the block
//   code = RN(v * gs / sf)           E2M1, nearest even, saturating at 6
//
// each a single rounding of the exact quotient (UE4M3: nearest even,
// saturating at 448; where sf = 0 the codes are the signed zeros of v * 0).
//
// How one rounding is reached in FP32.  For the scale, directed roundings
// bracket the exact t = amax * gs / 6: t_lo = RD(amax * RD(gs / 6)) <= t <=
// t_hi = RU(amax * RU(gs / 6)); rounding is monotonic, so when t_lo and t_hi
// round to the same code, that is the code of t.  Otherwise the bracket
// holds one rounding boundary m (the midpoint of the two codes) and the sign
// of amax * gs - 6m decides; 6m has at most 7 significant bits, so it is an
// FP32 number, amax * gs is split exactly into hi + lo by one FMA, and
// hi - 6m is exact (the two are within a factor of 2), so the sign of
// (hi - 6m) + lo is that of the exact difference.  The elements work the
// same way with a multiplier just below and one just above gs / sf (a
// per-code table): when the two code words of eight elements agree they are
// the codes of the exact quotients; where a pair of codes differs, the sign
// of |v| * gs - m * sf at the midpoint m between them decides (m * sf has at
// most 7 significant bits).  Ties (the exact quotient on the midpoint) go to
// the even code.  Where gs / sf itself is an FP32 number of at most 16
// significant bits, both multipliers are that value: the products are exact
// and the conversion rounds them once, ties included, with no exact step.
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

// E2M1 magnitude code (0..7) -> its value: 0, 0.5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  return c < 2 ? 0.5f * static_cast<float>(c)
               : ldexpf(1.0f + 0.5f * static_cast<float>(c & 1u), static_cast<int>(c >> 1) - 1);
}

// Per-kernel constants: gs and the bracket RD(gs / 6) <= gs / 6 <= RU(gs / 6).
struct Quantiser {
  float gs, c_lo, c_hi;
};
__device__ __forceinline__ Quantiser make_quantiser(float gs) {
  Quantiser q;
  q.gs = gs;
  q.c_lo = __fdiv_rd(gs, 6.0f);
  q.c_hi = __fdiv_ru(gs, 6.0f);
  return q;
}

// Multipliers of gs / q for a nonzero divisor q: where gs / q is an FP32
// number with at most 16 significant bits, both are that exact value, so
// |v| * (gs / q) is exact for any bf16 v (at most 8 + 16 bits) and the E2M1
// conversion's own nearest-even rounding is the single rounding, ties
// included; the two code words then always agree.  Otherwise a multiplier
// e_lo <= (gs / q)(1 - 2^-23) and one e_hi >= (gs / q)(1 + 2^-23): one
// round-to-nearest product |v| * e_lo stays strictly below |v| * gs / q and
// |v| * e_hi strictly above (for v != 0).
__device__ __forceinline__ float2 enc_pair(float gs, float q) {
  const float lo = __fdiv_rd(gs, q), hi = __fdiv_ru(gs, q);
  if (lo == hi && (__float_as_uint(lo) & 0xFFu) == 0u) return make_float2(lo, lo);
  return make_float2(__fmul_rd(lo, 0x1.fffffep-1f),   // 1 - 2^-23
                     __fmul_ru(hi, 0x1.000002p+0f));  // 1 + 2^-23
}

// enc[c] = the multipliers of gs / s_c for every UE4M3 code c ((0, 0) for
// c = 0).  Fill with all threads of the block, then synchronise.
constexpr int kEncLut = 128;
__device__ __forceinline__ void init_enc_lut(float2* lut, float gs, int tid, int nthreads) {
  for (int c = tid; c < kEncLut; c += nthreads) {
    const float s = c < 127 ? ue4m3_value(static_cast<uint32_t>(c)) : 0.0f;
    lut[c] = s != 0.0f ? enc_pair(gs, s) : make_float2(0.0f, 0.0f);
  }
}

struct BlockScale {
  uint32_t code;  // UE4M3 scale code (its value sf is decoded only where an
                  // element needs the exact step)
  float enc_lo;   // multipliers bracketing gs / sf
  float enc_hi;
};

// Sign of a * b - c for an FP32 number c within a factor of 2 of a * b:
// a * b = hi + lo exactly (one FMA), hi - c is exact, and (hi - c) + lo has
// the sign of the exact difference.
__device__ __forceinline__ float exact_diff_sign(float a, float b, float c) {
  const float hi = __fmul_rn(a, b);
  const float lo = __fmaf_rn(a, b, -hi);
  return __fadd_rn(__fsub_rn(hi, c), lo);
}

// The bracket [t_lo, t_hi] rounds to the adjacent codes lo < hi: decide at
// their midpoint m with the exact sign of amax * gs - 6m.
__device__ __forceinline__ uint32_t scale_code_at_boundary(float amax, float gs, uint32_t lo,
                                                           uint32_t hi) {
  const float six_m = __fmul_rn(__fadd_rn(ue4m3_value(lo), ue4m3_value(hi)), 3.0f);  // exact
  const float d = exact_diff_sign(amax, gs, six_m);
  if (d > 0.0f) return hi;
  if (d < 0.0f) return lo;
  return (lo & 1u) ? hi : lo;  // on the midpoint: the even code
}

__device__ __forceinline__ BlockScale block_scale(float amax, const Quantiser& q,
                                                  const float2* enc_lut) {
  const float t_lo = __fmul_rd(amax, q.c_lo);
  const float t_hi = __fmul_ru(amax, q.c_hi);
  const uint32_t both = e4m3x2_satfinite(t_lo, t_hi);  // t >= 0: nearest even, <= 448
  uint32_t code = both & 0xFFu;
  if (code != (both >> 8)) code = scale_code_at_boundary(amax, q.gs, code, both >> 8);
  BlockScale b;
  b.code = code;
  const float2 e = enc_lut[code];
  b.enc_lo = e.x;
  b.enc_hi = e.y;
  return b;
}

// The same multipliers from a 16-entry table per global scale, for kernels
// without room for kEncLut entries: a UE4M3 code with exponent field e and
// mantissa j has the value n 2^(E - 10), n = 8 + j and E = e for e >= 1, and
// n = j, E = 1 for e = 0.  So gs / sf = (gs / n) 2^(10 - E): the table holds
// enc_pair(gs, n) for n = 1..15, and the power of two is applied with a
// product rounded the same way, which keeps each bracketing multiplier on
// its side of (gs / sf)(1 -+ 2^-23) and an exact one exact.
struct Table16 {
  float gs, c_lo, c_hi, pad;
  float2 t[16];
};
// Fill with threads tid = 0..16 of the block (others return), then synchronise.
__device__ __forceinline__ void init_table16(Table16* q, float gs, int tid) {
  if (tid == 16) {
    q->gs = gs;
    q->c_lo = __fdiv_rd(gs, 6.0f);
    q->c_hi = __fdiv_ru(gs, 6.0f);
    q->pad = 0.0f;
  } else if (tid < 16) {
    q->t[tid] = tid > 0 ? enc_pair(gs, static_cast<float>(tid)) : make_float2(0.0f, 0.0f);
  }
}

__device__ __forceinline__ BlockScale block_scale_t16(float amax, const Table16& q) {
  const float t_lo = __fmul_rd(amax, q.c_lo);
  const float t_hi = __fmul_ru(amax, q.c_hi);
  const uint32_t both = e4m3x2_satfinite(t_lo, t_hi);
  uint32_t code = both & 0xFFu;
  if (code != (both >> 8)) code = scale_code_at_boundary(amax, q.gs, code, both >> 8);
  BlockScale b;
  b.code = code;
  const uint32_t e = code >> 3, j = code & 7u;
  const uint32_t n = e ? 8u + j : j;
  const uint32_t E = e ? e : 1u;
  const float pw = __uint_as_float((137u - E) << 23);  // 2^(10 - E), exact
  const float2 t = q.t[n];
  b.enc_lo = __fmul_rd(t.x, pw);
  b.enc_hi = __fmul_ru(t.y, pw);
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

// Eight bf16 values (uint4) times one multiplier, packed two-lane FP32
// multiplies (each lane one IEEE round-to-nearest multiply), to E2M1 codes.
__device__ __forceinline__ uint32_t codes8(const uint4& w, float enc) {
  const uint64_t e2 = f2_pack(enc, enc);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(f2_from_bf16x2(ws[i]), e2), v[2 * i], v[2 * i + 1]);
  return e2m1x8(v);
}

// The elements whose two bracketing codes differ (a nibble of lo ^ hi):
// decide each at the midpoint m between its two adjacent magnitudes with the
// exact sign of |v| * gs - m * sf.  4m for the midpoints above magnitude
// codes 0..6 (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5), five bits each.
constexpr uint64_t kE2m1Mid4 = 1ull | 3ull << 5 | 5ull << 10 | 7ull << 15 | 10ull << 20 |
                               14ull << 25 | 20ull << 30;
__device__ __forceinline__ uint32_t codes8_at_boundary(const uint4& w, uint32_t lo, uint32_t hi,
                                                       float gs, float sf) {
  uint32_t out = lo;
  uint32_t diff = lo ^ hi;
  while (diff != 0u) {
    const int j = (__ffs(static_cast<int>(diff)) - 1) >> 2;  // element with a differing code
    diff &= ~(0xFu << (4 * j));
    const uint32_t a = (lo >> (4 * j)) & 7u, b = (hi >> (4 * j)) & 7u;
    const uint32_t ma = a < b ? a : b;  // adjacent magnitudes ma, ma + 1
    const int word = j >> 1;
    uint32_t h = word == 0 ? w.x : (word == 1 ? w.y : (word == 2 ? w.z : w.w));
    h = (j & 1) ? (h >> 16) : h;
    const float mag = __uint_as_float((h & 0x7FFFu) << 16);  // |v|
    const float m = 0.25f * static_cast<float>((kE2m1Mid4 >> (5 * ma)) & 31u);
    const float d = exact_diff_sign(mag, gs, __fmul_rn(m, sf));  // m * sf exact
    const uint32_t pick = d > 0.0f ? ma + 1 : (d < 0.0f ? ma : ((ma & 1u) ? ma + 1 : ma));
    out = (out & ~(7u << (4 * j))) | (pick << (4 * j));  // the sign bit stays
  }
  return out;
}

// The codes of eight bf16 values of one block.
__device__ __forceinline__ uint32_t encode8(const uint4& w, const BlockScale& b, float gs) {
  const uint32_t lo = codes8(w, b.enc_lo);
  const uint32_t hi = codes8(w, b.enc_hi);
  return lo == hi ? lo : codes8_at_boundary(w, lo, hi, gs, ue4m3_value(b.code));
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
