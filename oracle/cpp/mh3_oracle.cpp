// mh3_oracle.cpp -- CPU oracle of the MiniMax-H3 BF16 pre-attention stage.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
// CPU-baseline / reference arm load this library.  It shares no code, header,
// table or helper with the CUDA library, and neither calls the other.
//
// Plain, slow, obviously correct C++: one function per step of the stage, in
// the order flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention runs them
// (summary paragraph), with the rounding points of the formula block of
// flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120 (lines n = ..., a = ...,
// a[i outside [0, rows)] = 0) for the first two steps.  Every value is a
// bf16 or FP32 number; every FP32 operation is one IEEE round-to-nearest-even
// operation (the library is built with FMA contraction off), and bf16() is
// round-to-nearest-even from FP32.
//
// Readings where the pages leave a step open:
//   * "FP32 sum of squares": the exact sum of the squares rounded once to
//     FP32 (computed exactly below with an integer accumulator per binary
//     exponent), i.e. the ideal FP32 result of any summation order;
//   * rmsnorm(x) * w = (x * r) * w with r = 1 / sqrt(ss / width + eps);
//   * AdaLN is an unfused multiply then add;
//   * the QKV accumulator ("FP32 accumulation") is the dot product summed in
//     double, in increasing k, rounded once to FP32, then rounded to bf16
//     before the Q/K RMSNorm; the products of two bf16 values are exact in
//     double, and the double sum of 5376 of them differs from the exact sum by
//     far less than an FP32 rounding step;
//   * the normalised head is rounded to bf16 before RoPE;
//   * RoPE pairs dims (j, j + 48) with cos in cache column j and sin in
//     column 48 + j; dims [96, 128) pass through;
//   * destination p of the pack owns the contiguous head block
//     [p * 56/P, (p + 1) * 56/P); the kind order is q, k, v.
//
// Bit patterns of bf16 values travel as uint16_t.  Tokens are independent, so
// any subset of tokens is computed exactly; OpenMP spreads tokens over cores.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ------------------------------------------------------------------ bf16 <-> FP32
float bf16_value(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round an FP32 value to the nearest bf16, ties to even (NaN stays NaN).
uint16_t bf16_round(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  const uint32_t keep = u >> 16;
  const uint32_t rest = u & 0xFFFFu;
  uint32_t r = keep;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) r = keep + 1;
  return static_cast<uint16_t>(r);
}

// ------------------------------------------------- exact FP32 sum of squares
// A bf16 value is s * 2^e with an integer s < 256 (the significand with its
// hidden bit) and e in [-133, 120].  Its square s^2 * 2^(2e) is added to the
// integer bin of exponent 2e; after all terms the bins are carried into one
// binary number, which is then rounded once to FP32 (nearest, ties to even).
class ExactSquareSum {
 public:
  static constexpr int kLow = -266;                  // smallest exponent 2e
  static constexpr int kBins = 560;                  // 2e up to 240, plus carries
  void add_square(uint16_t b) {
    const int E = (b >> 7) & 0xFF;
    const int mant = b & 0x7F;
    if (E == 0xFF) { non_finite_ = true; return; }
    int64_t s;
    int e;
    if (E == 0) { s = mant; e = -133; } else { s = 128 + mant; e = E - 134; }
    const int k = 2 * e - kLow;
    bins_[k] += s * s;                              // < 2^16 per term
    if (k < lo_) lo_ = k;
    if (k > hi_) hi_ = k;
  }
  float rounded() const {
    if (non_finite_) return NAN;
    if (hi_ < 0) return 0.0f;
    // carry the bins into single bits: bit[k] has weight 2^(k + kLow); bins
    // below lo_ are empty, and 64 more bits above hi_ hold every carry
    std::vector<uint8_t> bit(kBins + 64, 0);
    int64_t carry = 0;
    int top = -1;
    for (int k = lo_; k < hi_ + 64; ++k) {
      const int64_t t = (k < kBins ? bins_[k] : 0) + carry;
      bit[k] = static_cast<uint8_t>(t & 1);
      carry = t >> 1;
      if (bit[k]) top = k;
    }
    if (top < 0) return 0.0f;
    // FP32: 24 significant bits, but no bit below 2^-149 (subnormals)
    const int top_exp = top + kLow;
    int lsb_exp = top_exp - 23;
    if (lsb_exp < -149) lsb_exp = -149;
    const int lsb = lsb_exp - kLow;  // bin index of the last kept bit
    double kept = 0.0;                // the kept bits, exact in double (<= 24 bits)
    for (int k = top; k >= lsb && k >= 0; --k) kept = kept * 2.0 + bit[k];
    bool round_bit = false, sticky = false;
    if (lsb - 1 >= 0) round_bit = bit[lsb - 1] != 0;
    for (int k = lsb - 2; k >= 0; --k) sticky = sticky || bit[k];
    const bool odd = std::fmod(kept, 2.0) != 0.0;
    if (round_bit && (sticky || odd)) kept += 1.0;
    const double v = std::ldexp(kept, lsb_exp);  // exact; may reach 2^(top_exp+1)
    return v > 3.4028234663852886e38 ? INFINITY : static_cast<float>(v);
  }

 private:
  int64_t bins_[kBins] = {};
  int lo_ = kBins, hi_ = -1;  // range of bins that received a term
  bool non_finite_ = false;
};

float fp32_sum_of_squares(const uint16_t* v, int64_t n) {
  ExactSquareSum acc;
  for (int64_t i = 0; i < n; ++i) acc.add_square(v[i]);
  return acc.rounded();
}

// r = 1 / sqrt(ss / width + eps): three FP32 operations and an FP32 square root.
float rms_scale(float ss, int64_t width, float eps) {
  const float ms = ss / static_cast<float>(width);
  const float v = ms + eps;
  return 1.0f / std::sqrt(v);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- step 1
// Input RMSNorm (minimax_h3_mlp_fp8_sm120, formula block, line n = ...):
// n[t, k] = bf16((x[t, k] * r_t) * w[k]), r_t = 1 / sqrt(ss_t / H + eps),
// ss_t the FP32 sum of squares of row t.  x: [T, H]; w: [H]; n_out: [T, H];
// r_out: [T] (may be null) receives r_t.
void mh3o_input_rmsnorm(const uint16_t* x, int64_t T, int64_t H, const uint16_t* w, float eps,
                        uint16_t* n_out, float* r_out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const uint16_t* xr = x + t * H;
    const float r = rms_scale(fp32_sum_of_squares(xr, H), H, eps);
    if (r_out) r_out[t] = r;
    for (int64_t k = 0; k < H; ++k)
      n_out[t * H + k] = bf16_round((bf16_value(xr[k]) * r) * bf16_value(w[k]));
  }
}

// The same normalisation with a given r per row (no sum of squares): lets a
// test ask what n would have been had the FP32 sum of squares come out one
// rounding step higher or lower.
void mh3o_rmsnorm_apply(const uint16_t* x, int64_t T, int64_t H, const uint16_t* w,
                        const float* r, uint16_t* n_out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t k = 0; k < H; ++k)
      n_out[t * H + k] = bf16_round((bf16_value(x[t * H + k]) * r[t]) * bf16_value(w[k]));
}

// ---------------------------------------------------------------- step 2
// Indexed AdaLN with the guard (formula block, lines a = ... and
// a[i outside [0, rows)] = 0; minimax_h3_bf16_pre_attention, Parameters:
// adaln_scale / adaln_shift (row strides), adaln_index (int64, guarded)):
// i = index[t]; if 0 <= i < rows,
//   a[t, k] = bf16(shift[i, k] + n[t, k] * bf16(1 + scale[i, k]))
// (unfused multiply then add), else a[t, :] = +0.  Table row i starts at
// scale + i * scale_stride (elements).
void mh3o_indexed_adaln(const uint16_t* n, int64_t T, int64_t H, const uint16_t* scale,
                        int64_t scale_stride, const uint16_t* shift, int64_t shift_stride,
                        int64_t rows, const int64_t* index, uint16_t* a_out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const int64_t i = index[t];
    uint16_t* ar = a_out + t * H;
    if (!(i >= 0 && i < rows)) {
      for (int64_t k = 0; k < H; ++k) ar[k] = 0;  // +0.0
      continue;
    }
    const uint16_t* sc = scale + i * scale_stride;
    const uint16_t* sh = shift + i * shift_stride;
    for (int64_t k = 0; k < H; ++k) {
      const float g = bf16_value(bf16_round(1.0f + bf16_value(sc[k])));
      const float prod = bf16_value(n[t * H + k]) * g;
      ar[k] = bf16_round(bf16_value(sh[k]) + prod);
    }
  }
}

// ---------------------------------------------------------------- step 3
// QKV projection with FP32 accumulation (minimax_h3_bf16_pre_attention,
// summary; Parameters: qkv_weight, rows in the order [kind, head, d]):
// y[t, c] = bf16(FP32(sum_k a[t, k] * W[c, k])), the sum taken in double in
// increasing k.  a: [T, K]; W: [N, K]; y_out: [T, N].
//
// The operands are first widened to FP32 arrays (exact).  The loops then
// visit four tokens and four columns at a time so that sixteen independent
// sums advance together; each of the sixteen is still one plain running sum
// over k = 0, 1, ..., K-1, so the result is that of the textbook triple loop.
void mh3o_qkv_projection(const uint16_t* a, int64_t T, int64_t K, const uint16_t* W, int64_t N,
                         uint16_t* y_out) {
  std::vector<float> af(static_cast<size_t>(T * K)), wf(static_cast<size_t>(N * K));
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < T * K; ++i) af[i] = bf16_value(a[i]);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N * K; ++i) wf[i] = bf16_value(W[i]);
  const int64_t tb = (T + 3) / 4;
  const int64_t cb = (N + 3) / 4;
#pragma omp parallel for schedule(dynamic, 16) collapse(2)
  for (int64_t bt = 0; bt < tb; ++bt) {
    for (int64_t bc = 0; bc < cb; ++bc) {
      const int64_t t0 = bt * 4, c0 = bc * 4;
      const float* a0 = &af[(t0 + 0 < T ? t0 + 0 : t0) * K];
      const float* a1 = &af[(t0 + 1 < T ? t0 + 1 : t0) * K];
      const float* a2 = &af[(t0 + 2 < T ? t0 + 2 : t0) * K];
      const float* a3 = &af[(t0 + 3 < T ? t0 + 3 : t0) * K];
      const float* w0 = &wf[(c0 + 0 < N ? c0 + 0 : c0) * K];
      const float* w1 = &wf[(c0 + 1 < N ? c0 + 1 : c0) * K];
      const float* w2 = &wf[(c0 + 2 < N ? c0 + 2 : c0) * K];
      const float* w3 = &wf[(c0 + 3 < N ? c0 + 3 : c0) * K];
      // s<i><j>: token t0 + i, column c0 + j; every product is exact in double
      double s00 = 0, s01 = 0, s02 = 0, s03 = 0, s10 = 0, s11 = 0, s12 = 0, s13 = 0;
      double s20 = 0, s21 = 0, s22 = 0, s23 = 0, s30 = 0, s31 = 0, s32 = 0, s33 = 0;
      for (int64_t k = 0; k < K; ++k) {
        const double x0 = a0[k], x1 = a1[k], x2 = a2[k], x3 = a3[k];
        const double v0 = w0[k], v1 = w1[k], v2 = w2[k], v3 = w3[k];
        s00 += x0 * v0; s01 += x0 * v1; s02 += x0 * v2; s03 += x0 * v3;
        s10 += x1 * v0; s11 += x1 * v1; s12 += x1 * v2; s13 += x1 * v3;
        s20 += x2 * v0; s21 += x2 * v1; s22 += x2 * v2; s23 += x2 * v3;
        s30 += x3 * v0; s31 += x3 * v1; s32 += x3 * v2; s33 += x3 * v3;
      }
      const double s[4][4] = {{s00, s01, s02, s03}, {s10, s11, s12, s13},
                              {s20, s21, s22, s23}, {s30, s31, s32, s33}};
      for (int i = 0; i < 4 && t0 + i < T; ++i)
        for (int j = 0; j < 4 && c0 + j < N; ++j)
          y_out[(t0 + i) * N + c0 + j] = bf16_round(static_cast<float>(s[i][j]));
    }
  }
}

// ---------------------------------------------------------------- step 4
// Per-head RMSNorm (summary; Parameters: q_norm_weight / k_norm_weight,
// qk_eps): for each head vector v of width D,
// t_d = bf16((v_d * rr) * w[d]), rr = 1 / sqrt(ss / D + qk_eps), ss the FP32
// sum of squares.  y: [R, D] head vectors; w: [D]; t_out: [R, D].
void mh3o_head_rmsnorm(const uint16_t* y, int64_t R, int64_t D, const uint16_t* w, float qk_eps,
                       uint16_t* t_out) {
#pragma omp parallel for schedule(static)
  for (int64_t h = 0; h < R; ++h) {
    const uint16_t* v = y + h * D;
    const float rr = rms_scale(fp32_sum_of_squares(v, D), D, qk_eps);
    for (int64_t d = 0; d < D; ++d)
      t_out[h * D + d] = bf16_round((bf16_value(v[d]) * rr) * bf16_value(w[d]));
  }
}

// ---------------------------------------------------------------- step 5a
// Cache row of each token (Parameters: rope_positions): clamp(pos[tok], 0,
// S - 1) in int64, or the identity tok when positions is null.
void mh3o_rope_cache_rows(const int64_t* positions, const int64_t* tokens, int64_t T, int64_t S,
                          int64_t* rows_out) {
  for (int64_t t = 0; t < T; ++t) {
    if (!positions) {
      rows_out[t] = tokens[t];
      continue;
    }
    int64_t p = positions[tokens[t]];
    if (p < 0) p = 0;
    if (p > S - 1) p = S - 1;
    rows_out[t] = p;
  }
}

// ---------------------------------------------------------------- step 5b
// Partial split-half NeoX RoPE (Parameters: rope_cos_sin): for head vectors
// t of width D belonging to token tok (heads_per_token of them in a row),
// with half = RD / 2, c = cs[p, j], s = cs[p, half + j] (p = rows[tok]):
//   o_j        = bf16(t_j * c - t_{j+half} * s)
//   o_{j+half} = bf16(t_{j+half} * c + t_j * s)
// for j < half, and o_d = t_d for d >= RD.  t: [T * heads_per_token, D];
// cs: [S, RD]; rows: [T]; o_out like t.
void mh3o_rope_split_half(const uint16_t* t, int64_t T, int64_t heads_per_token, int64_t D,
                          const uint16_t* cs, int64_t RD, const int64_t* rows, uint16_t* o_out) {
  const int64_t half = RD / 2;
#pragma omp parallel for schedule(static)
  for (int64_t tok = 0; tok < T; ++tok) {
    const uint16_t* row = cs + rows[tok] * RD;
    for (int64_t h = 0; h < heads_per_token; ++h) {
      const uint16_t* v = t + (tok * heads_per_token + h) * D;
      uint16_t* o = o_out + (tok * heads_per_token + h) * D;
      for (int64_t j = 0; j < half; ++j) {
        const float c = bf16_value(row[j]);
        const float s = bf16_value(row[half + j]);
        const float a = bf16_value(v[j]);
        const float b = bf16_value(v[half + j]);
        o[j] = bf16_round(a * c - b * s);
        o[half + j] = bf16_round(b * c + a * s);
      }
      for (int64_t d = RD; d < D; ++d) o[d] = v[d];
    }
  }
}

// ---------------------------------------------------------------- step 6
// Destination-major pack (Parameters: out [P, M, 56 // P, 3, 128],
// ulysses_degree): the per-token result qkv[m, h, kind, d] ([M, NH, 3, D])
// goes to out[dst, m, hl, kind, d] with dst = h / (NH / P), hl = h % (NH / P).
void mh3o_ulysses_pack(const uint16_t* qkv, int64_t M, int64_t NH, int64_t D, int64_t P,
                       uint16_t* out) {
  const int64_t hp = NH / P;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t h = 0; h < NH; ++h) {
      const int64_t dst = h / hp, hl = h % hp;
      for (int64_t kind = 0; kind < 3; ++kind)
        for (int64_t d = 0; d < D; ++d)
          out[(((dst * M + m) * hp + hl) * 3 + kind) * D + d] =
              qkv[((m * NH + h) * 3 + kind) * D + d];
    }
}

// ------------------------------------------------------------- whole stage
// Every step for the tokens listed in `tokens` (T of them), in the order of
// the summary paragraph: input RMSNorm, indexed AdaLN, QKV projection, Q/K
// RMSNorm (qk_eps), RoPE, and the per-token result qkv[T, NH, 3, D] before
// the pack (the pack only moves these values).  x: [M, H]; W: [3*NH*D, H]
// with rows [kind, head, d]; cs: [S, RD]; positions: [M] or null (identity,
// which needs S >= M: returns 1 otherwise).  n_out, a_out: [T, H]; y_out:
// [T, 3*NH*D]; qkv_out: [T, NH, 3, D]; r_out: [T]; any output may be null
// except qkv_out.
int mh3o_pre_attention_tokens(const uint16_t* x, int64_t M, int64_t H, const uint16_t* xw,
                              const uint16_t* scale, int64_t scale_stride, const uint16_t* shift,
                              int64_t shift_stride, int64_t rows, const int64_t* index,
                              const uint16_t* W, int64_t NH, int64_t D, const uint16_t* qw,
                              const uint16_t* kw, const uint16_t* cs, int64_t S, int64_t RD,
                              const int64_t* positions, float eps, float qk_eps,
                              const int64_t* tokens, int64_t T, uint16_t* n_out, uint16_t* a_out,
                              uint16_t* y_out, uint16_t* qkv_out, float* r_out) {
  if (!positions && S < M) return 1;
  const int64_t N = 3 * NH * D;
  std::vector<uint16_t> xs(static_cast<size_t>(T * H)), n(static_cast<size_t>(T * H)),
      a(static_cast<size_t>(T * H)), y(static_cast<size_t>(T * N));
  std::vector<int64_t> idx(static_cast<size_t>(T)), crow(static_cast<size_t>(T));
  std::vector<float> r(static_cast<size_t>(T));
  for (int64_t t = 0; t < T; ++t) {
    std::memcpy(&xs[t * H], x + tokens[t] * H, static_cast<size_t>(H) * 2);
    idx[t] = index[tokens[t]];
  }
  mh3o_input_rmsnorm(xs.data(), T, H, xw, eps, n.data(), r.data());
  mh3o_indexed_adaln(n.data(), T, H, scale, scale_stride, shift, shift_stride, rows, idx.data(),
                     a.data());
  mh3o_qkv_projection(a.data(), T, H, W, N, y.data());
  // y[t] = [q heads | k heads | v heads], each [NH, D]
  std::vector<uint16_t> q(static_cast<size_t>(T * NH * D)), k(q.size()), tq(q.size()),
      tk(q.size()), oq(q.size()), ok(q.size());
  for (int64_t t = 0; t < T; ++t) {
    std::memcpy(&q[t * NH * D], &y[t * N], static_cast<size_t>(NH * D) * 2);
    std::memcpy(&k[t * NH * D], &y[t * N + NH * D], static_cast<size_t>(NH * D) * 2);
  }
  mh3o_head_rmsnorm(q.data(), T * NH, D, qw, qk_eps, tq.data());
  mh3o_head_rmsnorm(k.data(), T * NH, D, kw, qk_eps, tk.data());
  mh3o_rope_cache_rows(positions, tokens, T, S, crow.data());
  mh3o_rope_split_half(tq.data(), T, NH, D, cs, RD, crow.data(), oq.data());
  mh3o_rope_split_half(tk.data(), T, NH, D, cs, RD, crow.data(), ok.data());
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < NH; ++h) {
      uint16_t* o = qkv_out + ((t * NH + h) * 3) * D;
      std::memcpy(o, &oq[(t * NH + h) * D], static_cast<size_t>(D) * 2);
      std::memcpy(o + D, &ok[(t * NH + h) * D], static_cast<size_t>(D) * 2);
      std::memcpy(o + 2 * D, &y[t * N + 2 * NH * D + h * D], static_cast<size_t>(D) * 2);
    }
  if (n_out) std::memcpy(n_out, n.data(), n.size() * 2);
  if (a_out) std::memcpy(a_out, a.data(), a.size() * 2);
  if (y_out) std::memcpy(y_out, y.data(), y.size() * 2);
  if (r_out) std::memcpy(r_out, r.data(), r.size() * 4);
  return 0;
}

// Threads OpenMP will use (for reporting the CPU baseline's core count).
int mh3o_max_threads() {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
