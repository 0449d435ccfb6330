// mlp.cu -- the two GEMMs of the MiniMax-H3 MLP block with BF16 operands, on
// the CTA-pair tcgen05 GEMM of gemm_pair.cuh (formula block of
// flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120 without its FP8 lines;
// the norm/AdaLN before them is kernel 1 of the pre-attention stage):
//
//   h   = bf16(a @ fc1^T)               FP32 accumulation; h = [h_gate | h_up]
//   y   = bf16(bf16(silu(h_gate)) * h_up)                     (fc1 epilogue)
//   o   = bf16(y @ fc2^T)               FP32 accumulation
//   out = bf16(residual + bf16(gate[i] * o)),  gate 0 for i outside [0, rows)
//
// fc1 tiling: y column block t (128 columns) needs h_gate[:, 128t + j] and
// h_up[:, 128t + j].  CTA 0 of a pair loads fc1 rows [128t, 128t + 128)
// (gate) and CTA 1 rows [14336 + 128t, ...) (up), so accumulator columns
// [0, 128) are h_gate and [128, 256) h_up for the same j, and the SwiGLU of
// a token is local to the thread that owns its TMEM lane.  K = 5376 = 84
// k-blocks, 112 column blocks; y leaves through the staging buffer by 2-D TMA
// stores.  fc2 is the gated-residual policy of gated_residual_epi.cuh with
// K = 14336 = 224 k-blocks and the int64 AdaLN index.
//
// FP8 (W8A8) form, the page's own formula block: E4M3 a_q (kernel 1's E4M3
// form) and E4M3 weights with FP32 per-row scales, kind::f8f6f4 MMAs over
// 128-byte k-blocks (K = 5376 = 42 and 14336 = 112 of them), and
//   h   = bf16(RN(RN(acc * s_a[m]) * fc1_scale[c]))               (fc1 epilogue)
//   y   = bf16(bf16(silu(h_gate)) * h_up); amax_row(|y|) folded in by atomicMax
//   y_q = e4m3(y / s_y), s_y = RN(amax_row(|y|) / 448)           (y quantiser)
//   o   = bf16(RN(RN(acc * s_y[m]) * fc2_scale[c])), then the gated residual
// The y quantiser is a separate HBM-bound pass: s_y needs the whole row of
// y, which 112 different tiles produce.
#include "e4m3_rows.cuh"
#include "gated_residual_epi.cuh"

namespace mh3 {

namespace {

using namespace k2;

static_assert(kMlpInter % kHeadDim == 0, "y column blocks of 128");
static_assert(kMlpInter % BK == 0, "fc2 K must tile");

// silu(v) = v * (1 / (1 + exp(-v))) in FP32 from the fast exponential and
// reciprocal (__expf, __fdividef): branch-free, so the 32 outputs of a TMEM
// load interleave, and within a few FP32 ulps; the value is rounded to bf16
// at once, where those ulps move about one value in 10^4 by one bf16 step.
// For v < -87, 1 + exp(-v) exceeds 2^126 and the reciprocal is 0: silu = -0.
__device__ __forceinline__ float silu_f32(float v) {
  return __fmul_rn(v, __fdividef(1.0f, __fadd_rn(1.0f, __expf(-v))));
}

struct SwigluEpi {
  using Params = SwigluParams;
  static constexpr bool kFp8 = false;
  static constexpr int kKBlocks = kHidden / BK;          // 84
  static constexpr int kNTiles = kMlpInter / kHeadDim;    // 112
  __device__ static int b_row(int n_blk, int rank) {
    return (rank == 0 ? 0 : kMlpInter) + n_blk * kHeadDim;
  }
  __device__ static void prologue(float*, int, int, const Params&) {}

  __device__ static void tile(const gp::EpiCtx& c, const Params& p, int64_t row0, int n_blk) {
    const int lane = c.lane;
    const int64_t m0 = row0 + c.quad * 32;
    const int col0 = n_blk * kHeadDim;
    const uint32_t tl = c.tmem_acc + (static_cast<uint32_t>(c.quad * 32) << 16);
    // the previous store from this staging buffer must have read it
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t gv[32], uv[32];
      tmem_ld_x32(tl + 32 * q, gv);
      tmem_ld_x32(tl + kHeadDim + 32 * q, uv);
      tmem_wait_ld();
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float y2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int i = 8 * g + 2 * e + h;
            const float hg = round_bf16(__uint_as_float(gv[i]));
            const float hu = round_bf16(__uint_as_float(uv[i]));
            y2[h] = __fmul_rn(round_bf16(silu_f32(hg)), hu);
          }
          ow[e] = pack_bf16x2(y2[0], y2[1]);
        }
        st_shared_v4(stg_addr(c.stg, lane, 4 * q + g), make_uint4(ow[0], ow[1], ow[2], ow[3]));
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && m0 < p.M) {
      tma_store_2d(c.tm_out, c.stg, col0, static_cast<int32_t>(m0));
      tma_store_2d(c.tm_out, c.stg + kStgHalfBytes, col0 + 64, static_cast<int32_t>(m0));
      bulk_commit_group();
    }
  }
};

using Fc2Epi = gr::GatedResidualEpi<kMlpInter / BK, int64_t>;

// fc1 + SwiGLU with E4M3 operands: the rescaled accumulator, the same
// SwiGLU, and the row's largest |y| folded into y_amax.
struct Fc1Fp8Epi {
  using Params = SwigluParams;
  static constexpr bool kFp8 = true;
  static constexpr int kKBlocks = kHidden / 128;          // 42
  static constexpr int kNTiles = kMlpInter / kHeadDim;    // 112
  __device__ static int b_row(int n_blk, int rank) { return SwigluEpi::b_row(n_blk, rank); }
  __device__ static void prologue(float*, int, int, const Params&) {}

  __device__ static void tile(const gp::EpiCtx& c, const Params& p, int64_t row0, int n_blk) {
    const int lane = c.lane;
    const int64_t m0 = row0 + c.quad * 32;
    if (m0 >= p.M) return;  // no row of this warp is stored
    const int64_t m = m0 + lane;
    const float rs = m < p.M ? __ldg(p.row_scale + m) : 0.0f;
    const int col0 = n_blk * kHeadDim;
    const float* gs = p.col_scale + col0;               // gate rows' scales
    const float* us = p.col_scale + kMlpInter + col0;   // up rows' scales
    const uint32_t tl = c.tmem_acc + (static_cast<uint32_t>(c.quad * 32) << 16);
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
    float ymax = 0.0f;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t gv[32], uv[32];
      tmem_ld_x32(tl + 32 * q, gv);
      tmem_ld_x32(tl + kHeadDim + 32 * q, uv);
      tmem_wait_ld();
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int j0 = 32 * q + 8 * g;
        const float4 ga = __ldg(reinterpret_cast<const float4*>(gs + j0));
        const float4 gb = __ldg(reinterpret_cast<const float4*>(gs + j0 + 4));
        const float4 ua = __ldg(reinterpret_cast<const float4*>(us + j0));
        const float4 ub = __ldg(reinterpret_cast<const float4*>(us + j0 + 4));
        const float gsc[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
        const float usc[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float y2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int i = 8 * g + 2 * e + h;
            const float hg =
                round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(gv[i]), rs), gsc[2 * e + h]));
            const float hu =
                round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(uv[i]), rs), usc[2 * e + h]));
            y2[h] = round_bf16(__fmul_rn(round_bf16(silu_f32(hg)), hu));
            ymax = fmaxf(ymax, fabsf(y2[h]));
          }
          ow[e] = pack_bf16x2(y2[0], y2[1]);
        }
        st_shared_v4(stg_addr(c.stg, lane, 4 * q + g), make_uint4(ow[0], ow[1], ow[2], ow[3]));
      }
    }
    // |y| >= 0: its FP32 bits order as unsigned integers
    if (m < p.M) atomicMax(p.y_amax + m, __float_as_uint(ymax));
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(c.tm_out, c.stg, col0, static_cast<int32_t>(m0));
      tma_store_2d(c.tm_out, c.stg + kStgHalfBytes, col0 + 64, static_cast<int32_t>(m0));
      bulk_commit_group();
    }
  }
};

using Fc2Fp8Epi = gr::GatedResidualEpi<kMlpInter / 128, int64_t, true>;

// y_q = e4m3(y / s_y) per row: CTA b takes rows b, b + G, ...; the row's
// amax (FP32 bits, from fc1) is read by every thread, then replaced by s_y.
constexpr int kQyThreads = 256;
__global__ void __launch_bounds__(kQyThreads) quantize_y_kernel(const __nv_bfloat16* __restrict__ y,
                                                                int64_t M,
                                                                unsigned int* amax_then_scale,
                                                                uint8_t* __restrict__ y_q) {
  constexpr int kChunks = kMlpInter / 8;  // 1792 eight-element chunks per row
  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    const float amax = __uint_as_float(amax_then_scale[m]);
    __syncthreads();  // every thread has read the amax
    const e4m3r::RowScale rs = e4m3r::make_row_scale(amax);
    if (threadIdx.x == 0) amax_then_scale[m] = __float_as_uint(rs.s);
    const uint4* src = reinterpret_cast<const uint4*>(y + m * kMlpInter);
    uint2* dst = reinterpret_cast<uint2*>(y_q + m * kMlpInter);
    for (int c = threadIdx.x; c < kChunks; c += kQyThreads)
      dst[c] = e4m3r::quantize8(__ldcs(src + c), rs);
  }
}

}  // namespace

cudaError_t mlp_fc1_prepare_device(int* max_clusters) {
  return gp::gemm_pair_prepare<SwigluEpi>(max_clusters);
}

cudaError_t launch_mlp_fc1(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y,
                           const SwigluParams& p, int clusters, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  // no auxiliary input: the output map stands in for the unused operand
  return gp::gemm_pair_launch<SwigluEpi>(a, b, y, y, p, clusters, stream);
}

cudaError_t mlp_fc2_prepare_device(int* max_clusters) {
  return gp::gemm_pair_prepare<Fc2Epi>(max_clusters);
}

cudaError_t launch_mlp_fc2(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                           const CUtensorMap& residual, const GatedResidualParams<int64_t>& p,
                           int clusters, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  return gp::gemm_pair_launch<Fc2Epi>(a, b, out, residual, p, clusters, stream);
}

}  // namespace mh3

namespace mh3 {

cudaError_t mlp_fp8_fc1_prepare_device(int* max_clusters) {
  return gp::gemm_pair_prepare<Fc1Fp8Epi>(max_clusters);
}

cudaError_t launch_mlp_fp8_fc1(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y,
                               const SwigluParams& p, int clusters, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  return gp::gemm_pair_launch<Fc1Fp8Epi>(a, b, y, y, p, clusters, stream);
}

cudaError_t launch_mlp_quantize_y(const __nv_bfloat16* y, int64_t M, float* amax_then_scale,
                                  uint8_t* y_q, int num_sms, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  const int64_t want = static_cast<int64_t>(num_sms) * 8;
  const int64_t grid = M < want ? M : want;
  quantize_y_kernel<<<static_cast<unsigned>(grid), kQyThreads, 0, stream>>>(
      y, M, reinterpret_cast<unsigned int*>(amax_then_scale), y_q);
  return cudaGetLastError();
}

cudaError_t mlp_fp8_fc2_prepare_device(int* max_clusters) {
  return gp::gemm_pair_prepare<Fc2Fp8Epi>(max_clusters);
}

cudaError_t launch_mlp_fp8_fc2(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                               const CUtensorMap& residual, const GatedResidualParams<int64_t>& p,
                               int clusters, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  return gp::gemm_pair_launch<Fc2Fp8Epi>(a, b, out, residual, p, clusters, stream);
}

}  // namespace mh3
