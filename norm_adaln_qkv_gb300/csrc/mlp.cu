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
#include "gated_residual_epi.cuh"

namespace mh3 {

namespace {

using namespace k2;

static_assert(kMlpInter % kHeadDim == 0, "y column blocks of 128");
static_assert(kMlpInter % BK == 0, "fc2 K must tile");

// silu(v) = v / (1 + exp(-v)) in FP32 (expf, IEEE add and division).
__device__ __forceinline__ float silu_f32(float v) {
  return __fdiv_rn(v, __fadd_rn(1.0f, expf(-v)));
}

struct SwigluEpi {
  using Params = SwigluParams;
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
