// out_proj.cu -- the attention output projection with the fused gated
// residual, on the CTA-pair tcgen05 GEMM of gemm_pair.cuh:
//
//   o   = bf16(attn_out @ o_weight^T)                FP32 accumulation (TMEM)
//   out = bf16(residual + bf16(g * o)),  g = gate[gate_index[m]], or 0 when
//         gate_index[m] lies outside [0, gate_rows) (out = residual)
//
// (flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj, summary formula and
// Parameters: attn_out [M, 7168], gate [9, 5376] rows of the AdaLN plan,
// gate_index int32 [M], residual [M, 5376], out [M, 5376]; computed here with
// BF16 operands.)  A: attn_out, K = 7168 = 112 k-blocks; B: o_weight
// [5376, 7168], N = 5376 = 21 tiles of 256.  The epilogue is the gated
// residual policy of gated_residual_epi.cuh.
#include "gated_residual_epi.cuh"

namespace mh3 {

namespace {

static_assert(kAttnWidth % k2::BK == 0, "K must tile");
using OutProjEpi = gr::GatedResidualEpi<kAttnWidth / k2::BK, int32_t>;

}  // namespace

cudaError_t out_proj_prepare_device(int* max_clusters) {
  return gp::gemm_pair_prepare<OutProjEpi>(max_clusters);
}

cudaError_t launch_out_proj(const OutProjMaps& maps, const OutProjParams& p, int clusters,
                            cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  return gp::gemm_pair_launch<OutProjEpi>(maps.a, maps.b, maps.out, maps.residual, p, clusters,
                                          stream);
}

}  // namespace mh3
