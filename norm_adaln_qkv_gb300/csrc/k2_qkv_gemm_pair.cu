// k2_qkv_gemm_pair.cu -- kernel 2 of the pre-attention stage, CTA-pair form
// (M > 128): the QKV projection acc = workspace @ qkv_weight^T on the
// CTA-pair tcgen05 GEMM of gemm_pair.cuh, with the fused Q/K RMSNorm, RoPE
// and destination-major pack epilogue of k2_common.cuh
// (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention, summary and
// Parameters: qkv_weight, q/k_norm_weight, qk_eps, rope_cos_sin,
// rope_positions, out).
//
// A: workspace [M, 5376]; B: qkv_weight [21504, 5376] (rows in the order
// [kind, head, head_dim]); K = 5376 = 84 k-blocks; N = 21504 = 84 tiles of two
// heads of one kind.
#include "gemm_pair.cuh"

namespace mh3 {

namespace {

template <bool kE4m3>
struct QkvPairEpiT {
  using Params = QkvParams;
  static constexpr bool kFp8 = false;
  static constexpr bool kSplitTail = true;  // takes part in the split tail (p.sk_*)
  static constexpr int kKBlocks = k2::kKBlocks;  // 84
  static constexpr int kNTiles = k2::kNTiles;    // 84
  __device__ static int b_row(int n_blk, int rank) { return gp::contiguous_b_row(n_blk, rank); }

  // q then k norm weights, as FP32, into the epilogue scratch.
  __device__ static void prologue(float* scratch, int tid, int nthreads, const Params& p) {
    for (int i = tid; i < 2 * kHeadDim; i += nthreads) {
      const __nv_bfloat16 w = i < kHeadDim ? p.q_norm_weight[i] : p.k_norm_weight[i - kHeadDim];
      scratch[i] = __bfloat162float(w);
    }
  }

  __device__ static void tile(const gp::EpiCtx& c, const Params& p, int64_t row0, int n_blk) {
    k2::epilogue_block<kE4m3>(c.tmem_acc, c.quad, c.lane, c.stg, c.scratch, p, row0, n_blk,
                              c.tm_out);
  }
};
using QkvPairEpi = QkvPairEpiT<false>;
using QkvE4m3PairEpi = QkvPairEpiT<true>;

}  // namespace

int qkv_pair_smem_bytes() { return gp::kSmemAlloc; }

cudaError_t qkv_pair_prepare_device(int* max_clusters) {
  return gp::gemm_pair_prepare<QkvPairEpi>(max_clusters);
}

cudaError_t launch_qkv_pair(const QkvMaps& maps, const QkvParams& p, int clusters,
                            cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  // no auxiliary input: the output map stands in for the unused operand
  return gp::gemm_pair_launch<QkvPairEpi>(maps.a, maps.b, maps.out, maps.out, p, clusters, stream);
}

cudaError_t qkv_e4m3_prepare_device(int* max_clusters) {
  return gp::gemm_pair_prepare<QkvE4m3PairEpi>(max_clusters);
}

cudaError_t launch_qkv_e4m3(const QkvMaps& maps, const QkvParams& p, int clusters,
                            cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  return gp::gemm_pair_launch<QkvE4m3PairEpi>(maps.a, maps.b, maps.out, maps.out, p, clusters,
                                              stream);
}

}  // namespace mh3
