// common.cuh -- sizes, parameter blocks and small bf16 helpers shared by the
// two kernels and the C-ABI host code of the pre-attention stage.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mh3 {

// Fixed by flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention (Parameters:
// x [M, 5376], qkv_weight [21504, 5376], q/k_norm_weight [128],
// rope_cos_sin [S, 96], out [P, M, 56 // P, 3, 128]).
constexpr int kHidden = 5376;
constexpr int kHeads = 56;
constexpr int kHeadDim = 128;
constexpr int kQkvRows = 3 * kHeads * kHeadDim;  // 21504
constexpr int kKindCols = kHeads * kHeadDim;     // 7168 columns per q/k/v kind
constexpr int kRopeDims = 96;
constexpr int kRopeHalf = kRopeDims / 2;  // 48

// Device status codes (first writer wins): which bounded wait gave up.
enum : int {
  kStatusOk = 0,
  kStatusProducerEmpty = 0x101,
  kStatusMmaFull = 0x102,
  kStatusMmaTmemEmpty = 0x103,
  kStatusEpiTmemFull = 0x104,
  kStatusDrain = 0x105,
  kStatusRowFull = 0x106,
  kStatusEpiResidual = 0x107,
  kStatusSplitPartial = 0x108,  // an owner of a split tile waited for the other half's partial
};

struct NormAdalnParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* x_norm_weight;
  const __nv_bfloat16* scale;
  const __nv_bfloat16* shift;
  int64_t scale_stride;  // elements
  int64_t shift_stride;  // elements
  int64_t rows;
  const int64_t* index;
  __nv_bfloat16* workspace;
  int64_t M;
  float eps;
  int* status;  // device status word (bounded-wait timeouts)
  // NVFP4 form (act_q != nullptr): int32 indices; the quantised activation
  // replaces the bf16 workspace
  const int32_t* index32 = nullptr;
  uint8_t* act_q = nullptr;      // [M, 2688] packed E2M1
  uint8_t* act_sf = nullptr;     // UE4M3 scales, tiled atoms or row-major [M, 336]
  const float* act_gs = nullptr; // device [1]: activation global scale
  int sf_tiled = 1;
  // E4M3 form (a_q8 != nullptr, int64 indices): per token s = RN(amax|a| / 448)
  // and codes e4m3(a / s) replace the bf16 workspace
  uint8_t* a_q8 = nullptr;  // [M, 5376]
  float* a_s8 = nullptr;    // [M]
  // ints cleared by CTA 0 for the kernel that follows (the split-tail flags
  // of the QKV GEMM, which reads them only after this grid has completed)
  int* clear = nullptr;
  int clear_count = 0;
};

struct QkvParams {
  const int64_t* positions;  // [M] or nullptr (identity)
  const __nv_bfloat16* cos_sin;  // [S, 96]
  const __nv_bfloat16* q_norm_weight;  // [128]
  const __nv_bfloat16* k_norm_weight;  // [128]
  int64_t M;
  int64_t S;
  int heads_per_dst;  // 56 / P
  float qk_eps;
  int num_m_tiles;  // row blocks: of 128 rows (single-CTA form) or 256 (pair form)
  int num_tiles;    // num_m_tiles * 84
  const float* descales;  // e4m3 output mode: q, k, v dequantisation scales (device)
  int* status;  // device status word
  // NVFP4 stage: y = bf16(RN(alpha * acc)); alpha given (finite, > 0) or
  // derived on the device as RN(1 / RN(act_gs * w_gs))
  float alpha = 1.0f;
  const float* act_gs = nullptr;  // device [1]
  float w_gs = 0.0f;
  int test_stall = 0;  // test hook: the producer issues no loads (bounded waits run out)
  // Split tail of the CTA-pair form: tiles [0, sk_dp) whole, then tiles
  // sk_dp + j (j < sk_tail) split along K over clusters 2j (first half: its
  // FP32 partial goes to sk_partial, then its flag is set to sk_seq; the
  // flags are cleared before every launch) and 2j + 1 (second half: adds the
  // partial, then the epilogue).  sk_tail = 0: no split.
  int sk_dp = 0;
  int sk_tail = 0;
  float* sk_partial = nullptr;  // [sk_tail][2 CTAs][4 warps][256 columns][32 lanes]
  int* sk_flags = nullptr;      // [sk_tail][2][4]
  int sk_seq = 0;
  // The grid before this one is the stage's kernel 1, which writes A alone:
  // the pair form may load the weight boxes of its first stages before it
  // waits for that grid (0: wait first, as for a caller's kernel).
  int b_early = 0;
  // NVFP4 output mode of the NVFP4 stage: q, k, v global scales (device [3]),
  // codes [P, M, 56/P, 3, 64] and block scales [P, M, 56/P, 3, 8]
  const float* out_gs = nullptr;
  uint8_t* out_codes = nullptr;
  uint8_t* out_sf = nullptr;
};

// num_sms: SM count of the device (the kernel is persistent over rows).
cudaError_t launch_norm_adaln(const NormAdalnParams& p, int num_sms, cudaStream_t stream);

// Tensor maps are encoded by the host for each call.
struct QkvMaps {
  CUtensorMap a;    // workspace [M, 5376], box 64 x 128, 128-B swizzle
  CUtensorMap b;    // qkv_weight [21504, 5376], box 64 x 256 (single) / 64 x 128 (pair)
  CUtensorMap out;  // out as 4-D (d 128, slot 168/P, m M, dst P), box 64x1x32x1
};

// NVFP4 pre-attention, kernel 2: block-scaled FP4 CTA-pair GEMM with the
// QKV epilogue (two heads per 256 x 256 tile).
struct Nvfp4Maps {
  CUtensorMap a;    // act_q [M, 2688] bytes, box 128 B x 128 rows, 128-B swizzle
  CUtensorMap b;    // weight codes [21504, 2688] bytes, box 128 B x 128 rows, 128-B swizzle
  CUtensorMap sfa;  // act scales, tiled atoms as u32 (128, 84, ceil(M/128)), box 128 x 4 x 1
  CUtensorMap sfb;  // weight scales, tiled atoms as u32 (128, 84, 168), box 128 x 4 x 2
  CUtensorMap out;  // as QkvMaps::out (bf16) or the e4m3 byte map; out-projection: [M, 5376]
  CUtensorMap aux;  // out-projection: residual [M, 5376], box 64 x 32
};
// Output forms of the NVFP4 stage's GEMM.
constexpr int kOutBf16 = 0;
constexpr int kOutE4m3 = 1;
constexpr int kOutNvfp4 = 2;
cudaError_t nvfp4_qkv_prepare_device(int* max_clusters, int* max_clusters_e4m3,
                                     int* max_clusters_nvfp4);
cudaError_t launch_nvfp4_qkv(const Nvfp4Maps& maps, const QkvParams& p, int clusters, int out_mode,
                             cudaStream_t stream);

// W4A4 output projection with the gated residual (the same block-scaled GEMM):
//   o = bf16(RN(alpha * acc)), out = bf16(residual + bf16(g * o)).
//   a: attn codes [M, 3584] bytes; b: o_weight codes [5376, 3584]; scales tiled.
struct Nvfp4OutProjParams {
  int64_t M;
  int num_m_tiles;  // 256-row blocks
  int num_tiles;    // num_m_tiles * 21
  int* status;
  int test_stall = 0;
  float alpha = 1.0f;              // given (finite, > 0) or derived as in QkvParams
  const float* act_gs = nullptr;
  float w_gs = 0.0f;
  const __nv_bfloat16* gate;       // [gate_rows, 5376] view
  int64_t gate_stride;
  int64_t gate_rows;
  const int32_t* gate_index;       // [M]
};
cudaError_t nvfp4_out_proj_prepare_device(int* max_clusters);
cudaError_t launch_nvfp4_out_proj(const Nvfp4Maps& maps, const Nvfp4OutProjParams& p,
                                  int clusters, cudaStream_t stream);

// Standalone NVFP4 quantiser: rows x cols bf16 (cols a multiple of 64) ->
// packed codes [rows, cols/2] and scales (tiled atoms or row-major).
cudaError_t launch_nvfp4_quantize(const __nv_bfloat16* in, int64_t rows, int cols, const float* gs,
                                  uint8_t* codes, uint8_t* scales, bool tiled, int num_sms,
                                  cudaStream_t stream);

// ----------------------------------------- attention output projection
// out = bf16(residual + bf16(gate[gate_index[m]] * bf16(attn_out @ o_weight^T)))
constexpr int kAttnWidth = kHeads * kHeadDim;  // 7168

// Parameters of a GEMM whose epilogue applies the gated residual
// out = bf16(residual + bf16(gate[index[m]] * o)); IndexT is the index type.
template <typename IndexT>
struct GatedResidualParams {
  const __nv_bfloat16* gate;  // [gate_rows, 5376] view
  int64_t gate_stride;        // elements
  int64_t gate_rows;
  const IndexT* gate_index;   // [M]
  int64_t M;
  int num_m_tiles;  // 256-row blocks
  int num_tiles;    // num_m_tiles * 21
  int* status;
  int test_stall = 0;  // test hook: the producer issues no loads (bounded waits run out)
  // E4M3 operands (MLP fc2): o = bf16(RN(RN(acc * row_scale[m]) * col_scale[c]))
  const float* row_scale = nullptr;  // [M]
  const float* col_scale = nullptr;  // [5376]
};
using OutProjParams = GatedResidualParams<int32_t>;

struct OutProjMaps {
  CUtensorMap a;         // attn_out [M, 7168], box 64 x 128, 128-B swizzle
  CUtensorMap b;         // o_weight [5376, 7168], box 64 x 128, 128-B swizzle
  CUtensorMap out;       // out [M, 5376], box 64 x 32, 128-B swizzle (store)
  CUtensorMap residual;  // residual [M, 5376], box 64 x 32, 128-B swizzle (load)
};

cudaError_t out_proj_prepare_device(int* max_clusters);
cudaError_t launch_out_proj(const OutProjMaps& maps, const OutProjParams& p, int clusters,
                            cudaStream_t stream);

// ------------------------------------------------------------- the MLP block
constexpr int kMlpInter = 14336;  // SwiGLU width; fc1 rows [gate | up] = 28672

struct SwigluParams {
  int64_t M;
  int num_m_tiles;  // 256-row blocks
  int num_tiles;    // num_m_tiles * 112
  int* status;
  int test_stall = 0;  // test hook: the producer issues no loads (bounded waits run out)
  // E4M3 operands (FP8 block): h = bf16(RN(RN(acc * row_scale[m]) * col_scale[c])),
  // and the largest |y| of every row is folded into y_amax[m] (FP32 bits)
  const float* row_scale = nullptr;  // [M]
  const float* col_scale = nullptr;  // [28672]
  unsigned int* y_amax = nullptr;    // [M], zero before the launch
};

// fc1 + SwiGLU: y = bf16(bf16(silu(h_gate)) * h_up), h = bf16(a @ fc1^T).
//   a: workspace [M, 5376]; b: fc1 [28672, 5376]; out: y [M, 14336] (store).
cudaError_t mlp_fc1_prepare_device(int* max_clusters);
cudaError_t launch_mlp_fc1(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y,
                           const SwigluParams& p, int clusters, cudaStream_t stream);
// fc2 + gated residual: out = bf16(residual + bf16(gate[i] * bf16(y @ fc2^T))).
//   a: y [M, 14336]; b: fc2 [5376, 14336]; out, residual: [M, 5376].
// The FP8 (W8A8) block: fc1 on E4M3 operands with the rescale, SwiGLU and
// row amax of y; the y quantiser (s_y replaces the amax in place); fc2 on E4M3
// operands with the rescale and the gated residual.  a / b maps are uint8
// with 128-byte rows (box 128 x 128).
cudaError_t mlp_fp8_fc1_prepare_device(int* max_clusters);
cudaError_t launch_mlp_fp8_fc1(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y,
                               const SwigluParams& p, int clusters, cudaStream_t stream);
cudaError_t launch_mlp_quantize_y(const __nv_bfloat16* y, int64_t M, float* amax_then_scale,
                                  uint8_t* y_q, int num_sms, cudaStream_t stream);
cudaError_t mlp_fp8_fc2_prepare_device(int* max_clusters);
cudaError_t launch_mlp_fp8_fc2(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                               const CUtensorMap& residual, const GatedResidualParams<int64_t>& p,
                               int clusters, cudaStream_t stream);
cudaError_t mlp_fc2_prepare_device(int* max_clusters);
cudaError_t launch_mlp_fc2(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                           const CUtensorMap& residual, const GatedResidualParams<int64_t>& p,
                           int clusters, cudaStream_t stream);

// The pair form with e4m3 outputs: out as 4-D uint8 (d 128, slot, m, dst),
// box 128 x 1 x 32 x 1.
cudaError_t qkv_e4m3_prepare_device(int* max_clusters);
cudaError_t launch_qkv_e4m3(const QkvMaps& maps, const QkvParams& p, int clusters,
                            cudaStream_t stream);

// Standalone per-tensor e4m3 quantiser: out[i] = e4m3_sat(RN32(in[i] / *descale)).
cudaError_t launch_e4m3_quantize(const __nv_bfloat16* in, const float* descale, uint8_t* out,
                                 int64_t n, int num_sms, cudaStream_t stream);

// Single-CTA form (128 x 256 tiles), used for M <= 128.
int qkv_smem_bytes();
cudaError_t qkv_prepare_device();  // raise the dynamic shared-memory limit
cudaError_t launch_qkv(const QkvMaps& maps, const QkvParams& p, int grid, cudaStream_t stream);

// CTA-pair form (256 x 256 tiles on two SMs), used for M > 128.
int qkv_pair_smem_bytes();
// Raises the shared-memory limit and reports how many 2-CTA clusters can be
// resident at once (0: the pair form cannot run on this device).
cudaError_t qkv_pair_prepare_device(int* max_clusters);
cudaError_t launch_qkv_pair(const QkvMaps& maps, const QkvParams& p, int clusters,
                            cudaStream_t stream);

// --------------------------------------------------------------- bf16 bits
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Round an FP32 value to bf16 (nearest-even) and return it as FP32.
__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Two FP32 values -> packed bf16x2 (lo in bits 0-15), nearest-even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace mh3
