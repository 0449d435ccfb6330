// nvfp4_quantize.cu -- the NVFP4 block quantiser of nvfp4.cuh as a
// standalone kernel for any bf16 matrix (rows x cols, cols a multiple of 64):
// the weight preparation of the NVFP4 stage (the role of the page's
// quantize_minimax_h3_qkv_weight_nvfp4) and a direct check of the
// quantisation the stage's first kernel applies to the activation.
// One thread per (row, 64-element step): 128 B of input, 32 B of codes and
// one 4-byte scale word out.
#include "nvfp4.cuh"

namespace mh3 {

namespace {

__global__ void __launch_bounds__(256) nvfp4_quantize_kernel(const __nv_bfloat16* __restrict__ in,
                                                             int64_t rows, int cols,
                                                             const float* __restrict__ gs_ptr,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales,
                                                             int tiled) {
  const float gs = __ldg(gs_ptr);
  const fp4::Quantiser quant = fp4::make_quantiser(gs);
  __shared__ float2 enc_lut[fp4::kEncLut];
  fp4::init_enc_lut(enc_lut, gs, threadIdx.x, blockDim.x);
  __syncthreads();
  const int ksteps = cols / 64;
  // grid-stride over (row, step) items, the index pair advanced without a
  // division per item
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t stride_rows = stride / ksteps;
  const int stride_ks = static_cast<int>(stride - stride_rows * ksteps);
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t row = t0 / ksteps;
  int ks = static_cast<int>(t0 - row * ksteps);
  for (; row < rows; row += stride_rows, ks += stride_ks) {
    if (ks >= ksteps) {
      ks -= ksteps;
      if (++row >= rows) break;
    }
    const uint4* src = reinterpret_cast<const uint4*>(in + row * cols + ks * 64);
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldg(src + i);
    uint32_t q[8];
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float amax = fmaxf(fp4::amax8(v[2 * b]), fp4::amax8(v[2 * b + 1]));
      const fp4::BlockScale bs = fp4::block_scale(amax, quant, enc_lut);
      q[2 * b] = fp4::encode8(v[2 * b], bs, gs);
      q[2 * b + 1] = fp4::encode8(v[2 * b + 1], bs, gs);
      word |= bs.code << (8 * b);
    }
    uint4* dst = reinterpret_cast<uint4*>(codes + row * (cols / 2) + ks * 32);
    dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
    dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
    *reinterpret_cast<uint32_t*>(scales + fp4::scale_offset(row, ks, ksteps, tiled != 0)) = word;
  }
}

}  // namespace

cudaError_t launch_nvfp4_quantize(const __nv_bfloat16* in, int64_t rows, int cols, const float* gs,
                                  uint8_t* codes, uint8_t* scales, bool tiled, int num_sms,
                                  cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int64_t work = rows * (cols / 64);
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  nvfp4_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(in, rows, cols, gs, codes,
                                                                           scales, tiled ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace mh3
