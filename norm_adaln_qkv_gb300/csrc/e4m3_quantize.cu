// e4m3_quantize.cu -- the per-tensor e4m3 quantiser of e4m3.cuh as a
// standalone elementwise kernel: codes[i] = e4m3_sat(RN32(values[i] /
// descale)) for a bf16 tensor of any length (the conversion the stage's e4m3
// epilogue applies to each output tensor).  Grid-stride; eight elements per
// step when `values` is 16-byte and `codes` 8-byte aligned, one at a time
// otherwise.  HBM-bound: 3 bytes per element.
#include "e4m3.cuh"

namespace mh3 {

namespace {

__global__ void __launch_bounds__(256) e4m3_quantize_kernel(const __nv_bfloat16* __restrict__ in,
                                                            const float* __restrict__ descale,
                                                            uint8_t* __restrict__ out, int64_t n,
                                                            int vec) {
  const e4m3q::Divisor dv = e4m3q::make_divisor(__ldg(descale));
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (vec) {
    const int64_t n8 = n / 8;
    const uint4* in8 = reinterpret_cast<const uint4*>(in);
    uint2* out8 = reinterpret_cast<uint2*>(out);
    if (dv.fast) {
      for (int64_t i = tid; i < n8; i += stride) out8[i] = e4m3q::quantize8<true>(__ldg(in8 + i), dv);
    } else {
      for (int64_t i = tid; i < n8; i += stride) out8[i] = e4m3q::quantize8<false>(__ldg(in8 + i), dv);
    }
    done = n8 * 8;
  }
  const uint16_t* in1 = reinterpret_cast<const uint16_t*>(in);
  for (int64_t i = done + tid; i < n; i += stride) {
    const uint32_t w = __ldg(in1 + i);  // element in the low half, 0 above
    const uint32_t c = dv.fast ? e4m3q::quantize_word<true>(w, dv)
                               : e4m3q::quantize_word<false>(w, dv);
    out[i] = static_cast<uint8_t>(c & 0xFFu);
  }
}

}  // namespace

cudaError_t launch_e4m3_quantize(const __nv_bfloat16* in, const float* descale, uint8_t* out,
                                 int64_t n, int num_sms, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int vec = (reinterpret_cast<uintptr_t>(in) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(out) % 8 == 0) ? 1 : 0;
  const int64_t work = vec ? (n + 7) / 8 : n;
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  e4m3_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(in, descale, out, n, vec);
  return cudaGetLastError();
}

}  // namespace mh3
