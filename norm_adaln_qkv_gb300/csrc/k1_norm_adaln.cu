// k1_norm_adaln.cu -- kernel 1 of the pre-attention stage: input RMSNorm and
// indexed AdaLN, written to the BF16 [M, 5376] workspace.
//
// Formulas: flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, formula block
//   n = bf16(rmsnorm(x, eps) * x_norm_weight)   (FP32 sum of squares, rsqrt)
//   a = bf16(adaln_shift[i] + n * bf16(1 + adaln_scale[i])),  i = adaln_index[m]
//   a[i outside [0, rows)] = 0                  (device-side guard)
// which flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention runs as its
// first launch (summary; Parameters: adaln_scale, adaln_index; Notes).
//
// Design (HBM-bound row streaming): one CTA of 224 threads per token row.
// A row is 5376 bf16 = 672 16-byte vectors = 3 per thread, loaded up front
// with evict-first hints (x is read exactly once); many small CTAs per SM keep
// ~100 KB of loads in flight per SM.  The sum of squares is FP32: per-thread
// partial sums, a butterfly shuffle per warp, then the seven warp sums added
// in one fixed order by every thread, so all threads hold the same total.
// r = 1 / sqrt(ss/H + eps) and every elementwise step use IEEE
// round-to-nearest FP32 operations in the formula's order with no contraction
// into FMA.  The guard is an int64 compare: a bad index writes +0.0 and never
// forms a table address.  Workspace stores keep the default write-back policy
// so the GEMM that follows finds the rows in L2 when they fit.
#include "common.cuh"

namespace mh3 {

namespace {

constexpr int kVecPerRow = kHidden / 8;  // 672
constexpr int kThreads = 224;             // 7 warps
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = kVecPerRow / kThreads;  // 3
static_assert(kVecPerRow % kThreads == 0, "row must split evenly over the CTA");

__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) { return __ldcs(p); }

__device__ __forceinline__ void sq_acc(uint32_t u, float& a0, float& a1) {
  const float lo = bf16_lo(u), hi = bf16_hi(u);
  // bf16 squares are exact in FP32, so the fused form equals mul-then-add.
  a0 = __fmaf_rn(lo, lo, a0);
  a1 = __fmaf_rn(hi, hi, a1);
}

// One bf16 pair of the AdaLN output, in the formula's rounding order.
__device__ __forceinline__ uint32_t adaln_pair(uint32_t xu, uint32_t wu, uint32_t scu, uint32_t shu,
                                               float r) {
  float out[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float xv = h ? bf16_hi(xu) : bf16_lo(xu);
    const float wv = h ? bf16_hi(wu) : bf16_lo(wu);
    const float sc = h ? bf16_hi(scu) : bf16_lo(scu);
    const float sh = h ? bf16_hi(shu) : bf16_lo(shu);
    const float n = round_bf16(__fmul_rn(__fmul_rn(xv, r), wv));
    const float g = round_bf16(__fadd_rn(1.0f, sc));
    out[h] = __fadd_rn(sh, __fmul_rn(n, g));
  }
  return pack_bf16x2(out[0], out[1]);
}

__global__ void __launch_bounds__(kThreads) norm_adaln_kernel(const NormAdalnParams p) {
  __shared__ float warp_ss[kWarps];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int64_t m = blockIdx.x;

  const uint4* xr = reinterpret_cast<const uint4*>(p.x + m * kHidden);
  uint4 v[kVecPerThread];
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) v[i] = ld_stream_v4(xr + tid + kThreads * i);
  const int64_t idx = __ldg(p.index + m);

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    sq_acc(v[i].x, acc[0], acc[1]);
    sq_acc(v[i].y, acc[2], acc[3]);
    sq_acc(v[i].z, acc[0], acc[1]);
    sq_acc(v[i].w, acc[2], acc[3]);
  }
  float ss = __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, o));
  if (lane == 0) warp_ss[tid >> 5] = ss;
  __syncthreads();
  ss = __fadd_rn(__fadd_rn(__fadd_rn(warp_ss[0], warp_ss[1]), __fadd_rn(warp_ss[2], warp_ss[3])),
                 __fadd_rn(__fadd_rn(warp_ss[4], warp_ss[5]), warp_ss[6]));

  uint4* wr = reinterpret_cast<uint4*>(p.workspace + m * kHidden);
  if (idx < 0 || idx >= p.rows) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) wr[tid + kThreads * i] = z;
    return;
  }
  const float r =
      __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(kHidden)), p.eps)));

  const uint4* wv = reinterpret_cast<const uint4*>(p.x_norm_weight);
  const uint4* scr = reinterpret_cast<const uint4*>(p.scale + idx * p.scale_stride);
  const uint4* shr = reinterpret_cast<const uint4*>(p.shift + idx * p.shift_stride);
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    const int c = tid + kThreads * i;
    const uint4 w = __ldg(wv + c);
    const uint4 sc = __ldg(scr + c);
    const uint4 sh = __ldg(shr + c);
    uint4 o;
    o.x = adaln_pair(v[i].x, w.x, sc.x, sh.x, r);
    o.y = adaln_pair(v[i].y, w.y, sc.y, sh.y, r);
    o.z = adaln_pair(v[i].z, w.z, sc.z, sh.z, r);
    o.w = adaln_pair(v[i].w, w.w, sc.w, sh.w, r);
    wr[c] = o;
  }
}

}  // namespace

cudaError_t launch_norm_adaln(const NormAdalnParams& p, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  norm_adaln_kernel<<<static_cast<unsigned>(p.M), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mh3
