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
// Design (HBM-bound row streaming).  Persistent CTAs of 224 threads, several
// per SM; CTA b handles rows b, b + G, b + 2G, ...  One thread streams whole
// x rows (10752 B) into a ring of shared-memory row buffers with bulk async
// copies (evict-first: x is read exactly once), so the bytes in flight per SM
// are set by the ring depth, not by registers.  Each thread then owns 3
// 16-byte vectors of the row.  The sum of squares is FP32: per-thread
// partials, a butterfly shuffle per warp, then the seven warp sums added in
// one fixed order by every thread.  r = 1 / sqrt(ss/H + eps) uses IEEE
// division and square root; the elementwise steps are packed two-lane FP32
// operations (each lane one IEEE round-to-nearest operation, in the
// formula's order) and one bf16x2 add for bf16(1 + scale).  The squares and
// shift + n * g (whose product is exact) are fused multiply-adds that take
// their bf16 operands directly (fma.rn.f32.bf16: exact widening, one
// rounding), which saves the unpacking instructions.  The guard is an int64
// compare: a bad index writes +0.0 and never forms a table address.  Workspace stores keep the default
// write-back policy so the GEMM that follows finds the rows in L2 when they
// fit.  The ring wait is bounded (2 s) and records a status code instead of
// hanging.
//
// NVFP4 form (flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention,
// summary): int32 indices, and instead of the bf16 workspace the activation
// quantised per token in blocks of 16 (nvfp4.cuh): E2M1 codes [M, 2688] and
// UE4M3 scales.  A block is two neighbouring lanes' chunks (one shuffle for
// the amax), whose even lane stores the scale byte.  A guarded row gets zero
// codes and scales.
//
// E4M3 form (flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, formula block:
// a_q = e4m3(a / s_a), s_a = RN(amax_row(|a|) / 448)): int64 indices; the row
// amax is one more fixed-order CTA reduction, then each thread quantises its
// 24 values of a (e4m3_rows.cuh) and thread 0 stores s_a.  A guarded row gets
// zero codes and s_a = 0.
#include "common.cuh"
#include "e4m3_rows.cuh"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace mh3 {

namespace {

#ifndef MH3_K1_STAGES
#define MH3_K1_STAGES 4
#endif
#ifndef MH3_K1_CTAS_PER_SM
#define MH3_K1_CTAS_PER_SM 4
#endif

constexpr int kRowBytes = kHidden * 2;               // 10752
constexpr int kVecPerRow = kHidden / 8;              // 672 16-byte vectors
constexpr int kThreads = 224;                        // 7 warps
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = kVecPerRow / kThreads;  // 3
constexpr int kStages = MH3_K1_STAGES;
constexpr int kCtasPerSm = MH3_K1_CTAS_PER_SM;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
static_assert(kVecPerRow % kThreads == 0, "row must split evenly over the CTA");
static_assert(kRowBytes % 16 == 0, "bulk copies move multiples of 16 bytes");

// Bounded wait on one phase of a row-buffer barrier.
__device__ __noinline__ bool wait_row(uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(status, 0, kStatusRowFull);
      return false;
    }
  }
  return true;
}

// One bf16x2 word of x (as packed FP32), weight, scale and shift -> one
// bf16x2 word of a.
__device__ __forceinline__ uint32_t adaln_pair(uint64_t x2, uint32_t w, uint32_t sc, uint32_t sh,
                                               uint64_t r2) {
  // n = bf16((x * r) * w)
  const uint32_t n = f2_to_bf16x2(f2_mul(f2_mul(x2, r2), f2_from_bf16x2(w)));
  // g = bf16(1 + scale): one correctly rounded bf16 addition per lane
  const uint32_t g = bf16x2_add(0x3F803F80u, sc);
  // a = bf16(shift + n * g).  n and g are bf16, so n * g (at most 16
  // significant bits) is exact in FP32 and one fused multiply-add rounds
  // exactly as the multiply followed by the rounded add.
  return pack_bf16x2(fma_bf16_lo(n, g, bf16_lo(sh)), fma_bf16_hi(n, g, bf16_hi(sh)));
}

// NVFP4 outputs of one 8-element chunk (a in `o`): the block of 16 is this
// thread's chunk and its neighbour's (lanes 2b, 2b+1); the even lane stores
// the block's scale byte.  q: the chunk's code word; sf: its scale byte.
__device__ __forceinline__ void fp4_chunk(const uint4& o, int lane, uint32_t* q, uint8_t* sf,
                                          const fp4::Quantiser& qt, const float2* enc_lut) {
  float amax = fp4::amax8(o);
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  const fp4::BlockScale bs = fp4::block_scale(amax, qt, enc_lut);
  *q = fp4::encode8(o, bs, qt.gs);
  if ((lane & 1) == 0) *sf = static_cast<uint8_t>(bs.code);
}

constexpr int kModeBf16 = 0;  // bf16 workspace
constexpr int kModeFp4 = 1;   // NVFP4 codes and block scales
constexpr int kModeFp8 = 2;   // E4M3 codes and a per-token scale

template <int kMode>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) norm_adaln_kernel(const NormAdalnParams p) {
  constexpr bool kFp4 = kMode == kModeFp4;
  constexpr bool kFp8 = kMode == kModeFp8;
  __shared__ __align__(128) uint8_t rows_buf[kStages][kRowBytes];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ float warp_ss[kWarps];
  __shared__ float warp_amax[kFp8 ? kWarps : 1];
  __shared__ int go;
  __shared__ float2 enc_lut[kFp4 ? fp4::kEncLut : 1];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t first = blockIdx.x;
  const int64_t n_rows = (p.M - first + G - 1) / G;  // >= 1: the grid is at most M
  const uint32_t buf0 = smem_u32(&rows_buf[0][0]);
  const uint32_t bar0 = smem_u32(&full[0]);

  // kernel 2 may start its prologue (barriers, TMEM, tensor maps) now; it
  // waits for this grid's completion before it reads the workspace
  griddep_launch_dependents();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.clear_count; i += kThreads) p.clear[i] = 0;
  const float gs = kFp4 ? __ldg(p.act_gs) : 0.0f;
  const fp4::Quantiser quant = fp4::make_quantiser(gs);
  if (kFp4) fp4::init_enc_lut(enc_lut, gs, tid, kThreads);  // visible after the first barrier
  // scale byte of chunk j within its row's scales (row part added per row)
  int sf_off[kVecPerThread];
#pragma unroll
  for (int j = 0; j < kVecPerThread; ++j) {
    const int c = tid + kThreads * j;
    sf_off[j] = p.sf_tiled ? (c >> 3) * fp4::kAtomBytes + ((lane & 7) >> 1)
                           : (c >> 3) * 4 + ((lane & 7) >> 1);
  }

  uint64_t policy = 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
    policy = policy_evict_first();
    for (int64_t i = 0; i < kStages && i < n_rows; ++i) {
      mbar_arrive_expect_tx(bar0 + 8 * i, kRowBytes);
      bulk_load_1d(buf0 + i * kRowBytes, p.x + (first + i * G) * kHidden, kRowBytes, bar0 + 8 * i,
                   policy);
    }
  }
  __syncthreads();

  int64_t i = 0;
  for (; i < n_rows; ++i) {
    const int s = static_cast<int>(i % kStages);
    const uint32_t parity = static_cast<uint32_t>((i / kStages) & 1);
    const int64_t m = first + i * G;
    const int64_t idx = kFp4 ? static_cast<int64_t>(__ldg(p.index32 + m)) : __ldg(p.index + m);
    if (tid == 0) go = wait_row(bar0 + 8 * s, parity, p.status) ? 1 : 0;
    __syncthreads();
    if (!go) break;
    // already complete: gives every thread its own acquire of the copied row
    (void)mbar_try_wait(bar0 + 8 * s, parity);

    const uint32_t row = buf0 + s * kRowBytes;
    uint4 v[kVecPerThread];
    float lo = 0.0f, hi = 0.0f;  // two FP32 partial sums
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) {
      v[j] = ld_shared_v4(row + 16 * (tid + kThreads * j));
      lo = fma_bf16_lo(v[j].x, v[j].x, lo);
      hi = fma_bf16_hi(v[j].x, v[j].x, hi);
      lo = fma_bf16_lo(v[j].y, v[j].y, lo);
      hi = fma_bf16_hi(v[j].y, v[j].y, hi);
      lo = fma_bf16_lo(v[j].z, v[j].z, lo);
      hi = fma_bf16_hi(v[j].z, v[j].z, hi);
      lo = fma_bf16_lo(v[j].w, v[j].w, lo);
      hi = fma_bf16_hi(v[j].w, v[j].w, hi);
    }
    float ss = __fadd_rn(lo, hi);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, o));
    if (lane == 0) warp_ss[tid >> 5] = ss;
    __syncthreads();  // every thread holds its vectors; the warp sums are complete

    if (tid == 0 && i + kStages < n_rows) {
      // refill this buffer with row i + kStages (all reads of it are done)
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar0 + 8 * s, kRowBytes);
      bulk_load_1d(row, p.x + (first + (i + kStages) * G) * kHidden, kRowBytes, bar0 + 8 * s,
                   policy);
    }
    ss = __fadd_rn(__fadd_rn(__fadd_rn(warp_ss[0], warp_ss[1]), __fadd_rn(warp_ss[2], warp_ss[3])),
                   __fadd_rn(__fadd_rn(warp_ss[4], warp_ss[5]), warp_ss[6]));

    uint4* wr = reinterpret_cast<uint4*>(p.workspace + m * kHidden);
    uint32_t* qrow = kFp4 ? reinterpret_cast<uint32_t*>(p.act_q + m * (kHidden / 2)) : nullptr;
    uint8_t* sfrow = !kFp4 ? nullptr
                     : p.act_sf + (p.sf_tiled ? (m >> 7) * (kHidden / 64) * fp4::kAtomBytes +
                                                    (m & 31) * 16 + ((m >> 5) & 3) * 4
                                              : m * (kHidden / 16));
    if (idx < 0 || idx >= p.rows) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        if (kFp4) {
          qrow[tid + kThreads * j] = 0u;  // codes 0, scale 0
          if ((lane & 1) == 0) sfrow[sf_off[j]] = 0;
        } else if (kFp8)
          reinterpret_cast<uint2*>(p.a_q8 + m * kHidden)[tid + kThreads * j] = make_uint2(0u, 0u);
        else
          wr[tid + kThreads * j] = z;
      }
      if (kFp8 && tid == 0) p.a_s8[m] = 0.0f;
      continue;
    }
    const float r =
        __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(kHidden)), p.eps)));
    const uint64_t r2 = f2_pack(r, r);
    const uint4* wv = reinterpret_cast<const uint4*>(p.x_norm_weight);
    const uint4* scr = reinterpret_cast<const uint4*>(p.scale + idx * p.scale_stride);
    const uint4* shr = reinterpret_cast<const uint4*>(p.shift + idx * p.shift_stride);
    uint4 a8[kFp8 ? kVecPerThread : 1];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) {
      const int c = tid + kThreads * j;
      const uint4 w = __ldg(wv + c);
      const uint4 sc = __ldg(scr + c);
      const uint4 sh = __ldg(shr + c);
      uint4 o;
      o.x = adaln_pair(f2_from_bf16x2(v[j].x), w.x, sc.x, sh.x, r2);
      o.y = adaln_pair(f2_from_bf16x2(v[j].y), w.y, sc.y, sh.y, r2);
      o.z = adaln_pair(f2_from_bf16x2(v[j].z), w.z, sc.z, sh.z, r2);
      o.w = adaln_pair(f2_from_bf16x2(v[j].w), w.w, sc.w, sh.w, r2);
      if (kFp4) {
        fp4_chunk(o, lane, qrow + c, sfrow + sf_off[j], quant, enc_lut);
      } else if (kFp8) {
        a8[kFp8 ? j : 0] = o;
        amax = fmaxf(amax, e4m3r::amax8(o));
      } else {
        wr[c] = o;
      }
    }
    if (kFp8) {
      // row amax: warp butterflies, then the seven warp maxima (any order)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      if (lane == 0) warp_amax[tid >> 5] = amax;
      __syncthreads();
      amax = warp_amax[0];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, warp_amax[w]);
      const e4m3r::RowScale rs = e4m3r::make_row_scale(amax);
      uint2* q = reinterpret_cast<uint2*>(p.a_q8 + m * kHidden);
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j)
        q[tid + kThreads * j] = e4m3r::quantize8(a8[kFp8 ? j : 0], rs);
      if (tid == 0) p.a_s8[m] = rs.s;
    }
  }

  if (tid == 0 && i < n_rows) {
    // Stopped early: let the copies still in flight land before exiting.
    for (int64_t k = i; k < n_rows && k < i + kStages; ++k) {
      const int s = static_cast<int>(k % kStages);
      wait_row(bar0 + 8 * s, static_cast<uint32_t>((k / kStages) & 1), p.status);
    }
  }
}

}  // namespace

cudaError_t launch_norm_adaln(const NormAdalnParams& p, int num_sms, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  const int64_t want = static_cast<int64_t>(num_sms) * kCtasPerSm;
  const int64_t grid = p.M < want ? p.M : want;
  if (p.act_q != nullptr)
    norm_adaln_kernel<kModeFp4><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  else if (p.a_q8 != nullptr)
    norm_adaln_kernel<kModeFp8><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  else
    norm_adaln_kernel<kModeBf16><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mh3
