// k2_qkv_gemm.cu -- kernel 2 of the pre-attention stage, single-CTA form:
// the persistent QKV projection on the 5th-generation tensor cores with the
// per-head Q/K RMSNorm, the partial split-half RoPE and the destination-major
// pack fused into its epilogue (k2_common.cuh).  Used for M <= 128, where a
// CTA pair would compute half a tile of padding; larger M takes the pair
// form in k2_qkv_gemm_pair.cu.
//
// GEMM (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention, summary and
// Parameters: qkv_weight): acc[m, c] = sum_k a[m, k] * W[c, k], FP32 in TMEM,
// column c = kind*7168 + head*128 + d.
//
// Structure (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: A (workspace) 128x64 and B (weight) 256x64 bf16
//               boxes with 128-B swizzle into a 4-stage shared-memory ring;
//               the first tile's weight boxes start before kernel 1 ends.
//   warp 1      TMEM allocator and UMMA issuer: tcgen05.mma kind::f16,
//               M=128 N=256 K=16, four per 64-wide k-block, FP32 accumulator
//               in TMEM, double-buffered (2 x 256 columns) so the epilogue
//               of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue (k2_common.cuh).
// Every mbarrier wait is bounded: past a 2 s limit the waiting role records a
// code in the device status word, raises a CTA-wide abort flag, and all roles
// drain what they issued (TMA loads, UMMAs, TMA stores) before TMEM is freed
// and the CTA exits.
#include "k2_common.cuh"

namespace mh3 {

namespace {

using namespace k2;

constexpr int BM = 128;
constexpr int BN = kTileN;
#ifndef MH3_GROUP_M
#define MH3_GROUP_M 16
#endif
constexpr int kGroupM = MH3_GROUP_M;
constexpr int kThreads = 64 + kEpiWarps * 32;  // 192
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);

// Shared-memory layout (offsets from a 1024-B aligned base) for a ring of
// kStagesT stages whose A box holds kARowsT workspace rows.  The MMA always
// reads 128 A rows from a stage's A address; with kARowsT < 128 (the small-
// and tiny-M layouts, M <= kARowsT) the rows past the box lie in the
// following stages' A regions or in the B region, hold stale data, and
// produce accumulator rows >= M, which are never stored.  The shared memory
// freed this way buys one more stage of weight in flight.
template <int kStagesT, int kARowsT>
struct Layout {
  static constexpr int kStages = kStagesT;
  static constexpr int kARows = kARowsT;
  static constexpr int kABytes = kARowsT * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;  // 32 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffStg = kOffB + kStages * kBBytes;
  static constexpr int kOffBar = kOffStg + kEpiWarps * kStgWarpBytes;
  // full, empty, tmem full x2, tmem empty x2, drain
  static constexpr int kNumBars = 2 * kStages + 4 + 1;
  static constexpr int kOffTmemPtr = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemPtr + 4;
  static constexpr int kOffNormW = kOffBar + 256;  // 256 floats: q weights then k weights
  static constexpr int kSmemUsed = kOffNormW + 2 * kHeadDim * 4;
  static constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack for aligning the base
  static_assert(kOffAbort + 4 <= kOffNormW, "barrier block overflow");
  static_assert(kSmemAlloc <= 232448, "exceeds the 227 KB per-CTA limit");
  static_assert(kARows % 8 == 0 && kARows <= BM, "A box: whole 8-row swizzle atoms");
  static_assert(kOffA + (kStages - 1) * kABytes + BM * BK * 2 <= kSmemUsed,
                "the MMA's 128-row A reads stay inside the allocation");
};
using FullLayout = Layout<4, BM>;   // M <= 128
using SmallLayout = Layout<5, 48>;  // M <= 48
using TinyLayout = Layout<5, 16>;   // M <= 16
constexpr int kTinyRows = TinyLayout::kARows;
constexpr int kSmallRows = SmallLayout::kARows;

template <class L>
struct Smem {
  uint32_t base;  // shared address of the aligned base
  uint8_t* ptr;
  __device__ uint32_t a(int s) const { return base + L::kOffA + s * L::kABytes; }
  __device__ uint32_t b(int s) const { return base + L::kOffB + s * L::kBBytes; }
  __device__ uint32_t full(int s) const { return base + L::kOffBar + s * 8; }
  __device__ uint32_t empty(int s) const { return base + L::kOffBar + (L::kStages + s) * 8; }
  __device__ uint32_t tfull(int b) const { return base + L::kOffBar + (2 * L::kStages + b) * 8; }
  __device__ uint32_t tempty(int b) const {
    return base + L::kOffBar + (2 * L::kStages + 2 + b) * 8;
  }
  __device__ uint32_t drain() const { return base + L::kOffBar + (2 * L::kStages + 4) * 8; }
  __device__ uint32_t stg(int ew) const { return base + L::kOffStg + ew * kStgWarpBytes; }
  __device__ uint32_t* tmem_ptr() const {
    return reinterpret_cast<uint32_t*>(ptr + L::kOffTmemPtr);
  }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + L::kOffAbort);
  }
  __device__ float* norm_w() const { return reinterpret_cast<float*>(ptr + L::kOffNormW); }
};

template <class L>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_out, const QkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int kStages = L::kStages;
  Smem<L> sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    sm.base = (raw + 1023u) & ~1023u;
    sm.ptr = smem_raw + (sm.base - raw);
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(sm.full(s), 1);
      mbar_init(sm.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sm.tfull(b), 1);
      mbar_init(sm.tempty(b), kEpiWarps);
    }
    mbar_init(sm.drain(), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_out);
  }
  for (int i = threadIdx.x; i < 2 * kHeadDim; i += kThreads) {
    const __nv_bfloat16 w = i < kHeadDim ? p.q_norm_weight[i] : p.k_norm_weight[i - kHeadDim];
    sm.norm_w()[i] = __bfloat162float(w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(sm.tmem_ptr()), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_ptr();
  volatile int* abort_flag = sm.abort_flag();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t issued_mask = 0, issued_parity = 0;
      // The weight does not depend on kernel 1, which may still be running
      // (the workspace is its output): the first tile's weight boxes for the
      // whole ring go out at once, and only then does this thread wait for
      // kernel 1 and load the workspace boxes of those stages.
      int n_pre = 0;
      if (static_cast<int>(blockIdx.x) < p.num_tiles) {
        int m_blk, n_blk;
        tile_coords<kGroupM>(blockIdx.x, p.num_m_tiles, m_blk, n_blk);
        for (; n_pre < kStages; ++n_pre) {
          mbar_arrive_expect_tx(sm.full(n_pre), L::kStageBytes);
          tma_load_2d(sm.b(n_pre), &tm_b, sm.full(n_pre), n_pre * BK, n_blk * BN);
          issued_mask |= 1u << n_pre;
        }
        griddep_wait();
        for (int s = 0; s < n_pre; ++s)
          tma_load_2d(sm.a(s), &tm_a, sm.full(s), s * BK, m_blk * BM);
        phase = 1u;  // the ring has been filled once
      } else {
        griddep_wait();
      }
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int m_blk, n_blk;
        tile_coords<kGroupM>(t, p.num_m_tiles, m_blk, n_blk);
        for (int kb = t == static_cast<int>(blockIdx.x) ? n_pre : 0; kb < kKBlocks; ++kb) {
          if (!wait_phase<false>(sm.empty(stage), phase ^ 1u, abort_flag, p.status,
                                 kStatusProducerEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(sm.full(stage), L::kStageBytes);
          tma_load_2d(sm.a(stage), &tm_a, sm.full(stage), kb * BK, m_blk * BM);
          tma_load_2d(sm.b(stage), &tm_b, sm.full(stage), kb * BK, n_blk * BN);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every load this thread started land before the CTA can exit.
        for (int s = 0; s < kStages; ++s)
          if (issued_mask & (1u << s)) drain_wait(sm.full(s), (issued_parity >> s) & 1u, p.status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- UMMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!wait_phase<false>(sm.tempty(buf), (use & 1u) ^ 1u, abort_flag, p.status,
                               kStatusMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < kKBlocks; ++kb) {
          if (!wait_phase<false>(sm.full(stage), phase, abort_flag, p.status, kStatusMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sw128_kmajor_desc(sm.a(stage));
          const uint64_t b_desc = sw128_kmajor_desc(sm.b(stage));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // advance 16 elements (32 B) along K inside the swizzle atom
            umma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdesc, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(sm.empty(stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(sm.tfull(buf));
      }
      if (!ok) {
        umma_commit(sm.drain());
        drain_wait(sm.drain(), 0, p.status);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lane quadrant this warp may read
    const uint32_t stg = sm.stg(warp - 2);
    int it = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      bool ok = wait_phase<false>(sm.tfull(buf), use & 1u, abort_flag, p.status,
                                  kStatusEpiTmemFull);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      int m_blk, n_blk;
      tile_coords<kGroupM>(t, p.num_m_tiles, m_blk, n_blk);
      epilogue_block(tmem_base + static_cast<uint32_t>(buf * BN), quad, lane, stg, sm.norm_w(), p,
                     static_cast<int64_t>(m_blk) * BM, n_blk, &tm_out);
      // all TMEM reads of this accumulator are complete (tcgen05.wait::ld)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.tempty(buf));
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

int qkv_smem_bytes() {
  int m = FullLayout::kSmemAlloc;
  if (SmallLayout::kSmemAlloc > m) m = SmallLayout::kSmemAlloc;
  if (TinyLayout::kSmemAlloc > m) m = TinyLayout::kSmemAlloc;
  return m;
}

int qkv_a_box_rows(int64_t M) {
  return M <= kTinyRows ? kTinyRows : (M <= kSmallRows ? kSmallRows : BM);
}

cudaError_t qkv_prepare_device() {
  cudaError_t e = cudaFuncSetAttribute(qkv_gemm_kernel<FullLayout>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       FullLayout::kSmemAlloc);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qkv_gemm_kernel<SmallLayout>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, SmallLayout::kSmemAlloc);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(qkv_gemm_kernel<TinyLayout>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, TinyLayout::kSmemAlloc);
}

cudaError_t launch_qkv(const QkvMaps& maps, const QkvParams& p, int grid, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  // the A map's box height must be qkv_a_box_rows(p.M)
  if (p.M <= kTinyRows)
    return launch_k2(qkv_gemm_kernel<TinyLayout>, grid, kThreads, TinyLayout::kSmemAlloc, stream,
                     maps, p);
  if (p.M <= kSmallRows)
    return launch_k2(qkv_gemm_kernel<SmallLayout>, grid, kThreads, SmallLayout::kSmemAlloc, stream,
                     maps, p);
  return launch_k2(qkv_gemm_kernel<FullLayout>, grid, kThreads, FullLayout::kSmemAlloc, stream,
                   maps, p);
}

}  // namespace mh3
