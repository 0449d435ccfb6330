// k2_qkv_gemm_pair.cu -- kernel 2 of the pre-attention stage, CTA-pair form
// (M > 128): the persistent QKV projection computed by pairs of CTAs on two
// SMs with tcgen05 cta_group::2 MMAs, with the fused Q/K RMSNorm, RoPE and
// pack epilogue of k2_common.cuh.
//
// GEMM (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention, summary and
// Parameters: qkv_weight): acc[m, c] = sum_k a[m, k] * W[c, k], FP32 in TMEM,
// column c = kind*7168 + head*128 + d.
//
// A cluster of two CTAs owns a 256-row x 256-column output tile.  CTA r of
// the pair loads, per 64-wide k-block, rows [128r, 128r+128) of the tile's
// activation block (A) and columns [128r, 128r+128) of its weight block (B):
// 16 KB + 16 KB instead of the 16 KB + 32 KB one CTA needs for a 128x256
// tile, so each SM moves a third fewer bytes from L2 per FLOP and the
// shared-memory ring holds 6 k-blocks.  One thread of the even CTA issues
// M=256 N=256 K=16 MMAs that read A and B from both CTAs' shared memory and
// write the 128-row halves of the accumulator to each CTA's TMEM.
//
// Roles per CTA (192 threads):
//   warp 0      TMA producer (both CTAs): loads into its own ring, counting the
//               bytes on the even CTA's "full" barrier; waits on its own
//               "empty" barrier, which the MMA commit arrives on in both CTAs.
//   warp 1      TMEM allocation (both CTAs, collectively), UMMA issue and
//               commits (even CTA only).  Two 256-column accumulators.
//   warps 2..5  epilogue of this CTA's 128 rows; they report a drained
//               accumulator on the even CTA's "tmem empty" barrier.
// Every mbarrier wait is bounded (2 s): a role that gives up records a code
// in the device status word and raises the abort flag of both CTAs; aborting
// roles drain (MMA commit, store wait, a fixed grace period for copies that
// signal the other CTA) before the final cluster barrier and TMEM release.
#include "k2_common.cuh"

namespace mh3 {

namespace {

using namespace k2;

constexpr int BM = 128;           // rows per CTA
constexpr int kPairRows = 2 * BM;  // rows per pair tile
constexpr int BNC = kTileN / 2;   // weight rows (output columns) per CTA
constexpr int kStages = 6;
#ifndef MH3_GROUP_PAIRS
#define MH3_GROUP_PAIRS 8
#endif
constexpr int kGroupPairs = MH3_GROUP_PAIRS;
constexpr int kABytes = BM * BK * 2;   // 16 KB
constexpr int kBBytes = BNC * BK * 2;  // 16 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 64 + kEpiWarps * 32;  // 192
constexpr uint32_t kIdesc = idesc_bf16_f32(kPairRows, kTileN);
constexpr uint16_t kBothCtas = 0x3;
constexpr uint64_t kGraceNs = 50000000ull;  // 50 ms

// Shared-memory layout (offsets from a 1024-B aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffStg = kOffB + kStages * kBBytes;
constexpr int kOffBar = kOffStg + kEpiWarps * kStgWarpBytes;
constexpr int kNumBars = 2 * kStages + 4 + 1;  // full, empty, tmem full x2, tmem empty x2, drain
constexpr int kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemPtr + 4;
constexpr int kOffNormW = kOffBar + 256;  // 256 floats: q weights then k weights
constexpr int kSmemUsed = kOffNormW + 2 * kHeadDim * 4;
constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack for aligning the base
static_assert(kOffAbort + 4 <= kOffNormW, "barrier block overflow");
static_assert(kSmemAlloc <= 232448, "exceeds the 227 KB per-CTA limit");

struct Smem {
  uint32_t base;
  uint8_t* ptr;
  __device__ uint32_t a(int s) const { return base + kOffA + s * kABytes; }
  __device__ uint32_t b(int s) const { return base + kOffB + s * kBBytes; }
  __device__ uint32_t full(int s) const { return base + kOffBar + s * 8; }
  __device__ uint32_t empty(int s) const { return base + kOffBar + (kStages + s) * 8; }
  __device__ uint32_t tfull(int b) const { return base + kOffBar + (2 * kStages + b) * 8; }
  __device__ uint32_t tempty(int b) const { return base + kOffBar + (2 * kStages + 2 + b) * 8; }
  __device__ uint32_t drain() const { return base + kOffBar + (2 * kStages + 4) * 8; }
  __device__ uint32_t stg(int ew) const { return base + kOffStg + ew * kStgWarpBytes; }
  __device__ uint32_t tmem_ptr_addr() const { return base + kOffTmemPtr; }
  __device__ uint32_t* tmem_ptr() const { return reinterpret_cast<uint32_t*>(ptr + kOffTmemPtr); }
  __device__ uint32_t abort_addr() const { return base + kOffAbort; }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + kOffAbort);
  }
  __device__ float* norm_w() const { return reinterpret_cast<float*>(ptr + kOffNormW); }
};

struct PairCtx {
  volatile int* abort_flag;
  uint32_t peer_abort;  // shared::cluster address of the other CTA's abort flag
  int* status;
};

// Bounded wait; on failure also raises the other CTA's abort flag.
__device__ __forceinline__ bool pair_wait(const PairCtx& c, uint32_t bar, uint32_t parity,
                                          int code) {
  if (wait_phase<true>(bar, parity, c.abort_flag, c.status, code)) return true;
  st_shared_cluster_u32(c.peer_abort, 1u);
  return false;
}

// Fixed grace period for asynchronous work this thread cannot observe.
__device__ __noinline__ void grace_period() {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < kGraceNs) {
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    qkv_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a,
                         const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_out, const QkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    sm.base = (raw + 1023u) & ~1023u;
    sm.ptr = smem_raw + (sm.base - raw);
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(sm.full(s), 1);
      mbar_init(sm.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sm.tfull(b), 1);
      mbar_init(sm.tempty(b), 2 * kEpiWarps);
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
    tmem_alloc_pair(sm.tmem_ptr_addr(), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_ptr();
  PairCtx ctx{sm.abort_flag(), mapa_shared(sm.abort_addr(), rank ^ 1u), p.status};

  if (warp == 0) {
    // ------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      // the workspace is written by kernel 1, which may still be finishing
      griddep_wait();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        int pr, n_blk;
        tile_coords<kGroupPairs>(t, p.num_m_tiles, pr, n_blk);
        const int a_row = pr * kPairRows + static_cast<int>(rank) * BM;
        const int b_row = n_blk * kTileN + static_cast<int>(rank) * BNC;
        for (int kb = 0; kb < kKBlocks; ++kb) {
          if (!pair_wait(ctx, sm.empty(stage), phase ^ 1u, kStatusProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t leader_full = mapa_shared(sm.full(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(sm.full(stage), 2 * kStageBytes);
          tma_load_2d_pair(sm.a(stage), &tm_a, leader_full, kb * BK, a_row);
          tma_load_2d_pair(sm.b(stage), &tm_b, leader_full, kb * BK, b_row);
          issued_any = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && issued_any) grace_period();  // copies signal the even CTA
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------- UMMA issuer (even CTA only)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = cid; t < p.num_tiles && ok; t += ncl, ++it) {
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!pair_wait(ctx, sm.tempty(buf), (use & 1u) ^ 1u, kStatusMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kTileN);
        for (int kb = 0; kb < kKBlocks; ++kb) {
          if (!pair_wait(ctx, sm.full(stage), phase, kStatusMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sw128_kmajor_desc(sm.a(stage));
          const uint64_t b_desc = sw128_kmajor_desc(sm.b(stage));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // advance 16 elements (32 B) along K inside the swizzle atom
            umma_bf16_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdesc,
                           (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit_pair_multicast(sm.empty(stage), kBothCtas);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_multicast(sm.tfull(buf), kBothCtas);
      }
      if (!ok) {
        umma_commit_pair_multicast(sm.drain(), 0x1);
        drain_wait(sm.drain(), 0, p.status);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;  // TMEM lane quadrant this warp may read
    const uint32_t stg = sm.stg(warp - 2);
    int it = 0;
    for (int t = cid; t < p.num_tiles; t += ncl, ++it) {
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      bool ok = pair_wait(ctx, sm.tfull(buf), use & 1u, kStatusEpiTmemFull);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      int pr, n_blk;
      tile_coords<kGroupPairs>(t, p.num_m_tiles, pr, n_blk);
      epilogue_block(tmem_base + static_cast<uint32_t>(buf * kTileN), quad, lane, stg,
                     sm.norm_w(), p,
                     static_cast<int64_t>(pr) * kPairRows + static_cast<int64_t>(rank) * BM, n_blk,
                     &tm_out);
      // all TMEM reads of this accumulator are complete (tcgen05.wait::ld)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(sm.tempty(buf), 0));
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  // Neither CTA may leave while the other can still reach its shared memory
  // (MMA operand reads, barrier arrivals, copies counted on the even CTA).
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

int qkv_pair_smem_bytes() { return kSmemAlloc; }

cudaError_t qkv_pair_prepare_device(int* max_clusters) {
  *max_clusters = 0;
  cudaError_t e = cudaFuncSetAttribute(qkv_gemm_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  return cudaOccupancyMaxActiveClusters(max_clusters, qkv_gemm_pair_kernel, &cfg);
}

cudaError_t launch_qkv_pair(const QkvMaps& maps, const QkvParams& p, int clusters,
                            cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  return launch_k2(qkv_gemm_pair_kernel, 2 * clusters, kThreads, kSmemAlloc, stream, maps, p);
}

}  // namespace mh3
