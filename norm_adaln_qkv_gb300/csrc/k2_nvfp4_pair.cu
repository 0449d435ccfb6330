// k2_nvfp4_pair.cu -- kernel 2 of the NVFP4 pre-attention stage: the QKV
// projection with block-scaled FP4 operands on the CTA-pair tcgen05 MMA,
// with the Q/K RMSNorm, RoPE and destination-major pack epilogue of
// k2_common.cuh applied to y = bf16(RN(alpha * acc))
// (flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention, summary:
// NVFP4 operands, accumulator rescaled by alpha; Parameters: qkv_weight_q,
// qkv_weight_sf, qkv_weight_global_scale, act_global_scale, alpha).
//
// A: act_q [M, 2688] bytes (E2M1, two per byte); B: weight codes
// [21504, 2688]; both K-major with 128-byte swizzle, one 128-byte row = 256
// elements = one k-block (21 k-blocks).  Scales: 512-byte atoms of 128 rows
// x one 64-element step (row r at byte (r % 32) * 16 + (r / 32) * 4).
//
// A cluster of two CTAs owns a 256-row x 128-column tile (one head of one
// kind).  Per k-block CTA r loads its 128 A rows (16 KB), its 64 of the 128
// B rows (8 KB), and the 4 A-scale atoms of its rows (2 KB) and the 4
// B-scale atoms of all 128 B rows (2 KB), into a 6-stage ring, counted on
// two barriers of the even CTA (operands, scales).  The scales go from
// shared memory to both CTAs' TMEM by
// tcgen05.cp (pair form, 32x128b.warpx4: one copy = one K=64 step's 4
// columns of A or B scales).  A copy stalls the thread that issues it for
// over a hundred clocks, so four copy warps of the even CTA issue two copies
// each per k-block; once they have also seen the stage's operands land they
// commit to a per-stage "ready" barrier, the only one the MMA thread waits
// on (every wait or commit in that thread costs MMA issue time) before it
// issues four M=256 N=128 K=64 block-scaled MMAs.  With FP4 at four times the bf16 rate per clock a 256 x 128 tile
// reads 96 B of shared memory per clock per SM, inside the 128 B/clk budget,
// and two 128-column accumulators plus six 32-column scale slots fit the 512
// TMEM columns, so the epilogue of one tile overlaps the next tile's MMAs.
//
// Roles per CTA (352 threads): warp 0 operand TMA producer, warp 1 TMEM
// allocation
// and (even CTA) MMA issue, warps 2..5 the epilogue of the CTA's 128 rows,
// warps 6..9 (even CTA) the scale copies, warp 10 the scale TMA producer.  Bounded waits, abort flags and
// draining as in gemm_pair.cuh.
#include "gemm_pair.cuh"

namespace mh3 {

namespace {

using namespace k2;

constexpr int FBM = 128;                       // A rows per CTA
constexpr int kFTileN = 128;                   // one head
constexpr int kFBRows = kFTileN / 2;           // B rows per CTA
constexpr int kFBytesPerRow = 128;             // one k-block of one row
constexpr int kFKBlocks = kHidden / 256;       // 21
constexpr int kFNTiles = kQkvRows / kFTileN;   // 168
constexpr int kFStages = 6;
constexpr int kFABytes = FBM * kFBytesPerRow;       // 16 KB
constexpr int kFBBytes = kFBRows * kFBytesPerRow;   // 8 KB
constexpr int kFSfBytes = 4 * 512;                  // 4 atoms = 2 KB
constexpr int kFStageBytes = kFABytes + kFBBytes + 2 * kFSfBytes;  // 28 KB
constexpr uint32_t kFIdesc = idesc_fp4_f32(2 * FBM, kFTileN);
constexpr uint32_t kFTmemSf = 2 * kFTileN;     // scale slots start after the accumulators
constexpr uint32_t kFSfCols = 32;              // per slot: A scales 16 + B scales 16
constexpr int kFSfSlots = kFStages;            // scale slots (shared memory and TMEM), one per stage

constexpr int kFOffA = 0;
constexpr int kFOffB = kFOffA + kFStages * kFABytes;
constexpr int kFOffSfa = kFOffB + kFStages * kFBBytes;
constexpr int kFOffSfb = kFOffSfa + kFSfSlots * kFSfBytes;
constexpr int kFOffStg = kFOffSfb + kFSfSlots * kFSfBytes;
constexpr int kFOffBar = kFOffStg + kEpiWarps * kStgWarpBytes;
// per stage: operands full, empty, scales full, ready (scales in TMEM and
// operands landed); tmem full x2, tmem empty x2, drain, copy drain
constexpr int kFNumBars = 4 * kFStages + 4 + 1 + 1;
constexpr int kFOffTmemPtr = kFOffBar + kFNumBars * 8;
constexpr int kFOffAbort = kFOffTmemPtr + 4;
constexpr int kFOffScratch = kFOffBar + 512;
constexpr int kCpWarps = 4;  // scale-copy warps of the even CTA, one K step each
constexpr int kSfWarp = 2 + kEpiWarps + kCpWarps;                    // warp 10: scale loads
constexpr int kFThreads = 64 + kEpiWarps * 32 + kCpWarps * 32 + 32;  // 352
constexpr int kFSmemUsed = kFOffScratch + 1024;
constexpr int kFSmemAlloc = kFSmemUsed + 1024;
static_assert(kFOffAbort + 4 <= kFOffScratch, "barrier block overflow");
static_assert(kCpWarps == 4, "one copy warp per K=64 step of a k-block");
static_assert(kFSmemAlloc <= 232448, "exceeds the 227 KB per-CTA limit");
static_assert(kFTmemSf + kFSfSlots * kFSfCols <= kTmemCols, "TMEM budget");

static_assert(kHidden % 256 == 0 && kQkvRows % kFTileN == 0, "shapes must tile");

struct FSmem {
  uint32_t base;
  uint8_t* ptr;
  __device__ uint32_t a(int s) const { return base + kFOffA + s * kFABytes; }
  __device__ uint32_t b(int s) const { return base + kFOffB + s * kFBBytes; }
  __device__ uint32_t sfa(int s) const { return base + kFOffSfa + s * kFSfBytes; }
  __device__ uint32_t sfb(int s) const { return base + kFOffSfb + s * kFSfBytes; }
  __device__ uint32_t full(int s) const { return base + kFOffBar + s * 8; }
  __device__ uint32_t empty(int s) const { return base + kFOffBar + (kFStages + s) * 8; }
  __device__ uint32_t tfull(int b) const { return base + kFOffBar + (2 * kFStages + b) * 8; }
  __device__ uint32_t tempty(int b) const { return base + kFOffBar + (2 * kFStages + 2 + b) * 8; }
  __device__ uint32_t drain() const { return base + kFOffBar + (2 * kFStages + 4) * 8; }
  __device__ uint32_t cpdrain() const { return base + kFOffBar + (2 * kFStages + 5) * 8; }
  __device__ uint32_t sffull(int s) const { return base + kFOffBar + (2 * kFStages + 6 + s) * 8; }
  __device__ uint32_t ready(int s) const { return base + kFOffBar + (3 * kFStages + 6 + s) * 8; }
  __device__ uint32_t stg(int ew) const { return base + kFOffStg + ew * kStgWarpBytes; }
  __device__ uint32_t tmem_ptr_addr() const { return base + kFOffTmemPtr; }
  __device__ uint32_t* tmem_ptr() const { return reinterpret_cast<uint32_t*>(ptr + kFOffTmemPtr); }
  __device__ uint32_t abort_addr() const { return base + kFOffAbort; }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + kFOffAbort);
  }
  __device__ float* scratch() const { return reinterpret_cast<float*>(ptr + kFOffScratch); }
};

template <bool kE4m3>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFThreads, 1)
    nvfp4_qkv_kernel(const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_sfa,
                     const __grid_constant__ CUtensorMap tm_sfb,
                     const __grid_constant__ CUtensorMap tm_out, const QkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  FSmem sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    sm.base = (raw + 1023u) & ~1023u;
    sm.ptr = smem_raw + (sm.base - raw);
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the scale copies and MMAs
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFStages; ++s) {
      mbar_init(sm.full(s), 1);
      mbar_init(sm.empty(s), 1);
    }
    for (int s = 0; s < kFStages; ++s) {
      mbar_init(sm.sffull(s), 1);
      mbar_init(sm.ready(s), kCpWarps);
    }
    mbar_init(sm.cpdrain(), kCpWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(sm.tfull(b), 1);
      mbar_init(sm.tempty(b), 2 * kEpiWarps);
    }
    mbar_init(sm.drain(), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_sfa);
    prefetch_tmap(&tm_sfb);
    prefetch_tmap(&tm_out);
  }
  // q then k norm weights as FP32
  for (int i = threadIdx.x; i < 2 * kHeadDim; i += kFThreads) {
    const __nv_bfloat16 w = i < kHeadDim ? p.q_norm_weight[i] : p.k_norm_weight[i - kHeadDim];
    sm.scratch()[i] = __bfloat162float(w);
  }
  if (warp == 1) {
    tmem_alloc_pair(sm.tmem_ptr_addr(), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_ptr();
  gp::PairCtx ctx{sm.abort_flag(), mapa_shared(sm.abort_addr(), rank ^ 1u), p.status};

  if (warp == 0) {
    // ------------------------------------ operand producer (both CTAs)
    if (lane == 0) {
      griddep_wait();  // act_q / act_sf come from the kernel before this one
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        int pr, n_blk;
        tile_coords<gp::kGroupPairs, kFNTiles>(t, p.num_m_tiles, pr, n_blk);
        const int a_rg = pr * 2 + static_cast<int>(rank);  // 128-row group of A
        const int b_row = n_blk * kFTileN + static_cast<int>(rank) * kFBRows;
        for (int kb = 0; kb < kFKBlocks; ++kb) {
          if (!gp::pair_wait(ctx, sm.empty(stage), phase ^ 1u, kStatusProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t leader_full = mapa_shared(sm.full(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(sm.full(stage), 2 * (kFABytes + kFBBytes));
          tma_load_2d_pair(sm.a(stage), &tm_a, leader_full, kb * kFBytesPerRow, a_rg * FBM);
          tma_load_2d_pair(sm.b(stage), &tm_b, leader_full, kb * kFBytesPerRow, b_row);
          issued_any = true;
          if (++stage == kFStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && issued_any) gp::grace_period();  // copies signal the even CTA
    }
    __syncwarp();
  } else if (warp == 1) {
    // --------------------------------- scale copies + MMA issue (even CTA)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = cid; t < p.num_tiles && ok; t += ncl, ++it) {
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!gp::pair_wait(ctx, sm.tempty(buf), (use & 1u) ^ 1u, kStatusMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kFTileN);
        for (int kb = 0; kb < kFKBlocks; ++kb) {
          // the operands have landed and the scales are in both CTAs' TMEM
          // (the copy warps commit to `ready` only after seeing `full`)
          if (!gp::pair_wait(ctx, sm.ready(stage), phase, kStatusMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_cols = tmem_base + kFTmemSf + static_cast<uint32_t>(stage) * kFSfCols;
          const uint64_t a_desc = sw128_kmajor_desc(sm.a(stage));
          const uint64_t b_desc = sw128_kmajor_desc(sm.b(stage));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // 64 elements = 32 B along K inside the swizzle atom
            umma_fp4_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kFIdesc, sf_cols + 4 * k,
                          sf_cols + 16 + 4 * k, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit_pair_multicast(sm.empty(stage), gp::kBothCtas);
          if (++stage == kFStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_multicast(sm.tfull(buf), gp::kBothCtas);
      }
      if (!ok) {
        umma_commit_pair_multicast(sm.drain(), 0x1);
        drain_wait(sm.drain(), 0, p.status);
      }
    }
    __syncwarp();
  } else if (warp == kSfWarp) {
    // ---------------------- scale producer (both CTAs), on the stage ring
    if (lane == 0) {
      griddep_wait();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        int pr, n_blk;
        tile_coords<gp::kGroupPairs, kFNTiles>(t, p.num_m_tiles, pr, n_blk);
        const int a_rg = pr * 2 + static_cast<int>(rank);
        for (int kb = 0; kb < kFKBlocks; ++kb) {
          if (!gp::pair_wait(ctx, sm.empty(stage), phase ^ 1u, kStatusProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t leader_sffull = mapa_shared(sm.sffull(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(sm.sffull(stage), 4 * kFSfBytes);
          tma_load_3d_pair(sm.sfa(stage), &tm_sfa, leader_sffull, 0, 4 * kb, a_rg);
          tma_load_3d_pair(sm.sfb(stage), &tm_sfb, leader_sffull, 0, 4 * kb, n_blk);
          issued_any = true;
          if (++stage == kFStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && issued_any) gp::grace_period();
    }
    __syncwarp();
  } else if (warp >= 2 + kEpiWarps && warp < kSfWarp) {
    // ---------------------------------------- scale copies (even CTA only)
    // Copy warp k moves K step k's A-scale atom to columns [4k, 4k+4) and its
    // B-scale atom to [16+4k, 16+4k+4) of the stage's slot, in both CTAs.
    if (lane == 0 && rank == 0) {
      const int k = warp - 2 - kEpiWarps;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        for (int kb = 0; kb < kFKBlocks; ++kb) {
          if (!gp::pair_wait(ctx, sm.sffull(stage), phase, kStatusMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_cols =
              tmem_base + kFTmemSf + static_cast<uint32_t>(stage) * kFSfCols;
          tmem_cp_pair_32x128b_x4(sf_cols + 4 * k, rows16_desc(sm.sfa(stage) + 512 * k));
          tmem_cp_pair_32x128b_x4(sf_cols + 16 + 4 * k, rows16_desc(sm.sfb(stage) + 512 * k));
          // the MMA thread waits on `ready` alone: report only once the
          // operands of the stage have landed too
          if (!gp::pair_wait(ctx, sm.full(stage), phase, kStatusMmaFull)) {
            ok = false;
            break;
          }
          umma_commit_pair_multicast(sm.ready(stage), 0x1);
          if (++stage == kFStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every copy this warp issued has landed before TMEM can be released
      umma_commit_pair_multicast(sm.cpdrain(), 0x1);
      drain_wait(sm.cpdrain(), 0, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 2;
    const int quad = warp & 3;
    const uint32_t stg = sm.stg(ew);
    const float alpha = isfinite(p.alpha) && p.alpha > 0.0f
                            ? p.alpha
                            : __frcp_rn(__fmul_rn(__ldg(p.act_gs), p.w_gs));
    int it = 0;
    for (int t = cid; t < p.num_tiles; t += ncl, ++it) {
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      bool ok = gp::pair_wait(ctx, sm.tfull(buf), use & 1u, kStatusEpiTmemFull);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      int pr, n_blk;
      tile_coords<gp::kGroupPairs, kFNTiles>(t, p.num_m_tiles, pr, n_blk);
      const int kind = n_blk / kHeads;
      const int head = n_blk % kHeads;
      const int64_t m0 = static_cast<int64_t>(pr) * (2 * FBM) + static_cast<int64_t>(rank) * FBM +
                         quad * 32;
      const uint4* cs_row = rope_row(p, m0 + lane, kind);
      const uint32_t tcol = tmem_base + static_cast<uint32_t>(buf * kFTileN) +
                            (static_cast<uint32_t>(quad * 32) << 16);
      epilogue_head<kE4m3, true>(tcol, lane, stg, sm.scratch(), p, m0, kind, head, cs_row, alpha,
                                 &tm_out);
      // all TMEM reads of this accumulator are complete (tcgen05.wait::ld)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(sm.tempty(buf), 0));
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <bool kE4m3>
cudaError_t prepare_one(int* max_clusters) {
  *max_clusters = 0;
  cudaError_t e = cudaFuncSetAttribute(nvfp4_qkv_kernel<kE4m3>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmemAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = kFSmemAlloc;
  return cudaOccupancyMaxActiveClusters(max_clusters, nvfp4_qkv_kernel<kE4m3>, &cfg);
}

template <bool kE4m3>
cudaError_t launch_one(const Nvfp4Maps& m, const QkvParams& p, int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = kFSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MH3_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, nvfp4_qkv_kernel<kE4m3>, m.a, m.b, m.sfa, m.sfb, m.out, p);
}

}  // namespace

cudaError_t nvfp4_qkv_prepare_device(int* max_clusters, int* max_clusters_e4m3) {
  cudaError_t e = prepare_one<false>(max_clusters);
  if (e != cudaSuccess) return e;
  return prepare_one<true>(max_clusters_e4m3);
}

cudaError_t launch_nvfp4_qkv(const Nvfp4Maps& maps, const QkvParams& p, int clusters, bool e4m3,
                             cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  return e4m3 ? launch_one<true>(maps, p, clusters, stream)
              : launch_one<false>(maps, p, clusters, stream);
}

}  // namespace mh3
