// k2_nvfp4_pair.cu -- the block-scaled FP4 (NVFP4) CTA-pair GEMM: kernel 2
// of the NVFP4 pre-attention stage (the QKV projection, with the Q/K
// RMSNorm, RoPE and destination-major pack epilogue applied to
// y = bf16(RN(alpha * acc))), and, with another epilogue policy, the W4A4
// attention output projection with the gated residual
// (flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj, summary)
// (flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention, summary:
// NVFP4 operands, accumulator rescaled by alpha; Parameters: qkv_weight_q,
// qkv_weight_sf, qkv_weight_global_scale, act_global_scale, alpha).
//
// A: act_q [M, 2688] bytes (E2M1, two per byte); B: weight codes
// [21504, 2688]; both K-major with 128-byte swizzle, one 128-byte row = 256
// elements = one k-block (21 k-blocks).  Scales: 512-byte atoms of 128 rows
// x one 64-element step (row r at byte (r % 32) * 16 + (r / 32) * 4).
//
// A cluster of two CTAs owns a 256-row x 256-column tile (two heads of one
// kind).  Per k-block CTA r loads its 128 A rows (16 KB), its 128 of the 256
// B rows (16 KB), the 4 A-scale atoms of its rows (2 KB) and the 8 B-scale
// atoms of all 256 B rows (4 KB) into a 5-stage ring, counted on two
// barriers of the even CTA (scales, operands).  The scales go from shared
// memory to both CTAs' TMEM by tcgen05.cp (pair form, 32x128b.warpx4: one
// copy = one K=64 step's A scales, or half of its B scales).  A copy stalls
// the thread that issues it for over a hundred clocks, while copies issued
// by different warps overlap: the twelve copies of a k-block take about 1800
// clocks from one warp, 950 from two, 660 from three, against 512 clocks of
// MMA.  So kCpWarps copy warps of the even CTA share them; once they have
// also seen the stage's operands land they commit to a per-stage "ready"
// barrier, the only one the MMA thread waits on (every wait or commit in that
// thread costs MMA issue time) before it issues four M=256 N=256 K=64
// block-scaled MMAs.
//
// TMEM: one 256-column accumulator plus five 48-column scale slots (496 of
// 512 columns).  The epilogue drains its 32 lanes x 256 columns into
// registers at once, as packed bf16(RN(alpha * acc)) (128 registers), and
// releases the accumulator before it computes the two heads, so the next
// tile's MMAs overlap the epilogue's arithmetic and stores.
//
// Roles per CTA (12 warps, three warpgroups): warp 0 TMA producer, warp 1
// TMEM allocation and (even CTA) MMA issue, warps 4..7 (warpgroup 1) the
// epilogue of the CTA's 128 rows (warp w reads TMEM lanes 32 (w % 4) ...),
// warps 8..11 and, with six copy warps, 2..3 the scale copies (even CTA).
// Launched at 168 registers per thread; warpgroups 0 and 2 then give theirs
// down to 120 and the epilogue warpgroup takes 256, which its live row of y
// needs (each SM sub-partition holds one warp of each warpgroup: 256 + 2 x
// 120 <= 3 x 168).  Bounded waits, abort flags and draining as in
// gemm_pair.cuh.
#include "gemm_pair.cuh"

namespace mh3 {

namespace {

using namespace k2;

constexpr int FBM = 128;                       // A rows per CTA
constexpr int kFTileN = 256;                   // two heads
constexpr int kFBRows = kFTileN / 2;           // B rows per CTA
constexpr int kFBytesPerRow = 128;             // one k-block of one row
constexpr int kFNTilesPerKind = kKindCols / kFTileN;  // 28
constexpr int kFStages = 5;
constexpr int kFABytes = FBM * kFBytesPerRow;       // 16 KB
constexpr int kFBBytes = kFBRows * kFBytesPerRow;   // 16 KB
constexpr int kFSfaBytes = 4 * 512;                 // 4 atoms = 2 KB
constexpr int kFSfbBytes = 8 * 512;                 // 8 atoms = 4 KB
constexpr uint32_t kFIdesc = idesc_fp4_f32(2 * FBM, kFTileN);
constexpr uint32_t kFTmemSf = kFTileN;         // scale slots start after the accumulator
constexpr uint32_t kFSfCols = 48;              // per slot: A scales 16 + B scales 32
#ifndef MH3_FP4_CP_WARPS
#define MH3_FP4_CP_WARPS 6
#endif
constexpr int kCpWarps = MH3_FP4_CP_WARPS;     // scale-copy warps of the even CTA
constexpr int kFCopies = 12;                   // per k-block: 4 K steps x (A, B rows 0-127, 128-255)
#ifndef MH3_FP4_WARPS
#define MH3_FP4_WARPS 12
#endif
constexpr int kFWarps = MH3_FP4_WARPS;         // 12 (three warpgroups) or 16 (four)
constexpr int kFThreads = kFWarps * 32;
constexpr int kFEpiWarp0 = 4;                  // warpgroup 1
constexpr int kRegsLaunch = (65536 / kFThreads) / 8 * 8;  // 168 (12 warps), 128 (16)
constexpr int kRegsEpi = 256;
constexpr int kRegsOther = kFWarps == 12 ? 120 : 80;
constexpr int kWgs = kFWarps / 4;
static_assert(kFWarps == 12 || kFWarps == 16, "three or four warpgroups");
static_assert(kCpWarps >= 4 && kCpWarps <= kFWarps - 6 && kCpWarps <= kFCopies,
              "copy warps: 8.., plus 2..3");
static_assert(kEpiWarps == 4 && kFEpiWarp0 % 4 == 0, "the epilogue is one whole warpgroup");
static_assert(kRegsEpi + (kWgs - 1) * kRegsOther <= kWgs * kRegsLaunch,
              "per sub-partition register budget");
static_assert(128 * kRegsEpi + 128 * (kWgs - 1) * kRegsOther <= kFThreads * kRegsLaunch,
              "CTA register budget");

constexpr int kFOffA = 0;
constexpr int kFOffB = kFOffA + kFStages * kFABytes;
constexpr int kFOffSfa = kFOffB + kFStages * kFBBytes;
constexpr int kFOffSfb = kFOffSfa + kFStages * kFSfaBytes;
constexpr int kFOffStg = kFOffSfb + kFStages * kFSfbBytes;
constexpr int kFOffBar = kFOffStg + kEpiWarps * kStgWarpBytes;
// per stage: operands full, empty, scales full, ready (scales in TMEM and
// operands landed); tmem full, tmem empty, drain, copy drain; one per
// epilogue warp (loads into its staging buffer)
constexpr int kFNumBars = 4 * kFStages + 4 + kEpiWarps;
constexpr int kFOffTmemPtr = kFOffBar + kFNumBars * 8;
constexpr int kFOffAbort = kFOffTmemPtr + 4;
constexpr int kFOffScratch = kFOffBar + 256;  // norm weights (1 KB), NVFP4 output tables
constexpr int kFScratchTables = 256;           // float offset of the q, k, v Table16s
constexpr int kFSmemUsed = kFOffScratch + 1536;
static_assert(kFScratchTables * 4 + 3 * static_cast<int>(sizeof(fp4::Table16)) <= 1536,
              "scratch overflow");
constexpr int kFSmemAlloc = kFSmemUsed + 1024;
static_assert(kFOffAbort + 4 <= kFOffScratch, "barrier block overflow");
static_assert(kFSmemAlloc <= 232448, "exceeds the 227 KB per-CTA limit");
static_assert(kFTmemSf + kFStages * kFSfCols <= kTmemCols, "TMEM budget");
static_assert(kHidden % 256 == 0 && kQkvRows % kFTileN == 0, "shapes must tile");
static_assert(kKindCols % kFTileN == 0, "a tile must not straddle q/k/v");

struct FSmem {
  uint32_t base;
  uint8_t* ptr;
  __device__ uint32_t a(int s) const { return base + kFOffA + s * kFABytes; }
  __device__ uint32_t b(int s) const { return base + kFOffB + s * kFBBytes; }
  __device__ uint32_t sfa(int s) const { return base + kFOffSfa + s * kFSfaBytes; }
  __device__ uint32_t sfb(int s) const { return base + kFOffSfb + s * kFSfbBytes; }
  __device__ uint32_t full(int s) const { return base + kFOffBar + s * 8; }
  __device__ uint32_t empty(int s) const { return base + kFOffBar + (kFStages + s) * 8; }
  __device__ uint32_t sffull(int s) const { return base + kFOffBar + (2 * kFStages + s) * 8; }
  __device__ uint32_t ready(int s) const { return base + kFOffBar + (3 * kFStages + s) * 8; }
  __device__ uint32_t tfull() const { return base + kFOffBar + (4 * kFStages) * 8; }
  __device__ uint32_t tempty() const { return base + kFOffBar + (4 * kFStages + 1) * 8; }
  __device__ uint32_t drain() const { return base + kFOffBar + (4 * kFStages + 2) * 8; }
  __device__ uint32_t cpdrain() const { return base + kFOffBar + (4 * kFStages + 3) * 8; }
  __device__ uint32_t epi_bar(int ew) const { return base + kFOffBar + (4 * kFStages + 4 + ew) * 8; }
  __device__ uint32_t stg(int ew) const { return base + kFOffStg + ew * kStgWarpBytes; }
  __device__ uint32_t tmem_ptr_addr() const { return base + kFOffTmemPtr; }
  __device__ uint32_t* tmem_ptr() const { return reinterpret_cast<uint32_t*>(ptr + kFOffTmemPtr); }
  __device__ uint32_t abort_addr() const { return base + kFOffAbort; }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + kFOffAbort);
  }
  __device__ float* scratch() const { return reinterpret_cast<float*>(ptr + kFOffScratch); }
};

// This warp's 32 accumulator rows x 256 columns -> y = bf16(RN(alpha * acc)),
// two columns per register (y[i] = columns 2i, 2i + 1).
__device__ __forceinline__ void drain_accumulator(uint32_t tcol, float alpha, uint32_t (&y)[128]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t v[32];
    tmem_ld_x32(tcol + 32 * c, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i)
      y[16 * c + i] = pack_bf16x2(__fmul_rn(__uint_as_float(v[2 * i]), alpha),
                                  __fmul_rn(__uint_as_float(v[2 * i + 1]), alpha));
  }
}

// End of a role: neither CTA may leave while the other can still reach its
// shared memory (MMA operand reads, barrier arrivals, copies counted on the
// even CTA); warp 1 then releases TMEM.  Each role runs this copy of the tail
// itself, so that no code is shared by warps holding different register
// budgets.
__device__ __forceinline__ void finish_role(bool tmem_owner, uint32_t tmem_base) {
  tc_fence_before();
  cluster_sync_all();
  if (tmem_owner) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// What an epilogue warp gets for one tile whose accumulator it has drained
// into registers (y[i] = bf16 columns 2i, 2i + 1 of the 256, RN(alpha acc)).
struct FEpiCtx {
  int lane;
  int quad;          // TMEM lane quadrant (warp % 4)
  uint32_t rank;     // CTA of the pair
  uint32_t stg;      // this warp's staging buffer (8 KB)
  uint32_t epi_bar;  // this warp's own mbarrier
  uint32_t* epi_phase;
  const float* scratch;
  const CUtensorMap* tm_out;
  const CUtensorMap* tm_aux;
  const gp::PairCtx* pair;
};

// Epilogue policies (all members inline: warps with different register
// budgets may share no out-of-line code):
//   Params (with M, num_m_tiles, num_tiles, status, test_stall, alpha, act_gs,
//   w_gs), kKBlocks (K / 256), kNTiles (N / 256), prologue(), tile().

// The pre-attention QKV projection: Q/K RMSNorm, RoPE and pack per head,
// written as bf16, e4m3 or NVFP4 (kOut).
template <int kOut>
struct QkvFp4Epi {
  using Params = QkvParams;
  static constexpr int kKBlocks = kHidden / 256;      // 21
  static constexpr int kNTiles = kQkvRows / kFTileN;  // 84
  // q then k norm weights as FP32
  __device__ static __forceinline__ void prologue(float* scratch, int tid, const Params& p) {
    for (int i = tid; i < 2 * kHeadDim; i += kFThreads) {
      const __nv_bfloat16 w = i < kHeadDim ? p.q_norm_weight[i] : p.k_norm_weight[i - kHeadDim];
      scratch[i] = __bfloat162float(w);
    }
    if (kOut == kOutNvfp4 && tid < 96) {  // warp k fills the table of q, k or v
      fp4::Table16* t = reinterpret_cast<fp4::Table16*>(scratch + kFScratchTables);
      fp4::init_table16(t + (tid >> 5), __ldg(p.out_gs + (tid >> 5)), tid & 31);
    }
  }
  __device__ static __forceinline__ void tile(const uint32_t (&y)[128], const FEpiCtx& c,
                                              const Params& p, int pr, int n_blk) {
    const int kind = n_blk / kFNTilesPerKind;
    const int head0 = (n_blk % kFNTilesPerKind) * 2;
    const int64_t m0 = static_cast<int64_t>(pr) * (2 * FBM) + static_cast<int64_t>(c.rank) * FBM +
                       c.quad * 32;
    const uint4* cs_row = rope_row(p, m0 + c.lane, kind);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t yh[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) yh[i] = y[64 * j + i];
      epilogue_head_regs<kOut>(yh, c.lane, c.stg, c.scratch, p, m0, kind, head0 + j, cs_row,
                               c.tm_out,
                               reinterpret_cast<const fp4::Table16*>(c.scratch + kFScratchTables));
    }
  }
};

// The attention output projection with the gated residual (W4A4):
//   o = bf16(RN(alpha acc)),  out = bf16(residual + bf16(g * o)),
//   g = gate[gate_index[m]], or 0 for an index outside [0, gate_rows).
// Per warp and 128-column half: the residual block is TMA-loaded into the
// staging buffer, combined in place and TMA-stored to out (so out may alias
// residual: a block is read before the same warp writes it).
struct OutProjFp4Epi {
  using Params = Nvfp4OutProjParams;
  static constexpr int kKBlocks = kAttnWidth / 256;  // 28
  static constexpr int kNTiles = kHidden / kFTileN;  // 21
  __device__ static __forceinline__ void prologue(float*, int, const Params&) {}
  __device__ static __forceinline__ void tile(const uint32_t (&y)[128], const FEpiCtx& c,
                                              const Params& p, int pr, int n_blk) {
    const int64_t m0 = static_cast<int64_t>(pr) * (2 * FBM) + static_cast<int64_t>(c.rank) * FBM +
                       c.quad * 32;
    if (m0 >= p.M) return;  // no row of this warp is stored
    const int64_t m = m0 + c.lane;
    const uint4* grow = nullptr;
    if (m < p.M) {
      const int64_t gi = static_cast<int64_t>(__ldg(p.gate_index + m));
      if (gi >= 0 && gi < p.gate_rows)
        grow = reinterpret_cast<const uint4*>(p.gate + gi * p.gate_stride);
    }
    const uint64_t pol = policy_evict_first();
#pragma unroll
    for (int j = 0; j < 2; ++j) {  // unrolled: y stays in registers
      const int col0 = n_blk * kFTileN + j * kHeadDim;
      if (c.lane == 0) bulk_wait_group_read0();  // the previous store has read the staging
      __syncwarp();
      if (c.lane == 0) {
        mbar_arrive_expect_tx(c.epi_bar, 2 * kStgHalfBytes);
        tma_load_2d(c.stg, c.tm_aux, c.epi_bar, col0, static_cast<int32_t>(m0));
        tma_load_2d(c.stg + kStgHalfBytes, c.tm_aux, c.epi_bar, col0 + 64,
                    static_cast<int32_t>(m0));
      }
      wait_phase_inl<false>(c.epi_bar, *c.epi_phase, c.pair->abort_flag, c.pair->status,
                            kStatusEpiResidual);
      __syncwarp();
      *c.epi_phase ^= 1u;
#pragma unroll
      for (int chunk = 0; chunk < 16; ++chunk) {
        const uint32_t addr = stg_addr(c.stg, c.lane, chunk);
        const uint4 res = ld_shared_v4(addr);
        const uint4 gw = grow ? __ldg(grow + (col0 >> 3) + chunk) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t rw[4] = {res.x, res.y, res.z, res.w};
        const uint32_t gg[4] = {gw.x, gw.y, gw.z, gw.w};
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t yw = y[64 * j + 4 * chunk + e];
          const float r0 = __fadd_rn(bf16_lo(rw[e]), round_bf16(__fmul_rn(bf16_lo(gg[e]), bf16_lo(yw))));
          const float r1 = __fadd_rn(bf16_hi(rw[e]), round_bf16(__fmul_rn(bf16_hi(gg[e]), bf16_hi(yw))));
          ow[e] = pack_bf16x2(r0, r1);
        }
        st_shared_v4(addr, make_uint4(ow[0], ow[1], ow[2], ow[3]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (c.lane == 0) {
        tma_store_2d_hint(c.tm_out, c.stg, col0, static_cast<int32_t>(m0), pol);
        tma_store_2d_hint(c.tm_out, c.stg + kStgHalfBytes, col0 + 64, static_cast<int32_t>(m0),
                          pol);
        bulk_commit_group();
      }
    }
  }
};

template <class Epi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFThreads, 1)
    nvfp4_pair_kernel(const __grid_constant__ CUtensorMap tm_a,
                      const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_sfa,
                      const __grid_constant__ CUtensorMap tm_sfb,
                      const __grid_constant__ CUtensorMap tm_out,
                      const __grid_constant__ CUtensorMap tm_aux, const typename Epi::Params p) {
  constexpr int kFKBlocks = Epi::kKBlocks;
  constexpr int kFNTiles = Epi::kNTiles;
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
      mbar_init(sm.sffull(s), 1);
      mbar_init(sm.ready(s), kCpWarps);
    }
    mbar_init(sm.tfull(), 1);
    mbar_init(sm.tempty(), 2 * kEpiWarps);
    mbar_init(sm.drain(), 1);
    mbar_init(sm.cpdrain(), kCpWarps);
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(sm.epi_bar(w), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_sfa);
    prefetch_tmap(&tm_sfb);
    prefetch_tmap(&tm_out);
    prefetch_tmap(&tm_aux);
  }
  Epi::prologue(sm.scratch(), threadIdx.x, p);
  if (warp == 1) {
    tmem_alloc_pair(sm.tmem_ptr_addr(), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_ptr();
  gp::PairCtx ctx{sm.abort_flag(), mapa_shared(sm.abort_addr(), rank ^ 1u), p.status};

  // register split: the epilogue warpgroup takes what the others give up;
  // each side's roles sit inside its own branch
  __syncwarp();
  if ((warp >> 2) == kFEpiWarp0 / 4) {
    setmaxnreg_inc<kRegsEpi>();
    // ------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - kFEpiWarp0;
    const int quad = warp & 3;
    uint32_t epi_phase = 0;
    const FEpiCtx ec{lane, quad, rank, sm.stg(ew), sm.epi_bar(ew), &epi_phase, sm.scratch(),
                     &tm_out, &tm_aux, &ctx};
    const float alpha = isfinite(p.alpha) && p.alpha > 0.0f
                            ? p.alpha
                            : __frcp_rn(__fmul_rn(__ldg(p.act_gs), p.w_gs));
    int it = 0;
    for (int t = cid; t < p.num_tiles; t += ncl, ++it) {
      bool ok = gp::pair_wait_inl(ctx, sm.tfull(), static_cast<uint32_t>(it) & 1u, kStatusEpiTmemFull);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t y[128];
      drain_accumulator(tmem_base + (static_cast<uint32_t>(quad * 32) << 16), alpha, y);
      // every TMEM read of the accumulator is complete: the next tile may start
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(sm.tempty(), 0));
      int pr, n_blk;
      tile_coords<gp::kGroupPairs, kFNTiles>(t, p.num_m_tiles, pr, n_blk);
      Epi::tile(y, ec, p, pr, n_blk);
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
    finish_role(false, tmem_base);
    return;
  }
  setmaxnreg_dec<kRegsOther>();
  // copy warp index: 8.. -> 0.., then 2..3
  const int cw = warp >= 8 ? warp - 8 : warp + (kFWarps - 8) - 2;

  if (warp == 0) {
    // ------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      griddep_wait();  // act_q / act_sf come from the kernel before this one
      int stage = 0;
      uint32_t phase = 0;
      bool ok = p.test_stall == 0;
      bool issued_any = false;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        int pr, n_blk;
        tile_coords<gp::kGroupPairs, kFNTiles>(t, p.num_m_tiles, pr, n_blk);
        const int a_rg = pr * 2 + static_cast<int>(rank);  // 128-row group of A
        const int b_row = n_blk * kFTileN + static_cast<int>(rank) * kFBRows;
        for (int kb = 0; kb < kFKBlocks; ++kb) {
          if (!gp::pair_wait_inl(ctx, sm.empty(stage), phase ^ 1u, kStatusProducerEmpty)) {
            ok = false;
            break;
          }
          // scales first, on their own barrier: the copy warps can move them
          // into TMEM while the operands are still in flight
          const uint32_t leader_full = mapa_shared(sm.full(stage), 0);
          const uint32_t leader_sffull = mapa_shared(sm.sffull(stage), 0);
          if (rank == 0) {
            mbar_arrive_expect_tx(sm.sffull(stage), 2 * (kFSfaBytes + kFSfbBytes));
            mbar_arrive_expect_tx(sm.full(stage), 2 * (kFABytes + kFBBytes));
          }
          tma_load_3d_pair(sm.sfa(stage), &tm_sfa, leader_sffull, 0, 4 * kb, a_rg);
          tma_load_3d_pair(sm.sfb(stage), &tm_sfb, leader_sffull, 0, 4 * kb, 2 * n_blk);
          tma_load_2d_pair(sm.a(stage), &tm_a, leader_full, kb * kFBytesPerRow, a_rg * FBM);
          tma_load_2d_pair(sm.b(stage), &tm_b, leader_full, kb * kFBytesPerRow, b_row);
          issued_any = true;
          if (++stage == kFStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && issued_any) gp::grace_period_inl();  // copies signal the even CTA
    }
    __syncwarp();
    finish_role(false, tmem_base);
    return;
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issue (even CTA)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = cid; t < p.num_tiles && ok; t += ncl, ++it) {
        // the epilogue has drained the accumulator of the previous tile
        if (!gp::pair_wait_inl(ctx, sm.tempty(), (static_cast<uint32_t>(it) & 1u) ^ 1u,
                           kStatusMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < kFKBlocks; ++kb) {
          // the operands have landed and the scales are in both CTAs' TMEM
          // (the copy warps commit to `ready` only after seeing `full`)
          if (!gp::pair_wait_inl(ctx, sm.ready(stage), phase, kStatusMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_cols = tmem_base + kFTmemSf + static_cast<uint32_t>(stage) * kFSfCols;
          const uint64_t a_desc = sw128_kmajor_desc(sm.a(stage));
          const uint64_t b_desc = sw128_kmajor_desc(sm.b(stage));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // 64 elements = 32 B along K inside the swizzle atom; A scales of
            // step k in columns [4k, 4k+4), B scales in [16+8k, 16+8k+8)
            umma_fp4_pair(tmem_base, a_desc + 2 * k, b_desc + 2 * k, kFIdesc, sf_cols + 4 * k,
                          sf_cols + 16 + 8 * k, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit_pair_multicast(sm.empty(stage), gp::kBothCtas);
          if (++stage == kFStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_multicast(sm.tfull(), gp::kBothCtas);
      }
      if (!ok) {
        umma_commit_pair_multicast(sm.drain(), 0x1);
        drain_wait_inl(sm.drain(), 0, p.status);
      }
    }
    __syncwarp();
    finish_role(true, tmem_base);
    return;
  } else {
    // ---------------------------------------- scale copies (even CTA only)
    // Copy c of a k-block (K step k = c / 3) moves the A-scale atom of step k
    // to columns [4k, 4k+4), or one of its two B-scale atoms (rows 0-127,
    // 128-255) to [16+8k, 16+8k+4) or [16+8k+4, 16+8k+8), of the stage's
    // slot in both CTAs; copy warp cw issues copies cw, cw + kCpWarps, ...
    if (lane == 0 && rank == 0 && cw < kCpWarps) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        for (int kb = 0; kb < kFKBlocks; ++kb) {
          if (!gp::pair_wait_inl(ctx, sm.sffull(stage), phase, kStatusMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_cols =
              tmem_base + kFTmemSf + static_cast<uint32_t>(stage) * kFSfCols;
          // B-scale atoms arrive as [row group][step][512 B]
          for (int c = cw; c < kFCopies; c += kCpWarps) {
            const int k = c / 3, part = c - 3 * (c / 3);
            const uint32_t col = part == 0 ? 4u * k : 16u + 8u * k + 4u * (part - 1);
            const uint32_t src = part == 0 ? sm.sfa(stage) + 512 * k
                                           : sm.sfb(stage) + 2048 * (part - 1) + 512 * k;
            tmem_cp_pair_32x128b_x4(sf_cols + col, rows16_desc(src));
          }
          // the MMA thread waits on `ready` alone: report only once the
          // operands of the stage have landed too
          if (!gp::pair_wait_inl(ctx, sm.full(stage), phase, kStatusMmaFull)) {
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
      drain_wait_inl(sm.cpdrain(), 0, p.status);
    }
    __syncwarp();
    finish_role(false, tmem_base);
    return;
  }
}

template <class Epi>
cudaError_t prepare_one(int* max_clusters) {
  *max_clusters = 0;
  // The register split (setmaxnreg) is sized for a launch at exactly
  // kRegsLaunch registers per thread; with any other entry allocation an
  // `inc` could wait forever, so such a build is refused here.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, nvfp4_pair_kernel<Epi>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kRegsLaunch || fa.maxThreadsPerBlock < kFThreads)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(nvfp4_pair_kernel<Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kFSmemAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = kFSmemAlloc;
  return cudaOccupancyMaxActiveClusters(max_clusters, nvfp4_pair_kernel<Epi>, &cfg);
}

template <class Epi>
cudaError_t launch_one(const Nvfp4Maps& m, const typename Epi::Params& p, int clusters,
                       cudaStream_t stream) {
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
  // the QKV form has no auxiliary input: its output map stands in
  return cudaLaunchKernelEx(&cfg, nvfp4_pair_kernel<Epi>, m.a, m.b, m.sfa, m.sfb, m.out, m.aux, p);
}

}  // namespace

cudaError_t nvfp4_qkv_prepare_device(int* max_clusters, int* max_clusters_e4m3,
                                     int* max_clusters_nvfp4) {
  cudaError_t e = prepare_one<QkvFp4Epi<kOutBf16>>(max_clusters);
  if (e == cudaSuccess) e = prepare_one<QkvFp4Epi<kOutE4m3>>(max_clusters_e4m3);
  if (e == cudaSuccess) e = prepare_one<QkvFp4Epi<kOutNvfp4>>(max_clusters_nvfp4);
  return e;
}

cudaError_t launch_nvfp4_qkv(const Nvfp4Maps& maps, const QkvParams& p, int clusters, int out_mode,
                             cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  Nvfp4Maps m = maps;
  m.aux = maps.out;
  switch (out_mode) {
    case kOutE4m3: return launch_one<QkvFp4Epi<kOutE4m3>>(m, p, clusters, stream);
    case kOutNvfp4: return launch_one<QkvFp4Epi<kOutNvfp4>>(m, p, clusters, stream);
    default: return launch_one<QkvFp4Epi<kOutBf16>>(m, p, clusters, stream);
  }
}

cudaError_t nvfp4_out_proj_prepare_device(int* max_clusters) {
  return prepare_one<OutProjFp4Epi>(max_clusters);
}

cudaError_t launch_nvfp4_out_proj(const Nvfp4Maps& maps, const Nvfp4OutProjParams& p,
                                  int clusters, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  return launch_one<OutProjFp4Epi>(maps, p, clusters, stream);
}

}  // namespace mh3
