// gemm_pair.cuh -- the persistent CTA-pair GEMM main loop, shared by the QKV
// projection (kernel 2 of the pre-attention stage) and the attention output
// projection.  The epilogue is a policy class:
//
//   struct Epi {
//     using Params = ...;                    // has M, num_m_tiles, num_tiles, status
//     static constexpr bool kFp8;            // E4M3 operands (else bf16)
//     static constexpr int kKBlocks;         // K / 64 (bf16) or K / 128 (E4M3): 128-B rows
//     static constexpr int kNTiles;          // number of 256-column accumulator tiles
//     __device__ static int b_row(int n_blk, int rank);  // first B row CTA `rank` loads
//     __device__ static void prologue(float* scratch, int tid, int nthreads, const Params&);
//     __device__ static void tile(const EpiCtx&, const Params&, int64_t row0, int n_blk);
//   };
//
// A cluster of two CTAs owns a 256-row x 256-column output tile of
// C = A (M x K, K-major) x B^T (N x K, K-major).  CTA r of the pair loads, per
// 64-wide k-block, rows [128r, 128r+128) of the tile's A block and rows
// [128r, 128r+128) of its B block (16 KB + 16 KB, 128-B swizzle) into a
// 6-stage ring, counting the bytes on the even CTA's "full" barrier.  One
// thread of the even CTA issues tcgen05 cta_group::2 kind::f16 MMAs (M=256
// N=256 K=16) that read A and B from both CTAs' shared memory and write each
// CTA's 128-row half of the FP32 accumulator to its own TMEM (two 256-column
// buffers); the commits arrive on both CTAs' barriers by multicast.
//
// Roles per CTA (192 threads): warp 0 TMA producer (both CTAs), warp 1 TMEM
// allocation (both, collectively) and MMA issue (even CTA only), warps 2..5
// the epilogue of this CTA's 128 rows, which report a drained accumulator on
// the even CTA's "tmem empty" barrier.  Tiles are visited in groups of
// kGroupPairs row blocks (row block fastest) so that the operands in flight
// stay in L2.  Only the producer waits on the previous grid
// (griddepcontrol.wait) before it reads A.
//
// Every mbarrier wait is bounded (2 s): a role that gives up records a code
// in the device status word and raises the abort flag of both CTAs; aborting
// roles drain (MMA commit, store wait, a fixed grace period for copies that
// signal the other CTA) before the final cluster barrier and TMEM release.
#pragma once

#include <type_traits>

#include "k2_common.cuh"

namespace mh3 {
namespace gp {

using namespace k2;

constexpr int BM = 128;            // rows per CTA
constexpr int kPairRows = 2 * BM;  // rows per pair tile
constexpr int BNC = kTileN / 2;    // B rows (output columns) per CTA
constexpr int kStages = 6;
#ifndef MH3_GROUP_PAIRS
#define MH3_GROUP_PAIRS 8
#endif
#ifndef MH3_PAIR_L2_HINTS
#define MH3_PAIR_L2_HINTS 0
#endif
constexpr int kGroupPairs = MH3_GROUP_PAIRS;
constexpr int kABytes = BM * BK * 2;   // 16 KB
constexpr int kBBytes = BNC * BK * 2;  // 16 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 64 + kEpiWarps * 32;  // 192
constexpr uint32_t kIdesc = idesc_bf16_f32(kPairRows, kTileN);
constexpr uint32_t kIdescFp8 = idesc_e4m3_f32(kPairRows, kTileN);
constexpr uint16_t kBothCtas = 0x3;
constexpr uint64_t kGraceNs = 50000000ull;  // 50 ms

// Shared-memory layout (offsets from a 1024-B aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffStg = kOffB + kStages * kBBytes;
constexpr int kOffBar = kOffStg + kEpiWarps * kStgWarpBytes;
// full, empty, tmem full x2, tmem empty x2, drain, one per epilogue warp
constexpr int kNumBars = 2 * kStages + 4 + 1 + kEpiWarps;
constexpr int kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemPtr + 4;
constexpr int kOffScratch = kOffBar + 256;  // 1 KB of epilogue constants
constexpr int kScratchBytes = 1024;
constexpr int kSmemUsed = kOffScratch + kScratchBytes;
constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack for aligning the base
static_assert(kOffAbort + 4 <= kOffScratch, "barrier block overflow");
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
  __device__ uint32_t epi_bar(int ew) const { return base + kOffBar + (2 * kStages + 5 + ew) * 8; }
  __device__ uint32_t stg(int ew) const { return base + kOffStg + ew * kStgWarpBytes; }
  __device__ uint32_t tmem_ptr_addr() const { return base + kOffTmemPtr; }
  __device__ uint32_t* tmem_ptr() const { return reinterpret_cast<uint32_t*>(ptr + kOffTmemPtr); }
  __device__ uint32_t abort_addr() const { return base + kOffAbort; }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + kOffAbort);
  }
  __device__ float* scratch() const { return reinterpret_cast<float*>(ptr + kOffScratch); }
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
// The same without a subroutine call (for kernels with a register split).
__device__ __forceinline__ bool pair_wait_inl(const PairCtx& c, uint32_t bar, uint32_t parity,
                                              int code) {
  if (wait_phase_inl<true>(bar, parity, c.abort_flag, c.status, code)) return true;
  st_shared_cluster_u32(c.peer_abort, 1u);
  return false;
}

// Fixed grace period for asynchronous work this thread cannot observe.
__device__ __forceinline__ void grace_period_inl() {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < kGraceNs) {
  }
}
__device__ __noinline__ inline void grace_period() { grace_period_inl(); }

// The usual B split: the tile's 256 B rows, 128 per CTA of the pair.
__device__ __forceinline__ int contiguous_b_row(int n_blk, int rank) {
  return n_blk * kTileN + rank * BNC;
}

// What an epilogue warp gets for one 128-row x 256-column accumulator block.
struct EpiCtx {
  uint32_t tmem_acc;  // TMEM address of the block (lane 0, first column)
  int quad;           // TMEM lane quadrant this warp may read (warp % 4)
  int lane;
  uint32_t stg;       // this warp's staging buffer (8 KB, 128-B swizzled halves)
  uint32_t epi_bar;   // this warp's own mbarrier (for loads into its staging)
  uint32_t* epi_phase;  // its next phase parity
  const float* scratch;
  const CUtensorMap* tm_out;
  const CUtensorMap* tm_aux;
  const PairCtx* pair;
};


// Whether an epilogue policy takes part in the split tail (Params with the
// sk_* fields of QkvParams): policies opt in with kSplitTail = true.
template <class E, class = void>
struct split_tail : std::false_type {};
template <class E>
struct split_tail<E, std::void_t<decltype(E::kSplitTail)>> : std::bool_constant<E::kSplitTail> {};

// Policies whose Params say that the previous grid writes A alone (b_early)
// may have the weight boxes of the first stages loaded before the wait.
template <class E, class = void>
struct has_b_early : std::false_type {};
template <class E>
struct has_b_early<E, std::void_t<decltype(std::declval<typename E::Params>().b_early)>>
    : std::true_type {};

// One piece of a cluster's work: k-blocks [kb0, kb1) of tile t; role 0 is a
// whole tile, 1 the first half of a split tile (its partial is handed to the
// owner), 2 the second half (the owner: adds the partial, runs the epilogue).
struct Piece {
  int t, kb0, kb1, role;
};

// The pieces of cluster cid in order: whole tiles cid, cid + ncl, ... below
// `whole_end`, then its half of split tile whole_end + cid / 2 if cid < 2 *
// sk_tail.  The producer, the MMA issuer and the epilogue each walk their own
// copy.
template <class Epi>
struct Schedule {
  int t, ncl, whole_end, kkb;
  int tail_tile, tail_half;
  __device__ Schedule(const typename Epi::Params& p, int cid, int ncl_)
      : t(cid), ncl(ncl_), kkb(Epi::kKBlocks), tail_tile(-1), tail_half(0) {
    whole_end = p.num_tiles;
    if constexpr (split_tail<Epi>::value) {
      if (p.sk_tail > 0) {
        whole_end = p.sk_dp;
        if (cid < 2 * p.sk_tail) {
          tail_tile = p.sk_dp + cid / 2;
          tail_half = cid & 1;
        }
      }
    }
  }
  __device__ bool next(Piece& w) {
    if (t < whole_end) {
      w = Piece{t, 0, kkb, 0};
      t += ncl;
      return true;
    }
    if (tail_tile >= 0) {
      const int h = kkb / 2;
      w = Piece{tail_tile, tail_half * h, tail_half ? kkb : h, 1 + tail_half};
      tail_tile = -1;
      return true;
    }
    return false;
  }
};

// Split tail, first half: this warp's 32 accumulator rows x 256 columns to
// its partial slot ([column][lane], coalesced), then the flag (every lane's
// stores fenced, the warp synchronised, lane 0 releases the sequence value).
__device__ __forceinline__ void split_store(uint32_t tacc, float* slot, int* flag, int seq,
                                            int lane) {
#pragma unroll 1
  for (int c = 0; c < kTileN / 32; ++c) {
    uint32_t v[32];
    tmem_ld_x32(tacc + 32 * c, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) __stcg(slot + (32 * c + i) * 32 + lane, __uint_as_float(v[i]));
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) st_release_gpu(flag, seq);
}

// Split tail, second half: bounded wait for the partner's flag, then the
// accumulator becomes acc + partial (one FP32 addition per element) in TMEM.
// False when the wait gave up (status recorded, both CTAs' abort raised).
__device__ __forceinline__ bool split_add(uint32_t tacc, const float* slot, const int* flag,
                                          int seq, int lane, const PairCtx& ctx) {
  bool ok = true;
  if (lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 0; ld_acquire_gpu(flag) != seq; ++n) {
      if ((n & 63u) == 63u) {
        if (*ctx.abort_flag) {
          ok = false;
          break;
        }
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          *ctx.abort_flag = 1;
          st_shared_cluster_u32(ctx.peer_abort, 1u);
          atomicCAS(ctx.status, 0, kStatusSplitPartial);
          ok = false;
          break;
        }
      }
    }
  }
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  if (!ok) return false;
  (void)ld_acquire_gpu(flag);  // every lane's own acquire before it reads the partial
#pragma unroll 1
  for (int c = 0; c < kTileN / 32; ++c) {
    uint32_t v[32];
    float q[32];
    tmem_ld_x32(tacc + 32 * c, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) q[i] = __ldcg(slot + (32 * c + i) * 32 + lane);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__fadd_rn(__uint_as_float(v[i]), q[i]));
    tmem_st_x32(tacc + 32 * c, v);
  }
  tmem_wait_st();
  return true;
}

template <class Epi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_out,
                     const __grid_constant__ CUtensorMap tm_aux,
                     const typename Epi::Params p) {
  constexpr int kKB = Epi::kKBlocks;
  constexpr int kN = Epi::kNTiles;
  constexpr int kBKElems = Epi::kFp8 ? 128 : BK;  // elements in one 128-byte k-block row
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
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(sm.epi_bar(w), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_out);
    prefetch_tmap(&tm_aux);
  }
  Epi::prologue(sm.scratch(), threadIdx.x, kThreads, p);
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
      int stage = 0;
      uint32_t phase = 0;
      // test hook: issue nothing, so that the consumers' bounded waits run
      // out and the kernel reports a status code instead of hanging
      bool ok = p.test_stall == 0;
      bool issued_any = false;
#if MH3_PAIR_L2_HINTS
      // A blocks are read by every column tile of their group, B boxes by the
      // group's row blocks only: keep A, let B go first
      const uint64_t pol_a = policy_evict_last(), pol_b = policy_evict_first();
#endif
      Schedule<Epi> sched(p, cid, ncl);
      Piece w;
      bool have = ok && sched.next(w);
      // Stages of the first piece whose weight boxes go out before the wait
      // (the ring is fresh: no empty wait); their A boxes follow it.
      int pre = 0;
      if constexpr (has_b_early<Epi>::value) {
        if (have && p.b_early != 0) {
          int pr, n_blk;
          tile_coords<kGroupPairs, kN>(w.t, p.num_m_tiles, pr, n_blk);
          const int b_row = Epi::b_row(n_blk, static_cast<int>(rank));
          pre = w.kb1 - w.kb0 < kStages ? w.kb1 - w.kb0 : kStages;
          for (int s = 0; s < pre; ++s) {
            if (rank == 0) mbar_arrive_expect_tx(sm.full(s), 2 * kStageBytes);
            tma_load_2d_pair(sm.b(s), &tm_b, mapa_shared(sm.full(s), 0), (w.kb0 + s) * kBKElems,
                             b_row);
          }
        }
      }
      // A may be written by the kernel before this one, which may still be
      // finishing (programmatic dependent launch)
      griddep_wait();
      if (pre > 0) {
        int pr, n_blk;
        tile_coords<kGroupPairs, kN>(w.t, p.num_m_tiles, pr, n_blk);
        const int a_row = pr * kPairRows + static_cast<int>(rank) * BM;
        for (int s = 0; s < pre; ++s)
          tma_load_2d_pair(sm.a(s), &tm_a, mapa_shared(sm.full(s), 0), (w.kb0 + s) * kBKElems,
                           a_row);
        issued_any = true;
        stage = pre == kStages ? 0 : pre;
        phase = pre == kStages ? 1u : 0u;
      }
      for (; have; pre = 0, have = ok && sched.next(w)) {
        int pr, n_blk;
        tile_coords<kGroupPairs, kN>(w.t, p.num_m_tiles, pr, n_blk);
        const int a_row = pr * kPairRows + static_cast<int>(rank) * BM;
        const int b_row = Epi::b_row(n_blk, static_cast<int>(rank));
        for (int kb = w.kb0 + pre; kb < w.kb1; ++kb) {
          if (!pair_wait(ctx, sm.empty(stage), phase ^ 1u, kStatusProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t leader_full = mapa_shared(sm.full(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(sm.full(stage), 2 * kStageBytes);
#if MH3_PAIR_L2_HINTS
          tma_load_2d_pair_hint(sm.a(stage), &tm_a, leader_full, kb * kBKElems, a_row, pol_a);
          tma_load_2d_pair_hint(sm.b(stage), &tm_b, leader_full, kb * kBKElems, b_row, pol_b);
#else
          tma_load_2d_pair(sm.a(stage), &tm_a, leader_full, kb * kBKElems, a_row);
          tma_load_2d_pair(sm.b(stage), &tm_b, leader_full, kb * kBKElems, b_row);
#endif
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
      Schedule<Epi> sched(p, cid, ncl);
      Piece w;
      for (; ok && sched.next(w); ++it) {
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!pair_wait(ctx, sm.tempty(buf), (use & 1u) ^ 1u, kStatusMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kTileN);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!pair_wait(ctx, sm.full(stage), phase, kStatusMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sw128_kmajor_desc(sm.a(stage));
          const uint64_t b_desc = sw128_kmajor_desc(sm.b(stage));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // advance 32 B along K inside the swizzle atom (16 bf16 or 32 E4M3)
            // the piece's first MMA starts the accumulator
            const uint32_t acc = (kb != w.kb0 || k != 0) ? 1u : 0u;
            if constexpr (Epi::kFp8)
              umma_f8_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdescFp8, acc);
            else
              umma_bf16_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdesc, acc);
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
    const int ew = warp - 2;
    uint32_t epi_phase = 0;
    EpiCtx ec{0u, warp & 3, lane, sm.stg(ew), sm.epi_bar(ew), &epi_phase, sm.scratch(),
              &tm_out, &tm_aux, &ctx};
    int it = 0;
    Schedule<Epi> sched(p, cid, ncl);
    Piece w;
    for (; sched.next(w); ++it) {
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      bool ok = pair_wait(ctx, sm.tfull(buf), use & 1u, kStatusEpiTmemFull);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      int pr, n_blk;
      tile_coords<kGroupPairs, kN>(w.t, p.num_m_tiles, pr, n_blk);
      ec.tmem_acc = tmem_base + static_cast<uint32_t>(buf * kTileN);
      bool run = true;
      if constexpr (split_tail<Epi>::value) {
        if (w.role != 0) {
          // this warp's slot and flag: [split tile][CTA][TMEM lane quadrant]
          const int64_t slot_id =
              (static_cast<int64_t>(w.t - p.sk_dp) * 2 + static_cast<int64_t>(rank)) * 4 + ec.quad;
          float* slot = p.sk_partial + slot_id * (kTileN * 32);
          int* flag = p.sk_flags + slot_id;
          const uint32_t tq = ec.tmem_acc + (static_cast<uint32_t>(ec.quad * 32) << 16);
          if (w.role == 1) {
            split_store(tq, slot, flag, p.sk_seq, lane);
            run = false;  // the owner runs the epilogue of this tile
          } else {
            run = split_add(tq, slot, flag, p.sk_seq, lane, ctx);
          }
        }
      }
      if (run)
        Epi::tile(ec, p, static_cast<int64_t>(pr) * kPairRows + static_cast<int64_t>(rank) * BM,
                  n_blk);
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

// Host side: raise the shared-memory limit of one instantiation and report
// how many 2-CTA clusters of it can be resident at once.
template <class Epi>
inline cudaError_t gemm_pair_prepare(int* max_clusters) {
  *max_clusters = 0;
  cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<Epi>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  return cudaOccupancyMaxActiveClusters(max_clusters, gemm_pair_kernel<Epi>, &cfg);
}

// Launch with programmatic stream serialization, so that the prologue may
// overlap the end of the kernel before it on the stream.
template <class Epi>
inline cudaError_t gemm_pair_launch(const CUtensorMap& a, const CUtensorMap& b,
                                    const CUtensorMap& out, const CUtensorMap& aux,
                                    const typename Epi::Params& p, int clusters,
                                    cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MH3_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<Epi>, a, b, out, aux, p);
}

}  // namespace gp
}  // namespace mh3
