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
//   warp 0      TMA producer: per 64-wide k-block, the tile's workspace
//               rows and 256 weight rows (bf16, 128-B swizzle) into a
//               shared-memory ring.
//   warp 1      TMEM allocator and UMMA issuer: tcgen05.mma kind::f16,
//               M=128 N=256 K=16, four per 64-wide k-block, FP32 accumulator
//               in TMEM, double-buffered (2 x 256 columns) so the epilogue
//               of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue (k2_common.cuh).
//
// Schedules.  At these sizes the 84 tiles are fewer than the 152 SMs, and
// the work is streaming the 231 MB weight.  With the stream-K schedule (the
// handle path) the 84 x 84 (tile, k-block) units are cut into one
// contiguous range per CTA, so every SM streams an equal share.  A CTA whose
// range starts inside a tile writes that partial accumulator (FP32, its
// first range piece) to a global slot and raises a per-warp flag; the CTA
// that holds the tile's k-block 0 (and finishes its range with it) adds the
// following CTAs' partials into its TMEM accumulator, then runs the usual
// epilogue.  An owner only ever waits for other CTAs' first pieces, which
// they compute first, so no wait is circular; all CTAs are resident (one per
// SM, grid = SM count).  The sum is still the FP32 accumulation of the
// pages, in another order.  Without scratch (the allocation-free entry
// point) each CTA takes whole tiles.  The weight loads of the first ring
// stages go out before the wait on kernel 1 (they do not depend on it).
//
// Every wait is bounded: past a 2 s limit the waiting role records a code in
// the device status word, raises a CTA-wide abort flag, and all roles drain
// what they issued (TMA loads, UMMAs, TMA stores) before TMEM is freed and
// the CTA exits.
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

// Iterates this CTA's (tile, k-block) units in issue order: with stream-K a
// contiguous range of the num_tiles * 84 units, otherwise the tiles
// blockIdx.x, blockIdx.x + G, ... with all 84 k-blocks each.
template <bool kSK>
struct Units {
  int64_t u, u_end;  // stream-K range
  int t, kb;         // current tile and k-block
  int num_tiles;
  __device__ Units(const QkvParams& p) : num_tiles(p.num_tiles) {
    if (kSK) {
      const int64_t U = static_cast<int64_t>(p.num_tiles) * kKBlocks;
      u = static_cast<int64_t>(blockIdx.x) * U / gridDim.x;
      u_end = static_cast<int64_t>(blockIdx.x + 1) * U / gridDim.x;
      t = static_cast<int>(u / kKBlocks);
      kb = static_cast<int>(u % kKBlocks);
    } else {
      u = u_end = 0;
      t = blockIdx.x;
      kb = 0;
    }
  }
  __device__ bool valid() const { return kSK ? u < u_end : t < num_tiles; }
  __device__ bool last_of_piece() const { return kb == kKBlocks - 1 || (kSK && u + 1 == u_end); }
  __device__ bool first_of_piece(bool first_unit) const { return kb == 0 || first_unit; }
  __device__ void next() {
    if (kSK) ++u;
    if (++kb == kKBlocks) {
      kb = 0;
      t += kSK ? 1 : static_cast<int>(gridDim.x);
    }
  }
};

// Stream-K partial slots: [cta][warp][column][lane] FP32.
__device__ __forceinline__ float* sk_slot(const QkvParams& p, int cta, int quad) {
  return p.sk_partial + ((static_cast<int64_t>(cta) * 4 + quad) * BN) * 32;
}

// This warp's 32 accumulator rows x 256 columns -> its partial slot.
__device__ __forceinline__ void sk_store_partial(uint32_t tacc, float* slot, int lane) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t v[32];
    tmem_ld_x32(tacc + 32 * c, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) __stcg(slot + (32 * c + i) * 32 + lane, __uint_as_float(v[i]));
  }
}

// accumulator += partial slot (FP32 additions), in TMEM.
__device__ __forceinline__ void sk_add_partial(uint32_t tacc, const float* slot, int lane) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
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
}

// Bounded wait (lane 0) for a flag to become 1; false on abort or timeout.
__device__ __noinline__ bool sk_wait_flag(const int* flag, volatile int* abort_flag, int* status) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 0;; ++n) {
    if (ld_acquire_gpu(flag) != 0) return true;
    if ((n & 63u) == 63u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(status, 0, kStatusSkPartial);
        return false;
      }
    }
  }
}

template <class L, bool kSK>
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
      Units<kSK> it(p);
      // The weight does not depend on kernel 1: the first ring stages' weight
      // boxes go out at once, their workspace boxes after kernel 1 is done.
      int pre_t[kStages], pre_kb[kStages];
      int n_pre = 0;
      for (; n_pre < kStages && it.valid(); ++n_pre, it.next()) {
        int m_blk, n_blk;
        tile_coords<kGroupM>(it.t, p.num_m_tiles, m_blk, n_blk);
        pre_t[n_pre] = m_blk;
        pre_kb[n_pre] = it.kb;
        mbar_arrive_expect_tx(sm.full(n_pre), L::kStageBytes);
        tma_load_2d(sm.b(n_pre), &tm_b, sm.full(n_pre), it.kb * BK, n_blk * BN);
        issued_mask |= 1u << n_pre;
      }
      griddep_wait();  // kernel 1 writes the workspace
      for (int i = 0; i < n_pre; ++i)
        tma_load_2d(sm.a(i), &tm_a, sm.full(i), pre_kb[i] * BK, pre_t[i] * BM);
      stage = n_pre % kStages;
      phase = n_pre == kStages ? 1u : 0u;
      for (; it.valid() && ok; it.next()) {
        int m_blk, n_blk;
        tile_coords<kGroupM>(it.t, p.num_m_tiles, m_blk, n_blk);
        if (!wait_phase<false>(sm.empty(stage), phase ^ 1u, abort_flag, p.status,
                               kStatusProducerEmpty)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(sm.full(stage), L::kStageBytes);
        tma_load_2d(sm.a(stage), &tm_a, sm.full(stage), it.kb * BK, m_blk * BM);
        tma_load_2d(sm.b(stage), &tm_b, sm.full(stage), it.kb * BK, n_blk * BN);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
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
      int piece = 0;  // accumulator pieces started (whole tiles or stream-K parts)
      uint32_t d_tmem = tmem_base;
      bool first_unit = true;
      for (Units<kSK> it(p); it.valid(); it.next()) {
        const bool start = it.first_of_piece(first_unit);
        first_unit = false;
        if (start) {
          const int buf = piece & 1;
          const uint32_t use = static_cast<uint32_t>(piece >> 1);
          if (!wait_phase<false>(sm.tempty(buf), (use & 1u) ^ 1u, abort_flag, p.status,
                                 kStatusMmaTmemEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after();
          d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        }
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
          umma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdesc, (!start || k != 0) ? 1u : 0u);
        }
        umma_commit(sm.empty(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (it.last_of_piece()) {
          umma_commit(sm.tfull(piece & 1));
          ++piece;
        }
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
    Units<kSK> it(p);
    int piece = 0;
    while (it.valid()) {
      // the accumulator piece [k0, k1) of tile it.t
      const int t = it.t;
      const int k0 = it.kb;
      int k1;
      if (kSK) {
        const int64_t left = it.u_end - it.u;
        k1 = left < kKBlocks - k0 ? k0 + static_cast<int>(left) : kKBlocks;
      } else {
        k1 = kKBlocks;
      }
      for (int k = k0; k < k1; ++k) it.next();
      const int buf = piece & 1;
      const uint32_t use = static_cast<uint32_t>(piece >> 1);
      ++piece;
      bool ok = wait_phase<false>(sm.tfull(buf), use & 1u, abort_flag, p.status,
                                  kStatusEpiTmemFull);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      int m_blk, n_blk;
      tile_coords<kGroupM>(t, p.num_m_tiles, m_blk, n_blk);
      const uint32_t tacc = tmem_base + static_cast<uint32_t>(buf * BN) +
                            (static_cast<uint32_t>(quad * 32) << 16);
      const bool rows_used = static_cast<int64_t>(m_blk) * BM + quad * 32 < p.M;
      if (kSK && k0 > 0) {
        // not this tile's owner: hand the partial to the CTA that holds k-block 0
        if (rows_used) {
          sk_store_partial(tacc, sk_slot(p, blockIdx.x, quad), lane);
          __threadfence();
          __syncwarp();
          if (lane == 0) st_release_gpu(p.sk_flags + blockIdx.x * 4 + quad, 1);
        }
      } else {
        if (kSK && k1 < kKBlocks && rows_used) {
          // owner of a split tile: add the following CTAs' pieces of it
          const int64_t U = static_cast<int64_t>(p.num_tiles) * kKBlocks;
          const int64_t tile_end = static_cast<int64_t>(t + 1) * kKBlocks;
          bool got = true;
          for (int c = blockIdx.x + 1;
               c < static_cast<int>(gridDim.x) && static_cast<int64_t>(c) * U / gridDim.x < tile_end;
               ++c) {
            int* flag = p.sk_flags + c * 4 + quad;
            bool w = true;
            if (lane == 0) w = sk_wait_flag(flag, abort_flag, p.status);
            w = __shfl_sync(0xFFFFFFFFu, w ? 1 : 0, 0) != 0;
            if (!w) {
              got = false;
              break;
            }
            (void)ld_acquire_gpu(flag);  // every lane's own acquire of the partial
            __syncwarp();
            sk_add_partial(tacc, sk_slot(p, c, quad), lane);
            __syncwarp();
            if (lane == 0) flag[0] = 0;  // consumed: zero again for the next launch
          }
          if (!got) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.tempty(buf));
            break;
          }
        }
        epilogue_block(tmem_base + static_cast<uint32_t>(buf * BN), quad, lane, stg, sm.norm_w(),
                       p, static_cast<int64_t>(m_blk) * BM, n_blk, &tm_out);
      }
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

template <bool kSK>
cudaError_t prepare_layouts() {
  cudaError_t e = cudaFuncSetAttribute(qkv_gemm_kernel<FullLayout, kSK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       FullLayout::kSmemAlloc);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qkv_gemm_kernel<SmallLayout, kSK>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, SmallLayout::kSmemAlloc);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(qkv_gemm_kernel<TinyLayout, kSK>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, TinyLayout::kSmemAlloc);
}

cudaError_t qkv_prepare_device() {
  const cudaError_t e = prepare_layouts<false>();
  return e != cudaSuccess ? e : prepare_layouts<true>();
}

size_t qkv_sk_partial_bytes(int grid) { return static_cast<size_t>(grid) * 4 * BN * 32 * 4; }
size_t qkv_sk_flags_bytes(int grid) { return static_cast<size_t>(grid) * 4 * sizeof(int); }

template <bool kSK>
cudaError_t launch_layout(const QkvMaps& maps, const QkvParams& p, int grid, cudaStream_t stream) {
  // the A map's box height must be qkv_a_box_rows(p.M)
  if (p.M <= kTinyRows)
    return launch_k2(qkv_gemm_kernel<TinyLayout, kSK>, grid, kThreads, TinyLayout::kSmemAlloc,
                     stream, maps, p);
  if (p.M <= kSmallRows)
    return launch_k2(qkv_gemm_kernel<SmallLayout, kSK>, grid, kThreads, SmallLayout::kSmemAlloc,
                     stream, maps, p);
  return launch_k2(qkv_gemm_kernel<FullLayout, kSK>, grid, kThreads, FullLayout::kSmemAlloc,
                   stream, maps, p);
}

cudaError_t launch_qkv(const QkvMaps& maps, const QkvParams& p, int grid, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  if (p.sk_partial != nullptr) return launch_layout<true>(maps, p, grid, stream);
  return launch_layout<false>(maps, p, grid, stream);
}

}  // namespace mh3
