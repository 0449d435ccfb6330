// k2_qkv_gemm.cu -- kernel 2 of the pre-attention stage: the persistent QKV
// projection on the 5th-generation tensor cores, with the per-head Q/K
// RMSNorm, the partial split-half RoPE and the destination-major pack fused
// into its epilogue.
//
// What it computes (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention,
// summary and Parameters: qkv_weight, q/k_norm_weight, qk_eps, rope_cos_sin,
// rope_positions, out):
//   acc[m, c] = sum_k a[m, k] * W[c, k]            FP32 accumulator (TMEM)
//   y = bf16(acc); column c = kind*7168 + head*128 + d
//   kind q/k: t = bf16((y * rr) * w_kind[d]), rr = 1/sqrt(sum_d y^2/128 + qk_eps)
//             p = clamp(positions[m], 0, S-1) (or m); for j < 48:
//             o_j = bf16(t_j c_j - t_{j+48} s_j), o_{j+48} = bf16(t_{j+48} c_j + t_j s_j)
//             with c_j = cos_sin[p, j], s_j = cos_sin[p, 48 + j]; o_d = t_d, d >= 96
//   kind v:   o = y
//   out[head / (56/P), m, head % (56/P), kind, d] = o_d
//
// Structure (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: A (workspace) 128x64 and B (weight) 256x64 bf16
//               boxes with 128-B swizzle into a 4-stage shared-memory ring.
//   warp 1      TMEM allocator and UMMA issuer: tcgen05.mma kind::f16,
//               M=128 N=256 K=16, four per 64-wide k-block, FP32 accumulator
//               in TMEM, double-buffered (2 x 256 columns) so the epilogue
//               of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue: each thread owns one accumulator row (TMEM lane);
//               the per-head sum of squares and the (d, d+48) rotation pairs
//               are thread-local.  Results go through a 128-B-swizzled
//               staging buffer and leave by 4-D TMA stores straight into
//               out[P, M, 56/P, 3, 128]; rows past M are clipped by TMA.
// A 256-column tile is two heads of one kind (7168 / 256 = 28 tiles per
// kind), so a tile never mixes q, k and v.  Tiles are visited in groups of 16
// M-tiles (M fastest inside a group) so that the weight columns and the
// activation rows in flight stay in L2.
//
// Every mbarrier wait is bounded: past a 2 s limit the waiting role records a
// code in the device status word, raises a CTA-wide abort flag, and all roles
// drain what they issued (TMA loads, UMMAs, TMA stores) before TMEM is freed
// and the CTA exits.
#include <cstdio>

#include "common.cuh"
#include "ptx.cuh"

namespace mh3 {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int kStages = 4;
constexpr int kKBlocks = kHidden / BK;    // 84
constexpr int kNTiles = kQkvRows / BN;    // 84
constexpr int kNTilesPerKind = kKindCols / BN;  // 28
#ifndef MH3_GROUP_M
#define MH3_GROUP_M 16
#endif
#ifndef MH3_PREFETCH_NEXT_B
#define MH3_PREFETCH_NEXT_B 0
#endif
constexpr int kGroupM = MH3_GROUP_M;
constexpr int kABytes = BM * BK * 2;      // 16 KB
constexpr int kBBytes = BN * BK * 2;      // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + kEpiWarps * 32;  // 192
constexpr int kStgHalfBytes = 32 * 64 * 2;     // 32 rows x 64 cols bf16 = 4 KB
constexpr int kStgWarpBytes = 2 * kStgHalfBytes;  // one head (128 cols) per warp
constexpr uint32_t kTmemCols = 512;            // 2 accumulators x 256 columns
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);
constexpr uint64_t kWaitLimitNs = 2000000000ull;

static_assert(kHidden % BK == 0, "K must tile");
static_assert(kKindCols % BN == 0, "a tile must not straddle q/k/v");
static_assert(BN == 2 * kHeadDim, "two heads per tile");

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
  uint32_t base;  // shared address of the aligned base
  uint8_t* ptr;
  __device__ uint32_t a(int s) const { return base + kOffA + s * kABytes; }
  __device__ uint32_t b(int s) const { return base + kOffB + s * kBBytes; }
  __device__ uint32_t full(int s) const { return base + kOffBar + s * 8; }
  __device__ uint32_t empty(int s) const { return base + kOffBar + (kStages + s) * 8; }
  __device__ uint32_t tfull(int b) const { return base + kOffBar + (2 * kStages + b) * 8; }
  __device__ uint32_t tempty(int b) const { return base + kOffBar + (2 * kStages + 2 + b) * 8; }
  __device__ uint32_t drain() const { return base + kOffBar + (2 * kStages + 4) * 8; }
  __device__ uint32_t stg(int ew) const { return base + kOffStg + ew * kStgWarpBytes; }
  __device__ uint32_t* tmem_ptr() const { return reinterpret_cast<uint32_t*>(ptr + kOffTmemPtr); }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + kOffAbort);
  }
  __device__ float* norm_w() const { return reinterpret_cast<float*>(ptr + kOffNormW); }
};

// Bounded wait on one mbarrier phase; false when this CTA is aborting.
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        int* status, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(status, 0, code);
        return false;
      }
    }
  }
}

// Short bounded wait used only while draining after an abort.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(status, 0, kStatusDrain);
      return;
    }
  }
}

__device__ __forceinline__ void tile_coords(int t, int num_m_tiles, int& m_blk, int& n_blk) {
  const int group_tiles = kGroupM * kNTiles;
  const int g = t / group_tiles;
  const int first_m = g * kGroupM;
  const int gm = min(kGroupM, num_m_tiles - first_m);
  const int local = t - g * group_tiles;
  m_blk = first_m + local % gm;
  n_blk = local / gm;
}

// Staging address of 16-byte chunk `chunk` (0..15 over the head's 128
// columns) of row `row` (0..31): two 4 KB halves of 64 columns, each laid out
// as TMA's 128-byte swizzle expects (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t stg_addr(uint32_t stg, int row, int chunk) {
  const int half = chunk >> 3;
  const int c = chunk & 7;
  return stg + half * kStgHalfBytes + row * 128 + ((c ^ (row & 7)) << 4);
}

__device__ __forceinline__ float acc_to_y(uint32_t bits) { return round_bf16(__uint_as_float(bits)); }

// V head: o = bf16(acc).
__device__ __forceinline__ void epi_v_head(uint32_t tcol, uint32_t stg, int lane) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t v[32];
    tmem_ld_x32(tcol + 32 * c, v);
    tmem_wait_ld();
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint4 w;
      w.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]));
      w.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
      w.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]));
      w.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
      st_shared_v4(stg_addr(stg, lane, 4 * c + g), w);
    }
  }
}

// Q or K head: RMSNorm over the 128 columns, rotation of [0, 96), pass-through
// of [96, 128).
__device__ __forceinline__ void epi_qk_head(uint32_t tcol, uint32_t stg, int lane, const float* nw,
                                            const uint4* cs_row, float qk_eps) {
  // Pass 1: FP32 sum of squares of the bf16-rounded projection.
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t v[32];
    tmem_ld_x32(tcol + 32 * c, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float y0 = acc_to_y(v[i]), y1 = acc_to_y(v[i + 1]);
      const float y2 = acc_to_y(v[i + 2]), y3 = acc_to_y(v[i + 3]);
      s0 = __fmaf_rn(y0, y0, s0);
      s1 = __fmaf_rn(y1, y1, s1);
      s2 = __fmaf_rn(y2, y2, s2);
      s3 = __fmaf_rn(y3, y3, s3);
    }
  }
  const float ss = __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
  const float rr = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, 128.0f), qk_eps)));

  // Pass 2a: the rotated dims, 16 pairs (j, j + 48) at a time.
#pragma unroll
  for (int g = 0; g < 3; ++g) {
    uint32_t lo[16], hi[16];
    tmem_ld_x16(tcol + 16 * g, lo);
    tmem_ld_x16(tcol + kRopeHalf + 16 * g, hi);
    tmem_wait_ld();
    // cos for j in [16g, 16g+16): row elements [16g, 16g+16) = uint4 2g, 2g+1;
    // sin: elements [48+16g, ...) = uint4 6+2g, 7+2g.
    const uint4 cv[2] = {__ldg(cs_row + 2 * g), __ldg(cs_row + 2 * g + 1)};
    const uint4 sv[2] = {__ldg(cs_row + 6 + 2 * g), __ldg(cs_row + 7 + 2 * g)};
    uint32_t o1[8], o2[8];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const uint32_t cw = (&cv[i >> 3].x)[(i & 7) >> 1];
      const uint32_t sw = (&sv[i >> 3].x)[(i & 7) >> 1];
      float r1[2], r2[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = 16 * g + i + e;
        const float c = e ? bf16_hi(cw) : bf16_lo(cw);
        const float s = e ? bf16_hi(sw) : bf16_lo(sw);
        const float t1 = round_bf16(__fmul_rn(__fmul_rn(acc_to_y(lo[i + e]), rr), nw[j]));
        const float t2 =
            round_bf16(__fmul_rn(__fmul_rn(acc_to_y(hi[i + e]), rr), nw[j + kRopeHalf]));
        r1[e] = __fsub_rn(__fmul_rn(t1, c), __fmul_rn(t2, s));
        r2[e] = __fadd_rn(__fmul_rn(t2, c), __fmul_rn(t1, s));
      }
      o1[i >> 1] = pack_bf16x2(r1[0], r1[1]);
      o2[i >> 1] = pack_bf16x2(r2[0], r2[1]);
    }
    // columns [16g, 16g+16) are chunks 2g, 2g+1; [48+16g, ...) are 6+2g, 7+2g
    st_shared_v4(stg_addr(stg, lane, 2 * g), make_uint4(o1[0], o1[1], o1[2], o1[3]));
    st_shared_v4(stg_addr(stg, lane, 2 * g + 1), make_uint4(o1[4], o1[5], o1[6], o1[7]));
    st_shared_v4(stg_addr(stg, lane, 6 + 2 * g), make_uint4(o2[0], o2[1], o2[2], o2[3]));
    st_shared_v4(stg_addr(stg, lane, 7 + 2 * g), make_uint4(o2[4], o2[5], o2[6], o2[7]));
  }

  // Pass 2b: dims [96, 128) pass through the rotation.
  {
    uint32_t v[32];
    tmem_ld_x32(tcol + kRopeDims, v);
    tmem_wait_ld();
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 8 * g + 2 * e;
        const int d = kRopeDims + i;
        const float t0 = __fmul_rn(__fmul_rn(acc_to_y(v[i]), rr), nw[d]);
        const float t1 = __fmul_rn(__fmul_rn(acc_to_y(v[i + 1]), rr), nw[d + 1]);
        o[e] = pack_bf16x2(t0, t1);
      }
      st_shared_v4(stg_addr(stg, lane, 12 + g), make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    qkv_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
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
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int m_blk, n_blk;
        tile_coords(t, p.num_m_tiles, m_blk, n_blk);
        // Weight columns of this CTA's next tile, pulled into L2 one tile
        // ahead: in a wave every weight tile is touched for the first time,
        // and HBM latency would otherwise outrun the shared-memory ring.
        int n_next = -1;
        if (MH3_PREFETCH_NEXT_B && t + static_cast<int>(gridDim.x) < p.num_tiles) {
          int m_next;
          tile_coords(t + gridDim.x, p.num_m_tiles, m_next, n_next);
          if (n_next == n_blk) n_next = -1;
        }
        for (int kb = 0; kb < kKBlocks; ++kb) {
          if (n_next >= 0) tma_prefetch_l2_2d(&tm_b, kb * BK, n_next * BN);
          if (!wait_phase(sm.empty(stage), phase ^ 1u, abort_flag, p.status, kStatusProducerEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(sm.full(stage), kStageBytes);
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
        if (!wait_phase(sm.tempty(buf), (use & 1u) ^ 1u, abort_flag, p.status, kStatusMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < kKBlocks; ++kb) {
          if (!wait_phase(sm.full(stage), phase, abort_flag, p.status, kStatusMmaFull)) {
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
    const int ew = warp - 2;     // staging slot
    const int quad = warp & 3;   // TMEM lane quadrant this warp may read
    const int row = quad * 32 + lane;
    const uint32_t stg = sm.stg(ew);
    const float* nw_all = sm.norm_w();
    int it = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      bool ok = wait_phase(sm.tfull(buf), use & 1u, abort_flag, p.status, kStatusEpiTmemFull);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      int m_blk, n_blk;
      tile_coords(t, p.num_m_tiles, m_blk, n_blk);
      const int kind = n_blk / kNTilesPerKind;
      const int head0 = (n_blk % kNTilesPerKind) * 2;
      const int64_t m = static_cast<int64_t>(m_blk) * BM + row;
      int64_t prow = 0;
      if (kind < 2 && m < p.M) {
        if (p.positions) {
          const int64_t pv = __ldg(p.positions + m);
          prow = pv < 0 ? 0 : (pv >= p.S ? p.S - 1 : pv);
        } else {
          prow = m;
        }
      }
      const uint4* cs_row = reinterpret_cast<const uint4*>(p.cos_sin + prow * kRopeDims);
      const int m0 = m_blk * BM + quad * 32;
#pragma unroll 1
      for (int j = 0; j < 2; ++j) {
        const uint32_t tcol = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                              static_cast<uint32_t>(buf * BN + j * kHeadDim);
        // the previous store from this staging buffer must have read it
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        if (kind == 2)
          epi_v_head(tcol, stg, lane);
        else
          epi_qk_head(tcol, stg, lane, nw_all + kind * kHeadDim, cs_row, p.qk_eps);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && m0 < p.M) {
          const int head = head0 + j;
          const int dst = head / p.heads_per_dst;
          const int slot = (head % p.heads_per_dst) * 3 + kind;
          tma_store_4d(&tm_out, stg, 0, slot, m0, dst);
          tma_store_4d(&tm_out, stg + kStgHalfBytes, 64, slot, m0, dst);
          bulk_commit_group();
        }
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

int qkv_smem_bytes() { return kSmemAlloc; }

cudaError_t qkv_prepare_device() {
  return cudaFuncSetAttribute(qkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemAlloc);
}

cudaError_t launch_qkv(const QkvMaps& maps, const QkvParams& p, int grid, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  qkv_gemm_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(maps.a, maps.b, maps.out, p);
  return cudaGetLastError();
}

}  // namespace mh3
