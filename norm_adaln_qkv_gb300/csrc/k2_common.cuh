// k2_common.cuh -- pieces shared by the two forms of kernel 2 (one CTA per
// 128x256 tile, and a CTA pair per 256x256 tile): tile order, bounded
// mbarrier waits, and the fused epilogue of one 128-row x 256-column
// accumulator block held in TMEM.
//
// The epilogue computes, per token row m and per head of the tile
// (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention, summary and
// Parameters: q/k_norm_weight, qk_eps, rope_cos_sin, rope_positions, out):
//   y = bf16(acc)
//   kind q/k: t = bf16((y * rr) * w_kind[d]), rr = 1/sqrt(sum_d y^2/128 + qk_eps)
//             p = clamp(positions[m], 0, S-1) (or m); for j < 48:
//             o_j = bf16(t_j c_j - t_{j+48} s_j), o_{j+48} = bf16(t_{j+48} c_j + t_j s_j)
//             with c_j = cos_sin[p, j], s_j = cos_sin[p, 48 + j]; o_d = t_d, d >= 96
//   kind v:   o = y
//   out[head / (56/P), m, head % (56/P), kind, d] = o_d
// Each thread owns one accumulator row (one TMEM lane), so the per-head sum of
// squares and the (j, j+48) pairs are thread-local.  Results go through a
// 128-B-swizzled staging buffer (one head, 32 rows, per warp) and leave by
// 4-D TMA stores straight into out[P, M, 56/P, 3, 128]; rows past M are
// clipped by TMA and fully out-of-range boxes are skipped.
#pragma once

#include "common.cuh"
#include "e4m3.cuh"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace mh3 {
namespace k2 {

constexpr int BK = 64;                          // k-block: 64 bf16 = one 128-B swizzle row
constexpr int kKBlocks = kHidden / BK;          // 84
constexpr int kTileN = 256;                     // two heads of one kind
constexpr int kNTiles = kQkvRows / kTileN;      // 84
constexpr int kNTilesPerKind = kKindCols / kTileN;  // 28
constexpr int kEpiWarps = 4;
constexpr int kStgHalfBytes = 32 * 64 * 2;         // 32 rows x 64 cols bf16 = 4 KB
constexpr int kStgWarpBytes = 2 * kStgHalfBytes;  // one head (128 cols) per warp
constexpr uint32_t kTmemCols = 512;               // 2 accumulators x 256 columns
constexpr uint64_t kWaitLimitNs = 2000000000ull;
#ifndef MH3_PDL
#define MH3_PDL 1
#endif
#ifndef MH3_OUT_EVICT_FIRST
#define MH3_OUT_EVICT_FIRST 1
#endif
static_assert(kHidden % BK == 0, "K must tile");
static_assert(kKindCols % kTileN == 0, "a tile must not straddle q/k/v");
static_assert(kTileN == 2 * kHeadDim, "two heads per tile");

// Launch kernel 2 so that its prologue may overlap the end of the kernel
// before it on the stream (programmatic dependent launch); the producer's
// griddepcontrol.wait keeps the workspace reads behind that kernel.
template <typename Kernel>
inline cudaError_t launch_k2(Kernel kernel, int grid, int threads, int smem, cudaStream_t stream,
                             const QkvMaps& maps, const QkvParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MH3_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, maps.a, maps.b, maps.out, p);
}

// Bounded wait on one mbarrier phase; false when this CTA is aborting.
// (Inline form, for kernels whose warps hold different register budgets and
// so may not call shared subroutines; wait_phase is the out-of-line form.)
template <bool kClusterScope>
__device__ __forceinline__ bool wait_phase_inl(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* status, int code) {
  auto poll = [&]() {
    return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (poll()) return true;
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
template <bool kClusterScope>
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        int* status, int code) {
  return wait_phase_inl<kClusterScope>(bar, parity, abort_flag, status, code);
}

// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_wait_inl(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(status, 0, kStatusDrain);
      return;
    }
  }
}
__device__ __noinline__ inline void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  drain_wait_inl(bar, parity, status);
}

// Tile t -> (row block, column block): groups of kGroup row blocks, row
// block fastest inside a group, so that the weight columns and activation
// rows of the tiles in flight stay in L2.
template <int kGroup, int kN = kNTiles>
__device__ __forceinline__ void tile_coords(int t, int num_row_blocks, int& r_blk, int& n_blk) {
  const int group_tiles = kGroup * kN;
  const int g = t / group_tiles;
  const int first = g * kGroup;
  const int gm = min(kGroup, num_row_blocks - first);
  const int local = t - g * group_tiles;
  r_blk = first + local % gm;
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

// Two accumulator words -> the bf16-rounded projection y of both columns, as
// packed FP32.
__device__ __forceinline__ uint64_t acc2_to_y2(uint32_t a, uint32_t b) {
  return f2_from_bf16x2(f2_to_bf16x2(f2_pack(__uint_as_float(a), __uint_as_float(b))));
}

// Q or K head: RMSNorm over the 128 columns, rotation of [0, 96), pass-through
// of [96, 128).  Packed two-lane FP32 over neighbouring columns (d, d + 1):
// each lane is one IEEE round-to-nearest operation, in the order of the
// formulas (sum of squares in four partial sums over d % 4, d increasing;
// t = bf16((y * rr) * w); o = bf16(t_j c - t_{j+48} s), bf16(t_{j+48} c + t_j s)).
__device__ __forceinline__ void epi_qk_head(uint32_t tcol, uint32_t stg, int lane, const float* nw,
                                            const uint4* cs_row, float qk_eps) {
  auto nw2 = [&](int d) {
    const float2 w = *reinterpret_cast<const float2*>(nw + d);
    return f2_pack(w.x, w.y);
  };
  // Pass 1: FP32 sum of squares of the bf16-rounded projection.
  uint64_t s01 = 0, s23 = 0;  // (+0.0, +0.0)
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t v[32];
    tmem_ld_x32(tcol + 32 * c, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const uint64_t y01 = acc2_to_y2(v[i], v[i + 1]);
      const uint64_t y23 = acc2_to_y2(v[i + 2], v[i + 3]);
      s01 = f2_fma(y01, y01, s01);
      s23 = f2_fma(y23, y23, s23);
    }
  }
  float s0, s1, s2, s3;
  f2_unpack(s01, s0, s1);
  f2_unpack(s23, s2, s3);
  const float ss = __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
  const float rr = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, 128.0f), qk_eps)));
  const uint64_t rr2 = f2_pack(rr, rr);

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
      const int j = 16 * g + i;
      const uint64_t c2 = f2_from_bf16x2((&cv[i >> 3].x)[(i & 7) >> 1]);
      const uint64_t s2 = f2_from_bf16x2((&sv[i >> 3].x)[(i & 7) >> 1]);
      const uint64_t ta = f2_from_bf16x2(
          f2_to_bf16x2(f2_mul(f2_mul(acc2_to_y2(lo[i], lo[i + 1]), rr2), nw2(j))));
      const uint64_t tb = f2_from_bf16x2(f2_to_bf16x2(
          f2_mul(f2_mul(acc2_to_y2(hi[i], hi[i + 1]), rr2), nw2(j + kRopeHalf))));
      o1[i >> 1] = f2_to_bf16x2(f2_sub(f2_mul(ta, c2), f2_mul(tb, s2)));
      o2[i >> 1] = f2_to_bf16x2(f2_add(f2_mul(tb, c2), f2_mul(ta, s2)));
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
        o[e] = f2_to_bf16x2(
            f2_mul(f2_mul(acc2_to_y2(v[i], v[i + 1]), rr2), nw2(kRopeDims + i)));
      }
      st_shared_v4(stg_addr(stg, lane, 12 + g), make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

// e4m3 output mode: turn this thread's staged bf16 row (16 chunks over both
// halves) into 128 e4m3 codes (the quantiser of e4m3.cuh), written in place
// over the first half as one 128-byte swizzled row (the layout of a
// 128 x 32 byte box).  Only this thread's row is read or written.
template <bool kFast>
__device__ __forceinline__ void stage_row_to_e4m3(uint32_t stg, int lane,
                                                  const e4m3q::Divisor& dv) {
  uint4 w[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) w[c] = ld_shared_v4(stg_addr(stg, lane, c));
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // e4m3 chunk c = bf16 chunks 2c, 2c+1
    const uint2 a = e4m3q::quantize8<kFast>(w[2 * c], dv);
    const uint2 b = e4m3q::quantize8<kFast>(w[2 * c + 1], dv);
    st_shared_v4(stg_addr(stg, lane, c), make_uint4(a.x, a.y, b.x, b.y));
  }
}

__device__ __forceinline__ void stage_to_e4m3(uint32_t stg, int lane, float descale) {
  const e4m3q::Divisor dv = e4m3q::make_divisor(descale);
  if (dv.fast)
    stage_row_to_e4m3<true>(stg, lane, dv);
  else
    stage_row_to_e4m3<false>(stg, lane, dv);
}

// cos/sin row of token m for kind (q or k); v needs none.
__device__ __forceinline__ const uint4* rope_row(const QkvParams& p, int64_t m, int kind) {
  int64_t prow = 0;
  if (kind < 2 && m < p.M) {
    if (p.positions) {
      const int64_t pv = __ldg(p.positions + m);
      prow = pv < 0 ? 0 : (pv >= p.S ? p.S - 1 : pv);
    } else {
      prow = m;
    }
  }
  return reinterpret_cast<const uint4*>(p.cos_sin + prow * kRopeDims);
}

// The epilogue of one 128-column head for this warp's 32 accumulator rows.
//   tcol      TMEM address of the warp's lanes, first column of the head
//   m0        token row of the warp's first lane
// The previous store from the staging buffer is waited for first; the new
// one may still be in flight on return (bulk group of lane 0).
template <bool kE4m3>
__device__ __forceinline__ void epilogue_head(uint32_t tcol, int lane, uint32_t stg,
                                              const float* nw_all, const QkvParams& p, int64_t m0,
                                              int kind, int head, const uint4* cs_row,
                                              const CUtensorMap* tm_out) {
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
  if (kind == 2)
    epi_v_head(tcol, stg, lane);
  else
    epi_qk_head(tcol, stg, lane, nw_all + kind * kHeadDim, cs_row, p.qk_eps);
  if (kE4m3) stage_to_e4m3(stg, lane, __ldg(p.descales + kind));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && m0 < p.M) {
    const int dst = head / p.heads_per_dst;
    const int slot = (head % p.heads_per_dst) * 3 + kind;
    if (kE4m3) {
      tma_store_4d_hint(tm_out, stg, 0, slot, static_cast<int32_t>(m0), dst, policy_evict_first());
    } else if (MH3_OUT_EVICT_FIRST) {
      // out is written once and read by the next operation, not by this
      // one: evict-first keeps it from lingering dirty in L2
      const uint64_t pol = policy_evict_first();
      tma_store_4d_hint(tm_out, stg, 0, slot, static_cast<int32_t>(m0), dst, pol);
      tma_store_4d_hint(tm_out, stg + kStgHalfBytes, 64, slot, static_cast<int32_t>(m0), dst, pol);
    } else {
      tma_store_4d(tm_out, stg, 0, slot, static_cast<int32_t>(m0), dst);
      tma_store_4d(tm_out, stg + kStgHalfBytes, 64, slot, static_cast<int32_t>(m0), dst);
    }
    bulk_commit_group();
  }
}

// NVFP4 output mode: this thread's staged bf16 row (128 values of one head,
// token m) as 8 blocks of 16 -> 64 bytes of E2M1 codes and 8 UE4M3 scales
// (nvfp4.cuh, one rounding of each exact quotient), stored straight to
// global memory (row m < M only).
__device__ __forceinline__ void stage_row_to_nvfp4(uint32_t stg, int lane, const fp4::Table16& q,
                                                   uint8_t* codes, uint8_t* sf, bool store) {
  uint32_t cw[16];
  uint32_t sw[2] = {0u, 0u};
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const uint4 w0 = ld_shared_v4(stg_addr(stg, lane, 2 * b));
    const uint4 w1 = ld_shared_v4(stg_addr(stg, lane, 2 * b + 1));
    const float amax = fmaxf(fp4::amax8(w0), fp4::amax8(w1));
    const fp4::BlockScale bs = fp4::block_scale_t16(amax, q);
    cw[2 * b] = fp4::encode8(w0, bs, q.gs);
    cw[2 * b + 1] = fp4::encode8(w1, bs, q.gs);
    sw[b >> 2] |= bs.code << (8 * (b & 3));
  }
  if (store) {
    uint4* c4 = reinterpret_cast<uint4*>(codes);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      __stcs(c4 + i, make_uint4(cw[4 * i], cw[4 * i + 1], cw[4 * i + 2], cw[4 * i + 3]));
    __stcs(reinterpret_cast<uint2*>(sf), make_uint2(sw[0], sw[1]));
  }
}

// The epilogue of one head whose bf16 projection y is already in registers
// (y[i] holds columns 2i (low half) and 2i + 1): the same operations, in the
// same order, as epilogue_head on an accumulator in TMEM.  kOut: kOutBf16,
// kOutE4m3 (codes through the staging buffer and TMA) or kOutNvfp4 (codes
// and scales stored from registers; fq: the q, k, v quantiser tables).
template <int kOut>
__device__ __forceinline__ void epilogue_head_regs(const uint32_t (&y)[64], int lane, uint32_t stg,
                                                   const float* nw_all, const QkvParams& p,
                                                   int64_t m0, int kind, int head,
                                                   const uint4* cs_row,
                                                   const CUtensorMap* tm_out,
                                                   const fp4::Table16* fq = nullptr) {
  constexpr bool kE4m3 = kOut == kOutE4m3;
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
  if (kind == 2) {
#pragma unroll
    for (int c = 0; c < 16; ++c)
      st_shared_v4(stg_addr(stg, lane, c), make_uint4(y[4 * c], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3]));
  } else {
    // Packed two-lane FP32 (each lane one IEEE round-to-nearest operation, in
    // epi_qk_head's order): lane pairs are neighbouring columns (d, d + 1).
    const float* nw = nw_all + kind * kHeadDim;
    auto nw2 = [&](int d) {
      const float2 w = *reinterpret_cast<const float2*>(nw + d);
      return f2_pack(w.x, w.y);
    };
    // FP32 sum of squares: four partial sums over columns d % 4, d increasing
    uint64_t s01 = 0, s23 = 0;  // (+0.0, +0.0)
#pragma unroll
    for (int i = 0; i < kHeadDim / 4; ++i) {
      const uint64_t y01 = f2_from_bf16x2(y[2 * i]);
      const uint64_t y23 = f2_from_bf16x2(y[2 * i + 1]);
      s01 = f2_fma(y01, y01, s01);
      s23 = f2_fma(y23, y23, s23);
    }
    float s0, s1, s2, s3;
    f2_unpack(s01, s0, s1);
    f2_unpack(s23, s2, s3);
    const float ss = __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
    const float rr = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, 128.0f), p.qk_eps)));
    const uint64_t rr2 = f2_pack(rr, rr);
    // t = bf16((y * rr) * w) for the column pair (d, d + 1), back as FP32
    auto t2 = [&](int d) {
      return f2_from_bf16x2(f2_to_bf16x2(f2_mul(f2_mul(f2_from_bf16x2(y[d >> 1]), rr2), nw2(d))));
    };
    // rotated dims: chunk c (columns 8c..8c+7, c < 6) pairs with chunk c + 6
#pragma unroll
    for (int c = 0; c < 6; ++c) {
      const uint4 cv = __ldg(cs_row + c);
      const uint4 sv = __ldg(cs_row + 6 + c);
      const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
      const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
      uint32_t o1[4], o2[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const int j = 8 * c + 2 * e2;
        const uint64_t c2 = f2_from_bf16x2(cw[e2]);
        const uint64_t s2 = f2_from_bf16x2(sw[e2]);
        const uint64_t ta = t2(j), tb = t2(j + kRopeHalf);
        o1[e2] = f2_to_bf16x2(f2_sub(f2_mul(ta, c2), f2_mul(tb, s2)));
        o2[e2] = f2_to_bf16x2(f2_add(f2_mul(tb, c2), f2_mul(ta, s2)));
      }
      st_shared_v4(stg_addr(stg, lane, c), make_uint4(o1[0], o1[1], o1[2], o1[3]));
      st_shared_v4(stg_addr(stg, lane, c + 6), make_uint4(o2[0], o2[1], o2[2], o2[3]));
    }
    // dims [96, 128) pass through the rotation
#pragma unroll
    for (int c = 12; c < 16; ++c) {
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = 8 * c + 2 * e;
        o[e] = f2_to_bf16x2(f2_mul(f2_mul(f2_from_bf16x2(y[d >> 1]), rr2), nw2(d)));
      }
      st_shared_v4(stg_addr(stg, lane, c), make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
  if (kOut == kOutNvfp4) {
    // each thread reads back only its own staged row
    const int64_t m = m0 + lane;
    const int dst = head / p.heads_per_dst;
    const int slot = (head % p.heads_per_dst) * 3 + kind;
    const int64_t r = (static_cast<int64_t>(dst) * p.M + m) * (3 * p.heads_per_dst) + slot;
    stage_row_to_nvfp4(stg, lane, fq[kind], p.out_codes + r * 64, p.out_sf + r * 8, m < p.M);
    __syncwarp();  // the staging buffer is free again for the next head
    return;
  }
  if (kE4m3) stage_to_e4m3(stg, lane, __ldg(p.descales + kind));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && m0 < p.M) {
    const int dst = head / p.heads_per_dst;
    const int slot = (head % p.heads_per_dst) * 3 + kind;
    const uint64_t pol = policy_evict_first();
    if (kE4m3) {
      tma_store_4d_hint(tm_out, stg, 0, slot, static_cast<int32_t>(m0), dst, pol);
    } else {
      tma_store_4d_hint(tm_out, stg, 0, slot, static_cast<int32_t>(m0), dst, pol);
      tma_store_4d_hint(tm_out, stg + kStgHalfBytes, 64, slot, static_cast<int32_t>(m0), dst, pol);
    }
    bulk_commit_group();
  }
}

// The epilogue of one 128-row x 256-column accumulator block.
//   tmem_acc  TMEM address of the block (lane 0, first column)
//   quad      TMEM lane quadrant this warp may read (warp index % 4)
//   row0      token row of TMEM lane 0 of the block
//   n_blk     256-column block of the 21504 projection columns
// Returns after every TMEM read of the block has completed; the stores may
// still be in flight (bulk groups of this warp's lane 0).
template <bool kE4m3 = false>
__device__ __forceinline__ void epilogue_block(uint32_t tmem_acc, int quad, int lane, uint32_t stg,
                                               const float* nw_all, const QkvParams& p,
                                               int64_t row0, int n_blk, const CUtensorMap* tm_out) {
  const int kind = n_blk / kNTilesPerKind;
  const int head0 = (n_blk % kNTilesPerKind) * 2;
  const int64_t m0 = row0 + quad * 32;
  if (m0 >= p.M) return;  // this warp's rows are all past M: nothing is stored
  const int64_t m = m0 + lane;
  const uint4* cs_row = rope_row(p, m, kind);
#pragma unroll 1
  for (int j = 0; j < 2; ++j) {
    const uint32_t tcol = tmem_acc + (static_cast<uint32_t>(quad * 32) << 16) +
                          static_cast<uint32_t>(j * kHeadDim);
    epilogue_head<kE4m3>(tcol, lane, stg, nw_all, p, m0, kind, head0 + j, cs_row, tm_out);
  }
}

}  // namespace k2
}  // namespace mh3
