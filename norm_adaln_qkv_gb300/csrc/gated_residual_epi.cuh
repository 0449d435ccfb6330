// gated_residual_epi.cuh -- epilogue policy of the CTA-pair GEMM
// (gemm_pair.cuh) that applies the gated residual to the projection:
//
//   o   = bf16(acc)                                 acc: FP32 (TMEM)
//   out = bf16(residual + bf16(g * o)),  g = gate[index[m]], or 0 when the
//         index lies outside [0, gate_rows) (out = residual)
//
// With E4M3 operands (kFp8) the accumulator is rescaled first, the two
// factors in the order the MLP page prints them:
//   o   = bf16(RN(RN(acc * row_scale[m]) * col_scale[c]))
//
// (flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj, summary formula; the
// same last line as the formula block of
// flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120.)  N = 5376 = 21 tiles;
// K = 64 * KB; IndexT is int32 (output projection) or int64 (MLP).
//
// Per warp and per 128-column half of a tile: TMA-load the warp's 32 x 128
// residual block into its 128-B-swizzled staging buffer (one mbarrier per
// warp), combine it in place with the accumulator row of each thread and the
// gate row of that token (L1/L2-resident table), then TMA-store the block to
// out.  A block is loaded before the same block is stored by the same warp,
// so out may alias residual.  Rows past M are zero-filled on load and clipped
// on store; blocks that start past M are skipped.
#pragma once

#include "gemm_pair.cuh"

namespace mh3 {
namespace gr {

using namespace k2;

template <int KB, typename IndexT, bool kFp8T = false>
struct GatedResidualEpi {
  using Params = GatedResidualParams<IndexT>;
  static constexpr bool kFp8 = kFp8T;
  static constexpr int kKBlocks = KB;
  static constexpr int kNTiles = kHidden / kTileN;  // 21
  static_assert(kHidden % kTileN == 0, "output columns must tile");
  __device__ static int b_row(int n_blk, int rank) { return gp::contiguous_b_row(n_blk, rank); }

  __device__ static void prologue(float*, int, int, const Params&) {}

  __device__ static void tile(const gp::EpiCtx& c, const Params& p, int64_t row0, int n_blk) {
    const int lane = c.lane;
    const int64_t m0 = row0 + c.quad * 32;
    const int64_t m = m0 + lane;
    const bool block_live = m0 < p.M;  // warp-uniform
    const uint4* grow = nullptr;
    const float rs = kFp8T && m < p.M ? __ldg(p.row_scale + m) : 0.0f;
    if (m < p.M) {
      const int64_t gi = static_cast<int64_t>(__ldg(p.gate_index + m));
      if (gi >= 0 && gi < p.gate_rows)
        grow = reinterpret_cast<const uint4*>(p.gate + gi * p.gate_stride);
    }
    const uint64_t pol = policy_evict_first();
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
      const int col0 = n_blk * kTileN + j * kHeadDim;
      // the previous store from this staging buffer must have read it
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      if (block_live) {
        if (lane == 0) {
          mbar_arrive_expect_tx(c.epi_bar, 2 * kStgHalfBytes);
          tma_load_2d(c.stg, c.tm_aux, c.epi_bar, col0, static_cast<int32_t>(m0));
          tma_load_2d(c.stg + kStgHalfBytes, c.tm_aux, c.epi_bar, col0 + 64,
                      static_cast<int32_t>(m0));
        }
        wait_phase<false>(c.epi_bar, *c.epi_phase, c.pair->abort_flag, c.pair->status,
                          kStatusEpiResidual);
        __syncwarp();
        *c.epi_phase ^= 1u;
      }
      const uint32_t tcol = c.tmem_acc + (static_cast<uint32_t>(c.quad * 32) << 16) +
                            static_cast<uint32_t>(j * kHeadDim);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v[32];
        tmem_ld_x32(tcol + 32 * q, v);
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int chunk = 4 * q + g;  // 16-byte chunk of the 128 columns
          const uint32_t addr = stg_addr(c.stg, lane, chunk);
          const uint4 res = ld_shared_v4(addr);
          const uint4 gw = grow ? __ldg(grow + (col0 >> 3) + chunk) : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t rw[4] = {res.x, res.y, res.z, res.w};
          const uint32_t gg[4] = {gw.x, gw.y, gw.z, gw.w};
          float cs[8];
          if (kFp8T) {
            const float4 c0 = __ldg(reinterpret_cast<const float4*>(p.col_scale + col0 + 8 * chunk));
            const float4 c1 =
                __ldg(reinterpret_cast<const float4*>(p.col_scale + col0 + 8 * chunk + 4));
            cs[0] = c0.x; cs[1] = c0.y; cs[2] = c0.z; cs[3] = c0.w;
            cs[4] = c1.x; cs[5] = c1.y; cs[6] = c1.z; cs[7] = c1.w;
          }
          uint32_t ow[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float r2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float acc = __uint_as_float(v[8 * g + 2 * e + h]);
              if (kFp8T) acc = __fmul_rn(__fmul_rn(acc, rs), cs[2 * e + h]);
              const float o = round_bf16(acc);
              const float gv = h ? bf16_hi(gg[e]) : bf16_lo(gg[e]);
              const float rv = h ? bf16_hi(rw[e]) : bf16_lo(rw[e]);
              r2[h] = __fadd_rn(rv, round_bf16(__fmul_rn(gv, o)));
            }
            ow[e] = pack_bf16x2(r2[0], r2[1]);
          }
          st_shared_v4(addr, make_uint4(ow[0], ow[1], ow[2], ow[3]));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && block_live) {
        tma_store_2d_hint(c.tm_out, c.stg, col0, static_cast<int32_t>(m0), pol);
        tma_store_2d_hint(c.tm_out, c.stg + kStgHalfBytes, col0 + 64, static_cast<int32_t>(m0),
                          pol);
        bulk_commit_group();
      }
    }
  }
};

}  // namespace gr
}  // namespace mh3
