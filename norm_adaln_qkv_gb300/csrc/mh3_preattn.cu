// mh3_preattn.cu -- the C ABI of the pre-attention stage (declared in
// include/mh3_preattn.h): argument validation, the handle, TMA tensor-map
// encoding and the two launches.
//
// Validation follows flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention,
// Parameters: contiguous x/out/weights, AdaLN tables with unit column stride
// and a row stride that is a multiple of 8 elements with a 16-byte aligned
// base, rows >= 1, S >= 1, S >= M for identity positions, P in {1,2,4,8},
// qk_eps None -> eps.  Index and position VALUES are never validated on the
// host (no synchronising reduction): kernel 1 guards indices and kernel 2
// clamps positions (Notes; Parameters: adaln_index, rope_positions).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "mh3_preattn.h"
#include "common.cuh"

namespace mh3 {
// Workspace rows per stage of the single-CTA GEMM's A box for this M (its
// tiny-M ring loads fewer rows); defined with that kernel.
int qkv_a_box_rows(int64_t M);
}  // namespace mh3

using namespace mh3;

struct mh3_preattn_ctx {
  int device = 0;
  int num_sms = 0;
  int max_clusters = 0;  // resident 2-CTA clusters of the pair GEMM
  int out_proj_clusters = 0;  // the same for the output projection
  int e4m3_clusters = 0;      // ... the e4m3-output QKV GEMM
  int fc1_clusters = 0;       // ... and the two MLP GEMMs
  int fc2_clusters = 0;
  void* ws_y = nullptr;  // handle-owned MLP intermediate y [M, 14336]
  size_t ws_y_bytes = 0;
  int* d_status = nullptr;
  void* ws = nullptr;  // handle-owned workspace (grown on demand)
  size_t ws_bytes = 0;
  int nvfp4_clusters = 0;       // resident clusters of the NVFP4 GEMM (bf16 out)
  int nvfp4_e4m3_clusters = 0;  // ... and its e4m3-output form
  int nvfp4_fp4out_clusters = 0;  // ... and its NVFP4-output form
  int nvfp4_out_clusters = 0;   // ... and the W4A4 output projection
  void* act_q = nullptr;        // handle-owned NVFP4 stage-1 workspaces
  size_t act_q_bytes = 0;
  void* act_sf = nullptr;
  size_t act_sf_bytes = 0;
  int test_stall_next = 0;  // test hook for the next CTA-pair QKV GEMM launch (bf16 or NVFP4)
  void* sk_buf = nullptr;   // split-tail scratch of the pair form (flags, partials)
  size_t sk_bytes = 0;
  int fc1_fp8_clusters = 0;     // resident clusters of the FP8 MLP GEMMs
  int fc2_fp8_clusters = 0;
  void* fp8_aq = nullptr;       // handle-owned FP8 MLP workspaces
  size_t fp8_aq_bytes = 0;
  void* fp8_as = nullptr;
  size_t fp8_as_bytes = 0;
  void* fp8_yq = nullptr;
  size_t fp8_yq_bytes = 0;
  void* fp8_ys = nullptr;
  size_t fp8_ys_bytes = 0;
};

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MH3_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kMaxM = int64_t(1) << 30;  // TMA coordinates are 32-bit

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_ptr(const void* p, const char* name, uintptr_t align) {
  if (p == nullptr) return fail(MH3_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, align))
    return fail(MH3_ERR_ALIGNMENT, "%s must be %d-byte aligned", name, static_cast<int>(align));
  return MH3_OK;
}

bool valid_eps(float e) { return std::isfinite(e) && e > 0.0f; }
bool qk_eps_means_default(float e) { return std::isnan(e) || e < 0.0f; }

int check_M(int64_t M) {
  if (M < 0) return fail(MH3_ERR_INVALID_ARG, "M must be >= 0 (got %lld)", (long long)M);
  if (M > kMaxM) return fail(MH3_ERR_INVALID_ARG, "M must be <= 2^30 (got %lld)", (long long)M);
  return MH3_OK;
}

int check_norm_adaln_args(int64_t M, const mh3_bf16* x, const mh3_bf16* xw, const mh3_bf16* sc,
                          int64_t sc_stride, const mh3_bf16* sh, int64_t sh_stride, int64_t rows,
                          const void* idx, float eps, const mh3_bf16* ws, bool ws_required,
                          uintptr_t idx_align = 8) {
  int rc;
  if ((rc = check_M(M))) return rc;
  if (rows < 1) return fail(MH3_ERR_INVALID_ARG, "rows must be >= 1 (got %lld)", (long long)rows);
  if (!valid_eps(eps)) return fail(MH3_ERR_INVALID_ARG, "eps must be finite and > 0");
  const char* names[2] = {"scale_row_stride", "shift_row_stride"};
  const int64_t strides[2] = {sc_stride, sh_stride};
  for (int i = 0; i < 2; ++i) {
    if (strides[i] < kHidden)
      return fail(MH3_ERR_INVALID_ARG, "%s must be >= 5376 (got %lld)", names[i],
                  (long long)strides[i]);
    if (strides[i] % 8 != 0)
      return fail(MH3_ERR_ALIGNMENT, "%s must be a multiple of 8 elements (got %lld)", names[i],
                  (long long)strides[i]);
  }
  if ((rc = check_ptr(xw, "x_norm_weight", 16))) return rc;
  if ((rc = check_ptr(sc, "adaln_scale", 16))) return rc;
  if ((rc = check_ptr(sh, "adaln_shift", 16))) return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_ptr(x, "x", 16))) return rc;
  if ((rc = check_ptr(idx, "adaln_index", idx_align))) return rc;
  if (ws_required || ws != nullptr)
    if ((rc = check_ptr(ws, "workspace", 16))) return rc;
  return MH3_OK;
}

int check_qkv_args(int64_t M, const mh3_bf16* W, const mh3_bf16* qw, const mh3_bf16* kw,
                   const mh3_bf16* cs, int64_t S, const int64_t* pos, int P, const mh3_bf16* out) {
  int rc;
  if ((rc = check_M(M))) return rc;
  if (!(P == 1 || P == 2 || P == 4 || P == 8))
    return fail(MH3_ERR_INVALID_ARG, "P (ulysses_degree) must be 1, 2, 4 or 8 (got %d)", P);
  if (S < 1) return fail(MH3_ERR_INVALID_ARG, "S must be >= 1 (got %lld)", (long long)S);
  if (pos == nullptr && S < M)
    return fail(MH3_ERR_INVALID_ARG,
                "identity positions (NULL) need S >= M (S=%lld, M=%lld)", (long long)S,
                (long long)M);
  if ((rc = check_ptr(W, "qkv_weight", 16))) return rc;
  if ((rc = check_ptr(qw, "q_norm_weight", 2))) return rc;
  if ((rc = check_ptr(kw, "k_norm_weight", 2))) return rc;
  if ((rc = check_ptr(cs, "rope_cos_sin", 16))) return rc;
  if (M == 0) return MH3_OK;
  if (pos != nullptr && !aligned(pos, 8))
    return fail(MH3_ERR_ALIGNMENT, "rope_positions must be 8-byte aligned");
  if ((rc = check_ptr(out, "out", 16))) return rc;
  return MH3_OK;
}

int check_handle(mh3_preattn_t h) {
  if (h == nullptr) return fail(MH3_ERR_INVALID_ARG, "handle is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h->device)
    return fail(MH3_ERR_INVALID_ARG, "current device %d differs from the handle's device %d", dev,
                h->device);
  return MH3_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int encode_maps(QkvMaps& maps, int64_t M, const mh3_bf16* ws, const mh3_bf16* W, int P,
                mh3_bf16* out, unsigned b_box_rows, unsigned a_box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return fail(MH3_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  const cuuint32_t unit[4] = {1, 1, 1, 1};
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHidden), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHidden) * 2};
    const cuuint32_t box[2] = {64, a_box_rows};
    CUresult r = enc(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<mh3_bf16*>(ws), dims,
                     strides, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MH3_ERR_CUDA, "tensor map (workspace) failed: %d", (int)r);
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHidden),
                                static_cast<cuuint64_t>(kQkvRows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHidden) * 2};
    const cuuint32_t box[2] = {64, b_box_rows};
    CUresult r = enc(&maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<mh3_bf16*>(W), dims,
                     strides, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MH3_ERR_CUDA, "tensor map (qkv_weight) failed: %d", (int)r);
  }
  {
    // out[P, M, 56/P, 3, 128] as (d, slot = hl*3 + kind, m, dst)
    const int64_t slots = 3 * (kHeads / P);
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(slots),
                                static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(P)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                   static_cast<cuuint64_t>(slots) * kHeadDim * 2,
                                   static_cast<cuuint64_t>(M) * slots * kHeadDim * 2};
    const cuuint32_t box[4] = {64, 1, 32, 1};
    CUresult r = enc(&maps.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, out, dims, strides, box, unit,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MH3_ERR_CUDA, "tensor map (out) failed: %d", (int)r);
  }
  return MH3_OK;
}

// Grow a handle-owned buffer to `need` bytes with stream-ordered allocation.
int grow_buffer(void** buf, size_t* cap, size_t need, cudaStream_t s) {
  if (*cap >= need) return MH3_OK;
  if (*buf) {
    cudaError_t e = cudaFreeAsync(*buf, s);
    *buf = nullptr;
    *cap = 0;
    if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync (workspace)");
  }
  cudaError_t e = cudaMallocAsync(buf, need, s);
  if (e != cudaSuccess) {
    *buf = nullptr;
    return fail(MH3_ERR_OOM, "cudaMallocAsync of %zu B workspace failed: %s", need,
                cudaGetErrorString(e));
  }
  *cap = need;
  return MH3_OK;
}

// 2-D row-major uint8 tensor [rows, cols] (cols contiguous bytes), 128-B swizzle.
int encode_u8_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                 uint32_t box_cols, uint32_t box_rows, const char* what) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return fail(MH3_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t unit[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MH3_ERR_CUDA, "tensor map (%s) failed: %d", what, (int)r);
  return MH3_OK;
}

// 2-D row-major bf16 tensor [rows, cols] (cols contiguous), 128-B swizzle.
int encode_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows, const char* what) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return fail(MH3_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t unit[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MH3_ERR_CUDA, "tensor map (%s) failed: %d", what, (int)r);
  return MH3_OK;
}

int launch_stage1(cudaStream_t s, int num_sms, int* status, int64_t M, const mh3_bf16* x,
                  const mh3_bf16* xw, const mh3_bf16* sc, int64_t sc_stride, const mh3_bf16* sh,
                  int64_t sh_stride, int64_t rows, const int64_t* idx, float eps, mh3_bf16* ws,
                  int* clear = nullptr, int clear_count = 0) {
  NormAdalnParams p;
  p.clear = clear;
  p.clear_count = clear_count;
  p.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p.x_norm_weight = reinterpret_cast<const __nv_bfloat16*>(xw);
  p.scale = reinterpret_cast<const __nv_bfloat16*>(sc);
  p.shift = reinterpret_cast<const __nv_bfloat16*>(sh);
  p.scale_stride = sc_stride;
  p.shift_stride = sh_stride;
  p.rows = rows;
  p.index = idx;
  p.workspace = reinterpret_cast<__nv_bfloat16*>(ws);
  p.M = M;
  p.eps = eps;
  p.status = status;
  cudaError_t e = launch_norm_adaln(p, num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "norm/AdaLN launch");
  return MH3_OK;
}

// Scratch of the pair form's split tail, owned by a handle: one flag per
// (split tile, CTA, epilogue warp), then the FP32 partials.  The flags are
// cleared before every split launch, on the stream (inside a captured graph
// too): by kernel 1 of the same call, or by a memset when kernel 2 runs
// alone.  A partial's writer sets its flag to 1.
constexpr int kSplitMaxTiles = 128;  // more than half of any resident cluster count
constexpr size_t kSplitFlagBytes = kSplitMaxTiles * 8 * sizeof(int);
constexpr size_t kSplitSlotBytes = 8 * 256 * 32 * sizeof(float);  // 2 CTAs x 4 warps x 256 x 32
struct SplitScratch {
  void** buf;
  size_t* bytes;
};

// Tiles of the pair form's last wave that are split (0: no split): the last
// wave must hold at most half as many tiles as there are clusters.
int split_tiles(int64_t M, int max_clusters) {
  if (M <= 128 || max_clusters <= 0) return 0;
  const int tiles = static_cast<int>((M + 255) / 256) * (kQkvRows / 256);
  const int clusters = tiles < max_clusters ? tiles : max_clusters;
  const int rem = tiles % clusters;
  return tiles > clusters && rem > 0 && 2 * rem <= clusters && rem <= kSplitMaxTiles ? rem : 0;
}

// Grows the scratch to `tiles` split tiles; clears the flags on `s` when
// `clear` (otherwise kernel 1 of the call clears them).
int prepare_split(const SplitScratch& sk, int tiles, cudaStream_t s, bool clear) {
  const size_t need = kSplitFlagBytes + static_cast<size_t>(tiles) * kSplitSlotBytes;
  if (*sk.bytes < need) {
    if (*sk.buf) {
      cudaError_t e = cudaFreeAsync(*sk.buf, s);
      *sk.buf = nullptr;
      *sk.bytes = 0;
      if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync (split scratch)");
    }
    cudaError_t e = cudaMallocAsync(sk.buf, need, s);
    if (e != cudaSuccess) {
      *sk.buf = nullptr;
      return fail(MH3_ERR_OOM, "cudaMallocAsync of %zu B split scratch failed: %s", need,
                  cudaGetErrorString(e));
    }
    *sk.bytes = need;
  }
  if (!clear) return MH3_OK;
  cudaError_t e = cudaMemsetAsync(*sk.buf, 0, kSplitFlagBytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the split flags");
  return MH3_OK;
}

// Kernel 2: the CTA-pair form for M > 128 (when pairs can be resident), the
// single-CTA form otherwise.  With `sk`, a pair-form launch whose last wave
// holds at most half as many tiles as there are clusters splits those tiles
// along K over two clusters each (the last wave then takes half a tile).
// after_k1: the launch follows this stage's kernel 1 on the stream, so the
// pair form may fetch its first weight boxes before waiting for that grid.
int launch_stage2(cudaStream_t s, int num_sms, int max_clusters, int* status, int64_t M,
                  const mh3_bf16* ws, const mh3_bf16* W, const mh3_bf16* qw, const mh3_bf16* kw,
                  const mh3_bf16* cs, int64_t S, const int64_t* pos, int P, float qk_eps,
                  mh3_bf16* out, int* test_stall = nullptr, const SplitScratch* sk = nullptr,
                  bool after_k1 = false) {
  const bool pair = M > 128 && max_clusters > 0;
  QkvMaps maps;
  int rc = encode_maps(maps, M, ws, W, P, out, pair ? 128u : 256u,
                       pair ? 128u : static_cast<unsigned>(qkv_a_box_rows(M)));
  if (rc) return rc;
  QkvParams p;
  p.positions = pos;
  p.cos_sin = reinterpret_cast<const __nv_bfloat16*>(cs);
  p.q_norm_weight = reinterpret_cast<const __nv_bfloat16*>(qw);
  p.k_norm_weight = reinterpret_cast<const __nv_bfloat16*>(kw);
  p.M = M;
  p.S = S;
  p.heads_per_dst = kHeads / P;
  p.qk_eps = qk_eps;
  p.status = status;
  p.descales = nullptr;
  cudaError_t e;
  if (pair) {
    p.num_m_tiles = static_cast<int>((M + 255) / 256);
    p.num_tiles = p.num_m_tiles * (kQkvRows / 256);
    const int clusters = p.num_tiles < max_clusters ? p.num_tiles : max_clusters;
    // the caller has prepared the scratch for this M (prepare_split)
    const int rem = sk != nullptr ? split_tiles(M, max_clusters) : 0;
    if (rem > 0) {
      p.sk_dp = p.num_tiles - rem;
      p.sk_tail = rem;
      p.sk_flags = static_cast<int*>(*sk->buf);
      p.sk_partial = reinterpret_cast<float*>(static_cast<uint8_t*>(*sk->buf) + kSplitFlagBytes);
      p.sk_seq = 1;
    }
    if (test_stall != nullptr) {
      p.test_stall = *test_stall;
      *test_stall = 0;
    }
    p.b_early = after_k1 ? 1 : 0;
    e = launch_qkv_pair(maps, p, clusters, s);
  } else {
    p.num_m_tiles = static_cast<int>((M + 127) / 128);
    p.num_tiles = p.num_m_tiles * (kQkvRows / 256);
    const int grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
    e = launch_qkv(maps, p, grid, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "QKV GEMM launch");
  return MH3_OK;
}

}  // namespace

extern "C" {

const char* mh3_preattn_last_error(void) { return g_last_error.c_str(); }

size_t mh3_preattn_workspace_bytes(int64_t M) {
  return M <= 0 ? 0 : static_cast<size_t>(M) * kHidden * 2;
}

size_t mh3_preattn_out_bytes(int64_t M) {
  return M <= 0 ? 0 : static_cast<size_t>(M) * kQkvRows * 2;
}

int mh3_preattn_create(mh3_preattn_t* handle, int device) {
  if (handle == nullptr) return fail(MH3_ERR_INVALID_ARG, "handle pointer is NULL");
  *handle = nullptr;
  cudaError_t e = cudaSetDevice(device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(MH3_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                device, prop.major, prop.minor);
  if (static_cast<int>(prop.sharedMemPerBlockOptin) < qkv_smem_bytes())
    return fail(MH3_ERR_UNSUPPORTED, "device allows %zu B of shared memory per block, need %d",
                prop.sharedMemPerBlockOptin, qkv_smem_bytes());
  e = qkv_prepare_device();
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  int max_clusters = 0;
  e = qkv_pair_prepare_device(&max_clusters);
  if (e != cudaSuccess) return cuda_fail(e, "preparing the pair GEMM");
  int out_proj_clusters = 0;
  e = out_proj_prepare_device(&out_proj_clusters);
  if (e != cudaSuccess) return cuda_fail(e, "preparing the output-projection GEMM");
  int e4m3_clusters = 0;
  e = qkv_e4m3_prepare_device(&e4m3_clusters);
  if (e != cudaSuccess) return cuda_fail(e, "preparing the e4m3-output GEMM");
  int fc1_clusters = 0, fc2_clusters = 0;
  e = mlp_fc1_prepare_device(&fc1_clusters);
  if (e == cudaSuccess) e = mlp_fc2_prepare_device(&fc2_clusters);
  if (e != cudaSuccess) return cuda_fail(e, "preparing the MLP GEMMs");
  int nvfp4_clusters = 0, nvfp4_e4m3_clusters = 0, nvfp4_fp4out_clusters = 0;
  e = nvfp4_qkv_prepare_device(&nvfp4_clusters, &nvfp4_e4m3_clusters, &nvfp4_fp4out_clusters);
  if (e != cudaSuccess) return cuda_fail(e, "preparing the NVFP4 GEMM");
  int nvfp4_out_clusters = 0;
  e = nvfp4_out_proj_prepare_device(&nvfp4_out_clusters);
  if (e != cudaSuccess) return cuda_fail(e, "preparing the NVFP4 output projection");
  int fc1_fp8_clusters = 0, fc2_fp8_clusters = 0;
  e = mlp_fp8_fc1_prepare_device(&fc1_fp8_clusters);
  if (e == cudaSuccess) e = mlp_fp8_fc2_prepare_device(&fc2_fp8_clusters);
  if (e != cudaSuccess) return cuda_fail(e, "preparing the FP8 MLP GEMMs");
  mh3_preattn_ctx* h = new mh3_preattn_ctx();
  h->device = device;
  h->nvfp4_clusters = nvfp4_clusters;
  h->nvfp4_e4m3_clusters = nvfp4_e4m3_clusters;
  h->nvfp4_out_clusters = nvfp4_out_clusters;
  h->nvfp4_fp4out_clusters = nvfp4_fp4out_clusters;
  h->fc1_clusters = fc1_clusters;
  h->e4m3_clusters = e4m3_clusters;
  h->fc2_clusters = fc2_clusters;
  h->fc1_fp8_clusters = fc1_fp8_clusters;
  h->fc2_fp8_clusters = fc2_fp8_clusters;
  h->num_sms = prop.multiProcessorCount;
  h->max_clusters = max_clusters;
  h->out_proj_clusters = out_proj_clusters;
  e = cudaMalloc(&h->d_status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int));
  if (e != cudaSuccess) {
    if (h->d_status) cudaFree(h->d_status);
    delete h;
    return cuda_fail(e, "allocating the status word");
  }
  *handle = h;
  return MH3_OK;
}

int mh3_preattn_destroy(mh3_preattn_t h) {
  if (h == nullptr) return MH3_OK;
  int rc = MH3_OK;
  if (h->ws) {
    cudaError_t e = cudaFree(h->ws);
    if (e != cudaSuccess) rc = cuda_fail(e, "freeing the handle workspace");
  }
  for (void* buf : {h->ws_y, h->act_q, h->act_sf, h->fp8_aq, h->fp8_as, h->fp8_yq, h->fp8_ys,
                    h->sk_buf}) {
    if (buf == nullptr) continue;
    cudaError_t e = cudaFree(buf);
    if (e != cudaSuccess && rc == MH3_OK) rc = cuda_fail(e, "freeing the handle workspace");
  }
  if (h->d_status) {
    cudaError_t e = cudaFree(h->d_status);
    if (e != cudaSuccess && rc == MH3_OK) rc = cuda_fail(e, "freeing the status word");
  }
  delete h;
  return rc;
}

int mh3_preattn_validate(int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
                         const mh3_bf16* adaln_scale, int64_t scale_row_stride,
                         const mh3_bf16* adaln_shift, int64_t shift_row_stride, int64_t rows,
                         const int64_t* adaln_index, const mh3_bf16* qkv_weight,
                         const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
                         const mh3_bf16* rope_cos_sin, int64_t S, const int64_t* rope_positions,
                         int P, float eps, float qk_eps, const mh3_bf16* workspace,
                         const mh3_bf16* out) {
  int rc = check_norm_adaln_args(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                                 shift_row_stride, rows, adaln_index, eps, workspace, false);
  if (rc) return rc;
  if (!qk_eps_means_default(qk_eps) && !valid_eps(qk_eps))
    return fail(MH3_ERR_INVALID_ARG, "qk_eps must be finite and > 0 (or negative/NaN for eps)");
  return check_qkv_args(M, qkv_weight, q_norm_weight, k_norm_weight, rope_cos_sin, S,
                        rope_positions, P, out);
}

int mh3_preattn_run(mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* x,
                    const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                    int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                    int64_t shift_row_stride, int64_t rows, const int64_t* adaln_index,
                    const mh3_bf16* qkv_weight, const mh3_bf16* q_norm_weight,
                    const mh3_bf16* k_norm_weight, const mh3_bf16* rope_cos_sin, int64_t S,
                    const int64_t* rope_positions, int P, float eps, float qk_eps,
                    mh3_bf16* workspace, mh3_bf16* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = mh3_preattn_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                            shift_row_stride, rows, adaln_index, qkv_weight, q_norm_weight,
                            k_norm_weight, rope_cos_sin, S, rope_positions, P, eps, qk_eps,
                            workspace, out);
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float qk = qk_eps_means_default(qk_eps) ? eps : qk_eps;
  if (workspace == nullptr) {
    const size_t need = mh3_preattn_workspace_bytes(M);
    if (h->ws_bytes < need) {
      if (h->ws) {
        cudaError_t e = cudaFreeAsync(h->ws, s);
        h->ws = nullptr;
        h->ws_bytes = 0;
        if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync (workspace)");
      }
      cudaError_t e = cudaMallocAsync(&h->ws, need, s);
      if (e != cudaSuccess) {
        h->ws = nullptr;
        return fail(MH3_ERR_OOM, "cudaMallocAsync of %zu B workspace failed: %s", need,
                    cudaGetErrorString(e));
      }
      h->ws_bytes = need;
    }
    workspace = static_cast<mh3_bf16*>(h->ws);
  }
  // kernel 1 clears the split tail's flags (kernel 2 reads them only after
  // kernel 1 has completed)
  const SplitScratch sk{&h->sk_buf, &h->sk_bytes};
  const int split = split_tiles(M, h->max_clusters);
  if (split > 0 && (rc = prepare_split(sk, split, s, false))) return rc;
  rc = launch_stage1(s, h->num_sms, h->d_status, M, x, x_norm_weight, adaln_scale,
                     scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index, eps,
                     workspace, split > 0 ? static_cast<int*>(h->sk_buf) : nullptr,
                     split > 0 ? static_cast<int>(kSplitFlagBytes / sizeof(int)) : 0);
  if (rc) return rc;
  return launch_stage2(s, h->num_sms, h->max_clusters, h->d_status, M, workspace, qkv_weight,
                       q_norm_weight, k_norm_weight, rope_cos_sin, S, rope_positions, P, qk, out,
                       &h->test_stall_next, &sk, true);
}

int mh3_preattn_norm_adaln(mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* x,
                           const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                           int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                           int64_t shift_row_stride, int64_t rows, const int64_t* adaln_index,
                           float eps, mh3_bf16* workspace) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = check_norm_adaln_args(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                             shift_row_stride, rows, adaln_index, eps, workspace, true);
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  return launch_stage1(static_cast<cudaStream_t>(stream), h->num_sms, h->d_status, M, x,
                       x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                       shift_row_stride, rows, adaln_index, eps, workspace);
}

int mh3_preattn_qkv(mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* workspace,
                    const mh3_bf16* qkv_weight, const mh3_bf16* q_norm_weight,
                    const mh3_bf16* k_norm_weight, const mh3_bf16* rope_cos_sin, int64_t S,
                    const int64_t* rope_positions, int P, float qk_eps, mh3_bf16* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  if (!valid_eps(qk_eps)) return fail(MH3_ERR_INVALID_ARG, "qk_eps must be finite and > 0");
  rc = check_qkv_args(M, qkv_weight, q_norm_weight, k_norm_weight, rope_cos_sin, S,
                      rope_positions, P, out);
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_ptr(workspace, "workspace", 16))) return rc;
  const SplitScratch sk{&h->sk_buf, &h->sk_bytes};
  const int split = split_tiles(M, h->max_clusters);
  if (split > 0 && (rc = prepare_split(sk, split, static_cast<cudaStream_t>(stream), true)))
    return rc;
  return launch_stage2(static_cast<cudaStream_t>(stream), h->num_sms, h->max_clusters,
                       h->d_status, M, workspace, qkv_weight, q_norm_weight, k_norm_weight,
                       rope_cos_sin, S, rope_positions, P, qk_eps, out, &h->test_stall_next, &sk);
}

int mh3_preattn_set_test_stall(mh3_preattn_t h, int stall) {
  int rc = check_handle(h);
  if (rc) return rc;
  h->test_stall_next = stall != 0 ? 1 : 0;
  return MH3_OK;
}

int mh3_preattn_device_status(mh3_preattn_t h, void* stream, int* device_code) {
  if (h == nullptr || device_code == nullptr)
    return fail(MH3_ERR_INVALID_ARG, "handle or device_code is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, h->d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (v != 0) {
    e = cudaMemset(h->d_status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  }
  *device_code = v;
  return MH3_OK;
}

}  // extern "C"

// --------------------------------------------- attention output projection
namespace {

// The output projection's arguments other than the weight (BF16 and NVFP4).
int check_out_proj_args(int64_t M, const mh3_bf16* attn_out, const mh3_bf16* gate,
                        int64_t gate_row_stride, int64_t gate_rows, const int32_t* gate_index,
                        const mh3_bf16* residual, const mh3_bf16* out) {
  int rc;
  if ((rc = check_M(M))) return rc;
  if (gate_rows < 1)
    return fail(MH3_ERR_INVALID_ARG, "gate_rows must be >= 1 (got %lld)", (long long)gate_rows);
  if (gate_row_stride < kHidden)
    return fail(MH3_ERR_INVALID_ARG, "gate_row_stride must be >= 5376 (got %lld)",
                (long long)gate_row_stride);
  if (gate_row_stride % 8 != 0)
    return fail(MH3_ERR_ALIGNMENT, "gate_row_stride must be a multiple of 8 elements (got %lld)",
                (long long)gate_row_stride);
  if ((rc = check_ptr(gate, "gate", 16))) return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_ptr(attn_out, "attn_out", 16))) return rc;
  if ((rc = check_ptr(gate_index, "gate_index", 4))) return rc;
  if ((rc = check_ptr(residual, "residual", 16))) return rc;
  if ((rc = check_ptr(out, "out", 16))) return rc;
  const uintptr_t ro = reinterpret_cast<uintptr_t>(residual), oo = reinterpret_cast<uintptr_t>(out);
  const uintptr_t bytes = static_cast<uintptr_t>(M) * kHidden * 2;
  if (ro != oo && ro < oo + bytes && oo < ro + bytes)
    return fail(MH3_ERR_INVALID_ARG, "out may equal residual but must not partially overlap it");
  return MH3_OK;
}

}  // namespace

extern "C" int mh3_out_proj_validate(int64_t M, const mh3_bf16* attn_out, const mh3_bf16* o_weight,
                                     const mh3_bf16* gate, int64_t gate_row_stride,
                                     int64_t gate_rows, const int32_t* gate_index,
                                     const mh3_bf16* residual, const mh3_bf16* out) {
  int rc;
  if ((rc = check_ptr(o_weight, "o_weight", 16))) return rc;
  return check_out_proj_args(M, attn_out, gate, gate_row_stride, gate_rows, gate_index, residual,
                             out);
}

extern "C" int mh3_out_proj_run(mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* attn_out,
                                const mh3_bf16* o_weight, const mh3_bf16* gate,
                                int64_t gate_row_stride, int64_t gate_rows,
                                const int32_t* gate_index, const mh3_bf16* residual,
                                mh3_bf16* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = mh3_out_proj_validate(M, attn_out, o_weight, gate, gate_row_stride, gate_rows, gate_index,
                             residual, out);
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  if (h->out_proj_clusters <= 0)
    return fail(MH3_ERR_UNSUPPORTED, "no 2-CTA cluster of the output projection fits this device");
  OutProjMaps maps;
  if ((rc = encode_2d(&maps.a, attn_out, kAttnWidth, M, 64, 128, "attn_out"))) return rc;
  if ((rc = encode_2d(&maps.b, o_weight, kAttnWidth, kHidden, 64, 128, "o_weight"))) return rc;
  if ((rc = encode_2d(&maps.out, out, kHidden, M, 64, 32, "out"))) return rc;
  if ((rc = encode_2d(&maps.residual, residual, kHidden, M, 64, 32, "residual"))) return rc;
  OutProjParams p;
  p.gate = reinterpret_cast<const __nv_bfloat16*>(gate);
  p.gate_stride = gate_row_stride;
  p.gate_rows = gate_rows;
  p.gate_index = gate_index;
  p.M = M;
  p.status = h->d_status;
  p.num_m_tiles = static_cast<int>((M + 255) / 256);
  p.num_tiles = p.num_m_tiles * (kHidden / 256);
  const int clusters = p.num_tiles < h->out_proj_clusters ? p.num_tiles : h->out_proj_clusters;
  cudaError_t e = launch_out_proj(maps, p, clusters, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "output projection launch");
  return MH3_OK;
}

// ------------------------------------------------------- e4m3 output mode
extern "C" size_t mh3_preattn_out_e4m3_bytes(int64_t M) {
  return M <= 0 ? 0 : static_cast<size_t>(M) * kQkvRows;
}

// ------------------------------------------------------------ NVFP4 stage
namespace {

constexpr int kFp4KSteps = kHidden / 64;  // 84 scale words per token

int encode_tiled(CUtensorMap* map, CUtensorMapDataType type, uint32_t rank, const void* base,
                 const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                 CUtensorMapSwizzle swz, const char* what) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return fail(MH3_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  const cuuint32_t unit[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, type, rank, const_cast<void*>(base), dims, strides, box, unit,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MH3_ERR_CUDA, "tensor map (%s) failed: %d", what, (int)r);
  return MH3_OK;
}

// out[P, M, 56/P, 3, 128] as (d, slot, m, dst): bf16 (two 64-column boxes
// per head) or e4m3 bytes (one 128-byte box).
int encode_out_map(CUtensorMap* map, void* out, int64_t M, int P, bool e4m3) {
  const int64_t slots = 3 * (kHeads / P);
  const cuuint64_t es = e4m3 ? 1 : 2;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(slots),
                              static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(P)};
  const cuuint64_t strides[3] = {kHeadDim * es, static_cast<cuuint64_t>(slots) * kHeadDim * es,
                                 static_cast<cuuint64_t>(M) * slots * kHeadDim * es};
  const cuuint32_t box[4] = {e4m3 ? 128u : 64u, 1, 32, 1};
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return fail(MH3_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  const cuuint32_t unit[4] = {1, 1, 1, 1};
  CUresult r = enc(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   out, dims, strides, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MH3_ERR_CUDA, "tensor map (out) failed: %d", (int)r);
  return MH3_OK;
}

int check_fp4_stage1(int64_t M, const mh3_bf16* x, const mh3_bf16* xw, const mh3_bf16* sc,
                     int64_t sc_stride, const mh3_bf16* sh, int64_t sh_stride, int64_t rows,
                     const int32_t* idx, float eps, const float* act_gs) {
  int rc = check_norm_adaln_args(M, x, xw, sc, sc_stride, sh, sh_stride, rows, idx, eps, nullptr,
                                 false, 4);
  if (rc) return rc;
  if (M > 0 && (rc = check_ptr(act_gs, "act_global_scale", 4))) return rc;
  return MH3_OK;
}

int launch_fp4_stage1(cudaStream_t s, int num_sms, int* status, int64_t M, const mh3_bf16* x,
                      const mh3_bf16* xw, const mh3_bf16* sc, int64_t sc_stride,
                      const mh3_bf16* sh, int64_t sh_stride, int64_t rows, const int32_t* idx,
                      float eps, const float* act_gs, uint8_t* act_q, uint8_t* act_sf,
                      bool tiled) {
  NormAdalnParams p;
  p.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p.x_norm_weight = reinterpret_cast<const __nv_bfloat16*>(xw);
  p.scale = reinterpret_cast<const __nv_bfloat16*>(sc);
  p.shift = reinterpret_cast<const __nv_bfloat16*>(sh);
  p.scale_stride = sc_stride;
  p.shift_stride = sh_stride;
  p.rows = rows;
  p.index = nullptr;
  p.workspace = nullptr;
  p.M = M;
  p.eps = eps;
  p.status = status;
  p.index32 = idx;
  p.act_q = act_q;
  p.act_sf = act_sf;
  p.act_gs = act_gs;
  p.sf_tiled = tiled ? 1 : 0;
  cudaError_t e = launch_norm_adaln(p, num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 norm/AdaLN/quantisation launch");
  return MH3_OK;
}

// Kernel 2 of the NVFP4 stage on filled act_q / act_sf (tiled) buffers.
// The NVFP4 GEMM's arguments checked for any M: P, alpha (or the weight
// global scale it is derived from), the quantised weight and the norm
// weights.  *alpha_given reports whether alpha is used as given.
int check_fp4_gemm_fixed(int P, float alpha, float weight_global_scale, const uint8_t* weight_q,
                         const uint8_t* weight_sf, const mh3_bf16* q_norm_weight,
                         const mh3_bf16* k_norm_weight, bool* alpha_given) {
  if (!(P == 1 || P == 2 || P == 4 || P == 8))
    return fail(MH3_ERR_INVALID_ARG, "P (ulysses_degree) must be 1, 2, 4 or 8 (got %d)", P);
  *alpha_given = std::isfinite(alpha) && alpha > 0.0f;
  if (!*alpha_given && !(std::isfinite(weight_global_scale) && weight_global_scale > 0.0f))
    return fail(MH3_ERR_INVALID_ARG,
                "without alpha, weight_global_scale must be finite and > 0 (alpha is derived)");
  int rc;
  if ((rc = check_ptr(weight_q, "qkv_weight_q", 16))) return rc;
  if ((rc = check_ptr(weight_sf, "qkv_weight_sf", 16))) return rc;
  if ((rc = check_ptr(q_norm_weight, "q_norm_weight", 2))) return rc;
  if ((rc = check_ptr(k_norm_weight, "k_norm_weight", 2))) return rc;
  return MH3_OK;
}

// The NVFP4 GEMM's per-token arguments, checked when M > 0.
int check_fp4_gemm_rows(const mh3_bf16* rope_cos_sin, const void* out, const float* qkv_descale) {
  int rc;
  if ((rc = check_ptr(rope_cos_sin, "rope_cos_sin", 16))) return rc;
  if ((rc = check_ptr(out, "out", 16))) return rc;
  if (qkv_descale != nullptr && (rc = check_ptr(qkv_descale, "qkv_descale", 4))) return rc;
  return MH3_OK;
}

int launch_fp4_gemm(mh3_preattn_ctx* h, cudaStream_t s, int64_t M, const uint8_t* act_q,
                    const uint8_t* act_sf, const uint8_t* weight_q, const uint8_t* weight_sf,
                    float weight_global_scale, const float* act_global_scale, float alpha,
                    bool alpha_given, const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
                    const mh3_bf16* rope_cos_sin, int P, float eps, const float* qkv_descale,
                    void* out, const float* out_gs = nullptr, uint8_t* out_sf = nullptr) {
  // NVFP4 outputs when out_gs is given (out: the codes), else e4m3 when
  // qkv_descale is, else bf16
  const int mode = out_gs != nullptr ? kOutNvfp4 : (qkv_descale != nullptr ? kOutE4m3 : kOutBf16);
  const bool e4m3 = mode == kOutE4m3;
  const int max_clusters = mode == kOutNvfp4 ? h->nvfp4_fp4out_clusters
                           : e4m3            ? h->nvfp4_e4m3_clusters
                                             : h->nvfp4_clusters;
  if (max_clusters <= 0)
    return fail(MH3_ERR_UNSUPPORTED, "no 2-CTA cluster of the NVFP4 GEMM fits this device");
  int rc;
  Nvfp4Maps maps;
  {
    const cuuint64_t dims[2] = {kHidden / 2, static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {kHidden / 2};
    const cuuint32_t box[2] = {128, 128};
    if ((rc = encode_tiled(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, act_q, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, "act_q")))
      return rc;
  }
  {
    const cuuint64_t dims[2] = {kHidden / 2, kQkvRows};
    const cuuint64_t strides[1] = {kHidden / 2};
    const cuuint32_t box[2] = {128, 128};  // 128 of a tile's 256 B rows per CTA
    if ((rc = encode_tiled(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, weight_q, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, "qkv_weight_q")))
      return rc;
  }
  {
    // tiled scales as u32: (128 words of an atom, 84 steps, row groups)
    const cuuint64_t groups_a = static_cast<cuuint64_t>((M + 127) / 128);
    const cuuint64_t dims_a[3] = {128, kFp4KSteps, groups_a};
    const cuuint64_t dims_b[3] = {128, kFp4KSteps, kQkvRows / 128};
    const cuuint64_t strides[2] = {512, 512 * kFp4KSteps};
    const cuuint32_t box_a[3] = {128, 4, 1};  // one k-block: 4 steps of one row group
    const cuuint32_t box_b[3] = {128, 4, 2};  // ... of the tile's two row groups
    if ((rc = encode_tiled(&maps.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, act_sf, dims_a, strides,
                           box_a, CU_TENSOR_MAP_SWIZZLE_NONE, "act_sf")))
      return rc;
    if ((rc = encode_tiled(&maps.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, weight_sf, dims_b,
                           strides, box_b, CU_TENSOR_MAP_SWIZZLE_NONE, "qkv_weight_sf")))
      return rc;
  }
  if (mode == kOutNvfp4) {
    // the codes as a 4-D byte map (d 64, slot, m, dst); the NVFP4 form
    // stores from registers and never issues a TMA store through it
    const int64_t slots = 3 * (kHeads / P);
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(slots), static_cast<cuuint64_t>(M),
                                static_cast<cuuint64_t>(P)};
    const cuuint64_t strides[3] = {64, static_cast<cuuint64_t>(slots) * 64,
                                   static_cast<cuuint64_t>(M) * slots * 64};
    const cuuint32_t box[4] = {64, 1, 32, 1};
    if ((rc = encode_tiled(&maps.out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, out, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_NONE, "out_codes")))
      return rc;
  } else if ((rc = encode_out_map(&maps.out, out, M, P, e4m3))) {
    return rc;
  }
  QkvParams p;
  p.out_gs = out_gs;
  p.out_codes = mode == kOutNvfp4 ? static_cast<uint8_t*>(out) : nullptr;
  p.out_sf = out_sf;
  p.positions = nullptr;  // one cos/sin row per token
  p.cos_sin = reinterpret_cast<const __nv_bfloat16*>(rope_cos_sin);
  p.q_norm_weight = reinterpret_cast<const __nv_bfloat16*>(q_norm_weight);
  p.k_norm_weight = reinterpret_cast<const __nv_bfloat16*>(k_norm_weight);
  p.M = M;
  p.S = M;
  p.heads_per_dst = kHeads / P;
  p.qk_eps = eps;
  p.status = h->d_status;
  p.descales = qkv_descale;
  p.num_m_tiles = static_cast<int>((M + 255) / 256);
  p.num_tiles = p.num_m_tiles * (kQkvRows / 256);  // 256 x 256 pair tiles
  p.alpha = alpha_given ? alpha : -1.0f;
  p.act_gs = act_global_scale;
  p.w_gs = weight_global_scale;
  p.test_stall = h->test_stall_next;  // test hook: consumed by this launch
  h->test_stall_next = 0;
  const int clusters = p.num_tiles < max_clusters ? p.num_tiles : max_clusters;
  cudaError_t e = launch_nvfp4_qkv(maps, p, clusters, mode, s);
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 GEMM launch");
  return MH3_OK;
}

}  // namespace

extern "C" size_t mh3_nvfp4_codes_bytes(int64_t rows, int64_t cols) {
  return rows <= 0 || cols <= 0 ? 0 : static_cast<size_t>(rows) * static_cast<size_t>(cols) / 2;
}

extern "C" size_t mh3_nvfp4_scales_bytes(int64_t rows, int64_t cols, int tiled) {
  if (rows <= 0 || cols <= 0) return 0;
  if (!tiled) return static_cast<size_t>(rows) * static_cast<size_t>(cols / 16);
  return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>(cols / 64) * 512;
}

extern "C" int mh3_nvfp4_quantize(void* stream, int64_t rows, int64_t cols, const mh3_bf16* values,
                                  const float* global_scale, uint8_t* codes, uint8_t* scales,
                                  int tiled) {
  if (rows < 0) return fail(MH3_ERR_INVALID_ARG, "rows must be >= 0 (got %lld)", (long long)rows);
  if (cols <= 0 || cols % 64 != 0 || cols > (int64_t(1) << 24))
    return fail(MH3_ERR_INVALID_ARG, "cols must be a positive multiple of 64 up to 2^24 (got %lld)",
                (long long)cols);
  if (rows > (int64_t(1) << 40) / cols)
    return fail(MH3_ERR_INVALID_ARG, "rows x cols too large");
  if (rows == 0) return MH3_OK;
  int rc;
  if ((rc = check_ptr(values, "values", 16))) return rc;
  if ((rc = check_ptr(global_scale, "global_scale", 4))) return rc;
  if ((rc = check_ptr(codes, "codes", 16))) return rc;
  if ((rc = check_ptr(scales, "scales", 4))) return rc;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  e = launch_nvfp4_quantize(reinterpret_cast<const __nv_bfloat16*>(values), rows,
                            static_cast<int>(cols), global_scale, codes, scales, tiled != 0, sms,
                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 quantiser launch");
  return MH3_OK;
}

extern "C" int mh3_nvfp4_norm_quant(mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* x,
                                    const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                                    int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                                    int64_t shift_row_stride, int64_t rows,
                                    const int32_t* adaln_index, float eps,
                                    const float* act_global_scale, uint8_t* act_q,
                                    uint8_t* act_sf, int tiled) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = check_fp4_stage1(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                        shift_row_stride, rows, adaln_index, eps, act_global_scale);
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_ptr(act_q, "act_q", 16))) return rc;
  if ((rc = check_ptr(act_sf, "act_sf", 4))) return rc;
  return launch_fp4_stage1(static_cast<cudaStream_t>(stream), h->num_sms, h->d_status, M, x,
                           x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                           shift_row_stride, rows, adaln_index, eps, act_global_scale, act_q,
                           act_sf, tiled != 0);
}

extern "C" int mh3_nvfp4_preattn_run(
    mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
    const mh3_bf16* adaln_scale, int64_t scale_row_stride, const mh3_bf16* adaln_shift,
    int64_t shift_row_stride, int64_t rows, const int32_t* adaln_index, const uint8_t* weight_q,
    const uint8_t* weight_sf, float weight_global_scale, const float* act_global_scale,
    float alpha, const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
    const mh3_bf16* rope_cos_sin, int P, float eps, const float* qkv_descale, uint8_t* act_q,
    uint8_t* act_sf, void* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = check_fp4_stage1(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                        shift_row_stride, rows, adaln_index, eps, act_global_scale);
  if (rc) return rc;
  bool alpha_given = false;
  if ((rc = check_fp4_gemm_fixed(P, alpha, weight_global_scale, weight_q, weight_sf, q_norm_weight,
                                 k_norm_weight, &alpha_given)))
    return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_fp4_gemm_rows(rope_cos_sin, out, qkv_descale))) return rc;
  if (act_q != nullptr && (rc = check_ptr(act_q, "act_q", 16))) return rc;
  if (act_sf != nullptr && (rc = check_ptr(act_sf, "act_sf", 16))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (act_q == nullptr) {
    if ((rc = grow_buffer(&h->act_q, &h->act_q_bytes, mh3_nvfp4_codes_bytes(M, kHidden), s)))
      return rc;
    act_q = static_cast<uint8_t*>(h->act_q);
  }
  if (act_sf == nullptr) {
    if ((rc = grow_buffer(&h->act_sf, &h->act_sf_bytes, mh3_nvfp4_scales_bytes(M, kHidden, 1), s)))
      return rc;
    act_sf = static_cast<uint8_t*>(h->act_sf);
  }
  rc = launch_fp4_stage1(s, h->num_sms, h->d_status, M, x, x_norm_weight, adaln_scale,
                         scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index, eps,
                         act_global_scale, act_q, act_sf, true);
  if (rc) return rc;
  return launch_fp4_gemm(h, s, M, act_q, act_sf, weight_q, weight_sf, weight_global_scale,
                         act_global_scale, alpha, alpha_given, q_norm_weight, k_norm_weight,
                         rope_cos_sin, P, eps, qkv_descale, out);
}

extern "C" size_t mh3_preattn_out_nvfp4_bytes(int64_t M, int which) {
  if (M <= 0) return 0;
  const size_t rows = static_cast<size_t>(M) * kHeads * 3;  // (token, head, kind) rows of 128
  if (which == 0) return rows * (kHeadDim / 2);
  if (which == 1) return rows * (kHeadDim / 16);
  return 0;
}

extern "C" int mh3_nvfp4_preattn_run_nvfp4_out(
    mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
    const mh3_bf16* adaln_scale, int64_t scale_row_stride, const mh3_bf16* adaln_shift,
    int64_t shift_row_stride, int64_t rows, const int32_t* adaln_index, const uint8_t* weight_q,
    const uint8_t* weight_sf, float weight_global_scale, const float* act_global_scale,
    float alpha, const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
    const mh3_bf16* rope_cos_sin, int P, float eps, const float* qkv_global_scale,
    uint8_t* act_q, uint8_t* act_sf, uint8_t* out_codes, uint8_t* out_sf) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = check_fp4_stage1(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                        shift_row_stride, rows, adaln_index, eps, act_global_scale);
  if (rc) return rc;
  bool alpha_given = false;
  if ((rc = check_fp4_gemm_fixed(P, alpha, weight_global_scale, weight_q, weight_sf, q_norm_weight,
                                 k_norm_weight, &alpha_given)))
    return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_fp4_gemm_rows(rope_cos_sin, out_codes, nullptr))) return rc;
  if ((rc = check_ptr(qkv_global_scale, "qkv_global_scale", 4))) return rc;
  if ((rc = check_ptr(out_sf, "out_sf", 8))) return rc;
  if (act_q != nullptr && (rc = check_ptr(act_q, "act_q", 16))) return rc;
  if (act_sf != nullptr && (rc = check_ptr(act_sf, "act_sf", 16))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (act_q == nullptr) {
    if ((rc = grow_buffer(&h->act_q, &h->act_q_bytes, mh3_nvfp4_codes_bytes(M, kHidden), s)))
      return rc;
    act_q = static_cast<uint8_t*>(h->act_q);
  }
  if (act_sf == nullptr) {
    if ((rc = grow_buffer(&h->act_sf, &h->act_sf_bytes, mh3_nvfp4_scales_bytes(M, kHidden, 1), s)))
      return rc;
    act_sf = static_cast<uint8_t*>(h->act_sf);
  }
  rc = launch_fp4_stage1(s, h->num_sms, h->d_status, M, x, x_norm_weight, adaln_scale,
                         scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index, eps,
                         act_global_scale, act_q, act_sf, true);
  if (rc) return rc;
  return launch_fp4_gemm(h, s, M, act_q, act_sf, weight_q, weight_sf, weight_global_scale,
                         act_global_scale, alpha, alpha_given, q_norm_weight, k_norm_weight,
                         rope_cos_sin, P, eps, nullptr, out_codes, qkv_global_scale, out_sf);
}

extern "C" int mh3_nvfp4_qkv(mh3_preattn_t h, void* stream, int64_t M, const uint8_t* act_q,
                             const uint8_t* act_sf, const uint8_t* weight_q,
                             const uint8_t* weight_sf, float weight_global_scale,
                             const float* act_global_scale, float alpha,
                             const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
                             const mh3_bf16* rope_cos_sin, int P, float eps,
                             const float* qkv_descale, void* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  if ((rc = check_M(M))) return rc;
  if (!valid_eps(eps)) return fail(MH3_ERR_INVALID_ARG, "eps must be finite and > 0");
  bool alpha_given = false;
  if ((rc = check_fp4_gemm_fixed(P, alpha, weight_global_scale, weight_q, weight_sf, q_norm_weight,
                                 k_norm_weight, &alpha_given)))
    return rc;
  if (M == 0) return MH3_OK;
  if (!alpha_given && (rc = check_ptr(act_global_scale, "act_global_scale", 4))) return rc;
  if ((rc = check_ptr(act_q, "act_q", 16))) return rc;
  if ((rc = check_ptr(act_sf, "act_sf", 16))) return rc;
  if ((rc = check_fp4_gemm_rows(rope_cos_sin, out, qkv_descale))) return rc;
  return launch_fp4_gemm(h, static_cast<cudaStream_t>(stream), M, act_q, act_sf, weight_q,
                         weight_sf, weight_global_scale, act_global_scale, alpha, alpha_given,
                         q_norm_weight, k_norm_weight, rope_cos_sin, P, eps, qkv_descale, out);
}

// ---------------------------------------- NVFP4 (W4A4) output projection
namespace {

constexpr int kOutKSteps = kAttnWidth / 64;  // 112 scale words per token

int check_fp4_out_proj(int64_t M, const mh3_bf16* attn_out, const uint8_t* w_q,
                       const uint8_t* w_sf, float w_gs, const float* act_gs,
                       const mh3_bf16* gate, int64_t gate_row_stride, int64_t gate_rows,
                       const int32_t* gate_index, const mh3_bf16* residual, const mh3_bf16* out) {
  int rc;
  if (!(std::isfinite(w_gs) && w_gs > 0.0f))
    return fail(MH3_ERR_INVALID_ARG, "o_weight_global_scale must be finite and > 0");
  if ((rc = check_ptr(w_q, "o_weight_q", 16))) return rc;
  if ((rc = check_ptr(w_sf, "o_weight_sf", 16))) return rc;
  if ((rc = check_out_proj_args(M, attn_out, gate, gate_row_stride, gate_rows, gate_index,
                                residual, out)))
    return rc;
  if (M > 0 && (rc = check_ptr(act_gs, "act_global_scale", 4))) return rc;
  return MH3_OK;
}

}  // namespace

extern "C" int mh3_nvfp4_out_proj_validate(int64_t M, const mh3_bf16* attn_out,
                                           const uint8_t* o_weight_q, const uint8_t* o_weight_sf,
                                           float o_weight_global_scale,
                                           const float* act_global_scale, const mh3_bf16* gate,
                                           int64_t gate_row_stride, int64_t gate_rows,
                                           const int32_t* gate_index, const mh3_bf16* residual,
                                           const mh3_bf16* out) {
  return check_fp4_out_proj(M, attn_out, o_weight_q, o_weight_sf, o_weight_global_scale,
                            act_global_scale, gate, gate_row_stride, gate_rows, gate_index,
                            residual, out);
}

extern "C" int mh3_nvfp4_out_proj_run(mh3_preattn_t h, void* stream, int64_t M,
                                      const mh3_bf16* attn_out, const uint8_t* o_weight_q,
                                      const uint8_t* o_weight_sf, float o_weight_global_scale,
                                      const float* act_global_scale, const mh3_bf16* gate,
                                      int64_t gate_row_stride, int64_t gate_rows,
                                      const int32_t* gate_index, const mh3_bf16* residual,
                                      uint8_t* act_q, uint8_t* act_sf, mh3_bf16* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  if ((rc = check_fp4_out_proj(M, attn_out, o_weight_q, o_weight_sf, o_weight_global_scale,
                               act_global_scale, gate, gate_row_stride, gate_rows, gate_index,
                               residual, out)))
    return rc;
  if (M == 0) return MH3_OK;
  if (act_q != nullptr && (rc = check_ptr(act_q, "act_q", 16))) return rc;
  if (act_sf != nullptr && (rc = check_ptr(act_sf, "act_sf", 16))) return rc;
  if (h->nvfp4_out_clusters <= 0)
    return fail(MH3_ERR_UNSUPPORTED, "no 2-CTA cluster of the NVFP4 output projection fits");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (act_q == nullptr) {
    if ((rc = grow_buffer(&h->act_q, &h->act_q_bytes, mh3_nvfp4_codes_bytes(M, kAttnWidth), s)))
      return rc;
    act_q = static_cast<uint8_t*>(h->act_q);
  }
  if (act_sf == nullptr) {
    if ((rc = grow_buffer(&h->act_sf, &h->act_sf_bytes,
                          mh3_nvfp4_scales_bytes(M, kAttnWidth, 1), s)))
      return rc;
    act_sf = static_cast<uint8_t*>(h->act_sf);
  }
  Nvfp4Maps maps;
  {
    const cuuint64_t dims[2] = {kAttnWidth / 2, static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {kAttnWidth / 2};
    const cuuint32_t box[2] = {128, 128};
    if ((rc = encode_tiled(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, act_q, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, "act_q")))
      return rc;
  }
  {
    const cuuint64_t dims[2] = {kAttnWidth / 2, kHidden};
    const cuuint64_t strides[1] = {kAttnWidth / 2};
    const cuuint32_t box[2] = {128, 128};
    if ((rc = encode_tiled(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, o_weight_q, dims, strides,
                           box, CU_TENSOR_MAP_SWIZZLE_128B, "o_weight_q")))
      return rc;
  }
  {
    const cuuint64_t groups_a = static_cast<cuuint64_t>((M + 127) / 128);
    const cuuint64_t dims_a[3] = {128, kOutKSteps, groups_a};
    const cuuint64_t dims_b[3] = {128, kOutKSteps, kHidden / 128};
    const cuuint64_t strides[2] = {512, 512 * kOutKSteps};
    const cuuint32_t box_a[3] = {128, 4, 1};
    const cuuint32_t box_b[3] = {128, 4, 2};
    if ((rc = encode_tiled(&maps.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, act_sf, dims_a, strides,
                           box_a, CU_TENSOR_MAP_SWIZZLE_NONE, "act_sf")))
      return rc;
    if ((rc = encode_tiled(&maps.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, o_weight_sf, dims_b,
                           strides, box_b, CU_TENSOR_MAP_SWIZZLE_NONE, "o_weight_sf")))
      return rc;
  }
  if ((rc = encode_2d(&maps.out, out, kHidden, M, 64, 32, "out"))) return rc;
  if ((rc = encode_2d(&maps.aux, residual, kHidden, M, 64, 32, "residual"))) return rc;
  // 1. the activation's block-16 quantisation with act_global_scale (tiled scales)
  cudaError_t e = launch_nvfp4_quantize(reinterpret_cast<const __nv_bfloat16*>(attn_out), M,
                                        kAttnWidth, act_global_scale, act_q, act_sf, true,
                                        h->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 activation quantiser launch");
  // 2. the block-scaled GEMM with the gated residual
  Nvfp4OutProjParams p;
  p.M = M;
  p.num_m_tiles = static_cast<int>((M + 255) / 256);
  p.num_tiles = p.num_m_tiles * (kHidden / 256);
  p.status = h->d_status;
  p.alpha = -1.0f;  // derived on the device: RN(1 / RN(act_gs * w_gs))
  p.act_gs = act_global_scale;
  p.w_gs = o_weight_global_scale;
  p.gate = reinterpret_cast<const __nv_bfloat16*>(gate);
  p.gate_stride = gate_row_stride;
  p.gate_rows = gate_rows;
  p.gate_index = gate_index;
  p.test_stall = 0;
  const int clusters =
      p.num_tiles < h->nvfp4_out_clusters ? p.num_tiles : h->nvfp4_out_clusters;
  e = launch_nvfp4_out_proj(maps, p, clusters, s);
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 output projection launch");
  return MH3_OK;
}

extern "C" int mh3_e4m3_quantize(void* stream, int64_t n, const mh3_bf16* values,
                                 const float* descale, uint8_t* codes) {
  if (n < 0) return fail(MH3_ERR_INVALID_ARG, "n must be >= 0 (got %lld)", (long long)n);
  if (n == 0) return MH3_OK;
  int rc;
  if ((rc = check_ptr(values, "values", 2))) return rc;
  if ((rc = check_ptr(descale, "descale", 4))) return rc;
  if ((rc = check_ptr(codes, "codes", 1))) return rc;
  const uintptr_t v0 = reinterpret_cast<uintptr_t>(values), c0 = reinterpret_cast<uintptr_t>(codes);
  const uintptr_t v1 = v0 + static_cast<uintptr_t>(n) * 2, c1 = c0 + static_cast<uintptr_t>(n);
  if (v0 < c1 && c0 < v1) return fail(MH3_ERR_INVALID_ARG, "codes overlaps values");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  e = launch_e4m3_quantize(reinterpret_cast<const __nv_bfloat16*>(values), descale, codes, n, sms,
                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "e4m3 quantiser launch");
  return MH3_OK;
}

extern "C" int mh3_preattn_run_e4m3(
    mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
    const mh3_bf16* adaln_scale, int64_t scale_row_stride, const mh3_bf16* adaln_shift,
    int64_t shift_row_stride, int64_t rows, const int64_t* adaln_index,
    const mh3_bf16* qkv_weight, const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
    const mh3_bf16* rope_cos_sin, int64_t S, const int64_t* rope_positions, int P, float eps,
    float qk_eps, const float* qkv_descale, mh3_bf16* workspace, uint8_t* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  // the bf16 rules, with `out` checked as a 16-byte aligned buffer
  rc = mh3_preattn_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                            shift_row_stride, rows, adaln_index, qkv_weight, q_norm_weight,
                            k_norm_weight, rope_cos_sin, S, rope_positions, P, eps, qk_eps,
                            workspace, reinterpret_cast<const mh3_bf16*>(out));
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_ptr(qkv_descale, "qkv_descale", 4))) return rc;
  if (h->e4m3_clusters <= 0)
    return fail(MH3_ERR_UNSUPPORTED, "no 2-CTA cluster of the e4m3 GEMM fits this device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (workspace == nullptr) {
    if ((rc = grow_buffer(&h->ws, &h->ws_bytes, mh3_preattn_workspace_bytes(M), s))) return rc;
    workspace = static_cast<mh3_bf16*>(h->ws);
  }
  // the same split tail as the bf16 stage (the same accumulators, so the
  // codes are those of the bf16 outputs); kernel 1 clears its flags
  const SplitScratch sk{&h->sk_buf, &h->sk_bytes};
  const int split = split_tiles(M, h->e4m3_clusters);
  if (split > 0 && (rc = prepare_split(sk, split, s, false))) return rc;
  rc = launch_stage1(s, h->num_sms, h->d_status, M, x, x_norm_weight, adaln_scale,
                     scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index, eps,
                     workspace, split > 0 ? static_cast<int*>(h->sk_buf) : nullptr,
                     split > 0 ? static_cast<int>(kSplitFlagBytes / sizeof(int)) : 0);
  if (rc) return rc;
  QkvMaps maps;
  if ((rc = encode_2d(&maps.a, workspace, kHidden, M, 64, 128, "workspace"))) return rc;
  if ((rc = encode_2d(&maps.b, qkv_weight, kHidden, kQkvRows, 64, 128, "qkv_weight"))) return rc;
  if ((rc = encode_out_map(&maps.out, out, M, P, true))) return rc;
  QkvParams p;
  p.positions = rope_positions;
  p.cos_sin = reinterpret_cast<const __nv_bfloat16*>(rope_cos_sin);
  p.q_norm_weight = reinterpret_cast<const __nv_bfloat16*>(q_norm_weight);
  p.k_norm_weight = reinterpret_cast<const __nv_bfloat16*>(k_norm_weight);
  p.M = M;
  p.S = S;
  p.heads_per_dst = kHeads / P;
  p.qk_eps = qk_eps_means_default(qk_eps) ? eps : qk_eps;
  p.status = h->d_status;
  p.descales = qkv_descale;
  p.num_m_tiles = static_cast<int>((M + 255) / 256);
  p.num_tiles = p.num_m_tiles * (kQkvRows / 256);
  const int clusters = p.num_tiles < h->e4m3_clusters ? p.num_tiles : h->e4m3_clusters;
  if (split > 0) {
    p.sk_dp = p.num_tiles - split;
    p.sk_tail = split;
    p.sk_flags = static_cast<int*>(h->sk_buf);
    p.sk_partial = reinterpret_cast<float*>(static_cast<uint8_t*>(h->sk_buf) + kSplitFlagBytes);
    p.sk_seq = 1;
  }
  p.b_early = 1;  // kernel 1 just launched on this stream writes A alone
  cudaError_t e = launch_qkv_e4m3(maps, p, clusters, s);
  if (e != cudaSuccess) return cuda_fail(e, "e4m3 QKV GEMM launch");
  return MH3_OK;
}

// ------------------------------------------------------------- MLP block
extern "C" size_t mh3_mlp_workspace_y_bytes(int64_t M) {
  return M <= 0 ? 0 : static_cast<size_t>(M) * kMlpInter * 2;
}

extern "C" int mh3_mlp_validate(int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
                                const mh3_bf16* adaln_scale, int64_t scale_row_stride,
                                const mh3_bf16* adaln_shift, int64_t shift_row_stride,
                                const mh3_bf16* gate, int64_t gate_row_stride, int64_t rows,
                                const int64_t* adaln_index, const mh3_bf16* residual,
                                const mh3_bf16* fc1_weight, const mh3_bf16* fc2_weight,
                                float eps, const mh3_bf16* workspace_a,
                                const mh3_bf16* workspace_y, const mh3_bf16* out) {
  int rc = check_norm_adaln_args(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                                 shift_row_stride, rows, adaln_index, eps, workspace_a, false);
  if (rc) return rc;
  if (gate_row_stride < kHidden)
    return fail(MH3_ERR_INVALID_ARG, "gate_row_stride must be >= 5376 (got %lld)",
                (long long)gate_row_stride);
  if (gate_row_stride % 8 != 0)
    return fail(MH3_ERR_ALIGNMENT, "gate_row_stride must be a multiple of 8 elements (got %lld)",
                (long long)gate_row_stride);
  if ((rc = check_ptr(gate, "gate", 16))) return rc;
  if ((rc = check_ptr(fc1_weight, "fc1_weight", 16))) return rc;
  if ((rc = check_ptr(fc2_weight, "fc2_weight", 16))) return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_ptr(residual, "residual", 16))) return rc;
  if ((rc = check_ptr(out, "out", 16))) return rc;
  if (workspace_y != nullptr && (rc = check_ptr(workspace_y, "workspace_y", 16))) return rc;
  const uintptr_t bytes = static_cast<uintptr_t>(M) * kHidden * 2;
  const uintptr_t oo = reinterpret_cast<uintptr_t>(out);
  const uintptr_t cands[2] = {reinterpret_cast<uintptr_t>(residual), reinterpret_cast<uintptr_t>(x)};
  for (uintptr_t c : cands)
    if (c != oo && c < oo + bytes && oo < c + bytes)
      return fail(MH3_ERR_INVALID_ARG, "out may equal residual or x but must not partially overlap them");
  return MH3_OK;
}

extern "C" int mh3_mlp_run(mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* x,
                           const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                           int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                           int64_t shift_row_stride, const mh3_bf16* gate,
                           int64_t gate_row_stride, int64_t rows, const int64_t* adaln_index,
                           const mh3_bf16* residual, const mh3_bf16* fc1_weight,
                           const mh3_bf16* fc2_weight, float eps, mh3_bf16* workspace_a,
                           mh3_bf16* workspace_y, mh3_bf16* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = mh3_mlp_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                        shift_row_stride, gate, gate_row_stride, rows, adaln_index, residual,
                        fc1_weight, fc2_weight, eps, workspace_a, workspace_y, out);
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  if (h->fc1_clusters <= 0 || h->fc2_clusters <= 0)
    return fail(MH3_ERR_UNSUPPORTED, "no 2-CTA cluster of the MLP GEMMs fits this device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (workspace_a == nullptr) {
    if ((rc = grow_buffer(&h->ws, &h->ws_bytes, mh3_preattn_workspace_bytes(M), s))) return rc;
    workspace_a = static_cast<mh3_bf16*>(h->ws);
  }
  if (workspace_y == nullptr) {
    if ((rc = grow_buffer(&h->ws_y, &h->ws_y_bytes, mh3_mlp_workspace_y_bytes(M), s))) return rc;
    workspace_y = static_cast<mh3_bf16*>(h->ws_y);
  }
  rc = launch_stage1(s, h->num_sms, h->d_status, M, x, x_norm_weight, adaln_scale,
                     scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index, eps,
                     workspace_a);
  if (rc) return rc;
  const int pairs = static_cast<int>((M + 255) / 256);
  CUtensorMap ma, mb, my;
  if ((rc = encode_2d(&ma, workspace_a, kHidden, M, 64, 128, "workspace_a"))) return rc;
  if ((rc = encode_2d(&mb, fc1_weight, kHidden, 2 * kMlpInter, 64, 128, "fc1_weight"))) return rc;
  if ((rc = encode_2d(&my, workspace_y, kMlpInter, M, 64, 32, "workspace_y (store)"))) return rc;
  SwigluParams p1;
  p1.M = M;
  p1.num_m_tiles = pairs;
  p1.num_tiles = pairs * (kMlpInter / 128);
  p1.status = h->d_status;
  cudaError_t e = launch_mlp_fc1(ma, mb, my, p1, p1.num_tiles < h->fc1_clusters ? p1.num_tiles
                                                                                 : h->fc1_clusters, s);
  if (e != cudaSuccess) return cuda_fail(e, "MLP fc1 launch");
  CUtensorMap ya, wb, mo, mr;
  if ((rc = encode_2d(&ya, workspace_y, kMlpInter, M, 64, 128, "workspace_y (load)"))) return rc;
  if ((rc = encode_2d(&wb, fc2_weight, kMlpInter, kHidden, 64, 128, "fc2_weight"))) return rc;
  if ((rc = encode_2d(&mo, out, kHidden, M, 64, 32, "out"))) return rc;
  if ((rc = encode_2d(&mr, residual, kHidden, M, 64, 32, "residual"))) return rc;
  GatedResidualParams<int64_t> p2;
  p2.gate = reinterpret_cast<const __nv_bfloat16*>(gate);
  p2.gate_stride = gate_row_stride;
  p2.gate_rows = rows;
  p2.gate_index = adaln_index;
  p2.M = M;
  p2.num_m_tiles = pairs;
  p2.num_tiles = pairs * (kHidden / 256);
  p2.status = h->d_status;
  e = launch_mlp_fc2(ya, wb, mo, mr, p2, p2.num_tiles < h->fc2_clusters ? p2.num_tiles
                                                                         : h->fc2_clusters, s);
  if (e != cudaSuccess) return cuda_fail(e, "MLP fc2 launch");
  return MH3_OK;
}

// ----------------------------------------------------------- FP8 MLP block
extern "C" size_t mh3_mlp_fp8_workspace_bytes(int64_t M, int which) {
  if (M <= 0) return 0;
  switch (which) {
    case 0: return static_cast<size_t>(M) * kHidden;        // a_q, E4M3 [M, 5376]
    case 1: return static_cast<size_t>(M) * 4;              // a scale, FP32 [M]
    case 2: return static_cast<size_t>(M) * kMlpInter * 2;  // y, bf16 [M, 14336]
    case 3: return static_cast<size_t>(M) * kMlpInter;      // y_q, E4M3 [M, 14336]
    case 4: return static_cast<size_t>(M) * 4;              // y scale, FP32 [M]
    default: return 0;
  }
}

extern "C" int mh3_mlp_fp8_validate(
    int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
    int64_t scale_row_stride, const mh3_bf16* adaln_shift, int64_t shift_row_stride,
    const mh3_bf16* gate, int64_t gate_row_stride, int64_t rows, const int64_t* adaln_index,
    const mh3_bf16* residual, const uint8_t* fc1_weight_q, const float* fc1_weight_scale,
    const uint8_t* fc2_weight_q, const float* fc2_weight_scale, float eps,
    const uint8_t* workspace_a_q, const float* workspace_a_scale, const mh3_bf16* workspace_y,
    const uint8_t* workspace_y_q, const float* workspace_y_scale, const mh3_bf16* out) {
  int rc = mh3_mlp_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                            shift_row_stride, gate, gate_row_stride, rows, adaln_index, residual,
                            reinterpret_cast<const mh3_bf16*>(fc1_weight_q),
                            reinterpret_cast<const mh3_bf16*>(fc2_weight_q), eps, nullptr,
                            workspace_y, out);
  if (rc) return rc;
  if ((rc = check_ptr(fc1_weight_scale, "fc1_weight_scale", 16))) return rc;
  if ((rc = check_ptr(fc2_weight_scale, "fc2_weight_scale", 16))) return rc;
  if (M == 0) return MH3_OK;
  const void* ws[4] = {workspace_a_q, workspace_a_scale, workspace_y_q, workspace_y_scale};
  const char* names[4] = {"workspace_a_q", "workspace_a_scale", "workspace_y_q",
                          "workspace_y_scale"};
  for (int i = 0; i < 4; ++i)
    if (ws[i] != nullptr && (rc = check_ptr(ws[i], names[i], 16))) return rc;
  return MH3_OK;
}

extern "C" int mh3_mlp_fp8_run(
    mh3_preattn_t h, void* stream, int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
    const mh3_bf16* adaln_scale, int64_t scale_row_stride, const mh3_bf16* adaln_shift,
    int64_t shift_row_stride, const mh3_bf16* gate, int64_t gate_row_stride, int64_t rows,
    const int64_t* adaln_index, const mh3_bf16* residual, const uint8_t* fc1_weight_q,
    const float* fc1_weight_scale, const uint8_t* fc2_weight_q, const float* fc2_weight_scale,
    float eps, uint8_t* workspace_a_q, float* workspace_a_scale, mh3_bf16* workspace_y,
    uint8_t* workspace_y_q, float* workspace_y_scale, mh3_bf16* out) {
  int rc = check_handle(h);
  if (rc) return rc;
  rc = mh3_mlp_fp8_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                            shift_row_stride, gate, gate_row_stride, rows, adaln_index, residual,
                            fc1_weight_q, fc1_weight_scale, fc2_weight_q, fc2_weight_scale, eps,
                            workspace_a_q, workspace_a_scale, workspace_y, workspace_y_q,
                            workspace_y_scale, out);
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  if (h->fc1_fp8_clusters <= 0 || h->fc2_fp8_clusters <= 0)
    return fail(MH3_ERR_UNSUPPORTED, "no 2-CTA cluster of the FP8 MLP GEMMs fits this device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  struct Own {
    void** ptr;
    void** buf;
    size_t* cap;
    int which;
  } own[5] = {{reinterpret_cast<void**>(&workspace_a_q), &h->fp8_aq, &h->fp8_aq_bytes, 0},
              {reinterpret_cast<void**>(&workspace_a_scale), &h->fp8_as, &h->fp8_as_bytes, 1},
              {reinterpret_cast<void**>(&workspace_y), &h->ws_y, &h->ws_y_bytes, 2},
              {reinterpret_cast<void**>(&workspace_y_q), &h->fp8_yq, &h->fp8_yq_bytes, 3},
              {reinterpret_cast<void**>(&workspace_y_scale), &h->fp8_ys, &h->fp8_ys_bytes, 4}};
  for (const Own& o : own) {
    if (*o.ptr != nullptr) continue;
    if ((rc = grow_buffer(o.buf, o.cap, mh3_mlp_fp8_workspace_bytes(M, o.which), s))) return rc;
    *o.ptr = *o.buf;
  }
  // the y scale buffer first collects each row's amax (FP32 bits, from 0);
  // zeroed before kernel 1 so that kernel 1 and fc1 stay adjacent launches
  cudaError_t e = cudaMemsetAsync(workspace_y_scale, 0, mh3_mlp_fp8_workspace_bytes(M, 4), s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (y amax)");
  // kernel 1, E4M3 form: a_q and s_a
  NormAdalnParams p1;
  p1.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p1.x_norm_weight = reinterpret_cast<const __nv_bfloat16*>(x_norm_weight);
  p1.scale = reinterpret_cast<const __nv_bfloat16*>(adaln_scale);
  p1.shift = reinterpret_cast<const __nv_bfloat16*>(adaln_shift);
  p1.scale_stride = scale_row_stride;
  p1.shift_stride = shift_row_stride;
  p1.rows = rows;
  p1.index = adaln_index;
  p1.workspace = nullptr;
  p1.M = M;
  p1.eps = eps;
  p1.status = h->d_status;
  p1.a_q8 = workspace_a_q;
  p1.a_s8 = workspace_a_scale;
  e = launch_norm_adaln(p1, h->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "norm/AdaLN (E4M3) launch");
  const int pairs = static_cast<int>((M + 255) / 256);
  CUtensorMap ma, mb, my;
  if ((rc = encode_u8_2d(&ma, workspace_a_q, kHidden, M, 128, 128, "workspace_a_q"))) return rc;
  if ((rc = encode_u8_2d(&mb, fc1_weight_q, kHidden, 2 * kMlpInter, 128, 128, "fc1_weight_q")))
    return rc;
  if ((rc = encode_2d(&my, workspace_y, kMlpInter, M, 64, 32, "workspace_y (store)"))) return rc;
  SwigluParams q1;
  q1.M = M;
  q1.num_m_tiles = pairs;
  q1.num_tiles = pairs * (kMlpInter / 128);
  q1.status = h->d_status;
  q1.row_scale = workspace_a_scale;
  q1.col_scale = fc1_weight_scale;
  q1.y_amax = reinterpret_cast<unsigned int*>(workspace_y_scale);
  e = launch_mlp_fp8_fc1(ma, mb, my, q1, q1.num_tiles < h->fc1_fp8_clusters ? q1.num_tiles
                                                                            : h->fc1_fp8_clusters,
                         s);
  if (e != cudaSuccess) return cuda_fail(e, "FP8 MLP fc1 launch");
  e = launch_mlp_quantize_y(reinterpret_cast<const __nv_bfloat16*>(workspace_y), M,
                            workspace_y_scale, workspace_y_q, h->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "y quantiser launch");
  CUtensorMap ya, wb, mo, mr;
  if ((rc = encode_u8_2d(&ya, workspace_y_q, kMlpInter, M, 128, 128, "workspace_y_q"))) return rc;
  if ((rc = encode_u8_2d(&wb, fc2_weight_q, kMlpInter, kHidden, 128, 128, "fc2_weight_q")))
    return rc;
  if ((rc = encode_2d(&mo, out, kHidden, M, 64, 32, "out"))) return rc;
  if ((rc = encode_2d(&mr, residual, kHidden, M, 64, 32, "residual"))) return rc;
  GatedResidualParams<int64_t> q2;
  q2.gate = reinterpret_cast<const __nv_bfloat16*>(gate);
  q2.gate_stride = gate_row_stride;
  q2.gate_rows = rows;
  q2.gate_index = adaln_index;
  q2.M = M;
  q2.num_m_tiles = pairs;
  q2.num_tiles = pairs * (kHidden / 256);
  q2.status = h->d_status;
  q2.row_scale = workspace_y_scale;
  q2.col_scale = fc2_weight_scale;
  e = launch_mlp_fp8_fc2(ya, wb, mo, mr, q2, q2.num_tiles < h->fc2_fp8_clusters
                                                  ? q2.num_tiles
                                                  : h->fc2_fp8_clusters,
                         s);
  if (e != cudaSuccess) return cuda_fail(e, "FP8 MLP fc2 launch");
  return MH3_OK;
}

// ------------------------------------------------------ no-allocation variant
// The whole stage for callers that cannot call cudaMalloc (for example code
// running where a custom allocator owns all device memory, or inside a
// process whose allocation calls are forbidden after start-up): the BF16
// workspace lives in the file-scope array below, which the CUDA module
// reserves when it loads, so the call itself allocates nothing.
namespace {

constexpr int64_t kNoAllocMaxM = 1024;  // 1024 x 5376 bf16 = 10.5 MiB per device
static __device__ __align__(256) mh3_bf16 g_noalloc_workspace[kNoAllocMaxM * kHidden];

constexpr int kNoAllocMaxDevices = 64;
struct NoAllocDevice {
  bool ready = false;             // set only after a set-up that succeeded
  mh3_bf16* workspace = nullptr;  // device address of g_noalloc_workspace
  int num_sms = 0;
  int max_clusters = 0;
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// Per device, with that device current, until it succeeds once: the device
// address of the array (the host-side name is only a stand-in), the same
// device checks as mh3_preattn_create (sm_103a, enough opt-in shared memory
// per block), the GEMMs' shared-memory limits, and the SM count.  A failed
// set-up is not remembered: the next call tries again.
int noalloc_setup(int dev, NoAllocDevice& d) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (d.ready) return MH3_OK;
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(MH3_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                dev, prop.major, prop.minor);
  if (static_cast<int>(prop.sharedMemPerBlockOptin) < qkv_smem_bytes())
    return fail(MH3_ERR_UNSUPPORTED, "device allows %zu B of shared memory per block, need %d",
                prop.sharedMemPerBlockOptin, qkv_smem_bytes());
  mh3_bf16* ws = nullptr;
  if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ws), g_noalloc_workspace)) !=
      cudaSuccess)
    return cuda_fail(e, "cudaGetSymbolAddress (static workspace)");
  if ((e = qkv_prepare_device()) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  int clusters = 0;
  if ((e = qkv_pair_prepare_device(&clusters)) != cudaSuccess)
    return cuda_fail(e, "preparing the pair GEMM");
  d.workspace = ws;
  d.max_clusters = clusters;
  d.num_sms = prop.multiProcessorCount;
  d.ready = true;
  return MH3_OK;
}

}  // namespace

extern "C" int mh3_preattn_run_noalloc(
    void* stream, int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
    const mh3_bf16* adaln_scale, int64_t scale_row_stride, const mh3_bf16* adaln_shift,
    int64_t shift_row_stride, int64_t rows, const int64_t* adaln_index,
    const mh3_bf16* qkv_weight, const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
    const mh3_bf16* rope_cos_sin, int64_t S, const int64_t* rope_positions, int P, float eps,
    float qk_eps, mh3_bf16* out, int* device_status) {
  if (M > kNoAllocMaxM)
    return fail(MH3_ERR_INVALID_ARG,
                "M=%lld exceeds the %lld tokens the static workspace of "
                "mh3_preattn_run_noalloc holds; use mh3_preattn_run",
                (long long)M, (long long)kNoAllocMaxM);
  int rc = mh3_preattn_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                                shift_row_stride, rows, adaln_index, qkv_weight, q_norm_weight,
                                k_norm_weight, rope_cos_sin, S, rope_positions, P, eps, qk_eps,
                                nullptr, out);
  if (rc) return rc;
  if (M == 0) return MH3_OK;
  if ((rc = check_ptr(device_status, "device_status", 4))) return rc;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(MH3_ERR_UNSUPPORTED, "device index %d out of range", dev);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if ((rc = noalloc_setup(dev, d))) return rc;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the timeout code must start at zero for this call
  e = cudaMemsetAsync(device_status, 0, sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (device_status)");
  rc = launch_stage1(s, d.num_sms, device_status, M, x, x_norm_weight, adaln_scale,
                     scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index, eps,
                     d.workspace);
  if (rc) return rc;
  return launch_stage2(s, d.num_sms, d.max_clusters, device_status, M, d.workspace, qkv_weight,
                       q_norm_weight, k_norm_weight, rope_cos_sin, S, rope_positions, P,
                       qk_eps_means_default(qk_eps) ? eps : qk_eps, out, nullptr, nullptr, true);
}
