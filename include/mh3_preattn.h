/*
 * mh3_preattn.h -- C ABI of the MiniMax-H3 BF16 pre-attention stage on GB300
 * (sm_103a).
 *
 * The operation is the one the page
 * "flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention" defines (summary
 * paragraph, Parameters and Notes), with the norm/AdaLN formulas of the
 * formula block of "flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120":
 *
 *   n  = bf16(rmsnorm(x, eps) * x_norm_weight)       FP32 sum of squares
 *   a  = bf16(shift[i] + n * bf16(1 + scale[i]))     i = adaln_index[m]
 *   a  = 0 for the whole row when i is outside [0, rows)
 *   y  = bf16(a @ qkv_weight^T)                      FP32 accumulation
 *   q,k: per-head (128) RMSNorm with qk_eps and q/k_norm_weight, then the
 *        split-half rotation of dims [0, 96) by cache row
 *        p = clamp(positions[m], 0, S-1) (or p = m), dims [96, 128) unchanged
 *   out[dst, m, hl, kind, d], dst = head / (56/P), hl = head % (56/P),
 *        kind 0 = q, 1 = k, 2 = v
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers into the current device's
 *     memory.  bf16 values are stored as 16-bit patterns (mh3_bf16).  The
 *     library never takes ownership of caller memory and never frees it.
 *   - Every call validates all arguments on the host before it launches
 *     anything; on a validation error nothing is launched and the status is
 *     returned.  mh3_preattn_last_error() gives a message for the calling
 *     thread's last failure.
 *   - Launches go on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream), in stream order, with no host synchronisation
 *     and no host<->device copies.
 *   - Index and position VALUES are never errors: an adaln_index outside
 *     [0, rows) zeroes its row and a position outside [0, S) is clamped, on
 *     the device (page Notes and Parameters: adaln_index, rope_positions).
 *   - The kernels bound every wait they make; a wait that runs out records a
 *     code in the handle's device status word instead of hanging.  Read it
 *     with mh3_preattn_device_status().
 *   - Sizes: hidden H = 5376, heads NH = 56, head_dim D = 128, qkv rows
 *     N = 3*NH*D = 21504, rotary dims 96.  These are fixed by the page.
 */
#ifndef MH3_PREATTN_H
#define MH3_PREATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MH3_HIDDEN 5376
#define MH3_NUM_HEADS 56
#define MH3_HEAD_DIM 128
#define MH3_QKV_ROWS 21504
#define MH3_ROPE_DIMS 96

typedef uint16_t mh3_bf16; /* storage of one bfloat16 value */

typedef enum mh3_status {
  MH3_OK = 0,
  MH3_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad P, bad eps, S < M with identity positions */
  MH3_ERR_ALIGNMENT = 2,   /* a base pointer or row stride breaks the 16-byte rule */
  MH3_ERR_UNSUPPORTED = 3, /* device is not sm_103 / lacks the shared memory the GEMM needs */
  MH3_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (message has the CUDA error) */
  MH3_ERR_OOM = 5,         /* the handle could not grow its own workspace */
  MH3_ERR_DEVICE = 6       /* a kernel recorded a bounded-wait timeout (mh3_preattn_device_status) */
} mh3_status;

typedef struct mh3_preattn_ctx* mh3_preattn_t;

/* Create a handle bound to CUDA device `device` (made current for the call).
 * Caches the SM count, raises the GEMM's shared-memory limit and allocates a
 * 4-byte device status word.  No per-M state.  *handle is set only on MH3_OK.
 * The handle's own device buffers (the status word, the workspace it grows
 * when a call passes none, and the split-tail scratch) serve every call made
 * through it: calls through one handle on streams that may overlap on the GPU
 * race on them, so give each concurrent stream its own handle. */
int mh3_preattn_create(mh3_preattn_t* handle, int device);

/* Destroy a handle: frees its status word and its own workspace (if any).
 * The caller must ensure no launch that uses the handle is still running. */
int mh3_preattn_destroy(mh3_preattn_t handle);

/* Bytes of the BF16 [M, 5376] workspace: M * 5376 * 2.  0 when M <= 0. */
size_t mh3_preattn_workspace_bytes(int64_t M);

/* Bytes of out, [P, M, 56/P, 3, 128] BF16: M * 21504 * 2 (independent of P). */
size_t mh3_preattn_out_bytes(int64_t M);

/* Host-only validation of a full argument set (no device access, no launch).
 * Same rules and status codes as mh3_preattn_run; pointers are checked for
 * NULL and alignment only, never dereferenced.  Arguments as in
 * mh3_preattn_run. */
int mh3_preattn_validate(int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
                         const mh3_bf16* adaln_scale, int64_t scale_row_stride,
                         const mh3_bf16* adaln_shift, int64_t shift_row_stride, int64_t rows,
                         const int64_t* adaln_index, const mh3_bf16* qkv_weight,
                         const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
                         const mh3_bf16* rope_cos_sin, int64_t S, const int64_t* rope_positions,
                         int P, float eps, float qk_eps, const mh3_bf16* workspace,
                         const mh3_bf16* out);

/* The whole stage: kernel 1 (RMSNorm + indexed AdaLN into the workspace) then
 * kernel 2 (persistent QKV GEMM with the Q/K norm, RoPE and pack epilogue),
 * two launches on `stream` (page summary: "two kernel launches on the current
 * stream").
 *
 * Split tail: when M > 128 and the GEMM's last wave of 256 x 256 tiles holds
 * at most half as many tiles as there are resident CTA pairs, each of those
 * tiles is computed by two pairs, one per half of K; the first adds its FP32
 * partial to the second's accumulator (one FP32 addition per element, fixed
 * order, deterministic) before the epilogue.  Those tiles' accumulators are
 * summed in another order than a whole tile's, so their outputs may differ
 * from mh3_preattn_run_noalloc's (which never splits) within the stage's
 * tolerance.  The partials live in a scratch of the handle, grown with
 * stream-ordered cudaMallocAsync the first time a split size needs more
 * (even with a caller workspace): capture a split size into a graph after
 * one direct call at that size.  Its flags are cleared on the stream before
 * each such call, by kernel 1 of the same call (so a graph replay clears them
 * too), and runs of one handle on different streams race on the scratch.
 *
 *   M                 tokens, >= 0 (M == 0 launches nothing and returns MH3_OK)
 *   x                 [M, 5376] row-major, 16-byte aligned
 *   x_norm_weight     [5376], 16-byte aligned
 *   adaln_scale/shift [rows, 5376] views: unit column stride, row strides
 *                     scale_row_stride / shift_row_stride in ELEMENTS,
 *                     each >= 5376 and a multiple of 8 (16 bytes), base
 *                     16-byte aligned.  Column chunks of a wider
 *                     [rows, k*5376] projection qualify as they are
 *                     (Parameters: adaln_scale).
 *   rows              >= 1
 *   adaln_index       [M] int64, 8-byte aligned; any value (guarded)
 *   qkv_weight        [21504, 5376] row-major, rows in the order
 *                     [qkv_kind, head, head_dim] (Parameters: qkv_weight)
 *   q/k_norm_weight   [128] each
 *   rope_cos_sin      [S, 96] row-major, S >= 1; columns [0,48) cos, [48,96) sin
 *   rope_positions    [M] int64 or NULL.  NULL means row m uses cache row m
 *                     and requires S >= M (Parameters: rope_positions); it
 *                     needs no allocation, so it is graph-safe from the
 *                     first call.
 *   P                 destinations (ulysses_degree), one of 1, 2, 4, 8
 *   eps               input RMSNorm epsilon, finite and > 0
 *   qk_eps            Q/K RMSNorm epsilon; a negative value or NaN means
 *                     "use eps" (Parameters: qk_eps, None uses eps);
 *                     otherwise finite and > 0
 *   workspace         [M, 5376] BF16 scratch (overwritten), 16-byte aligned,
 *                     or NULL: the handle then uses its own buffer, grown
 *                     with stream-ordered cudaMallocAsync on `stream` when M
 *                     exceeds its size (Parameters: workspace).  With NULL,
 *                     runs of one handle on different streams race on that
 *                     buffer.
 *   out               [P, M, 56/P, 3, 128] contiguous BF16, 16-byte aligned,
 *                     caller-owned (Parameters: out)
 */
int mh3_preattn_run(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* x,
                    const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                    int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                    int64_t shift_row_stride, int64_t rows, const int64_t* adaln_index,
                    const mh3_bf16* qkv_weight, const mh3_bf16* q_norm_weight,
                    const mh3_bf16* k_norm_weight, const mh3_bf16* rope_cos_sin, int64_t S,
                    const int64_t* rope_positions, int P, float eps, float qk_eps,
                    mh3_bf16* workspace, mh3_bf16* out);

/* The whole stage with e4m3 outputs (out_mode "e4m3" of the page
 * "flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention", Parameters:
 * out_mode, q_descale / k_descale / v_descale).  Every output value is the
 * bf16 value of mh3_preattn_run divided by its kind's dequantisation scale
 * in FP32 and rounded to nearest-even e4m3, saturated to +-448:
 *   code = e4m3(o / descale[kind]),  o ~ code * descale[kind].
 *   qkv_descale   DEVICE pointer to 3 floats (q, k, v), read on the device
 *                 (no host synchronisation), 4-byte aligned
 *   out           [P, M, 56/P, 3, 128] bytes (e4m3 codes), the bf16 mode's
 *                 pack, 16-byte aligned; M * 21504 bytes
 * Other arguments and rules as in mh3_preattn_run.  Kernel 2 always runs in
 * its CTA-pair form here, with mh3_preattn_run's split tail for M > 128 (the
 * same accumulators, so the codes are those of mh3_preattn_run's outputs). */
int mh3_preattn_run_e4m3(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* x,
                         const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                         int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                         int64_t shift_row_stride, int64_t rows, const int64_t* adaln_index,
                         const mh3_bf16* qkv_weight, const mh3_bf16* q_norm_weight,
                         const mh3_bf16* k_norm_weight, const mh3_bf16* rope_cos_sin, int64_t S,
                         const int64_t* rope_positions, int P, float eps, float qk_eps,
                         const float* qkv_descale, mh3_bf16* workspace, uint8_t* out);

/* Bytes of the e4m3 out: M * 21504 (0 for M <= 0). */
size_t mh3_preattn_out_e4m3_bytes(int64_t M);

/* The e4m3 conversion of mh3_preattn_run_e4m3 on its own, for any bf16
 * tensor with one per-tensor dequantisation scale:
 *   codes[i] = e4m3(values[i] / *descale)   (FP32 quotient, nearest-even,
 *                                            saturated to +-448)
 *   stream   cudaStream_t or NULL (legacy default stream)
 *   n        number of elements, >= 0 (0 launches nothing)
 *   values   DEVICE, n bf16, 2-byte aligned
 *   descale  DEVICE pointer to one float, read on the device
 *   codes    DEVICE, n bytes, caller-owned; must not overlap `values`
 * Any alignment works; 16-byte aligned `values` with 8-byte aligned `codes`
 * take the vector path.  Returns MH3_ERR_INVALID_ARG for n < 0, a NULL
 * pointer with n > 0 or overlapping buffers, MH3_ERR_ALIGNMENT for an odd
 * `values` or a misaligned `descale`, MH3_ERR_CUDA for a failed launch.
 * Needs no handle. */
int mh3_e4m3_quantize(void* stream, int64_t n, const mh3_bf16* values, const float* descale,
                      uint8_t* codes);

/* Kernel 1 alone: workspace[m] = a (the formula block's n and a lines, with
 * the index guard).  Arguments as in mh3_preattn_run; workspace must not be
 * NULL. */
int mh3_preattn_norm_adaln(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* x,
                           const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                           int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                           int64_t shift_row_stride, int64_t rows, const int64_t* adaln_index,
                           float eps, mh3_bf16* workspace);

/* Kernel 2 alone: out = pack(rope(norm(bf16(workspace @ qkv_weight^T)))),
 * reading an already-filled workspace [M, 5376].  Arguments as in
 * mh3_preattn_run (qk_eps here must be finite and > 0: there is no eps to
 * fall back to); the same split tail, with the same handle scratch, whose
 * flags this call clears with a memset on the stream before kernel 2. */
int mh3_preattn_qkv(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* workspace,
                    const mh3_bf16* qkv_weight, const mh3_bf16* q_norm_weight,
                    const mh3_bf16* k_norm_weight, const mh3_bf16* rope_cos_sin, int64_t S,
                    const int64_t* rope_positions, int P, float qk_eps, mh3_bf16* out);

/* Test hook for failure detection: when `stall` is nonzero, the next launch
 * of a CTA-pair QKV GEMM through this handle (mh3_preattn_run or
 * mh3_preattn_qkv with M > 128, or the NVFP4 GEMM of mh3_nvfp4_preattn_run
 * or mh3_nvfp4_qkv) issues no operand loads.  Its consumers'
 * bounded waits then run out (about 2 s), the kernel records a nonzero code
 * in the device status word, drains and returns: the launch completes and the
 * context stays usable; `out` is not written.  The flag clears itself after
 * that launch.  No fault, trap or endless wait is involved. */
int mh3_preattn_set_test_stall(mh3_preattn_t handle, int stall);

/* Synchronise `stream`, then read and clear the handle's device status word.
 * *device_code receives 0 when no kernel recorded a timeout since the last
 * read, else a nonzero code (which wait gave up).  Returns MH3_OK, or
 * MH3_ERR_CUDA if the synchronisation or the copy failed. */
int mh3_preattn_device_status(mh3_preattn_t handle, void* stream, int* device_code);

/* The whole stage without any allocation, for callers that cannot call
 * cudaMalloc (a custom allocator owns all device memory, or allocation is
 * forbidden after start-up).  There is no counterpart of this call on the
 * pages; it is mh3_preattn_run with the workspace taken from a static device
 * array instead of the caller or a handle.
 *
 * The array holds at most 1024 tokens (1024 x 5376 bf16 = 10.5 MiB); it is
 * reserved on every GPU that loads the library and kept until the process
 * exits.  M > 1024 is rejected with MH3_ERR_INVALID_ARG before anything is
 * launched.  No cudaMalloc, cudaFree or other allocating call is made.
 *
 * The first call on a device does a one-time set-up on that device (it checks
 * the device as mh3_preattn_create does, looks up the array's device address,
 * raises the GEMMs' shared-memory limits and reads the SM count); make that
 * first call before any stream capture.  A set-up that fails is not kept:
 * the call returns its error and the next call on that device tries again.
 * Every call uses the same array, which keeps the last call's contents;
 * calls that overlap on the GPU (other streams, other threads) race on it.
 *
 *   device_status  caller-owned device int, 4-byte aligned: set to 0 on
 *                  `stream` before the kernels run, then to a nonzero code if
 *                  a kernel's bounded wait gives up (read it after a sync).
 *   other arguments as in mh3_preattn_run (no handle, no workspace).
 */
int mh3_preattn_run_noalloc(void* stream, int64_t M, const mh3_bf16* x,
                            const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                            int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                            int64_t shift_row_stride, int64_t rows, const int64_t* adaln_index,
                            const mh3_bf16* qkv_weight, const mh3_bf16* q_norm_weight,
                            const mh3_bf16* k_norm_weight, const mh3_bf16* rope_cos_sin,
                            int64_t S, const int64_t* rope_positions, int P, float eps,
                            float qk_eps, mh3_bf16* out, int* device_status);

/* ---------------------------------------------------------------------------
 * Attention output projection with the fused gated residual (the step after
 * attention), from the page "flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj"
 * (summary formula; Parameters: attn_out, gate, gate_index, residual, out),
 * computed here with BF16 operands on the same CTA-pair tcgen05 GEMM:
 *
 *   o   = bf16(attn_out @ o_weight^T)                 FP32 accumulation
 *   out = bf16(residual + bf16(g * o)),  g = gate[gate_index[m]]
 *   g   = 0 when gate_index[m] lies outside [0, gate_rows)   (out = residual)
 *
 *   M                 tokens, >= 0 (M == 0 launches nothing)
 *   attn_out          [M, 7168] row-major (7168 = 56 heads x 128), 16-B aligned
 *   o_weight          [5376, 7168] row-major, 16-B aligned
 *   gate              [gate_rows, 5376] view: unit column stride, row stride
 *                     gate_row_stride (elements, >= 5376, multiple of 8),
 *                     base 16-B aligned; a column chunk of the [rows, 6*5376]
 *                     modulation projection qualifies as it is
 *   gate_rows         >= 1
 *   gate_index        [M] int32, 4-B aligned; any value (guarded on the device)
 *   residual          [M, 5376] row-major, 16-B aligned
 *   out               [M, 5376] row-major, 16-B aligned; may be the same
 *                     buffer as residual (each block is read before it is
 *                     written), must not partially overlap it
 * One launch on `stream`; no host synchronisation.  Bounded waits report to
 * the handle's status word (mh3_preattn_device_status). */
int mh3_out_proj_run(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* attn_out,
                     const mh3_bf16* o_weight, const mh3_bf16* gate, int64_t gate_row_stride,
                     int64_t gate_rows, const int32_t* gate_index, const mh3_bf16* residual,
                     mh3_bf16* out);

/* Host-only validation of an mh3_out_proj_run argument set (no device
 * access, no launch); same rules and status codes. */
int mh3_out_proj_validate(int64_t M, const mh3_bf16* attn_out, const mh3_bf16* o_weight,
                          const mh3_bf16* gate, int64_t gate_row_stride, int64_t gate_rows,
                          const int32_t* gate_index, const mh3_bf16* residual,
                          const mh3_bf16* out);

/* ---------------------------------------------------------------------------
 * The MLP block with BF16 operands, after the formula block of the page
 * "flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120" without its FP8 lines:
 *
 *   n   = bf16(rmsnorm(x, eps) * x_norm_weight)
 *   a   = bf16(shift[i] + n * bf16(1 + scale[i]))     i = adaln_index[m]
 *   a   = 0 for the whole row when i is outside [0, rows)
 *   h   = bf16(a @ fc1_weight^T)                      [M, 28672], FP32 accumulation
 *   y   = bf16(bf16(silu(h_gate)) * h_up)             h_gate = h[:, :14336], h_up = h[:, 14336:]
 *   o   = bf16(y @ fc2_weight^T)                      [M, 5376], FP32 accumulation
 *   out = bf16(residual + bf16(gate[i] * o))          gate 0 (out = residual) for a bad i
 *
 * Three launches on `stream`: kernel 1 of the pre-attention stage into
 * workspace_a, fc1 with the SwiGLU epilogue into workspace_y, fc2 with the
 * gated-residual epilogue into out.  No host synchronisation.
 *
 *   x, x_norm_weight, adaln_scale/shift (+ row strides), rows, adaln_index, eps
 *                     as in mh3_preattn_run
 *   gate              [rows, 5376] view, row stride gate_row_stride (elements,
 *                     >= 5376, multiple of 8), base 16-B aligned
 *   residual          [M, 5376] row-major, 16-B aligned
 *   fc1_weight        [28672, 5376] row-major: rows [0, 14336) the gate
 *                     projection, rows [14336, 28672) the up projection
 *   fc2_weight        [5376, 14336] row-major
 *   workspace_a       [M, 5376] bf16 scratch or NULL (handle-owned)
 *   workspace_y       [M, 14336] bf16 scratch or NULL (handle-owned); with NULL
 *                     workspaces, runs of one handle on different streams race
 *   out               [M, 5376], 16-B aligned; may be residual or x itself
 *                     (both are read before out is written), must not
 *                     partially overlap either */
int mh3_mlp_run(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* x,
                const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                int64_t scale_row_stride, const mh3_bf16* adaln_shift, int64_t shift_row_stride,
                const mh3_bf16* gate, int64_t gate_row_stride, int64_t rows,
                const int64_t* adaln_index, const mh3_bf16* residual, const mh3_bf16* fc1_weight,
                const mh3_bf16* fc2_weight, float eps, mh3_bf16* workspace_a,
                mh3_bf16* workspace_y, mh3_bf16* out);

/* Host-only validation of an mh3_mlp_run argument set; same rules and codes. */
int mh3_mlp_validate(int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
                     const mh3_bf16* adaln_scale, int64_t scale_row_stride,
                     const mh3_bf16* adaln_shift, int64_t shift_row_stride, const mh3_bf16* gate,
                     int64_t gate_row_stride, int64_t rows, const int64_t* adaln_index,
                     const mh3_bf16* residual, const mh3_bf16* fc1_weight,
                     const mh3_bf16* fc2_weight, float eps, const mh3_bf16* workspace_a,
                     const mh3_bf16* workspace_y, const mh3_bf16* out);

/* Bytes of the MLP intermediate y, [M, 14336] bf16: M * 14336 * 2 (0 for M <= 0). */
size_t mh3_mlp_workspace_y_bytes(int64_t M);

/* ------------------------------------------------------- FP8 (W8A8) MLP block
 * The MLP block with E4M3 weights and per-token E4M3 activations, as the
 * formula block of the page "flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120"
 * defines it:
 *
 *   n   = bf16(rmsnorm(x, eps) * x_norm_weight)
 *   a   = bf16(adaln_shift[i] + n * bf16(1 + adaln_scale[i])),  0 for a bad i
 *   a_q = e4m3(a / s_a),  s_a = RN(amax_row(|a|) / 448)            per token
 *   h   = bf16(a_q @ fc1_weight_q^T * s_a * fc1_weight_scale)      FP32 accumulation
 *   y   = bf16(bf16(silu(h_gate)) * h_up)                          [M, 14336]
 *   y_q = e4m3(y / s_y),  s_y = RN(amax_row(|y|) / 448)            per token
 *   o   = bf16(y_q @ fc2_weight_q^T * s_y * fc2_weight_scale)      FP32 accumulation
 *   out = bf16(residual + bf16(gate[i] * o)),  gate 0 for a bad i
 *
 * e4m3(v / s) rounds the exact quotient once (nearest even, saturating at
 * +-448, sign kept); a row whose amax is 0 gets s = 0 and codes +0.  The
 * scale products are two FP32 roundings in the printed order.  Four kernels
 * and one memset run on `stream`: the norm/AdaLN/quantisation kernel, the
 * fc1 GEMM (tcgen05 kind::f8f6f4, SwiGLU epilogue, which also folds each
 * row's largest |y| into workspace_y_scale), the y quantiser (which then
 * replaces that amax by s_y), and the fc2 GEMM (gated-residual epilogue).
 *
 *   fc1_weight_q      E4M3 codes [28672, 5376] (rows [0, 14336) gate, the
 *                     rest up), 16-B aligned; fc1_weight_scale FP32 [28672]
 *   fc2_weight_q      E4M3 codes [5376, 14336]; fc2_weight_scale FP32 [5376]
 *   workspace_a_q     E4M3 [M, 5376] or NULL; workspace_a_scale FP32 [M] or NULL
 *   workspace_y       bf16 [M, 14336] or NULL
 *   workspace_y_q     E4M3 [M, 14336] or NULL; workspace_y_scale FP32 [M] or NULL
 *                     (NULL: handle-owned, grown on `stream`; runs of one
 *                     handle on different streams then race)
 *   other arguments as in mh3_mlp_run (int64 adaln_index, shared row count,
 *   out may be residual or x).  Returns MH3_OK or an error code; nothing is
 *   launched on an argument error. */
int mh3_mlp_fp8_run(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* x,
                    const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                    int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                    int64_t shift_row_stride, const mh3_bf16* gate, int64_t gate_row_stride,
                    int64_t rows, const int64_t* adaln_index, const mh3_bf16* residual,
                    const uint8_t* fc1_weight_q, const float* fc1_weight_scale,
                    const uint8_t* fc2_weight_q, const float* fc2_weight_scale, float eps,
                    uint8_t* workspace_a_q, float* workspace_a_scale, mh3_bf16* workspace_y,
                    uint8_t* workspace_y_q, float* workspace_y_scale, mh3_bf16* out);

/* Host-only validation of an mh3_mlp_fp8_run argument set; same rules and codes. */
int mh3_mlp_fp8_validate(int64_t M, const mh3_bf16* x, const mh3_bf16* x_norm_weight,
                         const mh3_bf16* adaln_scale, int64_t scale_row_stride,
                         const mh3_bf16* adaln_shift, int64_t shift_row_stride,
                         const mh3_bf16* gate, int64_t gate_row_stride, int64_t rows,
                         const int64_t* adaln_index, const mh3_bf16* residual,
                         const uint8_t* fc1_weight_q, const float* fc1_weight_scale,
                         const uint8_t* fc2_weight_q, const float* fc2_weight_scale, float eps,
                         const uint8_t* workspace_a_q, const float* workspace_a_scale,
                         const mh3_bf16* workspace_y, const uint8_t* workspace_y_q,
                         const float* workspace_y_scale, const mh3_bf16* out);

/* Bytes of one FP8 MLP workspace for M tokens: which = 0 a_q (M * 5376),
 * 1 a scale (M * 4), 2 y (M * 14336 * 2), 3 y_q (M * 14336), 4 y scale
 * (M * 4); 0 for M <= 0 or another `which`. */
size_t mh3_mlp_fp8_workspace_bytes(int64_t M, int which);

/* ------------------------------------------------------------ NVFP4 stage
 * The pre-attention stage with NVFP4 operands (page
 * "flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention", summary and
 * Parameters).  NVFP4 here: E2M1 element codes packed two per byte (element
 * 2j in the low nibble of byte j), one UE4M3 scale per block of 16
 * consecutive elements of a row, and an FP32 global scale gs, in the
 * FlashInfer block-16 convention the page
 * "flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj" prints in its summary:
 *   s    = ue4m3(amax * gs / 6)            amax = max |v| of the block
 *   code = e2m1(v * gs / s)                 (signed zero when s = 0)
 * each ONE rounding of the exact quotient, to nearest even, saturating at
 * 448 and 6; v ~ code * s / gs.
 * Scale layouts: row-major [rows, cols/16] (tiled = 0), or tiled (tiled = 1):
 * 512-byte atoms of 128 rows x 4 scales (one 64-element step), row r of an
 * atom at byte (r % 32) * 16 + (r / 32) * 4, atoms ordered [rows/128][cols/64]
 * (rows padded up to a multiple of 128; padding bytes are not written).  The
 * tiled layout is what the block-scaled GEMM reads, and is this library's
 * reading of the page's "128x4 swizzled" weight scales. */

/* Bytes of packed codes, rows * cols / 2, and of the scales of a rows x cols
 * matrix in the given layout (0 for rows <= 0 or cols <= 0). */
size_t mh3_nvfp4_codes_bytes(int64_t rows, int64_t cols);
size_t mh3_nvfp4_scales_bytes(int64_t rows, int64_t cols, int tiled);

/* Quantise a bf16 matrix (the weight preparation of the NVFP4 stage, in the
 * role of the page's quantize_minimax_h3_qkv_weight_nvfp4, and a standalone
 * activation quantiser):
 *   rows, cols     rows >= 0; cols a positive multiple of 64 (<= 2^24)
 *   values         DEVICE bf16 [rows, cols] row-major, 16-byte aligned
 *   global_scale   DEVICE pointer to one float gs, read on the device
 *   codes          DEVICE, rows * cols / 2 bytes, 16-byte aligned
 *   scales         DEVICE, mh3_nvfp4_scales_bytes(rows, cols, tiled) bytes
 * Returns MH3_ERR_INVALID_ARG / MH3_ERR_ALIGNMENT for bad arguments,
 * MH3_ERR_CUDA for a failed launch.  Needs no handle. */
int mh3_nvfp4_quantize(void* stream, int64_t rows, int64_t cols, const mh3_bf16* values,
                       const float* global_scale, uint8_t* codes, uint8_t* scales, int tiled);

/* Kernel 1 of the NVFP4 stage alone: the bf16 stage's n and a (input
 * RMSNorm, indexed AdaLN with the guard) quantised per token with the
 * activation global scale.  adaln_index is INT32 [M] here (Parameters:
 * adaln_index); a bad index gives zero codes and zero scales.
 *   act_global_scale  DEVICE pointer to one float (Parameters:
 *                     act_global_scale, read on the device)
 *   act_q             DEVICE [M, 2688] bytes, 16-byte aligned
 *   act_sf            DEVICE, mh3_nvfp4_scales_bytes(M, 5376, tiled) bytes
 * Other arguments as in mh3_preattn_norm_adaln. */
int mh3_nvfp4_norm_quant(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* x,
                         const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                         int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                         int64_t shift_row_stride, int64_t rows, const int32_t* adaln_index,
                         float eps, const float* act_global_scale, uint8_t* act_q,
                         uint8_t* act_sf, int tiled);

/* The whole NVFP4 stage: kernel 1 (norm, AdaLN, activation quantisation)
 * then the block-scaled FP4 GEMM (tcgen05 kind::mxf4nvf4) with
 *   y = bf16(RN(alpha * acc)),  acc = sum_k (qa sa)(qw sw)  (FP32)
 * and the bf16 stage's epilogue: per-head RMSNorm of q and k with eps (the
 * op has one eps), split-half RoPE of dims [0, 96) with row m of
 * rope_cos_sin for token m, and the destination-major pack.
 *   adaln_index          INT32 [M]
 *   weight_q             DEVICE [21504, 2688] codes of qkv_weight (rows in
 *                        [kind, head, d] order), 16-byte aligned
 *   weight_sf            DEVICE tiled scales of qkv_weight,
 *                        mh3_nvfp4_scales_bytes(21504, 5376, 1) bytes,
 *                        16-byte aligned
 *   weight_global_scale  host float: the weight's gs
 *   act_global_scale     DEVICE pointer to one float
 *   alpha                host float; finite and > 0 is used as given, any
 *                        other value (e.g. NaN) means alpha is derived on the
 *                        device as RN(1 / RN(act_gs * weight_global_scale))
 *                        (Parameters: alpha)
 *   rope_cos_sin         DEVICE bf16 [M, 96], 16-byte aligned
 *   P                    ulysses degree 1, 2, 4 or 8
 *   qkv_descale          NULL: bf16 out [P, M, 56/P, 3, 128]; else DEVICE
 *                        float [3] and out holds e4m3 codes of the same
 *                        shape (the conversion of mh3_preattn_run_e4m3)
 *   act_q, act_sf        stage-1 workspaces ([M, 2688] bytes and the tiled
 *                        scales of [M, 5376], each 16-byte aligned) or NULL
 *                        for handle-owned buffers (grown with
 *                        cudaMallocAsync on `stream`)
 *   out                  DEVICE, 16-byte aligned
 * The output shapes of the page's q, k, v are defined on the FP8 stage's
 * page, which is not available; this call writes the bf16 stage's packed
 * layout.  Returns as mh3_preattn_run; MH3_ERR_UNSUPPORTED when no CTA pair
 * of the GEMM fits the device. */
int mh3_nvfp4_preattn_run(mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* x,
                          const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale,
                          int64_t scale_row_stride, const mh3_bf16* adaln_shift,
                          int64_t shift_row_stride, int64_t rows, const int32_t* adaln_index,
                          const uint8_t* weight_q, const uint8_t* weight_sf,
                          float weight_global_scale, const float* act_global_scale, float alpha,
                          const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
                          const mh3_bf16* rope_cos_sin, int P, float eps,
                          const float* qkv_descale, uint8_t* act_q, uint8_t* act_sf, void* out);

/* Kernel 2 of the NVFP4 stage alone, on act_q / act_sf already filled by
 * mh3_nvfp4_norm_quant (tiled scales) or mh3_nvfp4_quantize (tiled).  act_q
 * and act_sf must be 16-byte aligned; act_global_scale is only read when
 * alpha is not given (finite and > 0).  Other arguments and rules as in
 * mh3_nvfp4_preattn_run. */
int mh3_nvfp4_qkv(mh3_preattn_t handle, void* stream, int64_t M, const uint8_t* act_q,
                  const uint8_t* act_sf, const uint8_t* weight_q, const uint8_t* weight_sf,
                  float weight_global_scale, const float* act_global_scale, float alpha,
                  const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight,
                  const mh3_bf16* rope_cos_sin, int P, float eps, const float* qkv_descale,
                  void* out);

/* The NVFP4 stage with NVFP4 outputs (out_mode "nvfp4" of the page
 * "flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention", Parameters:
 * out_mode, q_sf/k_sf/v_sf, q/k/v_global_scale).  The shapes are defined on
 * the FP8 stage's page, which is not available; this library's reading:
 * each output row of 128 values (one token, head and kind, after the Q/K
 * norm and RoPE, rounded to bf16 as in the bf16 output) is quantised in the
 * block-16 convention above with the global scale of its kind, and written
 * in the bf16 output's destination-major order:
 *   out_codes  DEVICE [P, M, 56/P, 3, 64] bytes (E2M1 codes, element 2j in
 *              the low nibble of byte j), 16-byte aligned,
 *              mh3_preattn_out_nvfp4_bytes(M, 0) bytes
 *   out_sf     DEVICE [P, M, 56/P, 3, 8] UE4M3 scales (block b covers
 *              elements 16b..16b+15), 8-byte aligned,
 *              mh3_preattn_out_nvfp4_bytes(M, 1) bytes
 *   qkv_global_scale  DEVICE float [3]: the q, k and v global scales
 * Other arguments and rules as in mh3_nvfp4_preattn_run (no qkv_descale,
 * no bf16 out). */
int mh3_nvfp4_preattn_run_nvfp4_out(
    mh3_preattn_t handle, void* stream, int64_t M, const mh3_bf16* x,
    const mh3_bf16* x_norm_weight, const mh3_bf16* adaln_scale, int64_t scale_row_stride,
    const mh3_bf16* adaln_shift, int64_t shift_row_stride, int64_t rows,
    const int32_t* adaln_index, const uint8_t* weight_q, const uint8_t* weight_sf,
    float weight_global_scale, const float* act_global_scale, float alpha,
    const mh3_bf16* q_norm_weight, const mh3_bf16* k_norm_weight, const mh3_bf16* rope_cos_sin,
    int P, float eps, const float* qkv_global_scale, uint8_t* act_q, uint8_t* act_sf,
    uint8_t* out_codes, uint8_t* out_sf);

/* Bytes of the NVFP4 outputs for M tokens: which = 0 the codes
 * (M * 10752), 1 the scales (M * 1344); 0 for M <= 0 or another `which`. */
size_t mh3_preattn_out_nvfp4_bytes(int64_t M, int which);

/* ---------------------------------------------------------------------------
 * The W4A4 attention output projection with the fused gated residual (page
 * "flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj", summary and
 * Parameters): attn_out is quantised to NVFP4 per token with the activation
 * global scale (the block-16 convention above), multiplied on the
 * block-scaled FP4 tensor cores (tcgen05 kind::mxf4nvf4, CTA pairs) by the
 * quantised o_weight, and the accumulator takes the gated residual:
 *
 *   acc   = sum_k (qa sa)(qw sw)                        FP32
 *   alpha = RN(1 / RN(act_gs * o_weight_global_scale))  (on the device)
 *   o     = bf16(RN(alpha * acc))
 *   out   = bf16(residual + bf16(g * o)),  g = gate[gate_index[m]], or 0 when
 *           gate_index[m] lies outside [0, gate_rows)    (out = residual)
 *
 * Two launches on `stream` (the activation quantiser, then the GEMM, which
 * starts its weight-independent set-up while the quantiser drains); no host
 * synchronisation.
 *   M                      tokens, >= 0 (M == 0 launches nothing)
 *   attn_out               DEVICE bf16 [M, 7168] row-major, 16-byte aligned
 *   o_weight_q             DEVICE [5376, 3584] E2M1 codes of o_weight (two
 *                          per byte), 16-byte aligned (mh3_nvfp4_quantize)
 *   o_weight_sf            DEVICE tiled scales of o_weight,
 *                          mh3_nvfp4_scales_bytes(5376, 7168, 1) bytes,
 *                          16-byte aligned
 *   o_weight_global_scale  host float, finite and > 0
 *   act_global_scale       DEVICE pointer to one float (read on the device)
 *   gate, gate_row_stride, gate_rows, gate_index, residual, out
 *                          as in mh3_out_proj_run (out may be residual)
 *   act_q, act_sf          workspaces: [M, 3584] code bytes and the tiled
 *                          scales of [M, 7168] (mh3_nvfp4_scales_bytes(M,
 *                          7168, 1) bytes: M * 448 when M is a multiple of
 *                          128), each 16-byte aligned, or NULL for
 *                          handle-owned buffers (grown with cudaMallocAsync
 *                          on `stream`); they hold the quantised activation
 *                          after the call
 * Returns MH3_ERR_INVALID_ARG / MH3_ERR_ALIGNMENT for bad arguments,
 * MH3_ERR_UNSUPPORTED when no CTA pair of the GEMM fits the device,
 * MH3_ERR_CUDA for a failed launch.  Bounded waits report to the handle's
 * status word (mh3_preattn_device_status). */
int mh3_nvfp4_out_proj_run(mh3_preattn_t handle, void* stream, int64_t M,
                           const mh3_bf16* attn_out, const uint8_t* o_weight_q,
                           const uint8_t* o_weight_sf, float o_weight_global_scale,
                           const float* act_global_scale, const mh3_bf16* gate,
                           int64_t gate_row_stride, int64_t gate_rows,
                           const int32_t* gate_index, const mh3_bf16* residual, uint8_t* act_q,
                           uint8_t* act_sf, mh3_bf16* out);

/* Host-only validation of an mh3_nvfp4_out_proj_run argument set (the
 * arguments other than the handle, the stream and the workspaces; no device
 * access); same rules and status codes. */
int mh3_nvfp4_out_proj_validate(int64_t M, const mh3_bf16* attn_out, const uint8_t* o_weight_q,
                                const uint8_t* o_weight_sf, float o_weight_global_scale,
                                const float* act_global_scale, const mh3_bf16* gate,
                                int64_t gate_row_stride, int64_t gate_rows,
                                const int32_t* gate_index, const mh3_bf16* residual,
                                const mh3_bf16* out);

/* Message of the calling thread's last failed call ("" if none). */
const char* mh3_preattn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MH3_PREATTN_H */
