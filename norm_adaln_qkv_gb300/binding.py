"""ctypes binding of the C ABI in include/mh3_preattn.h.

Argument marshalling only: every step of the stage runs in the CUDA library.
The functions keep the C names and take torch CUDA tensors (or raw integer
device pointers) plus sizes.  There is no fallback: if the library is missing
or a call fails, a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from . import inputs as _inputs

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmh3_preattn.so")

HIDDEN = _inputs.HIDDEN
NUM_HEADS = _inputs.NUM_HEADS
HEAD_DIM = _inputs.HEAD_DIM
QKV_ROWS = _inputs.QKV_ROWS
ROPE_DIMS = _inputs.ROPE_DIMS

STATUS = {0: "MH3_OK", 1: "MH3_ERR_INVALID_ARG", 2: "MH3_ERR_ALIGNMENT", 3: "MH3_ERR_UNSUPPORTED",
          4: "MH3_ERR_CUDA", 5: "MH3_ERR_OOM", 6: "MH3_ERR_DEVICE"}

# Every symbol include/mh3_preattn.h declares.
EXPORTS = ("mh3_preattn_create", "mh3_preattn_destroy", "mh3_preattn_workspace_bytes",
           "mh3_preattn_out_bytes", "mh3_preattn_validate", "mh3_preattn_run",
           "mh3_preattn_norm_adaln", "mh3_preattn_qkv", "mh3_preattn_device_status",
           "mh3_preattn_last_error", "mh3_preattn_run_noalloc", "mh3_out_proj_run",
           "mh3_out_proj_validate", "mh3_mlp_run", "mh3_mlp_validate",
           "mh3_mlp_workspace_y_bytes", "mh3_preattn_run_e4m3", "mh3_preattn_out_e4m3_bytes",
           "mh3_e4m3_quantize", "mh3_nvfp4_codes_bytes", "mh3_nvfp4_scales_bytes",
           "mh3_nvfp4_quantize", "mh3_nvfp4_norm_quant", "mh3_nvfp4_preattn_run", "mh3_nvfp4_qkv",
           "mh3_preattn_set_test_stall", "mh3_mlp_fp8_run", "mh3_mlp_fp8_validate",
           "mh3_mlp_fp8_workspace_bytes", "mh3_nvfp4_out_proj_run",
           "mh3_nvfp4_out_proj_validate", "mh3_nvfp4_preattn_run_nvfp4_out",
           "mh3_preattn_out_nvfp4_bytes")

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int
_f32 = ctypes.c_float

_SIGS = {
    "mh3_preattn_create": (_i32, [ctypes.POINTER(_vp), _i32]),
    "mh3_preattn_destroy": (_i32, [_vp]),
    "mh3_preattn_workspace_bytes": (ctypes.c_size_t, [_i64]),
    "mh3_preattn_out_bytes": (ctypes.c_size_t, [_i64]),
    "mh3_preattn_validate": (_i32, [_i64, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _vp,
                                    _vp, _i64, _vp, _i32, _f32, _f32, _vp, _vp]),
    "mh3_preattn_run": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp,
                               _vp, _vp, _i64, _vp, _i32, _f32, _f32, _vp, _vp]),
    "mh3_preattn_norm_adaln": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp,
                                      _f32, _vp]),
    "mh3_preattn_qkv": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _f32, _vp]),
    "mh3_preattn_device_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32)]),
    "mh3_preattn_last_error": (ctypes.c_char_p, []),
    "mh3_out_proj_run": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp]),
    "mh3_out_proj_validate": (_i32, [_i64, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp]),
    "mh3_mlp_run": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _i64, _i64, _vp, _vp,
                           _vp, _vp, _f32, _vp, _vp, _vp]),
    "mh3_mlp_validate": (_i32, [_i64, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _i64, _i64, _vp, _vp,
                                _vp, _vp, _f32, _vp, _vp, _vp]),
    "mh3_mlp_workspace_y_bytes": (ctypes.c_size_t, [_i64]),
    "mh3_preattn_run_e4m3": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp, _vp,
                                    _vp, _vp, _vp, _i64, _vp, _i32, _f32, _f32, _vp, _vp, _vp]),
    "mh3_preattn_out_e4m3_bytes": (ctypes.c_size_t, [_i64]),
    "mh3_e4m3_quantize": (_i32, [_vp, _i64, _vp, _vp, _vp]),
    "mh3_nvfp4_codes_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "mh3_nvfp4_scales_bytes": (ctypes.c_size_t, [_i64, _i64, _i32]),
    "mh3_nvfp4_quantize": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _i32]),
    "mh3_nvfp4_norm_quant": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp,
                                    _f32, _vp, _vp, _vp, _i32]),
    "mh3_preattn_set_test_stall": (_i32, [_vp, _i32]),
    "mh3_nvfp4_qkv": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _f32, _vp, _f32, _vp, _vp, _vp,
                             _i32, _f32, _vp, _vp]),
    "mh3_nvfp4_preattn_run": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp,
                                     _vp, _vp, _f32, _vp, _f32, _vp, _vp, _vp, _i32, _f32, _vp,
                                     _vp, _vp, _vp]),
    "mh3_preattn_run_noalloc": (_i32, [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp, _vp,
                                       _vp, _vp, _vp, _i64, _vp, _i32, _f32, _f32, _vp, _vp]),
    "mh3_mlp_fp8_run": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _i64, _i64,
                               _vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mh3_mlp_fp8_validate": (_i32, [_i64, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _i64, _i64, _vp,
                                    _vp, _vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mh3_mlp_fp8_workspace_bytes": (ctypes.c_size_t, [_i64, _i32]),
    "mh3_nvfp4_out_proj_run": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _f32, _vp, _vp, _i64, _i64,
                                      _vp, _vp, _vp, _vp, _vp]),
    "mh3_nvfp4_preattn_run_nvfp4_out": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i64,
                                               _i64, _vp, _vp, _vp, _f32, _vp, _f32, _vp, _vp,
                                               _vp, _i32, _f32, _vp, _vp, _vp, _vp, _vp]),
    "mh3_preattn_out_nvfp4_bytes": (ctypes.c_size_t, [_i64, _i32]),
    "mh3_nvfp4_out_proj_validate": (_i32, [_i64, _vp, _vp, _vp, _f32, _vp, _vp, _i64, _i64, _vp,
                                           _vp, _vp]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (built by norm_adaln_qkv_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run norm_adaln_qkv_gb300.build.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def last_error() -> str:
    return load().mh3_preattn_last_error().decode()


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what} failed: {STATUS.get(rc, rc)}: {last_error()}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _qk_eps_arg(qk_eps: Optional[float]) -> float:
    return -1.0 if qk_eps is None else float(qk_eps)


class Handle:
    """Owns an mh3_preattn_t for one device."""

    def __init__(self, device: Optional[int] = None):
        lib = load()
        if device is None:
            device = torch.cuda.current_device()
        self.device = device
        h = _vp()
        _check(lib.mh3_preattn_create(ctypes.byref(h), device), "mh3_preattn_create")
        self._h = h

    @property
    def ptr(self):
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value is not None:
            _check(load().mh3_preattn_destroy(self._h), "mh3_preattn_destroy")
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def device_status(self, stream=None) -> int:
        code = _i32(0)
        _check(load().mh3_preattn_device_status(self._h, _stream_ptr(stream), ctypes.byref(code)),
               "mh3_preattn_device_status")
        return code.value

    def set_test_stall(self, stall: bool = True) -> None:
        """Test hook: the next CTA-pair QKV GEMM launch issues no loads, so its
        bounded waits run out and it reports a status code."""
        _check(load().mh3_preattn_set_test_stall(self._h, 1 if stall else 0),
               "mh3_preattn_set_test_stall")


_handles = {}


def default_handle(device: Optional[int] = None) -> Handle:
    if device is None:
        device = torch.cuda.current_device()
    if device not in _handles:
        _handles[device] = Handle(device)
    return _handles[device]


def workspace_bytes(M: int) -> int:
    return load().mh3_preattn_workspace_bytes(M)


def out_bytes(M: int) -> int:
    return load().mh3_preattn_out_bytes(M)


def mh3_preattn_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                         shift_row_stride, rows, adaln_index, qkv_weight, q_norm_weight,
                         k_norm_weight, rope_cos_sin, S, rope_positions, P, eps, qk_eps,
                         workspace, out) -> int:
    """Host-only validation; returns the status code (pointers may be ints)."""
    return load().mh3_preattn_validate(
        M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale), scale_row_stride, _ptr(adaln_shift),
        shift_row_stride, rows, _ptr(adaln_index), _ptr(qkv_weight), _ptr(q_norm_weight),
        _ptr(k_norm_weight), _ptr(rope_cos_sin), S, _ptr(rope_positions), P, float(eps),
        _qk_eps_arg(qk_eps), _ptr(workspace), _ptr(out))


def mh3_preattn_run(handle: Handle, stream, M, x, x_norm_weight, adaln_scale, scale_row_stride,
                    adaln_shift, shift_row_stride, rows, adaln_index, qkv_weight, q_norm_weight,
                    k_norm_weight, rope_cos_sin, S, rope_positions, P, eps, qk_eps, workspace,
                    out) -> None:
    _check(load().mh3_preattn_run(
        handle.ptr, _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, rows, _ptr(adaln_index),
        _ptr(qkv_weight), _ptr(q_norm_weight), _ptr(k_norm_weight), _ptr(rope_cos_sin), S,
        _ptr(rope_positions), P, float(eps), _qk_eps_arg(qk_eps), _ptr(workspace), _ptr(out)),
        "mh3_preattn_run")


def mh3_preattn_run_noalloc(stream, M, x, x_norm_weight, adaln_scale, scale_row_stride,
                            adaln_shift, shift_row_stride, rows, adaln_index, qkv_weight,
                            q_norm_weight, k_norm_weight, rope_cos_sin, S, rope_positions, P, eps,
                            qk_eps, out, device_status) -> None:
    """The stage with the library's static workspace (M <= 1024); allocates
    nothing.  ``device_status`` is a caller-owned device int32 tensor."""
    _check(load().mh3_preattn_run_noalloc(
        _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, rows, _ptr(adaln_index),
        _ptr(qkv_weight), _ptr(q_norm_weight), _ptr(k_norm_weight), _ptr(rope_cos_sin), S,
        _ptr(rope_positions), P, float(eps), _qk_eps_arg(qk_eps), _ptr(out),
        _ptr(device_status)), "mh3_preattn_run_noalloc")


def mh3_out_proj_validate(M, attn_out, o_weight, gate, gate_row_stride, gate_rows, gate_index,
                          residual, out) -> int:
    """Host-only validation of an output-projection call; returns the status."""
    return load().mh3_out_proj_validate(M, _ptr(attn_out), _ptr(o_weight), _ptr(gate),
                                        gate_row_stride, gate_rows, _ptr(gate_index),
                                        _ptr(residual), _ptr(out))


def mh3_out_proj_run(handle: Handle, stream, M, attn_out, o_weight, gate, gate_row_stride,
                     gate_rows, gate_index, residual, out) -> None:
    _check(load().mh3_out_proj_run(handle.ptr, _stream_ptr(stream), M, _ptr(attn_out),
                                   _ptr(o_weight), _ptr(gate), gate_row_stride, gate_rows,
                                   _ptr(gate_index), _ptr(residual), _ptr(out)),
           "mh3_out_proj_run")


def minimax_h3_bf16_out_proj(attn_out, o_weight, gate, gate_index, residual, *,
                             out: Optional[torch.Tensor] = None, stream=None,
                             handle: Optional[Handle] = None) -> torch.Tensor:
    """Torch-tensor entry point of the output projection with the fused gated
    residual (argument names of flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj,
    BF16 weight); returns ``out`` (allocated when None; may be ``residual``)."""
    M = attn_out.shape[0]
    bf = torch.bfloat16
    _check_tensor(attn_out, "attn_out", bf, (M, NUM_HEADS * HEAD_DIM))
    _check_tensor(o_weight, "o_weight", bf, (HIDDEN, NUM_HEADS * HEAD_DIM))
    _check_tensor(gate, "gate", bf, contiguous=False)
    if gate.dim() != 2 or gate.shape[1] != HIDDEN or gate.stride(1) != 1:
        raise ValueError(f"gate must be [rows, {HIDDEN}] with stride(1) == 1")
    _check_tensor(gate_index, "gate_index", torch.int32, (M,))
    _check_tensor(residual, "residual", bf, (M, HIDDEN))
    if out is None:
        out = torch.empty_like(residual)
    _check_tensor(out, "out", bf, (M, HIDDEN))
    h = handle if handle is not None else default_handle(attn_out.device.index)
    mh3_out_proj_run(h, stream, M, attn_out, o_weight, gate, gate.stride(0), gate.shape[0],
                     gate_index, residual, out)
    return out


def mh3_mlp_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                     shift_row_stride, gate, gate_row_stride, rows, adaln_index, residual,
                     fc1_weight, fc2_weight, eps, workspace_a, workspace_y, out) -> int:
    """Host-only validation of an MLP call; returns the status code."""
    return load().mh3_mlp_validate(
        M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale), scale_row_stride, _ptr(adaln_shift),
        shift_row_stride, _ptr(gate), gate_row_stride, rows, _ptr(adaln_index), _ptr(residual),
        _ptr(fc1_weight), _ptr(fc2_weight), float(eps), _ptr(workspace_a), _ptr(workspace_y),
        _ptr(out))


def mh3_mlp_run(handle: Handle, stream, M, x, x_norm_weight, adaln_scale, scale_row_stride,
                adaln_shift, shift_row_stride, gate, gate_row_stride, rows, adaln_index, residual,
                fc1_weight, fc2_weight, eps, workspace_a, workspace_y, out) -> None:
    _check(load().mh3_mlp_run(
        handle.ptr, _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, _ptr(gate), gate_row_stride, rows,
        _ptr(adaln_index), _ptr(residual), _ptr(fc1_weight), _ptr(fc2_weight), float(eps),
        _ptr(workspace_a), _ptr(workspace_y), _ptr(out)), "mh3_mlp_run")


def mh3_mlp_fp8_validate(M, x, x_norm_weight, adaln_scale, scale_row_stride, adaln_shift,
                         shift_row_stride, gate, gate_row_stride, rows, adaln_index, residual,
                         fc1_weight_q, fc1_weight_scale, fc2_weight_q, fc2_weight_scale, eps,
                         workspace_a_q, workspace_a_scale, workspace_y, workspace_y_q,
                         workspace_y_scale, out) -> int:
    """Host-only validation of an FP8 MLP call; returns the status code."""
    return load().mh3_mlp_fp8_validate(
        M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale), scale_row_stride, _ptr(adaln_shift),
        shift_row_stride, _ptr(gate), gate_row_stride, rows, _ptr(adaln_index), _ptr(residual),
        _ptr(fc1_weight_q), _ptr(fc1_weight_scale), _ptr(fc2_weight_q), _ptr(fc2_weight_scale),
        float(eps), _ptr(workspace_a_q), _ptr(workspace_a_scale), _ptr(workspace_y),
        _ptr(workspace_y_q), _ptr(workspace_y_scale), _ptr(out))


def mh3_mlp_fp8_run(handle: Handle, stream, M, x, x_norm_weight, adaln_scale, scale_row_stride,
                    adaln_shift, shift_row_stride, gate, gate_row_stride, rows, adaln_index,
                    residual, fc1_weight_q, fc1_weight_scale, fc2_weight_q, fc2_weight_scale,
                    eps, workspace_a_q, workspace_a_scale, workspace_y, workspace_y_q,
                    workspace_y_scale, out) -> None:
    _check(load().mh3_mlp_fp8_run(
        handle.ptr, _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, _ptr(gate), gate_row_stride, rows,
        _ptr(adaln_index), _ptr(residual), _ptr(fc1_weight_q), _ptr(fc1_weight_scale),
        _ptr(fc2_weight_q), _ptr(fc2_weight_scale), float(eps), _ptr(workspace_a_q),
        _ptr(workspace_a_scale), _ptr(workspace_y), _ptr(workspace_y_q), _ptr(workspace_y_scale),
        _ptr(out)), "mh3_mlp_fp8_run")


def minimax_h3_mlp_fp8(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index, gate, residual,
                       fc1_weight_q, fc1_weight_scale, fc2_weight_q, fc2_weight_scale, *,
                       out: Optional[torch.Tensor] = None, workspace_a_q=None,
                       workspace_a_scale=None, workspace_y=None, workspace_y_q=None,
                       workspace_y_scale=None, eps: float = 1e-5, stream=None,
                       handle: Optional[Handle] = None) -> torch.Tensor:
    """Torch-tensor entry point of the FP8 MLP block (argument names of
    flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120); E4M3 weights are
    uint8 (or float8_e4m3fn) tensors; returns ``out`` (allocated when None)."""
    M = x.shape[0]
    if out is None:
        out = torch.empty_like(residual)
    h = handle if handle is not None else default_handle(x.device.index or 0)
    as_u8 = lambda t: None if t is None else t.view(torch.uint8)  # noqa: E731
    mh3_mlp_fp8_run(h, stream, M, x, x_norm_weight, adaln_scale, adaln_scale.stride(0),
                    adaln_shift, adaln_shift.stride(0), gate, gate.stride(0), adaln_scale.shape[0],
                    adaln_index, residual, as_u8(fc1_weight_q), fc1_weight_scale,
                    as_u8(fc2_weight_q), fc2_weight_scale, eps, as_u8(workspace_a_q),
                    workspace_a_scale, workspace_y, as_u8(workspace_y_q), workspace_y_scale, out)
    return out


def minimax_h3_bf16_mlp(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index, gate, residual,
                        fc1_weight, fc2_weight, *, out: Optional[torch.Tensor] = None,
                        workspace_a=None, workspace_y=None, eps: float = 1e-5, stream=None,
                        handle: Optional[Handle] = None) -> torch.Tensor:
    """Torch-tensor entry point of the MLP block (argument names of
    flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, BF16 weights); returns
    ``out`` (allocated when None; may be ``residual`` or ``x``)."""
    M = x.shape[0]
    bf = torch.bfloat16
    _check_tensor(x, "x", bf, (M, HIDDEN))
    _check_tensor(x_norm_weight, "x_norm_weight", bf, (HIDDEN,))
    for name, t in (("adaln_scale", adaln_scale), ("adaln_shift", adaln_shift), ("gate", gate)):
        _check_tensor(t, name, bf, contiguous=False)
        if t.dim() != 2 or t.shape[1] != HIDDEN or t.stride(1) != 1:
            raise ValueError(f"{name} must be [rows, {HIDDEN}] with stride(1) == 1")
    rows = adaln_scale.shape[0]
    if adaln_shift.shape[0] != rows or gate.shape[0] != rows:
        raise ValueError("adaln_scale, adaln_shift and gate must share one row count")
    _check_tensor(adaln_index, "adaln_index", torch.int64, (M,))
    _check_tensor(residual, "residual", bf, (M, HIDDEN))
    _check_tensor(fc1_weight, "fc1_weight", bf, (2 * 14336, HIDDEN))
    _check_tensor(fc2_weight, "fc2_weight", bf, (HIDDEN, 14336))
    if out is None:
        out = torch.empty_like(residual)
    _check_tensor(out, "out", bf, (M, HIDDEN))
    h = handle if handle is not None else default_handle(x.device.index)
    mh3_mlp_run(h, stream, M, x, x_norm_weight, adaln_scale, adaln_scale.stride(0), adaln_shift,
                adaln_shift.stride(0), gate, gate.stride(0), rows, adaln_index, residual,
                fc1_weight, fc2_weight, eps, workspace_a, workspace_y, out)
    return out


def mh3_preattn_run_e4m3(handle: Handle, stream, M, x, x_norm_weight, adaln_scale,
                         scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index,
                         qkv_weight, q_norm_weight, k_norm_weight, rope_cos_sin, S,
                         rope_positions, P, eps, qk_eps, qkv_descale, workspace, out) -> None:
    """The stage with e4m3 outputs; qkv_descale is a device float32 tensor [3]
    (q, k, v) and out a uint8 tensor of the bf16 mode's packed shape."""
    _check(load().mh3_preattn_run_e4m3(
        handle.ptr, _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, rows, _ptr(adaln_index),
        _ptr(qkv_weight), _ptr(q_norm_weight), _ptr(k_norm_weight), _ptr(rope_cos_sin), S,
        _ptr(rope_positions), P, float(eps), _qk_eps_arg(qk_eps), _ptr(qkv_descale),
        _ptr(workspace), _ptr(out)), "mh3_preattn_run_e4m3")


def mh3_e4m3_quantize(stream, values, descale, codes) -> None:
    """codes[i] = e4m3(values[i] / descale[0]) for a device bf16 tensor
    `values`, a device float32 tensor `descale` [1] and a device uint8 tensor
    `codes` of the same number of elements."""
    n = values.numel()
    if codes.numel() != n:
        raise ValueError("codes must have as many elements as values")
    _check(load().mh3_e4m3_quantize(_stream_ptr(stream), n, _ptr(values), _ptr(descale),
                                    _ptr(codes)), "mh3_e4m3_quantize")


def mh3_nvfp4_quantize(stream, values, global_scale, codes, scales, tiled: bool = True) -> None:
    """NVFP4 codes and block scales of a device bf16 matrix [rows, cols]
    (cols a multiple of 64); global_scale is a device float32 tensor [1]."""
    rows, cols = values.shape
    _check(load().mh3_nvfp4_quantize(_stream_ptr(stream), rows, cols, _ptr(values),
                                     _ptr(global_scale), _ptr(codes), _ptr(scales),
                                     1 if tiled else 0), "mh3_nvfp4_quantize")


def mh3_nvfp4_norm_quant(handle: Handle, stream, M, x, x_norm_weight, adaln_scale,
                         scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index, eps,
                         act_global_scale, act_q, act_sf, tiled: bool = True) -> None:
    _check(load().mh3_nvfp4_norm_quant(
        handle.ptr, _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, rows, _ptr(adaln_index),
        float(eps), _ptr(act_global_scale), _ptr(act_q), _ptr(act_sf), 1 if tiled else 0),
        "mh3_nvfp4_norm_quant")


def mh3_nvfp4_preattn_run(handle: Handle, stream, M, x, x_norm_weight, adaln_scale,
                          scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index,
                          weight_q, weight_sf, weight_global_scale, act_global_scale, alpha,
                          q_norm_weight, k_norm_weight, rope_cos_sin, P, eps, qkv_descale,
                          act_q, act_sf, out) -> None:
    """The NVFP4 stage; alpha None derives it on the device from the global
    scales; qkv_descale None writes bf16 out, else e4m3 codes."""
    _check(load().mh3_nvfp4_preattn_run(
        handle.ptr, _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, rows, _ptr(adaln_index),
        _ptr(weight_q), _ptr(weight_sf), float(weight_global_scale), _ptr(act_global_scale),
        float("nan") if alpha is None else float(alpha), _ptr(q_norm_weight),
        _ptr(k_norm_weight), _ptr(rope_cos_sin), P, float(eps), _ptr(qkv_descale), _ptr(act_q),
        _ptr(act_sf), _ptr(out)), "mh3_nvfp4_preattn_run")


def mh3_nvfp4_preattn_run_nvfp4_out(handle: Handle, stream, M, x, x_norm_weight, adaln_scale,
                                    scale_row_stride, adaln_shift, shift_row_stride, rows,
                                    adaln_index, weight_q, weight_sf, weight_global_scale,
                                    act_global_scale, alpha, q_norm_weight, k_norm_weight,
                                    rope_cos_sin, P, eps, qkv_global_scale, act_q, act_sf,
                                    out_codes, out_sf) -> None:
    _check(load().mh3_nvfp4_preattn_run_nvfp4_out(
        handle.ptr, _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, rows, _ptr(adaln_index),
        _ptr(weight_q), _ptr(weight_sf), float(weight_global_scale), _ptr(act_global_scale),
        float("nan") if alpha is None else float(alpha), _ptr(q_norm_weight), _ptr(k_norm_weight),
        _ptr(rope_cos_sin), P, float(eps), _ptr(qkv_global_scale), _ptr(act_q), _ptr(act_sf),
        _ptr(out_codes), _ptr(out_sf)), "mh3_nvfp4_preattn_run_nvfp4_out")


def mh3_nvfp4_qkv(handle: Handle, stream, M, act_q, act_sf, weight_q, weight_sf,
                  weight_global_scale, act_global_scale, alpha, q_norm_weight, k_norm_weight,
                  rope_cos_sin, P, eps, qkv_descale, out) -> None:
    _check(load().mh3_nvfp4_qkv(
        handle.ptr, _stream_ptr(stream), M, _ptr(act_q), _ptr(act_sf), _ptr(weight_q),
        _ptr(weight_sf), float(weight_global_scale), _ptr(act_global_scale),
        float("nan") if alpha is None else float(alpha), _ptr(q_norm_weight), _ptr(k_norm_weight),
        _ptr(rope_cos_sin), P, float(eps), _ptr(qkv_descale), _ptr(out)), "mh3_nvfp4_qkv")


def mh3_nvfp4_out_proj_validate(M, attn_out, o_weight_q, o_weight_sf, o_weight_global_scale,
                                act_global_scale, gate, gate_row_stride, gate_rows, gate_index,
                                residual, out) -> int:
    """Host-only validation of a W4A4 output-projection call; returns the status."""
    return load().mh3_nvfp4_out_proj_validate(
        M, _ptr(attn_out), _ptr(o_weight_q), _ptr(o_weight_sf), float(o_weight_global_scale),
        _ptr(act_global_scale), _ptr(gate), gate_row_stride, gate_rows, _ptr(gate_index),
        _ptr(residual), _ptr(out))


def mh3_nvfp4_out_proj_run(handle: Handle, stream, M, attn_out, o_weight_q, o_weight_sf,
                           o_weight_global_scale, act_global_scale, gate, gate_row_stride,
                           gate_rows, gate_index, residual, act_q, act_sf, out) -> None:
    _check(load().mh3_nvfp4_out_proj_run(
        handle.ptr, _stream_ptr(stream), M, _ptr(attn_out), _ptr(o_weight_q), _ptr(o_weight_sf),
        float(o_weight_global_scale), _ptr(act_global_scale), _ptr(gate), gate_row_stride,
        gate_rows, _ptr(gate_index), _ptr(residual), _ptr(act_q), _ptr(act_sf), _ptr(out)),
        "mh3_nvfp4_out_proj_run")


def minimax_h3_nvfp4_out_proj(attn_out, o_weight_q, o_weight_sf, o_weight_global_scale,
                              act_global_scale, gate, gate_index, residual, *,
                              out: Optional[torch.Tensor] = None,
                              act_q: Optional[torch.Tensor] = None,
                              act_sf: Optional[torch.Tensor] = None, stream=None,
                              handle: Optional[Handle] = None) -> torch.Tensor:
    """Torch-tensor entry point with the argument list of the page
    flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj; returns ``out``
    (allocated when None; may be ``residual``).  o_weight_sf is in this
    library's tiled layout (mh3_nvfp4_quantize with tiled=True); act_sf, when
    given, holds mh3_nvfp4_scales_bytes(M, 7168, 1) bytes."""
    M = attn_out.shape[0]
    bf = torch.bfloat16
    u8 = torch.uint8
    width = NUM_HEADS * HEAD_DIM
    _check_tensor(attn_out, "attn_out", bf, (M, width))
    _check_tensor(o_weight_q, "o_weight_q", u8, (HIDDEN, width // 2))
    _check_tensor(o_weight_sf, "o_weight_sf", u8)
    if o_weight_sf.numel() != int(load().mh3_nvfp4_scales_bytes(HIDDEN, width, 1)):
        raise ValueError("o_weight_sf must hold the tiled scales of [5376, 7168]")
    if isinstance(o_weight_global_scale, torch.Tensor):
        o_weight_global_scale = float(o_weight_global_scale.reshape(-1)[0])
    _check_tensor(act_global_scale, "act_global_scale", torch.float32, (1,))
    _check_tensor(gate, "gate", bf, contiguous=False)
    if gate.dim() != 2 or gate.shape[1] != HIDDEN or gate.stride(1) != 1:
        raise ValueError(f"gate must be [rows, {HIDDEN}] with stride(1) == 1")
    _check_tensor(gate_index, "gate_index", torch.int32, (M,))
    _check_tensor(residual, "residual", bf, (M, HIDDEN))
    if out is None:
        out = torch.empty_like(residual)
    _check_tensor(out, "out", bf, (M, HIDDEN))
    if act_q is not None:
        _check_tensor(act_q, "act_q", u8, (M, width // 2))
    if act_sf is not None:
        _check_tensor(act_sf, "act_sf", u8)
        if act_sf.numel() < int(load().mh3_nvfp4_scales_bytes(M, width, 1)):
            raise ValueError("act_sf is smaller than the tiled scales of [M, 7168]")
    h = handle if handle is not None else default_handle(attn_out.device.index)
    mh3_nvfp4_out_proj_run(h, stream, M, attn_out, o_weight_q, o_weight_sf,
                           o_weight_global_scale, act_global_scale, gate, gate.stride(0),
                           gate.shape[0], gate_index, residual, act_q, act_sf, out)
    return out


def mh3_preattn_norm_adaln(handle: Handle, stream, M, x, x_norm_weight, adaln_scale,
                           scale_row_stride, adaln_shift, shift_row_stride, rows, adaln_index,
                           eps, workspace) -> None:
    _check(load().mh3_preattn_norm_adaln(
        handle.ptr, _stream_ptr(stream), M, _ptr(x), _ptr(x_norm_weight), _ptr(adaln_scale),
        scale_row_stride, _ptr(adaln_shift), shift_row_stride, rows, _ptr(adaln_index),
        float(eps), _ptr(workspace)), "mh3_preattn_norm_adaln")


def mh3_preattn_qkv(handle: Handle, stream, M, workspace, qkv_weight, q_norm_weight,
                    k_norm_weight, rope_cos_sin, S, rope_positions, P, qk_eps, out) -> None:
    _check(load().mh3_preattn_qkv(
        handle.ptr, _stream_ptr(stream), M, _ptr(workspace), _ptr(qkv_weight),
        _ptr(q_norm_weight), _ptr(k_norm_weight), _ptr(rope_cos_sin), S, _ptr(rope_positions), P,
        float(qk_eps), _ptr(out)), "mh3_preattn_qkv")


def _check_tensor(t: torch.Tensor, name: str, dtype, shape=None, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(t.shape)})")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def minimax_h3_bf16_pre_attention(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index,
                                  qkv_weight, q_norm_weight, k_norm_weight, rope_cos_sin, *,
                                  ulysses_degree: int, out: torch.Tensor, eps: float = 1e-5,
                                  qk_eps: Optional[float] = None, rope_positions=None,
                                  workspace: Optional[torch.Tensor] = None, stream=None,
                                  handle: Optional[Handle] = None) -> torch.Tensor:
    """Torch-tensor entry point with the argument list of the page
    flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention; returns ``out``.

    Shapes/dtypes are checked here (tensor metadata only); every other rule
    is checked by the C library before it launches.
    """
    M = x.shape[0]
    P = int(ulysses_degree)
    bf = torch.bfloat16
    _check_tensor(x, "x", bf, (M, HIDDEN))
    _check_tensor(x_norm_weight, "x_norm_weight", bf, (HIDDEN,))
    for name, t in (("adaln_scale", adaln_scale), ("adaln_shift", adaln_shift)):
        _check_tensor(t, name, bf, contiguous=False)
        if t.dim() != 2 or t.shape[1] != HIDDEN or t.stride(1) != 1:
            raise ValueError(f"{name} must be [rows, {HIDDEN}] with stride(1) == 1")
    if adaln_scale.shape[0] != adaln_shift.shape[0]:
        raise ValueError("adaln_scale and adaln_shift must have the same row count")
    _check_tensor(adaln_index, "adaln_index", torch.int64, (M,))
    _check_tensor(qkv_weight, "qkv_weight", bf, (QKV_ROWS, HIDDEN))
    _check_tensor(q_norm_weight, "q_norm_weight", bf, (HEAD_DIM,))
    _check_tensor(k_norm_weight, "k_norm_weight", bf, (HEAD_DIM,))
    _check_tensor(rope_cos_sin, "rope_cos_sin", bf)
    if rope_cos_sin.dim() != 2 or rope_cos_sin.shape[1] != ROPE_DIMS:
        raise ValueError(f"rope_cos_sin must be [S, {ROPE_DIMS}]")
    if P not in (1, 2, 4, 8):
        raise ValueError("ulysses_degree must be 1, 2, 4 or 8")
    _check_tensor(out, "out", bf, (P, M, NUM_HEADS // P, 3, HEAD_DIM))
    if rope_positions is not None:
        _check_tensor(rope_positions, "rope_positions", torch.int64, (M,))
    if workspace is not None:
        _check_tensor(workspace, "workspace", bf, (M, HIDDEN))
    h = handle if handle is not None else default_handle(x.device.index)
    mh3_preattn_run(h, stream, M, x, x_norm_weight, adaln_scale, adaln_scale.stride(0),
                    adaln_shift, adaln_shift.stride(0), adaln_scale.shape[0], adaln_index,
                    qkv_weight, q_norm_weight, k_norm_weight, rope_cos_sin, rope_cos_sin.shape[0],
                    rope_positions, P, eps, qk_eps, workspace, out)
    return out

