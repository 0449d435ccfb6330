"""Python face of the C++ oracle (``oracle/cpp/mh3_oracle.cpp``).

TEST INFRASTRUCTURE ONLY (see the package docstring).  This module only moves
tensors in and out of the C++ functions: every step of the stage is computed
in C++.  Inputs are CPU tensors (bf16 values are passed as their bit
patterns); outputs are new CPU tensors.

Steps (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention, summary and
Parameters; the first two with the formula block of
flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120): input RMSNorm, indexed
AdaLN with the int64 guard, QKV projection with FP32 accumulation, per-head
Q/K RMSNorm, partial split-half RoPE with clamped positions, and the
destination-major pack.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import build as _build

BF16 = torch.bfloat16
_P = ctypes.c_void_p
_I = ctypes.c_int64
_F = ctypes.c_float

_lib = None


def lib() -> ctypes.CDLL:
    """The oracle library, compiled on first use."""
    global _lib
    if _lib is None:
        L = ctypes.CDLL(_build.build())
        sig = {
            "mh3o_input_rmsnorm": [_P, _I, _I, _P, _F, _P, _P],
            "mh3o_rmsnorm_apply": [_P, _I, _I, _P, _P, _P],
            "mh3o_indexed_adaln": [_P, _I, _I, _P, _I, _P, _I, _I, _P, _P],
            "mh3o_qkv_projection": [_P, _I, _I, _P, _I, _P],
            "mh3o_head_rmsnorm": [_P, _I, _I, _P, _F, _P],
            "mh3o_rope_cache_rows": [_P, _P, _I, _I, _P],
            "mh3o_rope_split_half": [_P, _I, _I, _I, _P, _I, _P, _P],
            "mh3o_ulysses_pack": [_P, _I, _I, _I, _I, _P],
            "mh3o_pre_attention_tokens": [_P, _I, _I, _P, _P, _I, _P, _I, _I, _P, _P, _I, _I,
                                          _P, _P, _P, _I, _I, _P, _F, _F, _P, _I, _P, _P, _P,
                                          _P, _P],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int if name == "mh3o_pre_attention_tokens" else None
        L.mh3o_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def threads() -> int:
    return int(lib().mh3o_max_threads())


def _bits(t: torch.Tensor) -> torch.Tensor:
    """Contiguous CPU int16 view of a bf16 tensor (its bit patterns)."""
    assert t.dtype == BF16, t.dtype
    return t.detach().cpu().contiguous().view(torch.int16)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _table(t: torch.Tensor):
    """(bits tensor, base pointer, row stride) of a [rows, H] table view whose
    rows may be strided (a column chunk of a wider tensor)."""
    assert t.dtype == BF16 and t.dim() == 2 and t.stride(1) == 1
    t = t.detach().cpu()
    base = t.view(torch.int16)
    return base, ctypes.c_void_p(base.data_ptr()), int(t.stride(0))


def _i64(t: torch.Tensor) -> torch.Tensor:
    return t.detach().cpu().to(torch.int64).contiguous()


# ------------------------------------------------------------------- steps
def input_rmsnorm(x: torch.Tensor, x_norm_weight: torch.Tensor, eps: float,
                  return_r: bool = False):
    """n = bf16((x * r) * w), r = 1 / sqrt(ss / H + eps), ss the FP32 sum of
    squares.  x: bf16 [..., H]; returns bf16 like x (and r, FP32 per row)."""
    shape = x.shape
    H = shape[-1]
    xb = _bits(x).reshape(-1, H)
    T = xb.shape[0]
    n = torch.empty((T, H), dtype=torch.int16)
    r = torch.empty((T,), dtype=torch.float32)
    lib().mh3o_input_rmsnorm(_ptr(xb), T, H, _ptr(_bits(x_norm_weight)), float(eps), _ptr(n),
                             _ptr(r))
    n = n.view(BF16).reshape(shape)
    return (n, r.reshape(shape[:-1])) if return_r else n


def rmsnorm_apply(x: torch.Tensor, x_norm_weight: torch.Tensor, r: torch.Tensor) -> torch.Tensor:
    """n = bf16((x * r) * w) for a given FP32 r per row."""
    H = x.shape[-1]
    xb = _bits(x).reshape(-1, H)
    T = xb.shape[0]
    rr = r.detach().cpu().to(torch.float32).contiguous().reshape(T)
    n = torch.empty((T, H), dtype=torch.int16)
    lib().mh3o_rmsnorm_apply(_ptr(xb), T, H, _ptr(_bits(x_norm_weight)), _ptr(rr), _ptr(n))
    return n.view(BF16).reshape(x.shape)


def indexed_adaln(n: torch.Tensor, adaln_scale: torch.Tensor, adaln_shift: torch.Tensor,
                  adaln_index: torch.Tensor) -> torch.Tensor:
    """a = bf16(shift[i] + n * bf16(1 + scale[i])), i = adaln_index[t]; rows
    with i outside [0, rows) are +0.  Tables may have any row stride."""
    T, H = n.shape
    sc_keep, sc, ss = _table(adaln_scale)
    sh_keep, sh, shs = _table(adaln_shift)
    idx = _i64(adaln_index)
    a = torch.empty((T, H), dtype=torch.int16)
    lib().mh3o_indexed_adaln(_ptr(_bits(n)), T, H, sc, ss, sh, shs, adaln_scale.shape[0],
                             _ptr(idx), _ptr(a))
    del sc_keep, sh_keep
    return a.view(BF16)


def qkv_projection(a: torch.Tensor, qkv_weight: torch.Tensor) -> torch.Tensor:
    """y = bf16(FP32(sum_k a[t, k] * W[c, k])).  a: [T, K]; W: [N, K]."""
    T, K = a.shape
    N = qkv_weight.shape[0]
    y = torch.empty((T, N), dtype=torch.int16)
    lib().mh3o_qkv_projection(_ptr(_bits(a)), T, K, _ptr(_bits(qkv_weight)), N, _ptr(y))
    return y.view(BF16)


def head_rmsnorm(y_heads: torch.Tensor, norm_weight: torch.Tensor, qk_eps: float) -> torch.Tensor:
    """t = bf16((y * rr) * w) per head vector (last dim D)."""
    D = y_heads.shape[-1]
    yb = _bits(y_heads).reshape(-1, D)
    t = torch.empty_like(yb)
    lib().mh3o_head_rmsnorm(_ptr(yb), yb.shape[0], D, _ptr(_bits(norm_weight)), float(qk_eps),
                            _ptr(t))
    return t.view(BF16).reshape(y_heads.shape)


def rope_cache_rows(positions: Optional[torch.Tensor], tokens: torch.Tensor, S: int) -> torch.Tensor:
    """clamp(positions[tok], 0, S - 1) in int64, or tok when positions is None."""
    tok = _i64(tokens)
    out = torch.empty_like(tok)
    pos = None if positions is None else _i64(positions)
    lib().mh3o_rope_cache_rows(_ptr(pos), _ptr(tok), tok.numel(), int(S), _ptr(out))
    return out


def rope_split_half(t: torch.Tensor, cos_sin: torch.Tensor, rows: torch.Tensor) -> torch.Tensor:
    """Split-half rotation of the first RD = cos_sin.shape[1] dims of each
    head.  t: bf16 [T, heads, D]; rows: int64 [T] cache rows."""
    T, heads, D = t.shape
    RD = cos_sin.shape[1]
    tb = _bits(t)
    o = torch.empty_like(tb)
    lib().mh3o_rope_split_half(_ptr(tb), T, heads, D, _ptr(_bits(cos_sin)), RD,
                               _ptr(_i64(rows)), _ptr(o))
    return o.view(BF16)


def ulysses_pack(tokens_qkv: torch.Tensor, P: int) -> torch.Tensor:
    """[M, NH, 3, D] -> out [P, M, NH/P, 3, D], head h to destination
    h // (NH/P), local head h % (NH/P)."""
    M, NH, K3, D = tokens_qkv.shape
    assert K3 == 3 and NH % P == 0
    out = torch.empty((P, M, NH // P, 3, D), dtype=torch.int16)
    lib().mh3o_ulysses_pack(_ptr(_bits(tokens_qkv)), M, NH, D, P, _ptr(out))
    return out.view(BF16)


def ulysses_unpack_rows(out: torch.Tensor, tokens: Sequence[int]) -> torch.Tensor:
    """Gather the per-token rows of a packed output back to [T, NH, 3, D]
    (data movement only, for comparing outputs token by token)."""
    P, M, hp, K3, D = out.shape
    idx = torch.as_tensor(list(tokens), dtype=torch.int64, device=out.device)
    sel = out.index_select(1, idx)
    return sel.permute(1, 0, 2, 3, 4).reshape(len(tokens), P * hp, K3, D)


# ------------------------------------------------------------- whole stage
@dataclass
class PreAttnTokens:
    tokens: torch.Tensor  # int64 [T] token ids evaluated
    n: torch.Tensor  # bf16 [T, H]   input RMSNorm output
    a: torch.Tensor  # bf16 [T, H]   workspace (AdaLN output)
    y: torch.Tensor  # bf16 [T, N]   QKV projection
    qkv: torch.Tensor  # bf16 [T, NH, 3, D] per-token outputs before the pack
    r: Optional[torch.Tensor] = None  # FP32 [T] input RMSNorm scale


def pre_attention_tokens(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index, qkv_weight,
                         q_norm_weight, k_norm_weight, rope_cos_sin, *, eps: float = 1e-5,
                         qk_eps: Optional[float] = None, rope_positions=None,
                         tokens: Optional[Sequence[int]] = None) -> PreAttnTokens:
    """Every step for the given tokens (default: all M).  Tokens are
    independent, so any subset is exact.  qk_eps None uses eps."""
    M, H = x.shape
    S, RD = rope_cos_sin.shape
    D = q_norm_weight.shape[0]
    N = qkv_weight.shape[0]
    NH = N // (3 * D)
    if rope_positions is None and S < M:
        raise ValueError("identity positions need S >= M")
    tok = torch.arange(M, dtype=torch.int64) if tokens is None else \
        torch.as_tensor(list(tokens), dtype=torch.int64)
    T = tok.numel()
    qk = eps if qk_eps is None else qk_eps
    xb = _bits(x)
    sc_keep, sc, ss = _table(adaln_scale)
    sh_keep, sh, shs = _table(adaln_shift)
    idx = _i64(adaln_index)
    pos = None if rope_positions is None else _i64(rope_positions)
    n = torch.empty((T, H), dtype=torch.int16)
    a = torch.empty((T, H), dtype=torch.int16)
    y = torch.empty((T, N), dtype=torch.int16)
    qkv = torch.empty((T, NH, 3, D), dtype=torch.int16)
    r = torch.empty((T,), dtype=torch.float32)
    rc = lib().mh3o_pre_attention_tokens(
        _ptr(xb), M, H, _ptr(_bits(x_norm_weight)), sc, ss, sh, shs, adaln_scale.shape[0],
        _ptr(idx), _ptr(_bits(qkv_weight)), NH, D, _ptr(_bits(q_norm_weight)),
        _ptr(_bits(k_norm_weight)), _ptr(_bits(rope_cos_sin)), S, RD, _ptr(pos), float(eps),
        float(qk), _ptr(tok), T, _ptr(n), _ptr(a), _ptr(y), _ptr(qkv), _ptr(r))
    del sc_keep, sh_keep
    if rc != 0:
        raise ValueError("identity positions need S >= M")
    return PreAttnTokens(tokens=tok, n=n.view(BF16), a=a.view(BF16), y=y.view(BF16),
                         qkv=qkv.view(BF16), r=r)


def pre_attention(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index, qkv_weight,
                  q_norm_weight, k_norm_weight, rope_cos_sin, *, ulysses_degree: int,
                  eps: float = 1e-5, qk_eps: Optional[float] = None, rope_positions=None):
    """The whole stage: out [P, M, NH/P, 3, D] (bf16) and the workspace a."""
    r = pre_attention_tokens(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index,
                             qkv_weight, q_norm_weight, k_norm_weight, rope_cos_sin,
                             eps=eps, qk_eps=qk_eps, rope_positions=rope_positions)
    return ulysses_pack(r.qkv, ulysses_degree), r.a
