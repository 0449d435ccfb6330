"""Oracle of ``flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention``.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Each function follows one step of the stage as the pages define it:

* input RMSNorm and indexed AdaLN: the formula block of
  ``flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120`` (lines ``n = ...``,
  ``a = ...``, ``a[i outside [0, rows)] = 0``), which the BF16 page shares
  (its summary lists the same input RMSNorm and indexed AdaLN);
* QKV projection with FP32 accumulation: ``minimax_h3_bf16_pre_attention``
  summary and Parameters: qkv_weight (row order [qkv_kind, head, head_dim]);
* per-head Q/K RMSNorm: summary, Parameters: q_norm_weight / k_norm_weight /
  qk_eps;
* partial split-half NeoX RoPE on dims [0, 96): Parameters: rope_cos_sin and
  rope_positions (clamp, identity);
* destination-major pack: Parameters: out ([P, M, 56 // P, 3, 128]) and
  ulysses_degree.

Readings where the pages are silent (each listed in the design notes):
the sum of squares is the exact sum rounded once to FP32; ``rmsnorm(x)*w`` is
``(x * r) * w`` with ``r = 1 / sqrt(ss / H + eps)``; AdaLN is an unfused
multiply then add; the QKV accumulator is rounded to BF16 before the Q/K
norm; the normalised head is rounded to BF16 before RoPE; the rotation pairs
(j, j + 48) with cos in column j and sin in column 48 + j; destination
``p`` owns the contiguous head block [p * 56/P, (p + 1) * 56/P).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import torch

F32 = torch.float32
F64 = torch.float64
BF16 = torch.bfloat16


def _f32_scalar(v: float) -> torch.Tensor:
    return torch.tensor(float(v), dtype=F32)


def _ideal_fp32_sum_of_squares(v_f32: torch.Tensor) -> torch.Tensor:
    """Sum of squares over the last dim: exact (float64) then rounded to FP32."""
    return (v_f32.to(F64) * v_f32.to(F64)).sum(-1).to(F32)


def _rms_scale(ss: torch.Tensor, width: int, eps: float) -> torch.Tensor:
    """r = 1 / sqrt(ss / width + eps), each step an FP32 operation."""
    ms = torch.div(ss, _f32_scalar(width))
    v = torch.add(ms, _f32_scalar(eps))
    return torch.div(torch.ones_like(v), torch.sqrt(v))


def input_rmsnorm(x: torch.Tensor, x_norm_weight: torch.Tensor, eps: float) -> torch.Tensor:
    """n = bf16(rmsnorm(x, eps) * x_norm_weight), FP32 sum of squares.

    x: bf16 [M, H]; x_norm_weight: bf16 [H].  Returns bf16 [M, H].
    """
    H = x.shape[-1]
    xf = x.to(F32)
    r = _rms_scale(_ideal_fp32_sum_of_squares(xf), H, eps)
    return torch.mul(torch.mul(xf, r[..., None]), x_norm_weight.to(F32)).to(BF16)


def indexed_adaln(n: torch.Tensor, adaln_scale: torch.Tensor, adaln_shift: torch.Tensor,
                  adaln_index: torch.Tensor) -> torch.Tensor:
    """a = bf16(shift[i] + n * bf16(1 + scale[i])), i = adaln_index[m];
    rows whose i lies outside [0, rows) are all zero (+0.0).

    n: bf16 [M, H]; adaln_scale / adaln_shift: bf16 [rows, H] (any row stride);
    adaln_index: int64 [M].  Returns bf16 [M, H].
    """
    rows = adaln_scale.shape[0]
    M, H = n.shape
    a = torch.zeros((M, H), dtype=BF16)
    valid = (adaln_index >= 0) & (adaln_index < rows)
    if bool(valid.any()):
        i = adaln_index[valid]
        g = torch.add(adaln_scale[i].to(F32), 1.0).to(BF16)
        prod = torch.mul(n[valid].to(F32), g.to(F32))
        a[valid] = torch.add(adaln_shift[i].to(F32), prod).to(BF16)
    return a


def qkv_projection(a: torch.Tensor, qkv_weight: torch.Tensor) -> torch.Tensor:
    """y = bf16(acc), acc[m, c] = sum_k a[m, k] * W[c, k] as an FP32 value.

    The products of two bf16 values are exact in float64 and the float64 sum
    of H of them is far inside FP32 resolution, so ``acc`` is the exact dot
    product rounded once to FP32.  a: bf16 [M, H]; W: bf16 [N, H].
    """
    acc = torch.matmul(a.to(F64), qkv_weight.to(F64).t()).to(F32)
    return acc.to(BF16)


def head_rmsnorm(y_heads: torch.Tensor, norm_weight: torch.Tensor, qk_eps: float) -> torch.Tensor:
    """t = bf16((y * rr) * w), rr = 1 / sqrt(sum_d y_d^2 / D + qk_eps), per head.

    y_heads: bf16 [..., D]; norm_weight: bf16 [D] (shared by all heads).
    """
    D = y_heads.shape[-1]
    yf = y_heads.to(F32)
    rr = _rms_scale(_ideal_fp32_sum_of_squares(yf), D, qk_eps)
    return torch.mul(torch.mul(yf, rr[..., None]), norm_weight.to(F32)).to(BF16)


def rope_cache_rows(positions: Optional[torch.Tensor], tokens: torch.Tensor, S: int) -> torch.Tensor:
    """Cache row of each token: clamp(positions[m], 0, S-1) in int64, or the
    identity m when positions is None (which requires S >= M; checked by the
    caller).  ``tokens`` are the token ids m being evaluated."""
    if positions is None:
        return tokens.to(torch.int64)
    p = positions[tokens].to(torch.int64)
    return torch.clamp(p, 0, S - 1)


def rope_split_half(t: torch.Tensor, cos_sin: torch.Tensor, rows: torch.Tensor) -> torch.Tensor:
    """Partial split-half NeoX rotation of the first RD = cos_sin.shape[1] dims.

    For j < RD/2 with c = cos_sin[p, j], s = cos_sin[p, RD/2 + j]:
      o_j        = bf16(t_j * c - t_{j+RD/2} * s)
      o_{j+RD/2} = bf16(t_{j+RD/2} * c + t_j * s)
    and o_d = t_d for d >= RD.  t: bf16 [T, heads, D]; rows: int64 [T].
    """
    RD = cos_sin.shape[1]
    half = RD // 2
    cs = cos_sin[rows].to(F32)
    c = cs[:, None, :half]
    s = cs[:, None, half:RD]
    tf = t.to(F32)
    t1 = tf[..., :half]
    t2 = tf[..., half:RD]
    o1 = torch.sub(torch.mul(t1, c), torch.mul(t2, s)).to(BF16)
    o2 = torch.add(torch.mul(t2, c), torch.mul(t1, s)).to(BF16)
    return torch.cat([o1, o2, t[..., RD:]], dim=-1)


def ulysses_pack(tokens_qkv: torch.Tensor, P: int) -> torch.Tensor:
    """[M, NH, 3, D] (kind order q, k, v) -> out [P, M, NH/P, 3, D] with
    head h going to destination h // (NH/P), local head h % (NH/P)."""
    M, NH, K3, D = tokens_qkv.shape
    assert NH % P == 0
    return tokens_qkv.reshape(M, P, NH // P, K3, D).permute(1, 0, 2, 3, 4).contiguous()


def ulysses_unpack_rows(out: torch.Tensor, tokens: Sequence[int]) -> torch.Tensor:
    """Inverse of the pack for selected tokens: out [P, M, NH/P, 3, D] ->
    [len(tokens), NH, 3, D]."""
    P, M, hp, K3, D = out.shape
    idx = torch.as_tensor(list(tokens), dtype=torch.int64, device=out.device)
    sel = out.index_select(1, idx)  # [P, T, hp, 3, D]
    return sel.permute(1, 0, 2, 3, 4).reshape(len(tokens), P * hp, K3, D)


@dataclass
class PreAttnTokens:
    tokens: torch.Tensor  # int64 [T] token ids evaluated
    n: torch.Tensor  # bf16 [T, H]   input RMSNorm output
    a: torch.Tensor  # bf16 [T, H]   workspace (AdaLN output)
    y: torch.Tensor  # bf16 [T, N]   QKV projection
    qkv: torch.Tensor  # bf16 [T, NH, 3, D] per-token outputs before the pack


def pre_attention_tokens(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index, qkv_weight,
                         q_norm_weight, k_norm_weight, rope_cos_sin, *, eps: float = 1e-5,
                         qk_eps: Optional[float] = None, rope_positions=None,
                         tokens: Optional[Sequence[int]] = None) -> PreAttnTokens:
    """Run every step for the given tokens (default: all M).  Rows are
    independent, so any subset is exact."""
    M = x.shape[0]
    S = rope_cos_sin.shape[0]
    if rope_positions is None and S < M:
        raise ValueError("identity positions need S >= M")
    if tokens is None:
        tok = torch.arange(M, dtype=torch.int64)
    else:
        tok = torch.as_tensor(list(tokens), dtype=torch.int64)
    qk = eps if qk_eps is None else qk_eps
    D = q_norm_weight.shape[0]
    N = qkv_weight.shape[0]
    NH = N // (3 * D)

    n = input_rmsnorm(x[tok], x_norm_weight, eps)
    a = indexed_adaln(n, adaln_scale, adaln_shift, adaln_index[tok])
    y = qkv_projection(a, qkv_weight)
    yk = y.reshape(len(tok), 3, NH, D)  # [q_all | k_all | v_all], each [head, d]
    rows = rope_cache_rows(rope_positions, tok, S)
    q = rope_split_half(head_rmsnorm(yk[:, 0], q_norm_weight, qk), rope_cos_sin, rows)
    k = rope_split_half(head_rmsnorm(yk[:, 1], k_norm_weight, qk), rope_cos_sin, rows)
    v = yk[:, 2]
    qkv = torch.stack([q, k, v], dim=2)  # [T, NH, 3, D]
    return PreAttnTokens(tokens=tok, n=n, a=a, y=y, qkv=qkv)


def pre_attention(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index, qkv_weight,
                  q_norm_weight, k_norm_weight, rope_cos_sin, *, ulysses_degree: int,
                  eps: float = 1e-5, qk_eps: Optional[float] = None, rope_positions=None):
    """The whole stage: returns out [P, M, NH/P, 3, D] (bf16) and the workspace a."""
    r = pre_attention_tokens(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index,
                             qkv_weight, q_norm_weight, k_norm_weight, rope_cos_sin,
                             eps=eps, qk_eps=qk_eps, rope_positions=rope_positions)
    return ulysses_pack(r.qkv, ulysses_degree), r.a
