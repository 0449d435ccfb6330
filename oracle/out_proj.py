"""Oracle of the attention output projection with the fused gated residual.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows ``flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj`` (summary:
``out = BF16(residual + BF16(gate[gate_index[m]] * o))``; rows whose
gate_index lies outside [0, rows) contribute gate = 0, so out = residual;
Parameters: attn_out [M, 7168], gate [9, 5376] rows of the AdaLN plan,
gate_index int32 [M], residual [M, 5376]), computed here with BF16 operands
instead of that page's NVFP4 ones.

Readings where the page is silent: ``o`` is the FP32 accumulator rounded to
bf16, as the ``o = bf16(...)`` line of the formula block of
``minimax_h3_mlp_fp8_sm120`` (whose last line is this same gated residual);
``gate * o`` is one FP32 multiply rounded to bf16 and the residual add one
FP32 add rounded to bf16.
"""
from __future__ import annotations

import torch

F32 = torch.float32
F64 = torch.float64
BF16 = torch.bfloat16


def out_projection(attn_out: torch.Tensor, o_weight: torch.Tensor) -> torch.Tensor:
    """o = bf16(acc), acc[m, c] = sum_k attn_out[m, k] * W[c, k] as an FP32
    value (exact float64 sum rounded once).  attn_out bf16 [M, K]; W bf16 [N, K]."""
    acc = torch.matmul(attn_out.to(F64), o_weight.to(F64).t()).to(F32)
    return acc.to(BF16)


def gated_residual(o: torch.Tensor, gate: torch.Tensor, gate_index: torch.Tensor,
                   residual: torch.Tensor) -> torch.Tensor:
    """out = bf16(residual + bf16(g * o)), g = gate[gate_index[m]], or 0 for
    an index outside [0, rows).  o, residual bf16 [M, N]; gate bf16 [rows, N]
    (any row stride); gate_index int [M]."""
    rows = gate.shape[0]
    M, N = o.shape
    g = torch.zeros((M, N), dtype=F32)
    valid = (gate_index >= 0) & (gate_index < rows)
    if bool(valid.any()):
        g[valid] = gate[gate_index[valid].to(torch.int64)].to(F32)
    go = torch.mul(g, o.to(F32)).to(BF16)
    return torch.add(residual.to(F32), go.to(F32)).to(BF16)


def out_proj_gated_residual(attn_out, o_weight, gate, gate_index, residual, tokens=None):
    """The whole operation for the given tokens (default: all M)."""
    if tokens is not None:
        idx = torch.as_tensor(list(tokens), dtype=torch.int64)
        attn_out, gate_index, residual = attn_out[idx], gate_index[idx], residual[idx]
    return gated_residual(out_projection(attn_out, o_weight), gate, gate_index, residual)
