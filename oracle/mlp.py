"""Oracle of the MiniMax-H3 MLP block, with BF16 operands.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the formula block of ``flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120``
without its FP8 quantisation lines (the weights and activations stay bf16):

    n   = bf16(rmsnorm(x, eps) * x_norm_weight)
    a   = bf16(adaln_shift[i] + n * bf16(1 + adaln_scale[i]))   (0 for a bad i)
    h   = bf16(a @ fc1_weight^T)              FP32 accumulation, [M, 28672]
    y   = bf16(bf16(silu(h_gate)) * h_up)     [M, 14336]
    o   = bf16(y @ fc2_weight^T)              FP32 accumulation, [M, 5376]
    out = bf16(residual + bf16(gate[i] * o))  (gate 0 for a bad i: out = residual)

Readings where the page is silent: h_gate is columns [0, 14336) of h and
h_up columns [14336, 28672) (the order the SwiGLU line names them);
silu(v) = v / (1 + exp(-v)) evaluated exactly and rounded once to FP32
before the bf16 rounding; the product bf16(silu) * h_up is one FP32
multiply.  The norm/AdaLN, projection and gated-residual steps are the ones
of oracle.preattn and oracle.out_proj.
"""
from __future__ import annotations

import torch

from .out_proj import gated_residual, out_projection
from .stage import indexed_adaln, input_rmsnorm

F32 = torch.float32
F64 = torch.float64
BF16 = torch.bfloat16


def swiglu(h: torch.Tensor) -> torch.Tensor:
    """y = bf16(bf16(silu(h_gate)) * h_up) for h = [h_gate | h_up] (bf16 [M, 2I])."""
    inter = h.shape[-1] // 2
    hg = h[..., :inter].to(F64)
    s = (hg / (1.0 + torch.exp(-hg))).to(F32).to(BF16)
    return torch.mul(s.to(F32), h[..., inter:].to(F32)).to(BF16)


def mlp_block(x, x_norm_weight, adaln_scale, adaln_shift, gate, adaln_index, residual,
              fc1_weight, fc2_weight, *, eps: float = 1e-5, tokens=None):
    """The whole block for the given tokens (default: all M); returns
    (out [T, 5376], a [T, 5376], y [T, I])."""
    if tokens is not None:
        idx = torch.as_tensor(list(tokens), dtype=torch.int64)
        x, adaln_index, residual = x[idx], adaln_index[idx], residual[idx]
    n = input_rmsnorm(x, x_norm_weight, eps)
    a = indexed_adaln(n, adaln_scale, adaln_shift, adaln_index)
    y = swiglu(out_projection(a, fc1_weight))
    out = gated_residual(out_projection(y, fc2_weight), gate, adaln_index, residual)
    return out, a, y
