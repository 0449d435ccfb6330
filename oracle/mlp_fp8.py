"""Oracle of the MiniMax-H3 FP8 (W8A8) MLP block.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the formula block of ``flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120``:

    n   = bf16(rmsnorm(x, eps) * x_norm_weight)
    a   = bf16(adaln_shift[i] + n * bf16(1 + adaln_scale[i]))    (0 for a bad i)
    a_q = e4m3(a / s_a),  s_a = RN(amax_row(|a|) / 448)          per token
    h   = bf16(a_q @ fc1_weight_q^T * s_a * fc1_weight_scale)     FP32 accumulation
    y   = bf16(bf16(silu(h_gate)) * h_up)
    y_q = e4m3(y / s_y),  s_y = RN(amax_row(|y|) / 448)          per token
    o   = bf16(y_q @ fc2_weight_q^T * s_y * fc2_weight_scale)     FP32 accumulation
    out = bf16(residual + bf16(gate[i] * o))                       (gate 0 for a bad i)

Readings where the page is silent:
* s = RN(amax / 448) is one FP32 division (amax is a bf16 value);
* e4m3(v / s) is one rounding of the exact quotient to e4m3 (nearest even,
  saturating at +-448; a negative value that rounds to zero gives -0); a row
  whose amax is 0 has s = 0 and codes +0.  The quotient is formed in float64:
  its one float64 rounding cannot move it across or onto an e4m3 rounding
  boundary (a bf16 numerator over an FP32 divisor that is not on a boundary
  lies at least 2^-32 of its size away from it, far more than 2^-53);
* the GEMMs sum the exact products of the e4m3 values (exact in float64),
  the sum rounded once to FP32 (acc); the two scale factors multiply in the
  printed order, each product one FP32 rounding:
  h = bf16(RN(RN(acc * s_a) * w_scale[c]));
* fc1's rows are [gate (14336) | up (14336)] with one FP32 scale per row,
  fc2's one scale per output row; silu and the gated residual are those of
  the BF16 block (oracle.mlp, oracle.out_proj).
"""
from __future__ import annotations

import torch

from .mlp import swiglu
from .out_proj import gated_residual
from .stage import indexed_adaln, input_rmsnorm

F32 = torch.float32
F64 = torch.float64
BF16 = torch.bfloat16
E4M3_MAX = 448.0


def e4m3_round(v: torch.Tensor) -> torch.Tensor:
    """Nearest e4m3 value of float64 values, ties to even, saturating at
    +-448 (three fraction bits at exponents >= -6, steps of 2^-9 below);
    the sign is kept on zero.  Returns float64."""
    v = v.to(F64)
    mag = v.abs()
    _, e = torch.frexp(mag)                          # mag = f * 2^e, f in [0.5, 1)
    lead = torch.clamp(e - 1, min=-6)
    step = torch.pow(2.0, (lead - 3).to(F64))
    q = torch.round(mag / step) * step               # exact scaling; round() ties to even
    q = torch.where(mag == 0, torch.zeros_like(q), torch.clamp(q, max=E4M3_MAX))
    return torch.where(torch.signbit(v), -q, q)


def e4m3_codes(v: torch.Tensor) -> torch.Tensor:
    """uint8 e4m3 (float8_e4m3fn) bit patterns of values already on the e4m3 grid."""
    return v.to(F32).to(torch.float8_e4m3fn).view(torch.uint8)


def e4m3_values(codes: torch.Tensor) -> torch.Tensor:
    return codes.view(torch.float8_e4m3fn).to(F64)


def row_scale(v: torch.Tensor) -> torch.Tensor:
    """s = RN(amax_row(|v|) / 448), FP32 [T], for bf16 v [T, K]."""
    amax = v.to(F32).abs().amax(dim=-1)
    return torch.div(amax, torch.tensor(E4M3_MAX, dtype=F32))


def quantize_rows(v: torch.Tensor):
    """(codes uint8 [T, K], s FP32 [T]): e4m3(v / s) per row with its scale."""
    s = row_scale(v)
    sd = s.to(F64).unsqueeze(-1)
    q = torch.where(sd == 0, v.to(F64) * 0.0, v.to(F64) / torch.where(sd == 0, 1.0, sd))
    q = torch.where(sd == 0, torch.zeros_like(q), q)  # an all-zero row: codes +0
    return e4m3_codes(e4m3_round(q)), s


def scaled_projection(codes: torch.Tensor, s_row: torch.Tensor, w_codes: torch.Tensor,
                      w_scale: torch.Tensor) -> torch.Tensor:
    """bf16(RN(RN(acc * s_row[m]) * w_scale[c])), acc = sum_k a[m,k] w[c,k]
    of the e4m3 values, exact, rounded once to FP32.  Returns bf16 [T, N]."""
    acc = (e4m3_values(codes) @ e4m3_values(w_codes).T).to(F32)
    t = torch.mul(acc, s_row.to(F32).unsqueeze(-1))
    return torch.mul(t, w_scale.to(F32).unsqueeze(0)).to(BF16)


def mlp_block_fp8(x, x_norm_weight, adaln_scale, adaln_shift, gate, adaln_index, residual,
                  fc1_q, fc1_scale, fc2_q, fc2_scale, *, eps: float = 1e-5, tokens=None):
    """The whole block for the given tokens (default: all M).  Returns a dict
    with out [T, 5376] and the intermediates a, a_q, s_a, y, y_q, s_y."""
    if tokens is not None:
        idx = torch.as_tensor(list(tokens), dtype=torch.int64)
        x, adaln_index, residual = x[idx], adaln_index[idx], residual[idx]
    n = input_rmsnorm(x, x_norm_weight, eps)
    a = indexed_adaln(n, adaln_scale, adaln_shift, adaln_index)
    a_q, s_a = quantize_rows(a)
    y = swiglu(scaled_projection(a_q, s_a, fc1_q, fc1_scale))
    y_q, s_y = quantize_rows(y)
    o = scaled_projection(y_q, s_y, fc2_q, fc2_scale)
    out = gated_residual(o, gate, adaln_index, residual)
    return dict(out=out, a=a, a_q=a_q, s_a=s_a, y=y, y_q=y_q, s_y=s_y)
