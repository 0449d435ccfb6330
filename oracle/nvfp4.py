"""Oracle of the NVFP4 pre-attention stage.

TEST INFRASTRUCTURE ONLY (see the package docstring).

flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention, summary and
Parameters: the same pre-norm and AdaLN as the bf16 stage; the normalised
activation a is quantised per token to NVFP4 (E2M1 codes, two per byte,
[M, 2688], and one UE4M3 scale per block of 16, [M, 336]) with the
activation global scale; the weight is quantised the same way with its own
global scale; the accumulator is rescaled by alpha = 1 / (act_global_scale *
qkv_weight_global_scale); then the bf16 stage's Q/K norm (with eps), RoPE
(rope_cos_sin is per token, [M, 96]) and outputs.

The block quantisation is the FlashInfer block-16 convention that
flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj prints in its summary:
  sf   = UE4M3(block_amax * act_global_scale / 6)
  code = RN(x * act_global_scale / sf)
each a single rounding of the exact quotient.  Readings:
* UE4M3 and E2M1 rounding is to nearest, ties to even; UE4M3 saturates at
  448, E2M1 at 6; E2M1 keeps the sign (a negative value that rounds to 0
  gives -0); where sf = 0 (the whole block rounds to a zero scale) the codes
  are the signed zeros of x * 0;
* the exact quotients are formed in float64: block_amax * gs and x * gs are
  exact there (8 + 24 significant bits), and the one float64 rounding of the
  division cannot move a value across, or onto, a UE4M3 or E2M1 rounding
  boundary: those boundaries (times 6, or times sf) have at most 7
  significant bits, so a numerator of at most 32 significant bits that is
  not equal to one differs from it by at least 2^-32 of its size, far more
  than a float64 rounding step (2^-53);
* packing: byte j holds elements 2j (low nibble) and 2j + 1 (high nibble);
* the GEMM sums the products (qa sa)(qw sw) exactly and rounds once to FP32
  (the FP32 accumulation of the bf16 stage's reading), then
  y = bf16(RN32(alpha * acc));
* the Q/K RMSNorm uses eps (the op has no separate qk_eps); positions are the
  token index (one cos/sin row per token).
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from .stage import (PreAttnTokens, head_rmsnorm, indexed_adaln, input_rmsnorm,
                    rope_split_half)

F32 = torch.float32
F64 = torch.float64
BF16 = torch.bfloat16
E2M1_VALUES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
UE4M3_MAX = 448.0
BLOCK = 16


def e2m1_codes(x: torch.Tensor) -> torch.Tensor:
    """4-bit E2M1 codes (uint8 0..15, sign in bit 3) of FP32/FP64 values:
    nearest of E2M1_VALUES by magnitude, ties to the even code, saturating."""
    mag = x.abs().to(F64)
    vals = torch.tensor(E2M1_VALUES, dtype=F64)
    d = (mag.unsqueeze(-1) - vals).abs()                       # distance to each value
    best = d.min(dim=-1, keepdim=True).values
    cand = d == best                                            # one or two nearest
    codes = torch.arange(8, dtype=torch.int64)
    # among equally near values take the even code (mantissa bit 0)
    score = torch.where(cand, (codes % 2) * 16 + codes, torch.full_like(codes, 1000))
    c = score.argmin(dim=-1)
    sign = torch.signbit(x.to(F64)).to(torch.int64)
    return (c + 8 * sign).to(torch.uint8)


def e2m1_values(codes: torch.Tensor) -> torch.Tensor:
    vals = torch.tensor(E2M1_VALUES, dtype=F64)
    c = codes.to(torch.int64)
    v = vals[c & 7]
    return torch.where((c & 8) != 0, -v, v)


def ue4m3_round(v: torch.Tensor) -> torch.Tensor:
    """Nearest UE4M3 value of non-negative float64 values, ties to even,
    saturating at 448: three fraction bits at exponents >= -6, steps of 2^-9
    below (subnormals).  Returns float64 values."""
    v = v.to(F64)
    _, e = torch.frexp(v)                         # v = f * 2^e, f in [0.5, 1)
    lead = torch.clamp(e - 1, min=-6)             # exponent of the leading bit
    step = torch.pow(2.0, (lead - 3).to(F64))     # spacing of UE4M3 values there
    q = torch.round(v / step) * step              # exact scaling; round() ties to even
    return torch.clamp(torch.where(v == 0, torch.zeros_like(v), q), max=UE4M3_MAX)


def ue4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """UE4M3 codes of non-negative values (rounded by ue4m3_round)."""
    return ue4m3_round(x.to(F64)).to(F32).to(torch.float8_e4m3fn).view(torch.uint8)


def ue4m3_values(codes: torch.Tensor) -> torch.Tensor:
    return codes.view(torch.float8_e4m3fn).to(F32)


def fp4_quantize(a: torch.Tensor, global_scale: float):
    """Per-row NVFP4 quantisation of bf16 a [T, K] (K a multiple of 16).
    Returns (codes uint8 [T, K/2] packed, scales uint8 [T, K/16] row-major).

    sf = UE4M3(amax * gs / 6) and code = E2M1(x * gs / sf), each one rounding
    of the exact quotient (see the module docstring)."""
    T, K = a.shape
    gs = float(torch.tensor(float(global_scale), dtype=F32))  # the FP32 value
    blocks = a.to(F64).reshape(T, K // BLOCK, BLOCK)
    amax = blocks.abs().amax(dim=-1)
    s = ue4m3_round((amax * gs) / 6.0)            # amax * gs exact; one rounding
    s_code = s.to(F32).to(torch.float8_e4m3fn).view(torch.uint8)
    sv = s.unsqueeze(-1)
    v = torch.where(sv == 0, blocks * 0.0, (blocks * gs) / torch.where(sv == 0, 1.0, sv))
    q = e2m1_codes(v).reshape(T, K)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).to(torch.uint8)
    return packed, s_code


def unpack_codes(packed: torch.Tensor) -> torch.Tensor:
    """[T, K/2] bytes -> [T, K] codes (element 2j from the low nibble)."""
    lo = packed & 0x0F
    hi = packed >> 4
    return torch.stack([lo, hi], dim=-1).reshape(packed.shape[0], -1)


def dequantize(packed: torch.Tensor, scales: torch.Tensor, global_scale: float) -> torch.Tensor:
    """FP64 values e2m1 * s / gs, [T, K]."""
    q = e2m1_values(unpack_codes(packed))
    s = ue4m3_values(scales).to(F64).repeat_interleave(BLOCK, dim=-1)
    return q * s / float(torch.tensor(float(global_scale), dtype=F32))


def block_products(packed: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """FP64 q * s per element (the factors the block-scaled MMA multiplies)."""
    q = e2m1_values(unpack_codes(packed))
    return q * ue4m3_values(scales).to(F64).repeat_interleave(BLOCK, dim=-1)


def nvfp4_projection(act_q, act_sf, w_q, w_sf, alpha: float) -> torch.Tensor:
    """y = bf16(RN32(alpha * RN32(sum_k (qa sa)(qw sw)))), [T, N] (bf16)."""
    acc = block_products(act_q, act_sf) @ block_products(w_q, w_sf).T  # FP64
    acc32 = acc.to(F32)
    return torch.mul(acc32, torch.tensor(float(alpha), dtype=F32)).to(BF16)


def alpha_from_scales(act_global_scale: float, weight_global_scale: float) -> float:
    """alpha = RN32(1 / RN32(act_gs * w_gs)) (Parameters: alpha)."""
    p = torch.mul(torch.tensor(float(act_global_scale), dtype=F32),
                  torch.tensor(float(weight_global_scale), dtype=F32))
    return float(torch.div(torch.tensor(1.0, dtype=F32), p))


def pre_attention_nvfp4_tokens(x, x_norm_weight, adaln_scale, adaln_shift, adaln_index,
                               w_q, w_sf, weight_global_scale, act_global_scale,
                               q_norm_weight, k_norm_weight, rope_cos_sin, *, eps: float = 1e-5,
                               alpha: Optional[float] = None,
                               tokens: Optional[Sequence[int]] = None) -> PreAttnTokens:
    """The NVFP4 stage for the given tokens (default all); w_q [21504, 2688]
    and w_sf [21504, 336] (row-major) are the quantised weight.  Returns the
    per-token outputs [T, 56, 3, 128] and the intermediates (n, a, y and the
    activation codes/scales as extra attributes)."""
    M = x.shape[0]
    tok = torch.arange(M) if tokens is None else torch.as_tensor(list(tokens), dtype=torch.int64)
    xs, idx = x[tok], adaln_index[tok].to(torch.int64)
    n = input_rmsnorm(xs, x_norm_weight, eps)
    a = indexed_adaln(n, adaln_scale, adaln_shift, idx)
    act_q, act_sf = fp4_quantize(a, act_global_scale)
    al = alpha_from_scales(act_global_scale, weight_global_scale) if alpha is None else alpha
    y = nvfp4_projection(act_q, act_sf, w_q, w_sf, al)       # [T, 21504]
    T = len(tok)
    y4 = y.view(T, 3, 56, 128)
    q = rope_split_half(head_rmsnorm(y4[:, 0], q_norm_weight, eps), rope_cos_sin, tok)
    k = rope_split_half(head_rmsnorm(y4[:, 1], k_norm_weight, eps), rope_cos_sin, tok)
    v = y4[:, 2]
    qkv = torch.stack([q, k, v], dim=2)                         # [T, 56, 3, 128]
    out = PreAttnTokens(tokens=tok, n=n, a=a, y=y, qkv=qkv)
    out.act_q, out.act_sf, out.alpha = act_q, act_sf, al
    return out


def out_proj_nvfp4(attn_out, o_weight_q, o_weight_sf, o_weight_global_scale: float,
                   act_global_scale: float, gate, gate_index, residual, *,
                   tokens: Optional[Sequence[int]] = None) -> dict:
    """The W4A4 attention output projection with the gated residual
    (flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj, summary and
    Parameters): attn_out bf16 [M, 7168] is quantised per token with
    act_global_scale (the block-16 convention above); o_weight_q [5376, 3584]
    and o_weight_sf [5376, 448] (row-major) are the quantised weight;
      o   = bf16(RN32(alpha * RN32(sum_k (qa sa)(qw sw)))),
      alpha = RN32(1 / RN32(act_gs * w_gs))   (the dequantisation the
              pre-attention page names alpha; this page derives it from the
              two global scales)
      out = bf16(residual + bf16(g * o)),  g = gate[gate_index[m]], 0 outside
            [0, rows).
    Returns the activation codes and scales, alpha, o and out for the given
    tokens (default all)."""
    from .out_proj import gated_residual
    if tokens is not None:
        t = torch.as_tensor(list(tokens), dtype=torch.int64)
        attn_out, gate_index, residual = attn_out[t], gate_index[t], residual[t]
    act_q, act_sf = fp4_quantize(attn_out, act_global_scale)
    al = alpha_from_scales(act_global_scale, o_weight_global_scale)
    o = nvfp4_projection(act_q, act_sf, o_weight_q, o_weight_sf, al)
    out = gated_residual(o, gate, gate_index, residual)
    return dict(act_q=act_q, act_sf=act_sf, alpha=al, o=o, out=out)


def quantize_outputs(qkv: torch.Tensor, global_scales: Sequence[float]):
    """NVFP4 outputs of the stage (minimax_h3_nvfp4_pre_attention,
    Parameters: out_mode "nvfp4", q/k/v_global_scale): every row of 128
    values (token t, head h, kind k) of the bf16 output qkv [T, H, 3, 128] is
    quantised with fp4_quantize and the global scale of its kind.  Returns
    codes uint8 [T, H, 3, 64] and scales uint8 [T, H, 3, 8]."""
    T, H, K3, D = qkv.shape
    codes = torch.empty((T, H, K3, D // 2), dtype=torch.uint8)
    scales = torch.empty((T, H, K3, D // BLOCK), dtype=torch.uint8)
    for kind in range(K3):
        c, s = fp4_quantize(qkv[:, :, kind, :].reshape(T * H, D), global_scales[kind])
        codes[:, :, kind] = c.view(T, H, D // 2)
        scales[:, :, kind] = s.view(T, H, D // BLOCK)
    return codes, scales
