"""Oracle of the e4m3 output mode of the pre-attention stage.

TEST INFRASTRUCTURE ONLY (see the package docstring).

flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention, Parameters:
out_mode ("e4m3") and q_descale / k_descale / v_descale ("per-tensor E4M3
dequantization scales").  The page defers the exact conventions to
minimax_h3_fp8_pre_attention, which is not among the pages, so this takes the
plainest reading: each output value is the bf16 value of the bf16 mode
divided by its tensor's dequantisation scale in FP32 (IEEE division), then
rounded to nearest-even e4m3 and saturated to +-448 (e4m3 has no infinity);
dequantising is code * descale.  The layout is the bf16 mode's
destination-major pack with one byte per element.
"""
from __future__ import annotations

import torch

E4M3_MAX = 448.0


def quantize_e4m3(values_bf16: torch.Tensor, descale: float) -> torch.Tensor:
    """uint8 e4m3 codes of bf16(values) / descale (FP32 quotient, RNE, saturated)."""
    q = torch.div(values_bf16.to(torch.float32), torch.tensor(float(descale), dtype=torch.float32))
    q = torch.clamp(q, -E4M3_MAX, E4M3_MAX)
    return q.to(torch.float8_e4m3fn).view(torch.uint8)


def dequantize_e4m3(codes: torch.Tensor, descale: float) -> torch.Tensor:
    """float32 values code * descale."""
    return codes.view(torch.float8_e4m3fn).to(torch.float32) * float(descale)


def quantize_packed(out_bf16: torch.Tensor, descales) -> torch.Tensor:
    """Packed bf16 out [P, M, NH/P, 3, D] -> packed e4m3 codes, kind k scaled
    by descales[k] (q, k, v)."""
    codes = torch.empty(out_bf16.shape, dtype=torch.uint8)
    for k in range(3):
        codes[:, :, :, k] = quantize_e4m3(out_bf16[:, :, :, k], descales[k])
    return codes
