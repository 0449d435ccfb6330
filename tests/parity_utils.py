"""Helpers shared by the GPU parity tests: moving a seeded workload to the
device, running the stage through the C ABI, and the comparison rules.

Tolerances (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention outputs):
* q/k/v: |gpu - ref| <= 2e-2 * |ref| + 2e-2 elementwise and mean |gpu - ref|
  <= 2e-3 over the compared elements;
* the bf16 workspace a: within 1 bf16 ulp of the oracle, widened only where
  the FP32 sum of squares (whose summation order the pages leave open) moves
  n across a bf16 rounding boundary.  Such a flip changes n by at most
  u_n = ulp(n_ref), so shift + n*g moves by at most |g|*u_n (g = bf16(1 +
  scale[i])), and rounding both sides to bf16 adds half an ulp of each
  result: |gpu - ref| <= |g|*u_n + ulp(a_ref)/2 + ulp(|a_ref| + |g|*u_n)/2.
  Without a flip the two sides run the same FP32 operations, so nearly
  every element must be bit-exact and all but a handful within 1 ulp;
* guard rows, clamped positions and the pack are compared bit for bit (zero
  rows by value, since +0 and -0 are both the zero the guard asks for).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import torch

import oracle
from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import HIDDEN, Workload

BF16 = torch.bfloat16


@dataclass
class DevWorkload:
    wl: Workload
    x: torch.Tensor
    xw: torch.Tensor
    mod: torch.Tensor
    scale: torch.Tensor
    shift: torch.Tensor
    idx: torch.Tensor
    W: torch.Tensor
    qw: torch.Tensor
    kw: torch.Tensor
    cs: torch.Tensor
    pos: Optional[torch.Tensor]

    @property
    def M(self):
        return self.wl.M

    @property
    def P(self):
        return self.wl.spec.P

    @property
    def S(self):
        return self.cs.shape[0]


def to_device(wl: Workload, dev="cuda") -> DevWorkload:
    mod = wl.adaln_mod.to(dev)
    sc, sh = wl.table_views(mod)
    return DevWorkload(
        wl=wl, x=wl.x.to(dev), xw=wl.x_norm_weight.to(dev), mod=mod, scale=sc, shift=sh,
        idx=wl.adaln_index.to(dev), W=wl.qkv_weight.to(dev), qw=wl.q_norm_weight.to(dev),
        kw=wl.k_norm_weight.to(dev), cs=wl.rope_cos_sin.to(dev),
        pos=None if wl.rope_positions is None else wl.rope_positions.to(dev))


def new_out(M: int, P: int, dev="cuda", fill: Optional[float] = None) -> torch.Tensor:
    o = torch.empty((P, M, 56 // P, 3, 128), dtype=BF16, device=dev)
    if fill is not None:
        o.fill_(fill)
    return o


def run_stage(h: binding.Handle, d: DevWorkload, out: torch.Tensor, workspace=None, P=None,
              positions="default", stream=None, qk_eps="default"):
    P = d.P if P is None else P
    pos = d.pos if positions == "default" else positions
    qk = d.wl.spec.qk_eps if qk_eps == "default" else qk_eps
    binding.mh3_preattn_run(
        h, stream, d.M, d.x, d.xw, d.scale, d.scale.stride(0), d.shift, d.shift.stride(0),
        d.scale.shape[0], d.idx, d.W, d.qw, d.kw, d.cs, d.S, pos, P, d.wl.spec.eps, qk,
        workspace, out)


def run_norm_adaln(h: binding.Handle, d: DevWorkload, ws: torch.Tensor, stream=None):
    binding.mh3_preattn_norm_adaln(
        h, stream, d.M, d.x, d.xw, d.scale, d.scale.stride(0), d.shift, d.shift.stride(0),
        d.scale.shape[0], d.idx, d.wl.spec.eps, ws)


def oracle_tokens(wl: Workload, tokens: Optional[Sequence[int]] = None) -> oracle.PreAttnTokens:
    sc, sh = wl.table_views()
    return oracle.pre_attention_tokens(
        wl.x, wl.x_norm_weight, sc, sh, wl.adaln_index, wl.qkv_weight, wl.q_norm_weight,
        wl.k_norm_weight, wl.rope_cos_sin, eps=wl.spec.eps, qk_eps=wl.spec.qk_eps,
        rope_positions=wl.rope_positions, tokens=tokens)


def ulp_bf16(v: torch.Tensor) -> torch.Tensor:
    av = v.abs().to(torch.float64).clamp_min(2.0 ** -126)
    return torch.pow(2.0, torch.floor(torch.log2(av)) - 7)


def check_outputs(gpu_tok: torch.Tensor, ref_tok: torch.Tensor, what: str) -> dict:
    """gpu_tok/ref_tok: [T, 56, 3, 128] bf16 (CPU).  Returns error stats."""
    g = gpu_tok.double()
    r = ref_tok.double()
    assert torch.isfinite(g).all(), f"{what}: non-finite output"
    err = (g - r).abs()
    bound = 2e-2 * r.abs() + 2e-2
    bad = err > bound
    stats = dict(max_abs=float(err.max()), mean_abs=float(err.mean()),
                 exact=float((gpu_tok.view(torch.int16) == ref_tok.view(torch.int16)).double().mean()),
                 n=int(err.numel()))
    assert not bool(bad.any()), (
        f"{what}: {int(bad.sum())} elements outside 2e-2*|ref|+2e-2; first at "
        f"{tuple(torch.nonzero(bad)[0].tolist())}: gpu={g[bad][0].item()} ref={r[bad][0].item()}")
    assert stats["mean_abs"] <= 2e-3, f"{what}: mean abs error {stats['mean_abs']}"
    return stats


def check_workspace(gpu_a: torch.Tensor, ref: oracle.PreAttnTokens, wl: Workload,
                    what: str) -> dict:
    """gpu_a: [T, H] bf16 (CPU) rows for ref.tokens."""
    a_ref = ref.a.double()
    a_gpu = gpu_a.double()
    sc, _ = wl.table_views()
    idx = wl.adaln_index[ref.tokens]
    rows = sc.shape[0]
    valid = (idx >= 0) & (idx < rows)
    g = torch.ones_like(a_ref)
    if bool(valid.any()):
        g[valid] = (sc[idx[valid]].float() + 1.0).to(BF16).double()
    shift_n = g.abs() * ulp_bf16(ref.n.double())
    allowed = shift_n + 0.5 * ulp_bf16(a_ref) + 0.5 * ulp_bf16(a_ref.abs() + shift_n)
    err = (a_gpu - a_ref).abs()
    assert torch.isfinite(a_gpu).all(), f"{what}: non-finite workspace"
    bad = err > allowed
    assert not bool(bad.any()), (
        f"{what}: {int(bad.sum())} workspace elements beyond the n-flip bound")
    exact = float((gpu_a.view(torch.int16) == ref.a.view(torch.int16)).double().mean())
    within1 = float((err <= ulp_bf16(a_ref)).double().mean())
    # guarded rows are +0.0 bit for bit
    if bool((~valid).any()):
        assert torch.all(gpu_a[~valid].view(torch.int16) == 0), f"{what}: guard row not +0"
    assert exact > 0.999, f"{what}: only {exact:.6f} of the workspace is bit-exact"
    assert within1 > 0.9999, f"{what}: only {within1:.6f} within 1 ulp"
    return dict(exact=exact, within_1ulp=within1)
