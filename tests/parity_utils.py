"""Helpers shared by the GPU parity tests: moving a seeded workload to the
device, running the stage through the C ABI, and the comparison rules.

Tolerances (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention outputs):
* q/k/v: |gpu - ref| <= 2e-2 * |ref| + 2e-2 elementwise and mean |gpu - ref|
  <= 2e-3 over the compared elements;
* the bf16 workspace a: every row bit-exact, or bit-exact against the
  oracle's own norm and AdaLN evaluated with an r = 1/sqrt(ss/H + eps) a few
  FP32 steps from the oracle's (the only freedom: the pages fix the type of
  the sum of squares, not its order); see check_workspace;
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


def untile(tiled: torch.Tensor, rows: int, cols: int) -> torch.Tensor:
    """Tiled NVFP4 scale atoms -> row-major [rows, cols/16] (the layout the
    C header states: row r of an atom at byte (r % 32) * 16 + (r / 32) * 4,
    atoms ordered [rows/128][cols/64])."""
    ks = cols // 64
    r = torch.arange(rows).view(-1, 1, 1)
    k = torch.arange(ks).view(1, -1, 1)
    j = torch.arange(4).view(1, 1, -1)
    off = ((r // 128) * ks + k) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + j
    return tiled.view(-1)[off.reshape(-1)].view(rows, ks * 4)


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


def _nudge(r: float, k: int) -> float:
    """The FP32 value k representable steps away from r (r > 0)."""
    b = torch.tensor([r], dtype=torch.float32).view(torch.int32) + k
    return float(b.view(torch.float32))


def check_workspace(gpu_a: torch.Tensor, ref: oracle.PreAttnTokens, wl: Workload,
                    what: str, max_steps: int = 96) -> dict:
    """gpu_a: [T, H] bf16 (CPU) rows for ref.tokens.

    Kernel 1 runs the oracle's FP32 operations after the sum of squares, so a
    row can differ from the oracle only through its FP32 sum of squares (the
    pages fix its type, not its order), i.e. through r = 1/sqrt(ss/H + eps).
    Every row must therefore be bit-exact, or equal bit for bit to the
    oracle's AdaLN applied to bf16((x * r') * w) for one r' a few FP32 steps
    from the oracle's r.  Guarded rows are +0.0 bit for bit.  Returns counts
    of exact rows, rows explained by a moved r, and the elements of those
    rows that lie more than one bf16 step from the oracle (with the largest
    distance in steps)."""
    assert torch.isfinite(gpu_a.double()).all(), f"{what}: non-finite workspace"
    sc, sh = wl.table_views()
    idx = wl.adaln_index[ref.tokens]
    rows = sc.shape[0]
    g_bits = gpu_a.contiguous().view(torch.int16)
    r_bits = ref.a.contiguous().view(torch.int16)
    same = (g_bits == r_bits).all(dim=1)
    moved = {}
    beyond, worst = 0, 0.0
    for t in torch.nonzero(~same).flatten().tolist():
        i = int(idx[t])
        assert 0 <= i < rows, f"{what}: guarded token {int(ref.tokens[t])} is not +0"
        x_row = wl.x[int(ref.tokens[t])].reshape(1, -1)
        r0 = float(ref.r[t])
        found = None
        for step in range(1, max_steps + 1):
            for k in (step, -step):
                n_alt = oracle.rmsnorm_apply(x_row, wl.x_norm_weight,
                                             torch.tensor([_nudge(r0, k)]))
                a_alt = oracle.indexed_adaln(n_alt, sc, sh, idx[t:t + 1])
                if torch.equal(a_alt.view(torch.int16)[0], g_bits[t]):
                    found = k
                    break
            if found is not None:
                break
        assert found is not None, (
            f"{what}: workspace row of token {int(ref.tokens[t])} is not the oracle's AdaLN "
            f"for any r within {max_steps} FP32 steps")
        moved[found] = moved.get(found, 0) + 1
        d = (gpu_a[t].double() - ref.a[t].double()).abs() / ulp_bf16(ref.a[t].double())
        beyond += int((d > 1).sum())
        worst = max(worst, float(d.max()))
    # guarded rows are +0.0 bit for bit
    bad = (idx < 0) | (idx >= rows)
    if bool(bad.any()):
        assert torch.all(g_bits[bad] == 0), f"{what}: guard row not +0"
    return dict(rows=int(len(same)), exact_rows=int(same.sum()),
                rows_with_moved_r=int((~same).sum()), r_steps=moved,
                elements_beyond_1ulp=beyond, max_ulps=worst)
