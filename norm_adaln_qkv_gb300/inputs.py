"""Seeded synthetic inputs for the MiniMax-H3 BF16 pre-attention stage.

This module only draws numbers and lays them out.  It holds none of the stage's
arithmetic (no normalisation, modulation, projection, rotation or packing), so
the CPU oracle and the CUDA path can both consume its tensors without sharing
any of the method.

The five workloads are DiT video latent grids at the sizes the
``flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention`` page implies
(hidden 5376, 56 heads of 128, fused QKV weight [21504, 5376], AdaLN tables
that may be column chunks of a [rows, 6*5376] modulation projection, int64
indices and positions, a [S, 96] cos/sin cache) and the M upper bound 149796
from ``flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120`` (Parameters: x).

Every tensor is drawn on the host from ``torch.Generator(seed)`` in a fixed
order (x, x_norm_weight, tables, index, qkv_weight, q/k norm weights,
positions), in FP32 and rounded to BF16 with ``.to(torch.bfloat16)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch

HIDDEN = 5376
NUM_HEADS = 56
HEAD_DIM = 128
QKV_ROWS = 3 * NUM_HEADS * HEAD_DIM  # 21504
ROPE_DIMS = 96
SEED_BASE = 20261202

INT64_MIN = -(2 ** 63)
INT64_MAX = 2 ** 63 - 1

# Chunk order of the [rows, 6*hidden] modulation projection: shift, scale, ...
SHIFT_CHUNK = 0
SCALE_CHUNK = 1


@dataclass(frozen=True)
class WorkloadSpec:
    """Sizes and recipe of one synthetic workload."""

    name: str
    cfg_id: int
    M: int
    grid: tuple  # (frames, height, width) of the latent grid
    rows: int
    P: int
    S: int
    eps: float
    qk_eps: Optional[float]
    x_std: float
    outlier_rate: float  # fraction of x elements set to +-200
    bad_index_rate: Optional[float]  # None: only the listed bad tokens
    bad_index_tokens: tuple = ()  # explicit (token, value) overrides
    table_layout: str = "separate"  # "separate" or "chunks"
    positions: str = "identity"  # "identity", "permutation", "arange_clamped"
    bad_position_rate: float = 0.0
    caller_workspace: bool = False
    index_mode: str = "uniform"  # "uniform" over [0, rows) or "zero"


WORKLOADS = {
    "c0": WorkloadSpec(
        name="tiny M=16 (1x4x4 grid), rows=2, P=1, identity positions S=16",
        cfg_id=0, M=16, grid=(1, 4, 4), rows=2, P=1, S=16, eps=1e-5, qk_eps=1e-5,
        x_std=1.0, outlier_rate=0.0, bad_index_rate=None,
        bad_index_tokens=((3, -1),), table_layout="separate", positions="identity"),
    "c1": WorkloadSpec(
        name="single-timestep DiT block M=1024 (4x16x16), rows=1, P=1, identity S=1024",
        cfg_id=1, M=1024, grid=(4, 16, 16), rows=1, P=1, S=1024, eps=1e-5, qk_eps=1e-6,
        x_std=1.0, outlier_rate=0.0, bad_index_rate=None, table_layout="separate",
        positions="identity", index_mode="zero"),
    "c2": WorkloadSpec(
        name="mid video block M=4096 (16x16x16), rows=9 strided chunks, P=2, permuted positions",
        cfg_id=2, M=4096, grid=(16, 16, 16), rows=9, P=2, S=4096, eps=1e-5, qk_eps=1e-5,
        x_std=1.0, outlier_rate=0.0, bad_index_rate=0.01, table_layout="chunks",
        positions="permutation"),
    "c3": WorkloadSpec(
        name="production video sequence M=32760 (21x30x52), rows=9, P=8, S=40000 clamped positions",
        cfg_id=3, M=32760, grid=(21, 30, 52), rows=9, P=8, S=40000, eps=1e-5, qk_eps=1e-5,
        x_std=math.sqrt(2.0), outlier_rate=1e-4, bad_index_rate=0.01, table_layout="chunks",
        positions="arange_clamped", bad_position_rate=1e-3, caller_workspace=True),
    "c4": WorkloadSpec(
        name="upper-bound sequence M=149796 (24x79x79 + 12), rows=9, P=4, identity S=149796",
        cfg_id=4, M=149796, grid=(24, 79, 79), rows=9, P=4, S=149796, eps=1e-5, qk_eps=1e-6,
        x_std=math.sqrt(2.0), outlier_rate=1e-4, bad_index_rate=0.01, table_layout="chunks",
        positions="identity", caller_workspace=True),
}

BAD_INDEX_CYCLE = (-1, 9, 2 ** 40)
BAD_POSITION_CYCLE = (-1, -(2 ** 40), INT64_MIN, "S", "S+1", 2 ** 40, INT64_MAX)


@dataclass
class Workload:
    """Host (CPU) tensors of one workload, plus its scalars.

    ``adaln_mod`` is the backing tensor of the AdaLN tables; ``table_views``
    cuts the scale/shift views out of it (on any device) with the row stride
    of the backing tensor, exactly as an engine passes column chunks.
    """

    spec: WorkloadSpec
    x: torch.Tensor
    x_norm_weight: torch.Tensor
    adaln_mod: torch.Tensor  # [rows, k*HIDDEN]
    scale_chunk: int
    shift_chunk: int
    separate_tables: bool
    adaln_index: torch.Tensor
    qkv_weight: torch.Tensor
    q_norm_weight: torch.Tensor
    k_norm_weight: torch.Tensor
    rope_cos_sin: torch.Tensor
    rope_positions: Optional[torch.Tensor]
    extras: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return self.spec.M

    def table_views(self, mod: Optional[torch.Tensor] = None):
        """(adaln_scale, adaln_shift) views of ``mod`` (default: the host tensor)."""
        mod = self.adaln_mod if mod is None else mod
        if self.separate_tables:
            # backing tensor is [2, rows, HIDDEN]: [0] = scale, [1] = shift
            return mod[0], mod[1]
        sc = mod[:, self.scale_chunk * HIDDEN:(self.scale_chunk + 1) * HIDDEN]
        sh = mod[:, self.shift_chunk * HIDDEN:(self.shift_chunk + 1) * HIDDEN]
        return sc, sh


def _normal(gen: torch.Generator, shape, std=1.0, mean=0.0) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float32)
    t.normal_(mean=mean, std=std, generator=gen)
    return t


def _x_bf16(gen: torch.Generator, M: int, std: float, chunk_rows: int = 8192) -> torch.Tensor:
    """[M, HIDDEN] bf16 drawn row-chunk by row-chunk (bounded host memory)."""
    x = torch.empty((M, HIDDEN), dtype=torch.bfloat16)
    for r0 in range(0, M, chunk_rows):
        r1 = min(M, r0 + chunk_rows)
        x[r0:r1] = _normal(gen, (r1 - r0, HIDDEN), std=std).to(torch.bfloat16)
    return x


def grid_coords(s: torch.Tensor, grid: tuple) -> tuple:
    """Row-major (frame, height, width) decode of cache row ``s``.

    Rows past F*H*W keep counting frames (the decode simply continues).
    """
    _, gh, gw = grid
    f = torch.div(s, gh * gw, rounding_mode="floor")
    h = torch.div(s, gw, rounding_mode="floor") % gh
    w = s % gw
    return f, h, w


def rope_cos_sin_cache(S: int, grid: tuple) -> torch.Tensor:
    """[S, 96] bf16 cache: columns [16a, 16a+16) hold cos(coord_a * 10000^(-j/16))
    for axis a in (frame, height, width), columns [48+16a, ...) the matching sin.

    This is how the synthetic cache is built (an input of the stage, computed
    in float64 on the host), not part of the stage.
    """
    s = torch.arange(S, dtype=torch.int64)
    coords = grid_coords(s, grid)
    j = torch.arange(16, dtype=torch.float64)
    inv_freq = torch.pow(torch.tensor(10000.0, dtype=torch.float64), -j / 16.0)
    cos_cols, sin_cols = [], []
    for c in coords:
        ang = c.to(torch.float64)[:, None] * inv_freq[None, :]
        cos_cols.append(torch.cos(ang))
        sin_cols.append(torch.sin(ang))
    cs = torch.cat(cos_cols + sin_cols, dim=1)
    return cs.to(torch.float32).to(torch.bfloat16).contiguous()


def make_workload(key: str, M: Optional[int] = None) -> Workload:
    """Draw workload ``key`` ("c0".."c4").  ``M`` overrides the token count
    (for smaller cases of the same recipe); S follows M for identity
    positions."""
    spec = WORKLOADS[key]
    if M is not None and M != spec.M:
        S = spec.S if spec.positions != "identity" else max(M, 1)
        spec = WorkloadSpec(**{**spec.__dict__, "M": M, "S": S})
    gen = torch.Generator().manual_seed(SEED_BASE + spec.cfg_id)
    Mv = spec.M

    # 1. x (with optional +-200 outliers)
    x = _x_bf16(gen, Mv, spec.x_std)
    n_out = int(round(spec.outlier_rate * Mv * HIDDEN))
    if n_out > 0:
        flat = torch.randint(0, Mv * HIDDEN, (n_out,), generator=gen, dtype=torch.int64)
        sign = torch.randint(0, 2, (n_out,), generator=gen, dtype=torch.int64) * 2 - 1
        x.view(-1)[flat] = (200.0 * sign).to(torch.bfloat16)

    # 2. x_norm_weight
    xw = (1.0 + 0.1 * _normal(gen, (HIDDEN,))).to(torch.bfloat16)

    # 3. AdaLN tables
    if spec.table_layout == "separate":
        mod = (0.1 * _normal(gen, (2, spec.rows, HIDDEN))).to(torch.bfloat16)
        separate = True
    else:
        mod = (0.1 * _normal(gen, (spec.rows, 6 * HIDDEN))).to(torch.bfloat16)
        separate = False

    # 4. adaln_index
    if spec.index_mode == "zero":
        idx = torch.zeros(Mv, dtype=torch.int64)
    else:
        idx = torch.randint(0, spec.rows, (Mv,), generator=gen, dtype=torch.int64)
    if spec.bad_index_rate:
        n_bad = int(round(spec.bad_index_rate * Mv))
        toks = torch.randperm(Mv, generator=gen)[:n_bad]
        for j, t in enumerate(toks.tolist()):
            idx[t] = BAD_INDEX_CYCLE[j % len(BAD_INDEX_CYCLE)]
    for t, v in spec.bad_index_tokens:
        if t < Mv:
            idx[t] = v

    # 5. fused QKV weight, engine order [q_all | k_all | v_all]
    w = (_normal(gen, (QKV_ROWS, HIDDEN)) / math.sqrt(HIDDEN)).to(torch.bfloat16)

    # 6. per-head norm weights
    qw = (1.0 + 0.1 * _normal(gen, (HEAD_DIM,))).to(torch.bfloat16)
    kw = (1.0 + 0.1 * _normal(gen, (HEAD_DIM,))).to(torch.bfloat16)

    # 7. positions
    pos = None
    if spec.positions == "permutation":
        pos = torch.randperm(Mv, generator=gen).to(torch.int64)
    elif spec.positions == "arange_clamped":
        pos = torch.arange(Mv, dtype=torch.int64)
        n_badp = int(round(spec.bad_position_rate * Mv))
        toks = torch.randperm(Mv, generator=gen)[:n_badp]
        for j, t in enumerate(toks.tolist()):
            v = BAD_POSITION_CYCLE[j % len(BAD_POSITION_CYCLE)]
            v = spec.S if v == "S" else (spec.S + 1 if v == "S+1" else v)
            pos[t] = v

    cs = rope_cos_sin_cache(spec.S, spec.grid)
    return Workload(
        spec=spec, x=x, x_norm_weight=xw, adaln_mod=mod,
        scale_chunk=SCALE_CHUNK, shift_chunk=SHIFT_CHUNK, separate_tables=separate,
        adaln_index=idx, qkv_weight=w, q_norm_weight=qw, k_norm_weight=kw,
        rope_cos_sin=cs, rope_positions=pos)


def special_rows(wl: Workload) -> list:
    """Tokens whose index is out of range or whose position is clamped."""
    rows = set()
    bad = (wl.adaln_index < 0) | (wl.adaln_index >= wl.spec.rows)
    rows.update(torch.nonzero(bad).flatten().tolist())
    if wl.rope_positions is not None:
        badp = (wl.rope_positions < 0) | (wl.rope_positions >= wl.spec.S)
        rows.update(torch.nonzero(badp).flatten().tolist())
    return sorted(rows)


def sample_rows(wl: Workload, every: int = 64, limit: Optional[int] = None) -> list:
    """Deterministic row sample: every ``every``-th row, the last row, and all
    special rows (guarded index, clamped position)."""
    M = wl.M
    rows = set(range(0, M, every))
    rows.add(M - 1)
    rows.update(special_rows(wl))
    out = sorted(rows)
    if limit is not None and len(out) > limit:
        keep = set(special_rows(wl)) | {M - 1}
        stride = max(1, len(out) // limit)
        out = sorted(set(out[::stride]) | keep)
    return out


# --------------------------------------------------- attention output projection
ATTN_WIDTH = NUM_HEADS * HEAD_DIM  # 7168
GATE_CHUNK = 2  # gate_msa: chunk 2 of the [rows, 6*hidden] modulation projection
BAD_GATE_CYCLE = (-1, 9, 2 ** 30)


@dataclass
class OutProjWorkload:
    """Host tensors of one out-projection case (shapes of
    flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj, Parameters: attn_out
    [M, 7168], o weight [5376, 7168], gate [9, 5376], gate_index int32 [M],
    residual [M, 5376])."""

    M: int
    attn_out: torch.Tensor
    o_weight: torch.Tensor
    adaln_mod: torch.Tensor  # [rows, 6*HIDDEN]; the gate is chunk GATE_CHUNK
    gate_index: torch.Tensor
    residual: torch.Tensor

    def gate_view(self, mod: Optional[torch.Tensor] = None) -> torch.Tensor:
        mod = self.adaln_mod if mod is None else mod
        return mod[:, GATE_CHUNK * HIDDEN:(GATE_CHUNK + 1) * HIDDEN]


def make_out_proj_workload(M: int, seed: int = SEED_BASE + 100, rows: int = 9,
                           bad_rate: float = 0.01) -> OutProjWorkload:
    """attn_out ~ N(0,1); o weight ~ N(0, 1/7168); modulation 0.1*N(0,1) with
    the gate as chunk 2 (row stride 6*5376); gate_index uniform in [0, rows)
    with bad_rate of the tokens set cyclically to -1, 9, 2^30; residual ~ N(0,1)."""
    gen = torch.Generator().manual_seed(seed)
    attn = torch.empty((M, ATTN_WIDTH), dtype=torch.bfloat16)
    for r0 in range(0, M, 8192):
        r1 = min(M, r0 + 8192)
        attn[r0:r1] = _normal(gen, (r1 - r0, ATTN_WIDTH)).to(torch.bfloat16)
    w = (_normal(gen, (HIDDEN, ATTN_WIDTH)) / math.sqrt(ATTN_WIDTH)).to(torch.bfloat16)
    mod = (0.1 * _normal(gen, (rows, 6 * HIDDEN))).to(torch.bfloat16)
    gi = torch.randint(0, rows, (M,), generator=gen, dtype=torch.int64).to(torch.int32)
    n_bad = int(round(bad_rate * M))
    if n_bad:
        toks = torch.randperm(M, generator=gen)[:n_bad]
        for j, t in enumerate(toks.tolist()):
            gi[t] = BAD_GATE_CYCLE[j % len(BAD_GATE_CYCLE)]
    res = torch.empty((M, HIDDEN), dtype=torch.bfloat16)
    for r0 in range(0, M, 8192):
        r1 = min(M, r0 + 8192)
        res[r0:r1] = _normal(gen, (r1 - r0, HIDDEN)).to(torch.bfloat16)
    return OutProjWorkload(M=M, attn_out=attn, o_weight=w, adaln_mod=mod, gate_index=gi,
                           residual=res)


# Global scales of the W4A4 output projection (448 * 6 / amax, Parameters of
# flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj): the calibration amax 8
# for attn_out ~ N(0, 1), and 6 sigma of the weight distribution N(0, 1/7168).
OUT_ACT_AMAX = 8.0


def out_proj_nvfp4_global_scales() -> Tuple[float, float]:
    """(act_global_scale, o_weight_global_scale)."""
    return 448.0 * 6.0 / OUT_ACT_AMAX, 448.0 * 6.0 / (6.0 / math.sqrt(ATTN_WIDTH))


# ------------------------------------------------------------- the MLP block
MLP_INTER = 14336  # SwiGLU width; fc1 has 2 * 14336 = 28672 rows [gate | up]
MLP_CHUNKS = (3, 4, 5)  # shift, scale, gate of the MLP in the [rows, 6*hidden] plan


@dataclass
class MlpWorkload:
    """Host tensors of one MLP-block case (shapes of
    flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, Parameters: x [M, 5376],
    tables [rows, 5376] sharing one row count, int64 adaln_index, residual
    [M, 5376], fc1 [28672, 5376], fc2 [5376, 14336]), with bf16 weights."""

    M: int
    x: torch.Tensor
    x_norm_weight: torch.Tensor
    adaln_mod: torch.Tensor  # [rows, 6*HIDDEN]
    adaln_index: torch.Tensor
    residual: torch.Tensor
    fc1_weight: torch.Tensor
    fc2_weight: torch.Tensor
    eps: float = 1e-5

    def tables(self, mod: Optional[torch.Tensor] = None):
        """(scale, shift, gate) views of the modulation tensor."""
        mod = self.adaln_mod if mod is None else mod
        sh, sc, gt = (mod[:, c * HIDDEN:(c + 1) * HIDDEN] for c in MLP_CHUNKS)
        return sc, sh, gt


def make_mlp_workload(M: int, seed: int = SEED_BASE + 200, rows: int = 9,
                      bad_rate: float = 0.01) -> MlpWorkload:
    """x, residual ~ N(0,1); x_norm_weight 1 + 0.1*N(0,1); modulation
    0.1*N(0,1); fc1 ~ N(0, 1/5376); fc2 ~ N(0, 1/14336); index uniform in
    [0, rows) with bad_rate of the tokens set cyclically to -1, 9, 2^40."""
    gen = torch.Generator().manual_seed(seed)
    x = _x_bf16(gen, M, 1.0)
    xw = (1.0 + 0.1 * _normal(gen, (HIDDEN,))).to(torch.bfloat16)
    mod = (0.1 * _normal(gen, (rows, 6 * HIDDEN))).to(torch.bfloat16)
    idx = torch.randint(0, rows, (M,), generator=gen, dtype=torch.int64)
    n_bad = int(round(bad_rate * M))
    if n_bad:
        toks = torch.randperm(M, generator=gen)[:n_bad]
        for j, t in enumerate(toks.tolist()):
            idx[t] = BAD_INDEX_CYCLE[j % len(BAD_INDEX_CYCLE)]
    res = _x_bf16(gen, M, 1.0)
    fc1 = (_normal(gen, (2 * MLP_INTER, HIDDEN)) / math.sqrt(HIDDEN)).to(torch.bfloat16)
    fc2 = (_normal(gen, (HIDDEN, MLP_INTER)) / math.sqrt(MLP_INTER)).to(torch.bfloat16)
    return MlpWorkload(M=M, x=x, x_norm_weight=xw, adaln_mod=mod, adaln_index=idx, residual=res,
                       fc1_weight=fc1, fc2_weight=fc2)


# ------------------------------------------------------- the FP8 MLP block
@dataclass
class MlpFp8Workload:
    """Host tensors of one FP8 MLP-block case (shapes of
    flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, Parameters): the
    bf16 activations and tables of the BF16 block, and E4M3 weights with one
    FP32 scale per output row (fc1 [28672, 5376] / [28672], rows [gate | up];
    fc2 [5376, 14336] / [5376]).  The weight codes are drawn directly as E4M3
    numbers (N(0, 1) * 32, rounded by torch's float8 conversion) and the
    scales as 1 / (32 sqrt(K)) * (1 + 0.1 N(0, 1)), so code * scale has the
    spread of the BF16 block's N(0, 1/K) weights."""

    M: int
    x: torch.Tensor
    x_norm_weight: torch.Tensor
    adaln_mod: torch.Tensor  # [rows, 6*HIDDEN]
    adaln_index: torch.Tensor
    residual: torch.Tensor
    fc1_q: torch.Tensor      # uint8 [28672, 5376]
    fc1_scale: torch.Tensor  # float32 [28672]
    fc2_q: torch.Tensor      # uint8 [5376, 14336]
    fc2_scale: torch.Tensor  # float32 [5376]
    eps: float = 1e-5

    def tables(self, mod: Optional[torch.Tensor] = None):
        """(scale, shift, gate) views of the modulation tensor."""
        mod = self.adaln_mod if mod is None else mod
        sh, sc, gt = (mod[:, c * HIDDEN:(c + 1) * HIDDEN] for c in MLP_CHUNKS)
        return sc, sh, gt


def _e4m3_codes(gen: torch.Generator, rows: int, cols: int, chunk_rows: int = 4096) -> torch.Tensor:
    out = torch.empty((rows, cols), dtype=torch.uint8)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        v = (_normal(gen, (r1 - r0, cols)) * 32.0).clamp(-448.0, 448.0)
        out[r0:r1] = v.to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def make_mlp_fp8_workload(M: int, seed: int = SEED_BASE + 300, rows: int = 9,
                          bad_rate: float = 0.01) -> MlpFp8Workload:
    """x, residual ~ N(0,1); x_norm_weight 1 + 0.1*N(0,1); modulation
    0.1*N(0,1); index uniform in [0, rows) with bad_rate of the tokens set
    cyclically to -1, 9, 2^40; E4M3 weights and FP32 row scales as described
    on MlpFp8Workload."""
    gen = torch.Generator().manual_seed(seed)
    x = _x_bf16(gen, M, 1.0)
    xw = (1.0 + 0.1 * _normal(gen, (HIDDEN,))).to(torch.bfloat16)
    mod = (0.1 * _normal(gen, (rows, 6 * HIDDEN))).to(torch.bfloat16)
    idx = torch.randint(0, rows, (M,), generator=gen, dtype=torch.int64)
    n_bad = int(round(bad_rate * M))
    if n_bad:
        toks = torch.randperm(M, generator=gen)[:n_bad]
        for j, t in enumerate(toks.tolist()):
            idx[t] = BAD_INDEX_CYCLE[j % len(BAD_INDEX_CYCLE)]
    res = _x_bf16(gen, M, 1.0)
    fc1_q = _e4m3_codes(gen, 2 * MLP_INTER, HIDDEN)
    fc1_s = (1.0 + 0.1 * _normal(gen, (2 * MLP_INTER,))) / (32.0 * math.sqrt(HIDDEN))
    fc2_q = _e4m3_codes(gen, HIDDEN, MLP_INTER)
    fc2_s = (1.0 + 0.1 * _normal(gen, (HIDDEN,))) / (32.0 * math.sqrt(MLP_INTER))
    return MlpFp8Workload(M=M, x=x, x_norm_weight=xw, adaln_mod=mod, adaln_index=idx,
                          residual=res, fc1_q=fc1_q, fc1_scale=fc1_s.to(torch.float32),
                          fc2_q=fc2_q, fc2_scale=fc2_s.to(torch.float32))


# ---------------------------------------------------------------- NVFP4 stage
# The NVFP4 op takes int32 AdaLN indices and one cos/sin row per token
# (flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention, Parameters).
BAD_INDEX32_CYCLE = (-1, 9, 2 ** 30)
NVFP4_ACT_AMAX = 8.0  # calibration amax of the normalised activation


@dataclass
class Nvfp4Workload:
    """A bf16-stage workload re-cut for the NVFP4 op: the same x, tables,
    weights and norm weights; int32 indices (out-of-range values -1, 9, 2^30);
    rope_cos_sin [M, 96] with row m for token m; global scales 448 * 6 / amax
    with the calibration amax 8 for the activation and 6 sigma of the weight
    distribution (N(0, 1/5376)) for the weight."""

    base: Workload
    adaln_index: torch.Tensor  # int32 [M]
    rope_cos_sin: torch.Tensor  # bf16 [M, 96]
    act_global_scale: float
    weight_global_scale: float

    @property
    def M(self) -> int:
        return self.base.M

    @property
    def eps(self) -> float:
        return self.base.spec.eps


def make_nvfp4_workload(key: str, M: Optional[int] = None) -> Nvfp4Workload:
    return nvfp4_from_workload(make_workload(key, M))


def nvfp4_from_workload(wl: Workload) -> Nvfp4Workload:
    """Re-cut an already drawn bf16-stage workload for the NVFP4 op."""
    idx = wl.adaln_index.clone()
    bad = (idx < 0) | (idx >= wl.spec.rows)
    for j, t in enumerate(torch.nonzero(bad).flatten().tolist()):
        idx[t] = BAD_INDEX32_CYCLE[j % len(BAD_INDEX32_CYCLE)]
    cs = rope_cos_sin_cache(max(wl.M, 1), wl.spec.grid)[:wl.M].contiguous()
    w_amax = 6.0 / math.sqrt(HIDDEN)
    return Nvfp4Workload(base=wl, adaln_index=idx.to(torch.int32), rope_cos_sin=cs,
                         act_global_scale=448.0 * 6.0 / NVFP4_ACT_AMAX,
                         weight_global_scale=448.0 * 6.0 / w_amax)
