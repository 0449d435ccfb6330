"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one step against a closed form, a library routine for a
special case, exact integer arithmetic, or an invariant, chosen so that a
plausible slip (mean vs sum, eps outside the root, a dropped weight, the
un-rounded AdaLN gain, a transposed weight, a wrong rotation sign or pairing,
a wrong head-to-destination map) fails at least one of them.

Every pin runs twice: on the C++ oracle (``oracle.stage``, the one the GPU
parity tests use) and on the PyTorch restatement (``oracle.preattn``).
"""
import math
import random
from fractions import Fraction

import pytest
import torch

import oracle
import oracle.preattn
import oracle.stage

BF16 = torch.bfloat16
F32 = torch.float32


def bf16_round(v: float) -> float:
    """Round a double to bf16 (via an exact FP32 when v is FP32-exact)."""
    return torch.tensor(v, dtype=torch.float64).to(F32).to(BF16).item()


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int16)


@pytest.fixture(params=["cpp", "torch"])
def O(request):
    """The oracle implementation under test."""
    return oracle.stage if request.param == "cpp" else oracle.preattn


def ulp_bf16(v: torch.Tensor) -> torch.Tensor:
    """Spacing of bf16 numbers at |v| (2^(e-7)); subnormal floor 2^-133."""
    av = v.abs().to(torch.float64).clamp_min(2.0 ** -126)
    e = torch.floor(torch.log2(av))
    return torch.pow(2.0, e - 7)


# ---------------------------------------------------------------- input RMSNorm
# flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, formula block, line n = ...

@pytest.mark.parametrize("c,eps", [(1.0, 1e-5), (2.0 ** -8, 1e-5), (-3.0, 1e-5),
                                   (2.0 ** -7, 1e-5), (0.5, 0.25)])
@pytest.mark.parametrize("H", [7, 5376])
def test_rmsnorm_constant_row_closed_form(c, eps, H, O):
    # x = c everywhere, w = 1: mean square is c^2, so n = bf16(c / sqrt(c^2 + eps)).
    x = torch.full((2, H), c, dtype=BF16)
    w = torch.ones(H, dtype=BF16)
    n = O.input_rmsnorm(x, w, eps)
    expect = bf16_round(c / math.sqrt(c * c + eps))
    assert torch.all(n.to(torch.float64) == expect), (n[0, 0].item(), expect)


def test_rmsnorm_weight_is_per_column(O):
    # c * r rounds to 1 - 3e-7, so n_k is w_k itself (w_k bf16): pins the weight
    # indexing and that the weight multiplies after the normalisation.
    H = 5376
    g = torch.Generator().manual_seed(1)
    w = (torch.rand(H, generator=g) * 4 - 2).to(BF16)
    x = torch.full((3, H), 4.0, dtype=BF16)
    n = O.input_rmsnorm(x, w, 1e-5)
    assert torch.equal(bits(n[1]), bits(w))


def test_rmsnorm_matches_torch_rms_norm(O):
    # Library routine for the scale = shift = 0 special case of the norm.
    g = torch.Generator().manual_seed(2)
    H = 5376
    x = (torch.randn(64, H, generator=g) * torch.logspace(-3, 2, 64)[:, None]).to(BF16)
    w = (1 + 0.1 * torch.randn(H, generator=g)).to(BF16)
    n = O.input_rmsnorm(x, w, 1e-5)
    ref = torch.nn.functional.rms_norm(x.float(), (H,), weight=w.float(), eps=1e-5).to(BF16)
    d = (n.double() - ref.double()).abs()
    assert torch.all(d <= ulp_bf16(ref.double()))
    assert (d == 0).double().mean() > 0.99


# --------------------------------------------------------------- indexed AdaLN
# formula block lines a = ... and a[i outside [0, rows)] = 0;
# minimax_h3_bf16_pre_attention, Parameters: adaln_index, adaln_scale.

@pytest.mark.parametrize("n,scale,shift,expect", [
    # 1 + 3*2^-9 rounds up to 1.0078125; 100 * 1.0078125 = 100.78125 -> 101
    # (the unrounded gain would give 100.5859375 -> 100.5)
    (100.0, 3 * 2.0 ** -9, 0.0, 101.0),
    # 1 + 2^-8 is a tie: round-to-even gives gain 1.0, so a = 100
    # (the unrounded gain would give 100.390625 -> 100.5)
    (100.0, 2.0 ** -8, 0.0, 100.0),
    (1.0, 0.5, 0.25, 1.75),
    (-2.0, -1.0, 0.375, 0.375),  # gain 0: a = shift
    (1.0, 0.0, 2.0 ** -9, 1.0),  # 1 + 2^-9 rounds back to 1.0
])
def test_adaln_rounding_points(n, scale, shift, expect, O):
    H = 16
    nt = torch.full((1, H), n, dtype=BF16)
    sc = torch.full((1, H), scale, dtype=BF16)
    sh = torch.full((1, H), shift, dtype=BF16)
    a = O.indexed_adaln(nt, sc, sh, torch.zeros(1, dtype=torch.int64))
    assert torch.all(a.double() == expect), (a[0, 0].item(), expect)


def test_adaln_selects_row_by_index(O):
    rows, H = 5, 8
    sc = torch.stack([torch.full((H,), i / 8.0) for i in range(rows)]).to(BF16)
    sh = torch.stack([torch.full((H,), -i / 4.0) for i in range(rows)]).to(BF16)
    n = torch.ones(rows, H, dtype=BF16)
    idx = torch.tensor([3, 0, 4, 1, 2], dtype=torch.int64)
    a = O.indexed_adaln(n, sc, sh, idx)
    for m, i in enumerate(idx.tolist()):
        # n = 1: a = -i/4 + (1 + i/8), exact in bf16 for these i
        assert torch.all(a[m].double() == -i / 4.0 + 1 + i / 8.0)


def test_adaln_guard_rows_are_positive_zero(O):
    rows, H = 3, 32
    g = torch.Generator().manual_seed(3)
    sc = torch.randn(rows, H, generator=g).to(BF16)
    sh = torch.randn(rows, H, generator=g).to(BF16)
    bad = [-1, rows, 2 ** 40, -(2 ** 63), 2 ** 63 - 1, -(2 ** 40)]
    idx = torch.tensor(bad + [0, 2], dtype=torch.int64)
    n = torch.randn(len(idx), H, generator=g).to(BF16)
    a = O.indexed_adaln(n, sc, sh, idx)
    assert torch.all(bits(a[: len(bad)]) == 0)
    assert torch.all(a[len(bad):] != 0)


def test_adaln_strided_chunks_equal_contiguous_tables(O):
    rows, H = 9, 64
    g = torch.Generator().manual_seed(4)
    mod = torch.randn(rows, 6 * H, generator=g).to(BF16)
    sh, sc = mod[:, 0:H], mod[:, H:2 * H]
    assert sc.stride(0) == 6 * H
    n = torch.randn(20, H, generator=g).to(BF16)
    idx = torch.randint(0, rows, (20,), generator=g)
    a1 = O.indexed_adaln(n, sc, sh, idx)
    a2 = O.indexed_adaln(n, sc.contiguous(), sh.contiguous(), idx)
    assert torch.equal(bits(a1), bits(a2))


# -------------------------------------------------------------- QKV projection
# minimax_h3_bf16_pre_attention summary (BF16 QKV projection) and the FP32
# accumulation of the formula block of minimax_h3_mlp_fp8_sm120.

def test_qkv_projection_exact_integers(O):
    # Small-integer operands: every dot product is an integer; compare with
    # Python integer arithmetic, rounded once to bf16.
    rnd = random.Random(5)
    M, H, N = 3, 40, 12
    A = [[rnd.randint(-3, 3) for _ in range(H)] for _ in range(M)]
    W = [[rnd.randint(-2, 2) for _ in range(H)] for _ in range(N)]
    y = O.qkv_projection(torch.tensor(A, dtype=BF16), torch.tensor(W, dtype=BF16))
    for m in range(M):
        for c in range(N):
            s = sum(A[m][k] * W[c][k] for k in range(H))
            assert y[m, c].item() == bf16_round(float(s)), (m, c)


def test_qkv_projection_accumulates_in_fp32_not_bf16(O):
    # 512 terms of 2^-9: exact sum 1.0.  A bf16 running sum stalls at 0.5.
    H = 512
    a = torch.ones(1, H, dtype=BF16)
    W = torch.full((2, H), 2.0 ** -9, dtype=BF16)
    y = O.qkv_projection(a, W)
    assert torch.all(y.double() == 1.0)


def test_qkv_projection_one_hot_weight_is_a_gather(O):
    g = torch.Generator().manual_seed(6)
    M, H, N = 5, 96, 48
    a = torch.randn(M, H, generator=g).to(BF16)
    perm = torch.randint(0, H, (N,), generator=g)
    W = torch.zeros(N, H, dtype=BF16)
    W[torch.arange(N), perm] = 1.0
    y = O.qkv_projection(a, W)
    assert torch.equal(bits(y), bits(a[:, perm]))


def test_qkv_projection_rounds_once_to_bf16(O):
    # Exact sum 1 + 2^-8 + 2^-20 must round up (above the tie), while
    # rounding an FP32-truncated or bf16-accumulated sum would give 1.0.
    a = torch.tensor([[1.0, 1.0, 1.0]], dtype=BF16)
    W = torch.tensor([[1.0, 2.0 ** -8, 2.0 ** -20]], dtype=BF16)
    y = O.qkv_projection(a, W)
    assert y.item() == 1.0078125


# ------------------------------------------------------------- per-head norm
# minimax_h3_bf16_pre_attention, Parameters: q_norm_weight, k_norm_weight, qk_eps.

@pytest.mark.parametrize("c,eps", [(2.0 ** -8, 1e-5), (3.0, 1e-6), (-0.25, 1e-2)])
def test_head_norm_constant_head_closed_form(c, eps, O):
    D = 128
    y = torch.full((2, 3, D), c, dtype=BF16)
    t = O.head_rmsnorm(y, torch.ones(D, dtype=BF16), eps)
    assert torch.all(t.double() == bf16_round(c / math.sqrt(c * c + eps)))


def test_head_norm_unit_weight_has_unit_mean_square(O):
    g = torch.Generator().manual_seed(7)
    y = (torch.randn(50, 7, 128, generator=g) * 3).to(BF16)
    t = O.head_rmsnorm(y, torch.ones(128, dtype=BF16), 1e-6)
    ms = (t.double() ** 2).mean(-1)
    assert torch.all((ms - 1).abs() < 1e-2)


def test_head_norm_zero_head_is_zero_and_matches_library(O):
    g = torch.Generator().manual_seed(8)
    y = torch.randn(10, 4, 128, generator=g).to(BF16)
    y[3, 2] = 0
    w = (1 + 0.1 * torch.randn(128, generator=g)).to(BF16)
    t = O.head_rmsnorm(y, w, 1e-5)
    assert torch.all(t[3, 2] == 0)
    ref = torch.nn.functional.rms_norm(y.float(), (128,), weight=w.float(), eps=1e-5).to(BF16)
    d = (t.double() - ref.double()).abs()
    assert torch.all(d <= ulp_bf16(ref.double()))


# ---------------------------------------------------------------------- RoPE
# minimax_h3_bf16_pre_attention, Parameters: rope_cos_sin, rope_positions.

def _cache_rows(angles: torch.Tensor, RD: int = 96) -> torch.Tensor:
    half = RD // 2
    return torch.cat([torch.cos(angles), torch.sin(angles)], -1).to(F32).to(BF16).reshape(-1, RD)


def test_rope_zero_angle_is_identity(O):
    g = torch.Generator().manual_seed(9)
    t = torch.randn(4, 3, 128, generator=g).to(BF16)
    cs = _cache_rows(torch.zeros(1, 48, dtype=torch.float64))
    o = O.rope_split_half(t, cs, torch.zeros(4, dtype=torch.int64))
    assert torch.equal(bits(o), bits(t))


def test_rope_quarter_turn_pairs_j_with_j_plus_48(O):
    # cos = 0, sin = 1: o_j = -t_{j+48}, o_{j+48} = t_j exactly.
    g = torch.Generator().manual_seed(10)
    t = torch.randn(2, 5, 128, generator=g).to(BF16)
    cs = torch.cat([torch.zeros(1, 48), torch.ones(1, 48)], -1).to(BF16)
    o = O.rope_split_half(t, cs, torch.zeros(2, dtype=torch.int64))
    assert torch.equal(bits(o[..., :48]), bits(-t[..., 48:96]))
    assert torch.equal(bits(o[..., 48:96]), bits(t[..., :48]))
    assert torch.equal(bits(o[..., 96:]), bits(t[..., 96:]))


def test_rope_equals_complex_multiplication(O):
    # Library routine: (t_j + i t_{j+48}) * (cos + i sin) in complex128.
    g = torch.Generator().manual_seed(11)
    T = 16
    t = torch.randn(T, 6, 128, generator=g).to(BF16)
    ang = torch.rand(T, 48, generator=g, dtype=torch.float64) * 6.3
    cs = _cache_rows(ang)
    rows = torch.arange(T)
    o = O.rope_split_half(t, cs, rows)
    csf = cs.double()
    z = torch.complex(t[..., :48].double(), t[..., 48:96].double())
    r = z * torch.complex(csf[:, None, :48], csf[:, None, 48:])
    ref = torch.cat([r.real, r.imag], -1)
    d = (o[..., :96].double() - ref).abs()
    # two FP32 roundings plus one bf16 rounding of the result
    assert torch.all(d <= ulp_bf16(ref) + 1e-6 * (t[..., :96].double().abs().amax() + 1))
    assert torch.equal(bits(o[..., 96:]), bits(t[..., 96:]))


def test_rope_preserves_pair_norm(O):
    g = torch.Generator().manual_seed(12)
    t = torch.randn(64, 4, 128, generator=g).to(BF16)
    ang = torch.rand(64, 48, generator=g, dtype=torch.float64) * 100
    cs = _cache_rows(ang)
    o = O.rope_split_half(t, cs, torch.arange(64)).double()
    td = t.double()
    csd = cs.double()
    lhs = o[..., :48] ** 2 + o[..., 48:96] ** 2
    rhs = (td[..., :48] ** 2 + td[..., 48:96] ** 2) * (csd[:, None, :48] ** 2 + csd[:, None, 48:] ** 2)
    assert torch.all((lhs - rhs).abs() <= 0.02 * rhs + 1e-4)


def test_rope_positions_identity_and_clamp(O):
    S = 10
    tok = torch.arange(6)
    assert torch.equal(O.rope_cache_rows(None, tok, S), tok)
    assert torch.equal(O.rope_cache_rows(torch.arange(6), tok, S), tok)
    pos = torch.tensor([-1, S, S + 1, -(2 ** 63), 2 ** 63 - 1, 2 ** 40], dtype=torch.int64)
    rows = O.rope_cache_rows(pos, tok, S)
    assert rows.tolist() == [0, S - 1, S - 1, 0, S - 1, S - 1]


# ---------------------------------------------------------------------- pack
# minimax_h3_bf16_pre_attention, Parameters: out, ulysses_degree.

@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_pack_places_head_by_contiguous_block(P, O):
    M, NH, D = 3, 56, 4
    # distinct 16-bit patterns (moved, never computed on) carry each element's
    # (m, h, kind, d)
    code = torch.zeros(M, NH, 3, D, dtype=torch.int16)
    for m in range(M):
        for h in range(NH):
            for k in range(3):
                for d in range(D):
                    code[m, h, k, d] = ((m * 64 + h) * 3 + k) * 4 + d
    out = O.ulysses_pack(code.view(BF16), P).view(torch.int16)
    assert tuple(out.shape) == (P, M, NH // P, 3, D)
    hp = NH // P
    for p in range(P):
        for m in range(M):
            for hl in range(hp):
                for k in range(3):
                    for d in range(D):
                        assert out[p, m, hl, k, d] == ((m * 64 + p * hp + hl) * 3 + k) * 4 + d


def test_pack_repack_equivalence_and_unpack(O):
    g = torch.Generator().manual_seed(13)
    qkv = torch.randn(5, 56, 3, 8, generator=g).to(BF16)
    base = O.ulysses_pack(qkv, 1)[0]
    for P in (2, 4, 8):
        o = O.ulysses_pack(qkv, P)
        rep = o.permute(1, 0, 2, 3, 4).reshape(5, 56, 3, 8)
        assert torch.equal(bits(rep), bits(base))
        assert torch.equal(bits(O.ulysses_unpack_rows(o, [4, 0, 2])), bits(qkv[[4, 0, 2]]))


# ----------------------------------------------------- whole stage, full sizes

def _full_size_one_hot_case(O, P: int, positions_zero_angle: bool = True):
    """a-level one-hot construction at the production sizes: W row
    c = kind*7168 + h*128 + d* (d* = code(h, kind)) reads input column 0,
    every other row is zero.  Each Q/K/V head then holds one non-zero value
    at d*, which the pack must deliver to out[h // (56/P), m, h % (56/P), kind, d*]."""
    H, NH, D = 5376, 56, 128
    N = 3 * NH * D
    M = 3
    code = lambda h, k: (h + 37 * k) % 96 if k < 2 else (h * 2 + 1) % 128  # noqa: E731
    W = torch.zeros(N, H, dtype=BF16)
    for k in range(3):
        for h in range(NH):
            W[k * NH * D + h * D + code(h, k), 0] = 1.0
    # x rows chosen so that a[:, 0] != 0: scale = shift = 0 reduces a to n.
    x = torch.full((M, H), 1.0, dtype=BF16)
    x[:, 0] = torch.tensor([2.0, -3.0, 0.5])
    xw = torch.ones(H, dtype=BF16)
    sc = torch.zeros(1, H, dtype=BF16)
    idx = torch.zeros(M, dtype=torch.int64)
    qw = torch.ones(D, dtype=BF16)
    cs = torch.cat([torch.ones(1, 48), torch.zeros(1, 48)], -1).to(BF16).repeat(4, 1)
    out, a = O.pre_attention(x, xw, sc, sc, idx, W, qw, qw, cs, ulysses_degree=P,
                                  rope_positions=torch.zeros(M, dtype=torch.int64))
    return out, a, code


@pytest.mark.parametrize("P", [1, 8])
def test_stage_one_hot_head_mapping_full_size(P, O):
    out, a, code = _full_size_one_hot_case(O, P)
    NH, hp = 56, 56 // P
    nz = out != 0
    assert int(nz.sum()) == 3 * NH * 3  # one value per (token, head, kind)
    for h in range(NH):
        p, hl = divmod(h, hp)
        for k in range(3):
            d = code(h, k)
            vals = out[p, :, hl, k, d].double()
            if k == 2:
                assert torch.equal(vals, a[:, 0].double())  # V: the gathered a value
            else:
                # one non-zero y in the head: rms norm gives sign(y) * sqrt(128 / (1 + 128 eps / y^2))
                yv = a[:, 0].double()
                expect = [bf16_round(math.copysign(1, v) / math.sqrt(1 / 128 + 1e-5 / (v * v)))
                          for v in yv.tolist()]
                assert vals.tolist() == expect


def test_stage_qk_eps_none_uses_eps_and_distinct_qk_eps_changes_qk_only(O):
    g = torch.Generator().manual_seed(14)
    H, NH, D = 64, 4, 16
    N = 3 * NH * D
    M = 4
    x = torch.randn(M, H, generator=g).to(BF16)
    xw = torch.ones(H, dtype=BF16)
    tab = (0.1 * torch.randn(2, H, generator=g)).to(BF16)
    idx = torch.tensor([0, 1, 0, 1])
    W = (torch.randn(N, H, generator=g) * 1e-3).to(BF16)  # tiny heads: eps matters
    qw = torch.ones(D, dtype=BF16)
    cs = _cache_rows(torch.rand(M, 6, generator=g, dtype=torch.float64), RD=12)
    kw = dict(ulysses_degree=2, eps=1e-4)
    o_none, _ = O.pre_attention(x, xw, tab, tab, idx, W, qw, qw, cs, qk_eps=None, **kw)
    o_same, _ = O.pre_attention(x, xw, tab, tab, idx, W, qw, qw, cs, qk_eps=1e-4, **kw)
    o_diff, _ = O.pre_attention(x, xw, tab, tab, idx, W, qw, qw, cs, qk_eps=1e-1, **kw)
    assert torch.equal(bits(o_none), bits(o_same))
    assert not torch.equal(o_none[:, :, :, :2], o_diff[:, :, :, :2])
    assert torch.equal(bits(o_none[:, :, :, 2]), bits(o_diff[:, :, :, 2]))


def test_stage_identity_positions_need_enough_cache_rows(O):
    H, D = 32, 16
    x = torch.ones(4, H, dtype=BF16)
    t = torch.zeros(1, H, dtype=BF16)
    W = torch.zeros(3 * 2 * D, H, dtype=BF16)
    w = torch.ones(D, dtype=BF16)
    cs = torch.zeros(3, 12, dtype=BF16)
    with pytest.raises(ValueError):
        O.pre_attention(x, torch.ones(H, dtype=BF16), t, t, torch.zeros(4, dtype=torch.int64),
                             W, w, w, cs, ulysses_degree=1)


def test_stage_rows_are_independent_subset_is_exact(O):
    g = torch.Generator().manual_seed(15)
    H, NH, D, M = 48, 4, 16, 9
    x = torch.randn(M, H, generator=g).to(BF16)
    xw = (1 + 0.1 * torch.randn(H, generator=g)).to(BF16)
    tab = (0.1 * torch.randn(3, H, generator=g)).to(BF16)
    idx = torch.tensor([0, 1, 2, -1, 3, 1, 0, 2, 1])
    W = (torch.randn(3 * NH * D, H, generator=g) / 7).to(BF16)
    qw = (1 + 0.1 * torch.randn(D, generator=g)).to(BF16)
    kw = (1 + 0.1 * torch.randn(D, generator=g)).to(BF16)
    cs = _cache_rows(torch.rand(12, 5, generator=g, dtype=torch.float64), RD=10)
    pos = torch.tensor([3, -4, 11, 12, 0, 5, 100, 7, 2])
    full = O.pre_attention_tokens(x, xw, tab, tab, idx, W, qw, kw, cs, rope_positions=pos)
    sub = O.pre_attention_tokens(x, xw, tab, tab, idx, W, qw, kw, cs, rope_positions=pos,
                                      tokens=[8, 3, 1])
    assert torch.equal(bits(sub.qkv), bits(full.qkv[[8, 3, 1]]))
    assert torch.all(full.qkv[3] == 0)  # guarded index: the whole token is zero
