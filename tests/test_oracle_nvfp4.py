"""Pins of the NVFP4 oracle (oracle/nvfp4.py) to facts that do not come from
the oracle (flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention, summary
and Parameters): hand-derived E2M1 and UE4M3 roundings, worked quantisation
examples, the E2M1 rounding bound, one-hot weights, and the bf16 stage's
oracle on inputs that NVFP4 represents exactly."""
from fractions import Fraction

import pytest
import torch

import oracle
from oracle import nvfp4 as f

BF16 = torch.bfloat16


def test_e2m1_hand_table():
    # value -> code, worked by hand: nearest of {0,.5,1,1.5,2,3,4,6}, ties to
    # the even code (0, 1.0, 2.0, 4.0 have even codes 0, 2, 4, 6), saturating
    cases = [(0.0, 0), (0.2, 0), (0.25, 0), (0.3, 1), (0.74, 1), (0.75, 2), (1.25, 2), (1.26, 3),
             (1.75, 4), (2.5, 4), (2.6, 5), (3.5, 6), (5.0, 6), (5.01, 7), (6.0, 7), (1e9, 7),
             (-0.25, 8), (-0.26, 9), (-1.75, 12), (-6.5, 15)]
    x = torch.tensor([c[0] for c in cases], dtype=torch.float64)
    assert f.e2m1_codes(x).tolist() == [c[1] for c in cases]
    assert f.e2m1_codes(torch.tensor([-0.0])).item() == 8  # sign kept on zero


def test_e2m1_is_the_nearest_value_brute_force():
    vals = [Fraction(v).limit_denominator() for v in f.E2M1_VALUES]
    g = torch.Generator().manual_seed(3)
    xs = torch.cat([torch.rand(400, generator=g, dtype=torch.float64) * 8,
                    torch.arange(0, 7.0, 0.125, dtype=torch.float64)])
    codes = f.e2m1_codes(xs)
    for x, c in zip(xs.tolist(), codes.tolist()):
        fx = Fraction(x)
        dist = [abs(fx - v) for v in vals]
        best = min(dist)
        near = [i for i, d in enumerate(dist) if d == best]
        want = near[0] if len(near) == 1 else [i for i in near if i % 2 == 0][0]
        if fx > 6:
            want = 7
        assert c == want, (x, c, want)


def test_ue4m3_brute_force():
    # all positive finite e4m3 values, enumerated from the format definition
    vals = []
    for code in range(0, 127):
        e, m = code >> 3, code & 7
        vals.append(Fraction(m, 8) * Fraction(1, 2 ** 6) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    g = torch.Generator().manual_seed(4)
    xs = torch.cat([torch.exp2(torch.rand(300, generator=g) * 20 - 11), torch.tensor([0.0, 448.0, 460.0, 1e6])])
    codes = f.ue4m3_codes(xs)
    for x, c in zip(xs.tolist(), codes.tolist()):
        fx = min(Fraction(x), Fraction(448))
        dist = [abs(fx - v) for v in vals]
        best = min(dist)
        near = [i for i, d in enumerate(dist) if d == best]
        want = near[0] if len(near) == 1 else [i for i in near if i % 2 == 0][0]
        assert c == want, (x, c, want)


def test_quantize_worked_examples():
    # block 0: amax 6, gs 1 -> t = 1, s = 1.0 (0x38), enc 1: codes are the values
    # block 1: amax 12, gs 1 -> s = 2.0 (0x40), enc 0.5: 12 -> 6 (7), -6 -> -3 (13), 1 -> 0.5 (1)
    b0 = [6.0, -3.0, 1.5, 0.5, -0.5, 2.0, 4.0, -1.0] + [0.0] * 8
    b1 = [12.0, -6.0, 1.0, 0.0] + [0.0] * 12
    a = torch.tensor([b0 + b1], dtype=BF16)
    q, s = f.fp4_quantize(a, 1.0)
    assert s.tolist() == [[0x38, 0x40]]
    codes = f.unpack_codes(q)[0].tolist()
    assert codes[:8] == [7, 13, 3, 1, 9, 4, 6, 10]
    assert codes[16:20] == [7, 13, 1, 0]
    # packing: element 0 in the low nibble
    assert q[0, 0].item() == 7 | (13 << 4)
    # gs = 336 (448 * 6 / 8), amax 8: t = 8/6 * 336 = 448 -> s = 448 (0x7E),
    # enc = 336/448 = 0.75; 8 -> 6 (7); 1 -> 0.75 -> tie .5/1 -> 1.0 (2)
    a2 = torch.tensor([[8.0, 1.0] + [0.0] * 14], dtype=BF16)
    q2, s2 = f.fp4_quantize(a2, 336.0)
    assert s2.item() == 0x7E and f.unpack_codes(q2)[0, :2].tolist() == [7, 2]
    # an all-zero block: scale 0, codes 0
    q3, s3 = f.fp4_quantize(torch.zeros(1, 32, dtype=BF16), 100.0)
    assert s3.tolist() == [[0, 0]] and int(q3.sum()) == 0


def test_quantize_error_bound():
    """Each element lands within half an E2M1 step of a * enc (or saturates)."""
    g = torch.Generator().manual_seed(5)
    a = (torch.randn(64, 256, generator=g) * 3).to(BF16)
    gs = 448.0 * 6 / 12.0
    q, s = f.fp4_quantize(a, gs)
    sv = f.ue4m3_values(s).to(torch.float64).repeat_interleave(16, dim=1)
    enc = torch.where(sv == 0, 0.0, torch.tensor(gs, dtype=torch.float32).double() / sv)
    scaled = a.double() * enc
    v = f.e2m1_values(f.unpack_codes(q))
    step = torch.where(v.abs() < 2, 0.5, torch.where(v.abs() < 4, 1.0, 2.0))
    err = (scaled - v).abs()
    sat = scaled.abs() > 6
    assert bool(((err <= step / 2 + 1e-6) | sat).all())
    # saturation only by the rounding of the block scale (at most 1/16 above 6)
    assert float(scaled.abs().max()) <= 6 * (1 + 1 / 16) + 1e-6


def test_alpha_closed_form():
    assert f.alpha_from_scales(2.0, 4.0) == 0.125
    assert f.alpha_from_scales(448.0 * 6, 1.0) == float(torch.tensor(1 / 2688.0, dtype=torch.float32))


def test_projection_one_hot_weight():
    g = torch.Generator().manual_seed(6)
    a = (torch.randn(5, 64, generator=g) * 2).to(BF16)
    aq, asf = f.fp4_quantize(a, 50.0)
    # weight row c: code 2 (1.0) at element k(c), scale 1.0 (0x38)
    N, K = 8, 64
    ks = torch.tensor([0, 1, 17, 33, 63, 5, 16, 48])
    codes = torch.zeros(N, K, dtype=torch.uint8)
    codes[torch.arange(N), ks] = 2
    wq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)
    wsf = torch.full((N, K // 16), 0x38, dtype=torch.uint8)
    y = f.nvfp4_projection(aq, asf, wq, wsf, 0.25)
    qa = f.e2m1_values(f.unpack_codes(aq))
    sa = f.ue4m3_values(asf).double()
    exp = torch.stack([qa[:, k] * sa[:, k // 16] for k in ks.tolist()], dim=1)
    assert torch.equal(y, (exp.float() * 0.25).to(BF16))


def _representable_inputs(M=6, H=64, N=12, seed=7):
    """bf16 a whose every 16-block has amax 6 and E2M1 values, and an E2M1
    weight with the same property: NVFP4 with unit global scales is exact."""
    g = torch.Generator().manual_seed(seed)
    def grid(rows, cols):
        c = torch.randint(0, 16, (rows, cols), generator=g, dtype=torch.uint8)
        c[:, ::16] = 7  # amax 6 in every block
        return f.e2m1_values(c).float()
    return grid(M, H), grid(N, H)


def test_projection_matches_bf16_oracle_on_exact_inputs():
    a, w = _representable_inputs()
    aq, asf = f.fp4_quantize(a.to(BF16), 1.0)
    wq, wsf = f.fp4_quantize(w.to(BF16), 1.0)
    assert torch.equal(f.dequantize(aq, asf, 1.0), a.double())
    assert asf.unique().tolist() == [0x38]
    y = f.nvfp4_projection(aq, asf, wq, wsf, 1.0)
    assert torch.equal(y.view(torch.int16), oracle.qkv_projection(a.to(BF16), w.to(BF16)).view(torch.int16))


def test_stage_matches_bf16_oracle_when_nvfp4_is_exact():
    """The NVFP4 stage composes the bf16 stage's oracle steps: its GEMM equals
    the bf16 GEMM of the dequantised operands (with an exactly representable
    weight), and its tail is the bf16 Q/K norm (eps) and RoPE (token-index
    positions)."""
    g = torch.Generator().manual_seed(8)
    M, H = 3, 5376
    # zero AdaLN tables: a = n
    codes = torch.randint(0, 16, (M, H), generator=g, dtype=torch.uint8)
    codes[:, ::16] = 7
    x = f.e2m1_values(codes).float()
    x = x.to(BF16)
    xw = torch.ones(H, dtype=BF16)
    sc = torch.zeros(1, H, dtype=BF16)
    sh = torch.zeros(1, H, dtype=BF16)
    idx = torch.zeros(M, dtype=torch.int32)
    n = oracle.input_rmsnorm(x, xw, 1e-30)
    wc = torch.randint(0, 16, (21504, H), generator=g, dtype=torch.uint8)
    wc[:, ::16] = 7
    w = f.e2m1_values(wc).to(BF16)
    wq, wsf = f.fp4_quantize(w, 1.0)
    cs = torch.randn(M, 96, generator=g).to(BF16)
    qn = (1 + 0.1 * torch.randn(128, generator=g)).to(BF16)
    kn = (1 + 0.1 * torch.randn(128, generator=g)).to(BF16)
    got = f.pre_attention_nvfp4_tokens(x, xw, sc, sh, idx, wq, wsf, 1.0, 1.0, qn, kn, cs,
                                       eps=1e-30)
    # zero tables: a = n (by value; shift 0 turns -0 into +0)
    assert torch.equal(got.a.float(), n.float())
    # the NVFP4 GEMM equals the bf16 oracle's GEMM of the dequantised operands
    # (e2m1 * ue4m3 values are exact in bf16; the weight dequantises to w)
    a_deq = f.dequantize(got.act_q, got.act_sf, 1.0).to(BF16)
    assert torch.equal(f.dequantize(wq, wsf, 1.0).to(BF16).view(torch.int16), w.view(torch.int16))
    y_ref = oracle.qkv_projection(a_deq, w)
    assert torch.equal(got.y.view(torch.int16), y_ref.view(torch.int16))
    # the norm/RoPE tail: the bf16 oracle's own functions, eps for the Q/K norm
    y4 = y_ref.view(M, 3, 56, 128)
    for kind, wn in ((0, qn), (1, kn)):
        t = oracle.rope_split_half(oracle.head_rmsnorm(y4[:, kind], wn, 1e-30), cs, torch.arange(M))
        assert torch.equal(got.qkv[:, :, kind].view(torch.int16), t.view(torch.int16))
    assert torch.equal(got.qkv[:, :, 2].view(torch.int16), y4[:, 2].view(torch.int16))


# ------------------------------------------------ single rounding at midpoints
# flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj, summary: the block-16
# convention sf = UE4M3(block_amax * act_global_scale / 6) and
# code = RN(x * act_global_scale / sf), one rounding of each exact quotient.
# The cases below are built so that the exact quotient lies within one FP32
# step of a rounding boundary: there the old two-rounding order
# (RN32(RN32(amax / 6) * gs), RN32(x * RN32(gs / sf))) gives another code,
# and exact rational arithmetic decides which one the formula means.

import numpy as np  # noqa: E402

UE4M3_ALL = [(c, (Fraction(c & 7, 8) * Fraction(1, 64)) if (c >> 3) == 0 else
              (1 + Fraction(c & 7, 8)) * Fraction(2) ** ((c >> 3) - 7)) for c in range(127)]
E2M1_ALL = [(c, Fraction(v).limit_denominator()) for c, v in enumerate(f.E2M1_VALUES)]


def _nearest(q: Fraction, table, top):
    """Code of the nearest table value to q >= 0, ties to the even code,
    values above the largest saturating to it."""
    if q >= top:
        return table[-1][0]
    best = min(abs(q - v) for _, v in table)
    near = [c for c, v in table if abs(q - v) == best]
    return near[0] if len(near) == 1 else [c for c in near if c % 2 == 0][0]


def _f32(v) -> float:
    return float(np.float32(v))


def _f32_steps(v: float, k: int) -> float:
    return float(np.array([v], dtype=np.float32).view(np.int32).__add__(k).view(np.float32)[0])


def _scale_cases():
    cases = []
    mids = [(UE4M3_ALL[c][1] + UE4M3_ALL[c + 1][1]) / 2 for c in (8, 9, 13, 44, 57, 70, 100)]
    for m in mids:
        for amax in (1.5, 3.0, 5.25, 7.0, 9.5, 11.0, 13.0, 19.0, 23.0, 29.0, 37.0, 53.0):
            g0 = _f32(float(6 * m) / amax)
            for k in range(-3, 4):
                gs = _f32_steps(g0, k)
                exact = _nearest(Fraction(amax) * Fraction(gs) / 6, UE4M3_ALL, Fraction(448))
                t2 = _f32(np.float32(_f32(np.float32(amax) / np.float32(6.0))) * np.float32(gs))
                two = _nearest(Fraction(t2), UE4M3_ALL, Fraction(448))
                if exact != two:
                    cases.append((amax, gs, exact, two))
    return cases


def test_scale_is_one_rounding_of_the_exact_quotient():
    cases = _scale_cases()
    assert len(cases) >= 5, len(cases)
    for amax, gs, exact, two in cases:
        a = torch.tensor([[amax] + [0.0] * 15], dtype=BF16)
        _, s = f.fp4_quantize(a, gs)
        assert s.item() == exact != two, (amax, gs, s.item(), exact, two)


def test_scale_exact_ties_go_to_even():
    # amax * 1 / 6 = 1.0625, halfway between 1.0 (0x38) and 1.125 (0x39): even -> 1.0
    # 7.125 / 6 = 1.1875, halfway between 1.125 (0x39) and 1.25 (0x3A): even -> 1.25
    a = torch.tensor([[6.375] + [0.0] * 15 + [7.125] + [0.0] * 15], dtype=BF16)
    _, s = f.fp4_quantize(a, 1.0)
    assert s.tolist() == [[0x38, 0x3A]]


def _element_cases():
    cases = []
    for sf_code in (0x39, 0x3B, 0x3D, 0x3F, 0x4B, 0x2D):
        sf = UE4M3_ALL[sf_code][1]
        for lo, hi in zip(E2M1_ALL[:-1], E2M1_ALL[1:]):
            me = (lo[1] + hi[1]) / 2
            for x in (0.3125, 0.5625, 0.8125, 1.0625, 1.4375, 1.8125, 2.6875, 3.0625):
                g0 = _f32(float(me * sf) / x)
                for k in range(-3, 4):
                    gs = _f32_steps(g0, k)
                    exact = _nearest(Fraction(x) * Fraction(gs) / sf, E2M1_ALL, Fraction(6))
                    enc = np.float32(np.float32(gs) / np.float32(float(sf)))
                    two = _nearest(Fraction(_f32(np.float32(x) * enc)), E2M1_ALL, Fraction(6))
                    if exact == two:
                        continue
                    # a block whose amax gives exactly this sf at this gs
                    amax = float(torch.tensor(float(6 * sf) / gs).to(BF16))
                    if amax < x or _nearest(Fraction(amax) * Fraction(gs) / 6, UE4M3_ALL,
                                            Fraction(448)) != sf_code:
                        continue
                    cases.append((x, amax, gs, sf_code, exact, two))
    return cases


def test_element_code_is_one_rounding_of_the_exact_quotient():
    cases = _element_cases()
    assert len(cases) >= 5, len(cases)
    for x, amax, gs, sf_code, exact, two in cases:
        a = torch.tensor([[x, -x, amax] + [0.0] * 13], dtype=BF16)
        q, s = f.fp4_quantize(a, gs)
        codes = f.unpack_codes(q)[0].tolist()
        assert s.item() == sf_code
        assert codes[0] == exact != two, (x, gs, codes[0], exact, two)
        assert codes[1] == exact | 8  # the same magnitude, sign kept


# ---------------------------------------------- W4A4 output projection
def _exact_out_proj_inputs(M, K, N, gs_a, gs_w, seed):
    """attn_out and o_weight whose every 16-block is e2m1 values times a
    power of two p (one 6 per block) divided by the global scale: the block
    scale is then p exactly and every code is the e2m1 value, so NVFP4 is
    lossless."""
    g = torch.Generator().manual_seed(seed)
    def grid(rows, gs):
        c = torch.randint(0, 16, (rows, K), generator=g, dtype=torch.uint8)
        c[:, ::16] = 7                                           # amax 6
        p = torch.exp2(torch.randint(-2, 3, (rows, K // 16), generator=g).double())
        v = f.e2m1_values(c) * p.repeat_interleave(16, dim=1) / gs
        return v.to(BF16)
    return grid(M, gs_a), grid(N, gs_w)


def test_out_proj_nvfp4_equals_bf16_out_proj_when_exact():
    """With lossless operands and power-of-two global scales (alpha exact),
    the W4A4 projection with the gated residual is the BF16 output
    projection's oracle bit for bit, bad gate indices included."""
    from oracle import out_proj as op
    M, K, N = 7, 128, 40
    gs_a, gs_w = 4.0, 0.5
    a, w = _exact_out_proj_inputs(M, K, N, gs_a, gs_w, seed=21)
    wq, wsf = f.fp4_quantize(w, gs_w)
    assert torch.equal(f.dequantize(wq, wsf, gs_w), w.double())
    g = torch.Generator().manual_seed(22)
    gate = torch.randn(3, N, generator=g).to(BF16)
    gi = torch.tensor([0, 2, -1, 1, 3, 2, 2 ** 30], dtype=torch.int32)
    res = torch.randn(M, N, generator=g).to(BF16)
    got = f.out_proj_nvfp4(a, wq, wsf, gs_w, gs_a, gate, gi, res)
    assert got["alpha"] == 0.5
    assert torch.equal(f.dequantize(got["act_q"], got["act_sf"], gs_a), a.double())
    ref = op.out_proj_gated_residual(a, w, gate, gi, res)
    assert torch.equal(got["out"].view(torch.int16), ref.view(torch.int16))
    for m in (2, 6):  # bad index: out is the residual
        assert torch.equal(got["out"][m].view(torch.int16), res[m].view(torch.int16))


def test_out_proj_nvfp4_token_subset_is_row_subset():
    g = torch.Generator().manual_seed(23)
    M, K, N = 9, 64, 24
    a = torch.randn(M, K, generator=g).to(BF16)
    w = (torch.randn(N, K, generator=g) / 8).to(BF16)
    wq, wsf = f.fp4_quantize(w, 448.0 * 6 / 0.75)
    gate = torch.randn(2, N, generator=g).to(BF16)
    gi = torch.tensor([0, 1, 1, 0, -1, 1, 0, 1, 2], dtype=torch.int32)
    res = torch.randn(M, N, generator=g).to(BF16)
    full = f.out_proj_nvfp4(a, wq, wsf, 448.0 * 6 / 0.75, 336.0, gate, gi, res)
    sub = f.out_proj_nvfp4(a, wq, wsf, 448.0 * 6 / 0.75, 336.0, gate, gi, res, tokens=[8, 3, 4])
    assert torch.equal(sub["out"].view(torch.int16), full["out"][[8, 3, 4]].view(torch.int16))
    assert torch.equal(sub["act_q"], full["act_q"][[8, 3, 4]])


def test_output_quantisation_is_lossless_per_kind():
    """Rows built to be exact in NVFP4 under their own kind's global scale
    (three different scales) dequantise back bit for bit; a kind read with
    another kind's scale, or a row landing in another (token, head, kind)
    slot, would not."""
    g = torch.Generator().manual_seed(31)
    T, H = 3, 5
    gss = (4.0, 0.25, 64.0)
    qkv = torch.empty(T, H, 3, 128, dtype=BF16)
    for kind, gs in enumerate(gss):
        c = torch.randint(0, 16, (T * H, 128), generator=g, dtype=torch.uint8)
        c[:, ::16] = 7
        p = torch.exp2(torch.randint(-3, 3, (T * H, 8), generator=g).double()).repeat_interleave(16, 1)
        qkv[:, :, kind] = (f.e2m1_values(c) * p / gs).to(BF16).view(T, H, 128)
    codes, sf = f.quantize_outputs(qkv, gss)
    assert codes.shape == (T, H, 3, 64) and sf.shape == (T, H, 3, 8)
    for kind, gs in enumerate(gss):
        deq = f.dequantize(codes[:, :, kind].reshape(T * H, 64), sf[:, :, kind].reshape(T * H, 8), gs)
        assert torch.equal(deq, qkv[:, :, kind].reshape(T * H, 128).double()), kind
    # the three kinds' scales differ by the ratio of their global scales
    assert not torch.equal(sf[:, :, 0], sf[:, :, 1])
