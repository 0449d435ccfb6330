"""Pins of the FP8 MLP oracle (oracle/mlp_fp8.py) to facts that do not come
from the oracle: the e4m3 grid enumerated from the format definition, hand
roundings and ties, the per-token scale's closed form, quotients built to sit
one FP32 step from an e4m3 rounding boundary (where an FP32 division followed
by a second rounding gives another code than the formula's single rounding),
one-hot weights, and the guard
(flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, formula block)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mlp_fp8 as f8

BF16 = torch.bfloat16
F32 = torch.float32

# all non-negative finite e4m3 values, from the format: exponent bias 7,
# subnormals m/8 * 2^-6, the top code (S.1111.111) is NaN
E4M3 = [(c, (Fraction(c & 7, 8) * Fraction(1, 64)) if (c >> 3) == 0 else
         (1 + Fraction(c & 7, 8)) * Fraction(2) ** ((c >> 3) - 7)) for c in range(127)]


def nearest_code(q: Fraction) -> int:
    """Code of the nearest e4m3 value to q (ties to the even code), saturating."""
    sign = 0x80 if q < 0 else 0
    a = abs(q)
    if a >= 448:
        return sign | 126
    best = min(abs(a - v) for _, v in E4M3)
    near = [c for c, v in E4M3 if abs(a - v) == best]
    return sign | (near[0] if len(near) == 1 else [c for c in near if c % 2 == 0][0])


def test_e4m3_hand_table():
    # value -> code: 1.0 = 0x38; 1.0625 ties between 1.0 and 1.125 -> 1.0 (even);
    # 1.1875 ties between 1.125 and 1.25 -> 1.25 (0x3A); 464 and 1e6 saturate to 448;
    # 2^-10 ties between 0 and 2^-9 -> 0; 3*2^-10 ties between 2^-9 and 2^-8 -> 2^-8
    cases = [(1.0, 0x38), (1.0625, 0x38), (1.1875, 0x3A), (448.0, 0x7E), (464.0, 0x7E),
             (1e6, 0x7E), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (2.0 ** -9, 0x01),
             (-1.0, 0xB8), (-2.0 ** -11, 0x80), (0.0, 0x00), (-0.0, 0x80)]
    v = torch.tensor([c[0] for c in cases], dtype=torch.float64)
    assert f8.e4m3_codes(f8.e4m3_round(v)).tolist() == [c[1] for c in cases]


def test_e4m3_is_the_nearest_value_brute_force():
    g = torch.Generator().manual_seed(31)
    v = torch.cat([torch.exp2(torch.rand(400, generator=g, dtype=torch.float64) * 20 - 11) *
                   torch.sign(torch.rand(400, generator=g, dtype=torch.float64) - 0.5),
                   torch.arange(-8, 8, 0.0625, dtype=torch.float64)])
    got = f8.e4m3_codes(f8.e4m3_round(v)).tolist()
    for x, c in zip(v.tolist(), got):
        if x == 0:
            continue
        assert c == nearest_code(Fraction(x)), (x, c, nearest_code(Fraction(x)))


def test_row_scale_closed_form_and_amax_element_maps_to_448():
    g = torch.Generator().manual_seed(32)
    a = (torch.randn(8, 64, generator=g) * torch.logspace(-2, 2, 8)[:, None]).to(BF16)
    codes, s = f8.quantize_rows(a)
    amax = a.float().abs().amax(-1)
    assert torch.equal(s, (amax / torch.tensor(448.0)).to(F32))
    # the element of largest magnitude lands at +-448 (exactly, or saturated)
    arg = a.float().abs().argmax(-1)
    c = codes[torch.arange(8), arg]
    assert bool(((c == 0x7E) | (c == 0xFE)).all())


SINGLE_ROUNDING_CASES = [(1.03125, 1.375), (1.171875, 1.5625), (1.6171875, 2.15625),
                         (1.6875, 2.25), (1.8984375, 2.53125)]


@pytest.mark.parametrize("a,amax", SINGLE_ROUNDING_CASES)
def test_quantisation_rounds_the_exact_quotient_once(a, amax):
    # a / s lies just above the midpoint 336 of 320 and 352, but the FP32
    # quotient RN32(a / s) lands on 336 and its e4m3 rounding would go to 320
    row = torch.tensor([[amax, a, -a] + [0.0] * 13], dtype=BF16)
    codes, s = f8.quantize_rows(row)
    exact = nearest_code(Fraction(a) / Fraction(float(s[0])))
    q32 = np.float32(np.float32(a) / np.float32(s[0]))
    twice = nearest_code(Fraction(float(q32)))
    assert exact != twice
    assert codes[0, 1].item() == exact and codes[0, 2].item() == exact | 0x80


def test_zero_row_has_zero_scale_and_codes():
    row = torch.zeros(2, 32, dtype=BF16)
    row[1, 5] = -0.0
    codes, s = f8.quantize_rows(row)
    assert s.tolist() == [0.0, 0.0]
    assert int(codes.sum()) == 0


def test_scaled_projection_one_hot_closed_form():
    g = torch.Generator().manual_seed(33)
    a = (torch.randn(4, 64, generator=g) * 3).to(BF16)
    codes, s = f8.quantize_rows(a)
    ks = torch.tensor([0, 7, 33, 63, 5])
    w = torch.zeros(5, 64, dtype=torch.uint8)
    w[torch.arange(5), ks] = 0x38                      # e4m3 1.0
    ws = torch.tensor([0.125, 1.0, 3.0, 0.5, 2.0 ** -20], dtype=F32)
    h = f8.scaled_projection(codes, s, w, ws)
    av = f8.e4m3_values(codes[:, ks]).to(F32)           # exact e4m3 values, [4, 5]
    expect = torch.mul(torch.mul(av, s[:, None]), ws[None, :]).to(BF16)
    assert torch.equal(h.view(torch.int16), expect.view(torch.int16))


def test_projection_accumulates_exact_products():
    # codes 0x38 (1.0) and 0x30 (0.5) times 0x20 (0.125): small sums exact in FP32
    a = torch.full((1, 256), 0x38, dtype=torch.uint8)
    a[0, ::2] = 0x30
    w = torch.full((3, 256), 0x20, dtype=torch.uint8)
    h = f8.scaled_projection(a, torch.tensor([1.0]), w, torch.ones(3))
    assert h.double().tolist() == [[24.0, 24.0, 24.0]]  # 128 * (0.5 + 1.0) * 0.125


def test_block_guard_token_returns_the_residual():
    g = torch.Generator().manual_seed(34)
    H, I = 64, 32
    x = torch.randn(3, H, generator=g).to(BF16)
    xw = torch.ones(H, dtype=BF16)
    tab = (0.1 * torch.randn(2, H, generator=g)).to(BF16)
    gate = torch.randn(2, H, generator=g).to(BF16)
    idx = torch.tensor([0, -1, 1])
    res = torch.randn(3, H, generator=g).to(BF16)
    fc1 = torch.randint(0, 0x70, (2 * I, H), generator=g).to(torch.uint8)
    fc2 = torch.randint(0, 0x70, (H, I), generator=g).to(torch.uint8)
    ws1 = torch.rand(2 * I, generator=g) * 1e-2
    ws2 = torch.rand(H, generator=g) * 1e-2
    r = f8.mlp_block_fp8(x, xw, tab, tab, gate, idx, res, fc1, ws1, fc2, ws2)
    assert torch.equal(r["out"][1].view(torch.int16), res[1].view(torch.int16))
    assert int(r["a_q"][1].sum()) == 0 and r["s_a"][1].item() == 0.0
    assert not torch.equal(r["out"][0], res[0])
