"""Pins of the e4m3 output-mode oracle (oracle/e4m3.py): closed-form codes of
the e4m3 format (bias 7, 3 mantissa bits, largest finite 448, no infinity),
round-to-nearest-even ties, saturation, and the per-kind scales."""
import math

import torch

from oracle import e4m3

BF16 = torch.bfloat16


def code(v: float, descale: float = 1.0) -> int:
    return int(e4m3.quantize_e4m3(torch.tensor([v], dtype=BF16), descale)[0])


def by_hand(v: float) -> int:
    """e4m3 bits of an exactly representable normal value, from the format."""
    s = 0x80 if v < 0 else 0
    a = abs(v)
    if a == 0:
        return s
    e = math.floor(math.log2(a))
    if e < -6:  # subnormal: value = m * 2^-9
        return s | int(round(a / 2 ** -9))
    m = a / 2 ** e - 1.0
    return s | ((e + 7) << 3) | int(round(m * 8))


def test_exact_values_have_their_format_codes():
    for v in [1.0, 1.125, 1.875, 2.0, 3.5, 448.0, 0.015625, 2 ** -9, 3 * 2 ** -9, -6.0, 240.0]:
        assert code(v) == by_hand(v), v


def test_largest_finite_and_saturation():
    assert code(448.0) == 0x7E
    assert code(480.0) == 0x7E and code(1e6) == 0x7E  # beyond 448 saturates
    assert code(-1e6) == 0xFE


def test_round_to_nearest_even_on_ties():
    # spacing in [1, 2) is 1/8: 1.0625 is halfway between 1.0 (even) and 1.125
    assert code(1.0625) == by_hand(1.0)
    # 1.1875 is halfway between 1.125 (odd mantissa 1) and 1.25 (even 2)
    assert code(1.1875) == by_hand(1.25)
    assert code(1.07) == by_hand(1.125)  # above the tie


def test_descale_divides_and_dequantize_inverts_exact_codes():
    assert code(3.0, descale=0.5) == by_hand(6.0)
    assert code(3.0, descale=4.0) == by_hand(0.75)
    c = e4m3.quantize_e4m3(torch.tensor([1.5, -0.25, 448.0], dtype=BF16), 2.0)
    assert e4m3.dequantize_e4m3(c, 2.0).tolist() == [1.5, -0.25, 448.0]


def test_packed_uses_the_scale_of_each_kind():
    out = torch.full((2, 3, 4, 3, 8), 3.0, dtype=BF16)
    codes = e4m3.quantize_packed(out, (1.0, 0.5, 4.0))
    assert torch.all(codes[:, :, :, 0] == by_hand(3.0))
    assert torch.all(codes[:, :, :, 1] == by_hand(6.0))
    assert torch.all(codes[:, :, :, 2] == by_hand(0.75))
