"""CPU checks of the comparison rules the GPU parity tests apply.

* The workspace rule accepts a row whose FP32 sum of squares was taken in
  another order (emulated here in plain FP32, on the CPU), and rejects a row
  with any other change.
* bf16(1 + scale) computed as an FP32 addition rounded to bf16 (the oracle)
  equals the single rounding of the exact sum (a bf16 addition, as kernel 1
  does it) for every finite bf16 scale, so the AdaLN gain is not a source of
  difference between the two.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from norm_adaln_qkv_gb300.inputs import make_workload
from parity_utils import check_workspace

BF16 = torch.bfloat16


def _reordered_workspace(wl, ref):
    """Kernel-1-like workspace: the sum of squares in FP32 over 224 strided
    partials, then the oracle's own FP32 steps from that r."""
    x = wl.x.float().numpy()
    T, H = x.shape
    sq = (x * x).astype(np.float32)
    part = np.zeros((T, 224), dtype=np.float32)
    for j in range(H // 224):
        part += sq[:, j * 224:(j + 1) * 224]
    ss = np.zeros(T, dtype=np.float32)
    for j in range(224):
        ss = (ss + part[:, j]).astype(np.float32)
    ms = (ss / np.float32(H)).astype(np.float32)
    r = (np.float32(1.0) / np.sqrt((ms + np.float32(wl.spec.eps)).astype(np.float32))).astype(
        np.float32)
    n = oracle.rmsnorm_apply(wl.x, wl.x_norm_weight, torch.from_numpy(r))
    sc, sh = wl.table_views()
    return oracle.indexed_adaln(n, sc, sh, wl.adaln_index), torch.from_numpy(r)


def test_workspace_rule_accepts_reordered_sum_and_rejects_other_changes():
    wl = make_workload("c2", M=300)
    ref = oracle.pre_attention_tokens(*_args(wl), **_kw(wl))
    a, r = _reordered_workspace(wl, ref)
    assert not torch.equal(r, ref.r)  # the order does move r in some rows
    st = check_workspace(a, ref, wl, "reordered")
    assert st["exact_rows"] + st["rows_with_moved_r"] == 300
    # one element moved by one bf16 step in an otherwise exact row
    t = st["rows"] - 1
    while not torch.equal(a[t].view(torch.int16), ref.a[t].view(torch.int16)) or \
            not (0 <= int(wl.adaln_index[t]) < wl.spec.rows):
        t -= 1
    bad = a.clone()
    bad.view(torch.int16)[t, 17] += 1
    with pytest.raises(AssertionError):
        check_workspace(bad, ref, wl, "planted")
    # a guarded row that is not +0
    g = int(torch.nonzero((wl.adaln_index < 0) | (wl.adaln_index >= wl.spec.rows))[0])
    bad = a.clone()
    bad[g, 5] = -0.0
    with pytest.raises(AssertionError):
        check_workspace(bad, ref, wl, "guard")


def _args(wl):
    sc, sh = wl.table_views()
    return (wl.x, wl.x_norm_weight, sc, sh, wl.adaln_index, wl.qkv_weight, wl.q_norm_weight,
            wl.k_norm_weight, wl.rope_cos_sin)


def _kw(wl):
    return dict(eps=wl.spec.eps, qk_eps=wl.spec.qk_eps, rope_positions=wl.rope_positions)


def _bf16_nearest(q: Fraction) -> Fraction:
    """Nearest bf16 value of an exact rational (ties to even), normal range."""
    if q == 0:
        return q
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    step = Fraction(2) ** (max(e, -126) - 7)
    k = a / step
    lo = k.numerator // k.denominator
    rem = k - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * lo * step


def test_gain_fp32_then_bf16_equals_single_rounding_for_every_bf16_scale():
    codes = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    s = codes.view(BF16)
    fin = torch.isfinite(s.float())
    s = s[fin]
    two_step = (1.0 + s.float()).to(BF16).double()  # FP32 add, then bf16
    vals = s.double().tolist()
    got = two_step.tolist()
    for v, g in zip(vals, got):
        want = _bf16_nearest(1 + Fraction(v))
        assert Fraction(g) == want, (v, g, float(want))
