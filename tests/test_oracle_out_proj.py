"""Pins of the out-projection oracle (oracle/out_proj.py) to facts that do
not come from the oracle: exact integer sums, one-hot gathers, the guard
(out = residual), and a hand-derived case where rounding gate * o to bf16
before the residual add changes the result
(flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj, summary formula)."""
import random

import torch

from oracle import out_proj as op

BF16 = torch.bfloat16


def bits(t):
    return t.contiguous().view(torch.int16)


def bf16_round(v: float) -> float:
    return torch.tensor(v, dtype=torch.float64).to(torch.float32).to(BF16).item()


def test_unit_gate_zero_residual_is_the_projection_exact_integers():
    rnd = random.Random(31)
    M, K, N = 4, 48, 10
    A = [[rnd.randint(-3, 3) for _ in range(K)] for _ in range(M)]
    W = [[rnd.randint(-2, 2) for _ in range(K)] for _ in range(N)]
    gate = torch.ones(2, N, dtype=BF16)
    out = op.out_proj_gated_residual(torch.tensor(A, dtype=BF16), torch.tensor(W, dtype=BF16), gate,
                                     torch.zeros(M, dtype=torch.int32),
                                     torch.zeros(M, N, dtype=BF16))
    for m in range(M):
        for c in range(N):
            s = sum(A[m][k] * W[c][k] for k in range(K))
            assert out[m, c].item() == bf16_round(float(s)), (m, c)


def test_one_hot_weight_gathers_the_input_columns():
    g = torch.Generator().manual_seed(32)
    M, K, N = 6, 40, 24
    a = torch.randn(M, K, generator=g).to(BF16)
    pi = torch.randint(0, K, (N,), generator=g)
    W = torch.zeros(N, K, dtype=BF16)
    W[torch.arange(N), pi] = 1.0
    out = op.out_proj_gated_residual(a, W, torch.ones(1, N, dtype=BF16),
                                     torch.zeros(M, dtype=torch.int32), torch.zeros(M, N, dtype=BF16))
    assert torch.equal(bits(out), bits(a[:, pi]))


def test_guarded_index_returns_the_residual_bit_for_bit():
    g = torch.Generator().manual_seed(33)
    M, K, N, rows = 7, 32, 16, 9
    a = torch.randn(M, K, generator=g).to(BF16)
    W = torch.randn(N, K, generator=g).to(BF16)
    gate = torch.randn(rows, N, generator=g).to(BF16)
    res = torch.randn(M, N, generator=g).to(BF16)
    idx = torch.tensor([-1, rows, 2 ** 30, -(2 ** 31), 2 ** 31 - 1, 0, 8], dtype=torch.int32)
    out = op.out_proj_gated_residual(a, W, gate, idx, res)
    assert torch.equal(bits(out[:5]), bits(res[:5]))
    assert not torch.equal(bits(out[5:]), bits(res[5:]))


def test_gate_times_o_is_rounded_before_the_residual_add():
    # o = 3 (one-hot), g = 1 + 2^-7: g*o = 3.0234375 is a bf16 tie between
    # 3.015625 and 3.03125 -> round-to-even 3.03125; -1.5 + 3.03125 = 1.53125.
    # Adding the unrounded 3.0234375 would give 1.5234375 instead.
    K, N = 8, 2
    a = torch.zeros(1, K, dtype=BF16)
    a[0, 0] = 3.0
    W = torch.zeros(N, K, dtype=BF16)
    W[:, 0] = 1.0
    gate = torch.full((1, N), 1.0078125, dtype=BF16)
    res = torch.full((1, N), -1.5, dtype=BF16)
    out = op.out_proj_gated_residual(a, W, gate, torch.zeros(1, dtype=torch.int32), res)
    assert torch.all(out.double() == 1.53125)


def test_gate_row_is_selected_by_index_and_strided_views_match():
    g = torch.Generator().manual_seed(34)
    M, K, N, rows = 5, 16, 32, 9
    a = torch.randn(M, K, generator=g).to(BF16)
    W = torch.randn(N, K, generator=g).to(BF16)
    mod = torch.randn(rows, 6 * N, generator=g).to(BF16)
    gate = mod[:, 2 * N:3 * N]
    res = torch.randn(M, N, generator=g).to(BF16)
    idx = torch.tensor([3, 0, 8, 3, 1], dtype=torch.int32)
    out = op.out_proj_gated_residual(a, W, gate, idx, res)
    out2 = op.out_proj_gated_residual(a, W, gate.contiguous(), idx, res)
    assert torch.equal(bits(out), bits(out2))
    # rows 0 and 3 share gate row 3 and differ only through their inputs
    o = op.out_projection(a, W)
    for m, i in enumerate(idx.tolist()):
        one = op.gated_residual(o[m:m + 1], gate[i:i + 1], torch.zeros(1, dtype=torch.int32),
                                res[m:m + 1])
        assert torch.equal(bits(out[m:m + 1]), bits(one))


def test_token_subset_is_exact():
    g = torch.Generator().manual_seed(35)
    M, K, N = 9, 24, 16
    a = torch.randn(M, K, generator=g).to(BF16)
    W = torch.randn(N, K, generator=g).to(BF16)
    gate = torch.randn(3, N, generator=g).to(BF16)
    res = torch.randn(M, N, generator=g).to(BF16)
    idx = torch.tensor([0, 1, 2, -1, 1, 0, 2, 5, 1], dtype=torch.int32)
    full = op.out_proj_gated_residual(a, W, gate, idx, res)
    sub = op.out_proj_gated_residual(a, W, gate, idx, res, tokens=[8, 3, 0])
    assert torch.equal(bits(sub), bits(full[[8, 3, 0]]))


def test_projection_is_rounded_to_bf16_before_the_gate():
    # acc = 1 + 2^-8 + 2^-20 rounds (above the tie) to o = 1.0078125; with
    # g = 1.5, g*o = 1.51171875 is a tie -> even 1.515625.  Gating the
    # unrounded accumulator would give 1.50586... -> 1.5078125.
    K, N = 4, 3
    a = torch.tensor([[1.0, 1.0, 1.0, 0.0]], dtype=BF16)
    W = torch.tensor([[1.0, 2.0 ** -8, 2.0 ** -20, 0.0]] * N, dtype=BF16)
    gate = torch.full((1, N), 1.5, dtype=BF16)
    out = op.out_proj_gated_residual(a, W, gate, torch.zeros(1, dtype=torch.int32),
                                     torch.zeros(1, N, dtype=BF16))
    assert torch.all(out.double() == 1.515625)
