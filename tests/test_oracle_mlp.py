"""Pins of the MLP-block oracle (oracle/mlp.py) to facts that do not come
from the oracle: torch's silu for the activation, a hand-derived case that
fails if h_gate and h_up are swapped, one-hot weights, and the guard
(flashinfer.diffusion_ops.minimax_h3_mlp_fp8_sm120, formula block)."""
import torch

from oracle import mlp

BF16 = torch.bfloat16


def bits(t):
    return t.contiguous().view(torch.int16)


def test_swiglu_matches_torch_silu_times_up():
    g = torch.Generator().manual_seed(51)
    h = (torch.randn(64, 2 * 96, generator=g) * 4).to(BF16)
    y = mlp.swiglu(h)
    ref = (torch.nn.functional.silu(h[:, :96].double()).float().to(BF16).float()
           * h[:, 96:].float()).to(BF16)
    assert torch.equal(bits(y), bits(ref))


def test_swiglu_gate_half_comes_first():
    # h_gate = 2, h_up = 3: silu(2) = 1.76159... -> bf16 1.7578125; times 3 =
    # 5.2734375 -> bf16 5.28125.  With the halves swapped: silu(3) = 2.85772...
    # -> 2.859375; times 2 = 5.71875.
    h = torch.tensor([[2.0, 3.0]], dtype=BF16)
    assert mlp.swiglu(h).item() == 5.28125


def test_swiglu_closed_forms():
    h = torch.tensor([[0.0, 7.0, 20.0, -20.0, 5.0, 0.0, 2.5, 1.0]], dtype=BF16)
    y = mlp.swiglu(h)
    assert y[0, 0].item() == 0.0                # silu(0) = 0
    assert y[0, 1].item() == 0.0                # h_up = 0
    assert y[0, 2].item() == 50.0               # silu(20) rounds to 20; 20 * 2.5
    assert -1e-7 < y[0, 3].item() < 0           # silu(-20) = -4.1e-8


def test_block_one_hot_weights_and_guard():
    g = torch.Generator().manual_seed(52)
    M, H, I = 6, 32, 8
    x = torch.randn(M, H, generator=g).to(BF16)
    xw = torch.ones(H, dtype=BF16)
    rows = 3
    mod = (0.1 * torch.randn(rows, 6 * H, generator=g)).to(BF16)
    shift, scale, gate = mod[:, 0:H], mod[:, H:2 * H], mod[:, 2 * H:3 * H]
    idx = torch.tensor([0, 2, -1, 1, rows, 0], dtype=torch.int64)
    res = torch.randn(M, H, generator=g).to(BF16)
    # fc1: gate row j reads input column j, up row j reads column I + j
    fc1 = torch.zeros(2 * I, H, dtype=BF16)
    fc1[torch.arange(I), torch.arange(I)] = 1.0
    fc1[I + torch.arange(I), I + torch.arange(I)] = 1.0
    # fc2: output column c reads y column c % I
    fc2 = torch.zeros(H, I, dtype=BF16)
    fc2[torch.arange(H), torch.arange(H) % I] = 1.0
    out, a, y = mlp.mlp_block(x, xw, scale, shift, gate, idx, res, fc1, fc2, eps=1e-5)
    # one-hot fc1: y_j = bf16(bf16(silu(a_j)) * a_{I+j}) with torch's silu
    exp_y = (torch.nn.functional.silu(a[:, :I].double()).float().to(BF16).float()
             * a[:, I:2 * I].float()).to(BF16)
    assert torch.equal(bits(y), bits(exp_y))
    # guarded tokens: zero activation, zero gate -> out is the residual
    for m in (2, 4):
        assert torch.all(bits(a[m]) == 0)
        assert torch.equal(bits(out[m]), bits(res[m]))
    # one-hot fc2: o_c = y_{c % I} exactly
    o = y[:, torch.arange(H) % I]
    ok = [0, 1, 3, 5]
    gg = gate[idx[ok]].float()
    exp_out = (res[ok].float() + (gg * o[ok].float()).to(BF16).float()).to(BF16)
    assert torch.equal(bits(out[ok]), bits(exp_out))


def test_block_token_subset_is_exact():
    g = torch.Generator().manual_seed(53)
    M, H, I = 7, 24, 6
    x = torch.randn(M, H, generator=g).to(BF16)
    xw = (1 + 0.1 * torch.randn(H, generator=g)).to(BF16)
    mod = (0.1 * torch.randn(2, 3 * H, generator=g)).to(BF16)
    sh, sc, gt = mod[:, :H], mod[:, H:2 * H], mod[:, 2 * H:]
    idx = torch.tensor([0, 1, -1, 1, 0, 2, 1])
    res = torch.randn(M, H, generator=g).to(BF16)
    fc1 = (torch.randn(2 * I, H, generator=g) / 5).to(BF16)
    fc2 = (torch.randn(H, I, generator=g) / 3).to(BF16)
    full = mlp.mlp_block(x, xw, sc, sh, gt, idx, res, fc1, fc2)[0]
    sub = mlp.mlp_block(x, xw, sc, sh, gt, idx, res, fc1, fc2, tokens=[6, 2, 0])[0]
    assert torch.equal(bits(sub), bits(full[[6, 2, 0]]))
