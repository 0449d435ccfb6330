"""A tiny, fully specified input of the stage with shrunken sizes
(H=24, 4 heads of 8, 6 rotary dims, rows=3, P=2), built from integers so it
is identical on every machine."""
import torch

BF16 = torch.bfloat16


def _ramp(n, mod, scale, off=0):
    return torch.tensor([((i * 7 + off) % mod - mod // 2) * scale for i in range(n)],
                        dtype=torch.float32).to(BF16)


def tiny_inputs():
    H, NH, D, RD, rows, M, S = 24, 4, 8, 6, 3, 5, 6
    x = _ramp(M * H, 23, 0.125).reshape(M, H)
    xw = (1 + _ramp(H, 5, 0.0625, 1).float()).to(BF16)
    mod = _ramp(rows * 3 * H, 11, 0.03125, 2).reshape(rows, 3 * H)
    shift, scale = mod[:, 0:H], mod[:, H:2 * H]
    idx = torch.tensor([0, 2, -1, 1, 3], dtype=torch.int64)
    W = _ramp(3 * NH * D * H, 13, 0.0625, 3).reshape(3 * NH * D, H)
    qw = (1 + _ramp(D, 3, 0.125, 4).float()).to(BF16)
    kw = (1 + _ramp(D, 3, 0.125, 5).float()).to(BF16)
    cs = torch.tensor([[((s * 3 + j) % 9 - 4) * 0.25 for j in range(RD)] for s in range(S)],
                      dtype=torch.float32).to(BF16)
    pos = torch.tensor([5, -2, 0, 9, 3], dtype=torch.int64)
    args = (x, xw, scale, shift, idx, W, qw, kw, cs)
    kw_ = dict(ulysses_degree=2, eps=1e-5, qk_eps=1e-3, rope_positions=pos)
    return args, kw_
