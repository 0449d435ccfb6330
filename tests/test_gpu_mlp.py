"""GPU parity of the BF16 MLP block (mh3_mlp_run, through the C ABI) against
the CPU oracle (oracle/mlp.py)."""
import pytest
import torch

from oracle import mlp
from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import make_mlp_workload

from parity_utils import check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle(cuda_lib):
    h = binding.Handle(torch.cuda.current_device())
    yield h
    torch.cuda.synchronize()
    h.close()


def _dev(w):
    mod = w.adaln_mod.cuda()
    sc, sh, gt = w.tables(mod)
    return dict(x=w.x.cuda(), xw=w.x_norm_weight.cuda(), mod=mod, sc=sc, sh=sh, gt=gt,
                idx=w.adaln_index.cuda(), res=w.residual.cuda(), fc1=w.fc1_weight.cuda(),
                fc2=w.fc2_weight.cuda())


def _run(h, d, M, out, wa=None, wy=None, x=None, res=None):
    x = d["x"] if x is None else x
    res = d["res"] if res is None else res
    binding.mh3_mlp_run(h, None, M, x, d["xw"], d["sc"], d["sc"].stride(0), d["sh"],
                        d["sh"].stride(0), d["gt"], d["gt"].stride(0), d["sc"].shape[0], d["idx"],
                        res, d["fc1"], d["fc2"], 1e-5, wa, wy, out)


def _oracle(w, tokens=None):
    sc, sh, gt = w.tables()
    return mlp.mlp_block(w.x, w.x_norm_weight, sc, sh, gt, w.adaln_index, w.residual,
                         w.fc1_weight, w.fc2_weight, eps=1e-5, tokens=tokens)


def _flat(t):
    return t.reshape(t.shape[0], 1, 1, -1)


@pytest.mark.parametrize("M", [16, 300, 2048])
def test_full_parity(handle, M):
    w = make_mlp_workload(M)
    d = _dev(w)
    out = torch.full((M, 5376), float("nan"), dtype=torch.bfloat16, device="cuda")
    wy = torch.full((M, 14336), float("nan"), dtype=torch.bfloat16, device="cuda")
    _run(handle, d, M, out, wy=wy)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    ref_out, _, ref_y = _oracle(w)
    sty = check_outputs(_flat(wy.cpu()), _flat(ref_y), f"mlp y M={M}")
    sto = check_outputs(_flat(out.cpu()), _flat(ref_out), f"mlp out M={M}")
    assert sty["exact"] > 0.98 and sto["exact"] > 0.98, (sty, sto)
    bad = (w.adaln_index < 0) | (w.adaln_index >= 9)
    if bool(bad.any()):
        assert torch.equal(out.cpu()[bad].view(torch.int16), w.residual[bad].view(torch.int16))
    print(M, sty, sto)


def test_production_size_sampled_parity_and_guard(handle):
    M = 32760
    w = make_mlp_workload(M)
    d = _dev(w)
    out = torch.empty((M, 5376), dtype=torch.bfloat16, device="cuda")
    _run(handle, d, M, out)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    bad = (w.adaln_index < 0) | (w.adaln_index >= 9)
    tokens = sorted(set(range(0, M, 128)) | {M - 1} | set(torch.nonzero(bad).flatten()[:16].tolist()))
    ref_out = _oracle(w, tokens)[0]
    st = check_outputs(_flat(out[tokens].cpu()), _flat(ref_out), "mlp sampled M=32760")
    assert st["exact"] > 0.98, st
    badd = bad.cuda()
    assert torch.equal(out[badd].view(torch.int16), d["res"][badd].view(torch.int16))
    assert bool(torch.isfinite(out).all())


def test_in_place_on_residual_or_x_and_handle_workspaces(handle):
    M = 520
    w = make_mlp_workload(M)
    d = _dev(w)
    ref = torch.empty((M, 5376), dtype=torch.bfloat16, device="cuda")
    wa = torch.empty((M, 5376), dtype=torch.bfloat16, device="cuda")
    wy = torch.empty((M, 14336), dtype=torch.bfloat16, device="cuda")
    _run(handle, d, M, ref, wa=wa, wy=wy)
    handle_ws = torch.empty_like(ref)
    _run(handle, d, M, handle_ws)  # handle-owned workspaces
    res_io = d["res"].clone()
    _run(handle, d, M, res_io, res=res_io)  # out is the residual
    x_io = d["x"].clone()
    _run(handle, d, M, x_io, x=x_io)  # out is x
    torch.cuda.synchronize()
    for t in (handle_ws, res_io, x_io):
        assert torch.equal(t.view(torch.int16), ref.view(torch.int16))
    assert handle.device_status() == 0
