"""GPU parity of the attention output projection with the fused gated
residual (mh3_out_proj_run, through the C ABI) against the CPU oracle."""
import pytest
import torch

from oracle import out_proj as op
from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import make_out_proj_workload

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
    return dict(a=w.attn_out.cuda(), W=w.o_weight.cuda(), mod=mod, gate=w.gate_view(mod),
                gi=w.gate_index.cuda(), res=w.residual.cuda())


def _run(h, d, M, out):
    g = d["gate"]
    binding.mh3_out_proj_run(h, None, M, d["a"], d["W"], g, g.stride(0), g.shape[0], d["gi"],
                             d["res"], out)


def _cmp(gpu, ref, what):
    # [T, 5376] -> the [T, 56, 3, 128]-free comparison rules of the stage outputs
    return check_outputs(gpu.view(gpu.shape[0], 1, 1, -1), ref.view(ref.shape[0], 1, 1, -1), what)


@pytest.mark.parametrize("M", [16, 1, 300, 4096])
def test_full_parity(handle, M):
    w = make_out_proj_workload(M)
    d = _dev(w)
    out = torch.full((M, 5376), float("nan"), dtype=torch.bfloat16, device="cuda")
    _run(handle, d, M, out)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    ref = op.out_proj_gated_residual(w.attn_out, w.o_weight, w.gate_view(), w.gate_index,
                                     w.residual)
    st = _cmp(out.cpu(), ref, f"out_proj M={M}")
    assert st["exact"] > 0.99, st
    bad = (w.gate_index < 0) | (w.gate_index >= 9)
    if bool(bad.any()):
        assert torch.equal(out.cpu()[bad].view(torch.int16), w.residual[bad].view(torch.int16))
    print(M, st)


def test_production_size_sampled_parity_and_guard(handle):
    M = 32760
    w = make_out_proj_workload(M)
    d = _dev(w)
    out = torch.empty((M, 5376), dtype=torch.bfloat16, device="cuda")
    _run(handle, d, M, out)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    bad = (w.gate_index < 0) | (w.gate_index >= 9)
    tokens = sorted(set(range(0, M, 64)) | {M - 1} | set(torch.nonzero(bad).flatten()[:32].tolist()))
    ref = op.out_proj_gated_residual(w.attn_out, w.o_weight, w.gate_view(), w.gate_index,
                                     w.residual, tokens=tokens)
    st = _cmp(out[tokens].cpu(), ref, "out_proj sampled M=32760")
    assert st["exact"] > 0.99, st
    badd = bad.cuda()
    assert int(bad.sum()) > 0
    assert torch.equal(out[badd].view(torch.int16), d["res"][badd].view(torch.int16))
    assert bool(torch.isfinite(out).all())


def test_in_place_on_the_residual_matches(handle):
    M = 700
    w = make_out_proj_workload(M)
    d = _dev(w)
    out = torch.empty((M, 5376), dtype=torch.bfloat16, device="cuda")
    _run(handle, d, M, out)
    inplace = d["res"].clone()
    d2 = dict(d, res=inplace)
    _run(handle, d2, M, inplace)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), inplace.view(torch.int16))


def test_one_hot_weight_unit_gate_zero_residual_is_an_exact_gather(handle):
    g = torch.Generator().manual_seed(41)
    M = 333
    a = torch.randn(M, 7168, generator=g).to(torch.bfloat16)
    pi = torch.randint(0, 7168, (5376,), generator=g)
    W = torch.zeros(5376, 7168, dtype=torch.bfloat16)
    W[torch.arange(5376), pi] = 1.0
    gate = torch.ones(1, 5376, dtype=torch.bfloat16)
    d = dict(a=a.cuda(), W=W.cuda(), gate=gate.cuda(), gi=torch.zeros(M, dtype=torch.int32).cuda(),
             res=torch.zeros(M, 5376, dtype=torch.bfloat16).cuda())
    out = torch.empty((M, 5376), dtype=torch.bfloat16, device="cuda")
    _run(handle, d, M, out)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().view(torch.int16), a[:, pi].view(torch.int16))


def test_zero_tokens_and_invalid_arguments(handle):
    w = make_out_proj_workload(8)
    d = _dev(w)
    out = torch.full((8, 5376), 3.0, dtype=torch.bfloat16, device="cuda")
    g = d["gate"]
    binding.mh3_out_proj_run(handle, None, 0, None, d["W"], g, g.stride(0), 9, None, None, None)
    with pytest.raises(RuntimeError, match="gate_rows"):
        binding.mh3_out_proj_run(handle, None, 8, d["a"], d["W"], g, g.stride(0), 0, d["gi"],
                                 d["res"], out)
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    assert handle.device_status() == 0
