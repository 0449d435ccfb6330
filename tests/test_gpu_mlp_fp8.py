"""GPU parity of the FP8 (W8A8) MLP block (flashinfer.diffusion_ops.
minimax_h3_mlp_fp8_sm120, formula block) through the C ABI, against the oracle
(oracle/mlp_fp8.py):

* the quantised activation: codes and per-token scale bit for bit against
  the oracle's quantiser applied to the bf16 activation kernel 1 writes;
* y against the oracle's fc1 + SwiGLU on the GPU's own codes (same operands
  of the contraction: only the FP32 summation order and expf differ);
* y's codes and scale bit for bit against the oracle's quantiser applied to
  the GPU's y;
* out against the oracle's fc2 + gated residual on the GPU's own y codes, and
  against the oracle's whole block, under the stage's bar
  (|d| <= 2e-2 |ref| + 2e-2, mean <= 2e-3); guarded tokens bit for bit equal
  to the residual.
"""
import pytest
import torch

from oracle import mlp_fp8 as f8
from oracle import out_proj as op
from oracle.mlp import swiglu
from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import make_mlp_fp8_workload

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


@pytest.fixture(scope="module")
def handle(cuda_lib):
    h = binding.Handle(torch.cuda.current_device())
    yield h
    torch.cuda.synchronize()
    h.close()


@pytest.fixture(scope="module")
def weights():
    w = make_mlp_fp8_workload(1)
    return dict(fc1_q=w.fc1_q.cuda(), fc1_s=w.fc1_scale.cuda(), fc2_q=w.fc2_q.cuda(),
                fc2_s=w.fc2_scale.cuda(), host=w)


def _bar(g, r, what, exact_min=None):
    g, r = g.double(), r.double()
    assert torch.isfinite(g).all(), what
    err = (g - r).abs()
    bad = err > 2e-2 * r.abs() + 2e-2
    assert not bool(bad.any()), (what, int(bad.sum()), float(err.max()))
    assert float(err.mean()) <= 2e-3, (what, float(err.mean()))
    ex = float((g == r).double().mean())
    if exact_min is not None:
        assert ex >= exact_min, (what, ex)
    return ex


def _run(handle, wl, wt, out=None, same_residual=False):
    M = wl.M
    dev = "cuda"
    mod = wl.adaln_mod.to(dev)
    sc, sh, gt = wl.tables(mod)
    x, xw, idx = wl.x.to(dev), wl.x_norm_weight.to(dev), wl.adaln_index.to(dev)
    res = wl.residual.to(dev)
    ws = dict(aq=torch.full((M, 5376), 0xEE, dtype=torch.uint8, device=dev),
              as_=torch.full((M,), -1.0, device=dev),
              y=torch.empty((M, 14336), dtype=BF16, device=dev),
              yq=torch.full((M, 14336), 0xEE, dtype=torch.uint8, device=dev),
              ys=torch.full((M,), -1.0, device=dev))
    if same_residual:
        out = res
    elif out is None:
        out = torch.full((M, 5376), float("nan"), dtype=BF16, device=dev)
    binding.mh3_mlp_fp8_run(handle, None, M, x, xw, sc, sc.stride(0), sh, sh.stride(0), gt,
                            gt.stride(0), sc.shape[0], idx, res, wt["fc1_q"], wt["fc1_s"],
                            wt["fc2_q"], wt["fc2_s"], wl.eps, ws["aq"], ws["as_"], ws["y"],
                            ws["yq"], ws["ys"], out)
    # the bf16 activation of the same kernel arithmetic (kernel 1, bf16 form)
    a = torch.empty((M, 5376), dtype=BF16, device=dev)
    binding.mh3_preattn_norm_adaln(handle, None, M, x, xw, sc, sc.stride(0), sh, sh.stride(0),
                                   sc.shape[0], idx, wl.eps, a)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    return {k: v.cpu() for k, v in ws.items()}, a.cpu(), out.cpu()


@pytest.mark.parametrize("M", [300, 16, 257])
def test_fp8_mlp_parity(handle, weights, M):
    base = weights["host"]
    wl = make_mlp_fp8_workload(M)
    wl.fc1_q, wl.fc1_scale, wl.fc2_q, wl.fc2_scale = base.fc1_q, base.fc1_scale, base.fc2_q, \
        base.fc2_scale
    ws, a, out = _run(handle, wl, weights)
    sc, sh, gt = wl.tables()
    # 1. quantised activation, bit for bit
    aq, s_a = f8.quantize_rows(a)
    assert torch.equal(ws["as_"], s_a)
    assert torch.equal(ws["aq"], aq), int((ws["aq"] != aq).sum())
    # 2. y from the GPU's own codes
    y_ref = swiglu(f8.scaled_projection(ws["aq"], ws["as_"], wl.fc1_q, wl.fc1_scale))
    _bar(ws["y"], y_ref, f"y M={M}", exact_min=0.95)
    # 3. y codes and scale, bit for bit on the GPU's y
    yq, s_y = f8.quantize_rows(ws["y"])
    assert torch.equal(ws["ys"], s_y)
    assert torch.equal(ws["yq"], yq), int((ws["yq"] != yq).sum())
    # 4. out from the GPU's own y codes
    o = f8.scaled_projection(ws["yq"], ws["ys"], wl.fc2_q, wl.fc2_scale)
    ref_own = op.gated_residual(o, gt, wl.adaln_index, wl.residual)
    _bar(out, ref_own, f"out (own codes) M={M}", exact_min=0.95)
    # 5. the whole block against the oracle end to end
    full = f8.mlp_block_fp8(wl.x, wl.x_norm_weight, sc, sh, gt, wl.adaln_index, wl.residual,
                            wl.fc1_q, wl.fc1_scale, wl.fc2_q, wl.fc2_scale, eps=wl.eps)
    _bar(out, full["out"], f"out (oracle block) M={M}")
    # guarded tokens: out is the residual bit for bit, codes and scales zero
    bad = (wl.adaln_index < 0) | (wl.adaln_index >= gt.shape[0])
    if bool(bad.any()):
        assert torch.equal(out[bad].view(torch.int16), wl.residual[bad].view(torch.int16))
        assert int(ws["aq"][bad].sum()) == 0 and bool((ws["as_"][bad] == 0).all())


def test_fp8_mlp_in_place_on_residual_and_handle_workspaces(handle, weights):
    base = weights["host"]
    wl = make_mlp_fp8_workload(200, seed=777)
    wl.fc1_q, wl.fc1_scale, wl.fc2_q, wl.fc2_scale = base.fc1_q, base.fc1_scale, base.fc2_q, \
        base.fc2_scale
    _, _, ref = _run(handle, wl, weights)
    # the same call writing over the residual, with handle-owned workspaces
    dev = "cuda"
    mod = wl.adaln_mod.to(dev)
    sc, sh, gt = wl.tables(mod)
    res = wl.residual.to(dev)
    binding.mh3_mlp_fp8_run(handle, None, wl.M, wl.x.to(dev), wl.x_norm_weight.to(dev), sc,
                            sc.stride(0), sh, sh.stride(0), gt, gt.stride(0), sc.shape[0],
                            wl.adaln_index.to(dev), res, weights["fc1_q"], weights["fc1_s"],
                            weights["fc2_q"], weights["fc2_s"], wl.eps, None, None, None, None,
                            None, res)
    torch.cuda.synchronize()
    assert torch.equal(res.cpu().view(torch.int16), ref.view(torch.int16))


def test_fp8_mlp_invalid_arguments_and_empty(handle, weights):
    wl = make_mlp_fp8_workload(8)
    dev = "cuda"
    mod = wl.adaln_mod.to(dev)
    sc, sh, gt = wl.tables(mod)
    out = torch.full((8, 5376), 3.0, dtype=BF16, device=dev)
    args = [wl.x.to(dev), wl.x_norm_weight.to(dev), sc, sc.stride(0), sh, sh.stride(0), gt,
            gt.stride(0), sc.shape[0], wl.adaln_index.to(dev), wl.residual.to(dev),
            weights["fc1_q"], weights["fc1_s"], weights["fc2_q"], weights["fc2_s"], 1e-5,
            None, None, None, None, None, out]
    bad = list(args)
    bad[3] = 5375  # scale row stride below 5376
    with pytest.raises(RuntimeError, match="MH3_ERR_INVALID_ARG"):
        binding.mh3_mlp_fp8_run(handle, None, 8, *bad)
    bad = list(args)
    bad[12] = None  # missing fc1 scales
    with pytest.raises(RuntimeError, match="MH3_ERR_INVALID_ARG"):
        binding.mh3_mlp_fp8_run(handle, None, 8, *bad)
    binding.mh3_mlp_fp8_run(handle, None, 0, *args)  # M = 0: nothing to do
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())


def test_fp8_mlp_production_size_sampled(handle, weights):
    """M = 32760 in the bench's launch configuration; the oracle on a sample
    of tokens (every 512th, the last, and the guarded ones)."""
    base = weights["host"]
    wl = make_mlp_fp8_workload(32760)
    wl.fc1_q, wl.fc1_scale, wl.fc2_q, wl.fc2_scale = base.fc1_q, base.fc1_scale, base.fc2_q, \
        base.fc2_scale
    ws, a, out = _run(handle, wl, weights)
    sc, sh, gt = wl.tables()
    bad = (wl.adaln_index < 0) | (wl.adaln_index >= gt.shape[0])
    tokens = sorted(set(range(0, wl.M, 512)) | {wl.M - 1} |
                    set(torch.nonzero(bad).flatten().tolist()[:24]))
    t = torch.tensor(tokens)
    aq, s_a = f8.quantize_rows(a[t])
    assert torch.equal(ws["aq"][t], aq) and torch.equal(ws["as_"][t], s_a)
    yq, s_y = f8.quantize_rows(ws["y"][t])
    assert torch.equal(ws["yq"][t], yq) and torch.equal(ws["ys"][t], s_y)
    full = f8.mlp_block_fp8(wl.x, wl.x_norm_weight, sc, sh, gt, wl.adaln_index, wl.residual,
                            wl.fc1_q, wl.fc1_scale, wl.fc2_q, wl.fc2_scale, eps=wl.eps,
                            tokens=tokens)
    _bar(out[t], full["out"], "out (oracle block) M=32760 sampled")
    assert torch.equal(out[bad].view(torch.int16), wl.residual[bad].view(torch.int16))
    assert bool(torch.isfinite(out.double()).all())
