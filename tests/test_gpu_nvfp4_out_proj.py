"""GPU parity of the W4A4 attention output projection with the fused gated
residual (flashinfer.diffusion_ops.minimax_h3_nvfp4_out_proj, summary and
Parameters) through the C ABI, against the oracle (oracle/nvfp4.py):

* the weight quantised by the library's quantiser at K = 7168: codes and
  scales bit for bit against the oracle's quantiser;
* the activation codes and scales the call leaves in act_q / act_sf, bit for
  bit against the oracle's quantisation of attn_out (the same bf16 input, so
  every decision is the same);
* out against the oracle's whole operation under the stage's bar
  (|d| <= 2e-2 |ref| + 2e-2, mean <= 2e-3): the contraction has the same
  operands on both sides, only the FP32 summation order differs; tokens with
  a bad gate index bit for bit equal to the residual.
"""
import pytest
import torch

from oracle import nvfp4 as f
from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import make_out_proj_workload, out_proj_nvfp4_global_scales

from parity_utils import check_outputs, untile

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16
N, K = 5376, 7168
ACT_GS, W_GS = out_proj_nvfp4_global_scales()


@pytest.fixture(scope="module")
def handle(cuda_lib):
    h = binding.Handle(torch.cuda.current_device())
    yield h
    torch.cuda.synchronize()
    h.close()


@pytest.fixture(scope="module")
def weight(cuda_lib):
    """o_weight of the seeded workload, quantised on the GPU (tiled scales)
    and checked against the oracle's quantiser."""
    W = make_out_proj_workload(1).o_weight
    q = torch.empty(N, K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.full((binding.load().mh3_nvfp4_scales_bytes(N, K, 1),), 0xEE, dtype=torch.uint8,
                    device="cuda")
    g = torch.tensor([W_GS], dtype=torch.float32, device="cuda")
    binding.mh3_nvfp4_quantize(None, W.cuda(), g, q, sf, True)
    torch.cuda.synchronize()
    ref_q, ref_s = f.fp4_quantize(W, W_GS)
    assert torch.equal(untile(sf.cpu(), N, K), ref_s)
    assert torch.equal(q.cpu(), ref_q), int((q.cpu() != ref_q).sum())
    return dict(W=W, q=ref_q, sf=ref_s, q_dev=q, sf_dev=sf)


def _workload(M, weight, seed=None):
    w = make_out_proj_workload(M) if seed is None else make_out_proj_workload(M, seed=seed)
    w.o_weight = weight["W"]
    return w


def _run(h, w, weight, out=None, act_q=None, act_sf=None, same_residual=False):
    M = w.M
    mod = w.adaln_mod.cuda()
    gate = w.gate_view(mod)
    res = w.residual.cuda()
    if act_q is None:
        act_q = torch.full((M, K // 2), 0xEE, dtype=torch.uint8, device="cuda")
    if act_sf is None:
        act_sf = torch.full((max(binding.load().mh3_nvfp4_scales_bytes(M, K, 1), 1),), 0xEE,
                            dtype=torch.uint8, device="cuda")
    if same_residual:
        out = res
    elif out is None:
        out = torch.full((M, N), float("nan"), dtype=BF16, device="cuda")
    gs = torch.tensor([ACT_GS], dtype=torch.float32, device="cuda")
    binding.mh3_nvfp4_out_proj_run(h, None, M, w.attn_out.cuda(), weight["q_dev"],
                                   weight["sf_dev"], W_GS, gs, gate, gate.stride(0),
                                   gate.shape[0], w.gate_index.cuda(), res, act_q, act_sf, out)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    return act_q.cpu(), act_sf.cpu(), out.cpu()


def _cmp(gpu, ref, what):
    return check_outputs(gpu.view(gpu.shape[0], 1, 1, -1), ref.view(ref.shape[0], 1, 1, -1), what)


def _bad(w):
    return (w.gate_index < 0) | (w.gate_index >= w.adaln_mod.shape[0])


@pytest.mark.parametrize("M", [300, 16, 1, 257])
def test_parity(handle, weight, M):
    w = _workload(M, weight)
    aq, asf, out = _run(handle, w, weight)
    ref = f.out_proj_nvfp4(w.attn_out, weight["q"], weight["sf"], W_GS, ACT_GS, w.gate_view(),
                           w.gate_index, w.residual)
    assert torch.equal(untile(asf, M, K), ref["act_sf"])
    assert torch.equal(aq, ref["act_q"]), int((aq != ref["act_q"]).sum())
    st = _cmp(out, ref["out"], f"nvfp4 out_proj M={M}")
    assert st["exact"] > 0.95, st
    bad = _bad(w)
    if bool(bad.any()):
        assert torch.equal(out[bad].view(torch.int16), w.residual[bad].view(torch.int16))
    print(M, st)


def test_in_place_handle_workspaces_and_torch_entry(handle, weight):
    """out written over the residual with handle-owned workspaces, and the
    torch entry point, are bit-identical to the call with caller workspaces."""
    w = _workload(200, weight, seed=4242)
    _, _, ref = _run(handle, w, weight)
    mod = w.adaln_mod.cuda()
    gate = w.gate_view(mod)
    res = w.residual.cuda()
    gs = torch.tensor([ACT_GS], dtype=torch.float32, device="cuda")
    binding.mh3_nvfp4_out_proj_run(handle, None, w.M, w.attn_out.cuda(), weight["q_dev"],
                                   weight["sf_dev"], W_GS, gs, gate, gate.stride(0),
                                   gate.shape[0], w.gate_index.cuda(), res, None, None, res)
    torch.cuda.synchronize()
    assert torch.equal(res.cpu().view(torch.int16), ref.view(torch.int16))
    got = binding.minimax_h3_nvfp4_out_proj(w.attn_out.cuda(), weight["q_dev"], weight["sf_dev"],
                                            torch.tensor([W_GS]), gs, gate, w.gate_index.cuda(),
                                            w.residual.cuda(), handle=handle)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu().view(torch.int16), ref.view(torch.int16))


def test_invalid_arguments_and_empty(handle, weight):
    w = _workload(8, weight)
    mod = w.adaln_mod.cuda()
    gate = w.gate_view(mod)
    gs = torch.tensor([ACT_GS], dtype=torch.float32, device="cuda")
    out = torch.full((8, N), 3.0, dtype=BF16, device="cuda")
    args = [w.attn_out.cuda(), weight["q_dev"], weight["sf_dev"], W_GS, gs, gate,
            gate.stride(0), gate.shape[0], w.gate_index.cuda(), w.residual.cuda(), None, None,
            out]
    for i, v, code in ((3, float("nan"), "MH3_ERR_INVALID_ARG"),     # weight global scale
                       (3, 0.0, "MH3_ERR_INVALID_ARG"),
                       (6, 5375, "MH3_ERR_INVALID_ARG"),              # gate row stride
                       (7, 0, "MH3_ERR_INVALID_ARG"),                 # gate rows
                       (4, None, "MH3_ERR_INVALID_ARG"),              # act_global_scale
                       (2, None, "MH3_ERR_INVALID_ARG")):             # weight scales
        bad = list(args)
        bad[i] = v
        with pytest.raises(RuntimeError, match=code):
            binding.mh3_nvfp4_out_proj_run(handle, None, 8, *bad)
    bad = list(args)
    bad[10] = weight["q_dev"][:, 1:]  # act_q not 16-byte aligned
    with pytest.raises(RuntimeError, match="MH3_ERR_ALIGNMENT"):
        binding.mh3_nvfp4_out_proj_run(handle, None, 8, *bad)
    res = args[9]
    bad = list(args)
    bad[12] = res.view(-1)[8:].view(-1)  # partial overlap of out with the residual
    with pytest.raises(RuntimeError, match="MH3_ERR_INVALID_ARG"):
        binding.mh3_nvfp4_out_proj_run(handle, None, 8, *bad)
    binding.mh3_nvfp4_out_proj_run(handle, None, 0, *args)  # M = 0: nothing to do
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())


def test_production_size_sampled(handle, weight):
    """M = 32760 in the bench's launch configuration; the oracle on a sample
    of tokens (every 512th, the last, and the guarded ones); every code and
    scale against the oracle's quantiser on the same sample."""
    w = _workload(32760, weight)
    aq, asf, out = _run(handle, w, weight)
    bad = _bad(w)
    tokens = sorted(set(range(0, w.M, 512)) | {w.M - 1} |
                    set(torch.nonzero(bad).flatten().tolist()[:24]))
    ref = f.out_proj_nvfp4(w.attn_out, weight["q"], weight["sf"], W_GS, ACT_GS, w.gate_view(),
                           w.gate_index, w.residual, tokens=tokens)
    t = torch.tensor(tokens)
    assert torch.equal(aq[t], ref["act_q"])
    assert torch.equal(untile(asf, w.M, K)[t], ref["act_sf"])
    st = _cmp(out[t], ref["out"], "nvfp4 out_proj M=32760 sampled")
    assert st["exact"] > 0.95, st
    assert torch.equal(out[bad].view(torch.int16), w.residual[bad].view(torch.int16))
    assert bool(torch.isfinite(out.double()).all())
