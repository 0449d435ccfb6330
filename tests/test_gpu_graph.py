"""The stage is stream-ordered and allocation-free when the caller passes the
workspaces, or once the handle's own buffers have grown to the call's M, so
it can be captured in a CUDA graph and replayed: the replayed outputs equal
a direct call bit for bit (bf16 stage, e4m3 outputs and the NVFP4 stage)."""
import pytest
import torch

from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import make_nvfp4_workload, make_workload

from parity_utils import new_out, run_stage, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle(cuda_lib):
    h = binding.Handle(torch.cuda.current_device())
    yield h
    torch.cuda.synchronize()
    h.close()


def _capture_and_replay(fn, replays=3):
    """Warm up on a side stream, capture fn(stream) into a graph, replay."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(torch.cuda.current_stream())
    return g


def test_bf16_stage_replays_from_a_cuda_graph(handle):
    wl = make_workload("c2", M=300)
    d = to_device(wl)
    ws = torch.empty(d.M, 5376, dtype=torch.bfloat16, device="cuda")
    ref = new_out(d.M, d.P)
    run_stage(handle, d, ref, workspace=ws)
    out = new_out(d.M, d.P)
    g = _capture_and_replay(lambda s: run_stage(handle, d, out, workspace=ws, stream=s))
    for _ in range(3):
        out.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert handle.device_status() == 0


def test_e4m3_stage_replays_from_a_cuda_graph(handle):
    wl = make_workload("c3", M=257)
    d = to_device(wl)
    ws = torch.empty(d.M, 5376, dtype=torch.bfloat16, device="cuda")
    ds = torch.tensor([1 / 64, 1 / 48, 1 / 128], dtype=torch.float32, device="cuda")

    def call(out, stream):
        binding.mh3_preattn_run_e4m3(
            handle, stream, d.M, d.x, d.xw, d.scale, d.scale.stride(0), d.shift,
            d.shift.stride(0), d.scale.shape[0], d.idx, d.W, d.qw, d.kw, d.cs, d.S, d.pos, d.P,
            wl.spec.eps, wl.spec.qk_eps, ds, ws, out)

    shape = (d.P, d.M, 56 // d.P, 3, 128)
    ref = torch.empty(shape, dtype=torch.uint8, device="cuda")
    call(ref, None)
    out = torch.empty_like(ref)
    g = _capture_and_replay(lambda s: call(out, s))
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert handle.device_status() == 0


def test_nvfp4_stage_replays_from_a_cuda_graph(handle):
    w = make_nvfp4_workload("c2", 300)
    b = w.base
    mod = b.adaln_mod.cuda()
    sc, sh = b.table_views(mod)
    x, xw, idx = b.x.cuda(), b.x_norm_weight.cuda(), w.adaln_index.cuda()
    qw, kw, cs = b.q_norm_weight.cuda(), b.k_norm_weight.cuda(), w.rope_cos_sin.cuda()
    gsa = torch.tensor([w.act_global_scale], dtype=torch.float32, device="cuda")
    gsw = torch.tensor([w.weight_global_scale], dtype=torch.float32, device="cuda")
    lib = binding.load()
    wq = torch.empty(21504, 2688, dtype=torch.uint8, device="cuda")
    wsf = torch.empty(lib.mh3_nvfp4_scales_bytes(21504, 5376, 1), dtype=torch.uint8, device="cuda")
    binding.mh3_nvfp4_quantize(None, b.qkv_weight.cuda(), gsw, wq, wsf, True)
    M, P = w.M, b.spec.P
    aq = torch.empty(M, 2688, dtype=torch.uint8, device="cuda")
    asf = torch.empty(lib.mh3_nvfp4_scales_bytes(M, 5376, 1), dtype=torch.uint8, device="cuda")

    def call(out, stream):
        binding.mh3_nvfp4_preattn_run(handle, stream, M, x, xw, sc, sc.stride(0), sh, sh.stride(0),
                                      sc.shape[0], idx, wq, wsf, w.weight_global_scale, gsa, None,
                                      qw, kw, cs, P, w.eps, None, aq, asf, out)

    ref = new_out(M, P)
    call(ref, None)
    out = new_out(M, P)
    g = _capture_and_replay(lambda s: call(out, s))
    out.fill_(0.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert handle.device_status() == 0


def test_handle_workspace_is_capturable_once_grown(cuda_lib):
    """With workspace NULL the handle's own buffer serves; once a call has
    grown it to at least M, a captured call allocates nothing and replays
    bit-identically (a fresh handle, so the first call does the growing)."""
    h = binding.Handle(torch.cuda.current_device())
    try:
        wl = make_workload("c2", M=300)
        d = to_device(wl)
        ref = new_out(d.M, d.P)
        run_stage(h, d, ref)  # grows the handle workspace to M
        torch.cuda.synchronize()
        out = new_out(d.M, d.P)
        g = _capture_and_replay(lambda s: run_stage(h, d, out, stream=s))
        out.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert h.device_status() == 0
    finally:
        torch.cuda.synchronize()
        h.close()


def test_nvfp4_handle_buffers_are_capturable_once_grown(cuda_lib):
    h = binding.Handle(torch.cuda.current_device())
    try:
        w = make_nvfp4_workload("c2", 300)
        b = w.base
        mod = b.adaln_mod.cuda()
        sc, sh = b.table_views(mod)
        x, xw, idx = b.x.cuda(), b.x_norm_weight.cuda(), w.adaln_index.cuda()
        qw, kw, cs = b.q_norm_weight.cuda(), b.k_norm_weight.cuda(), w.rope_cos_sin.cuda()
        gsa = torch.tensor([w.act_global_scale], dtype=torch.float32, device="cuda")
        gsw = torch.tensor([w.weight_global_scale], dtype=torch.float32, device="cuda")
        lib = binding.load()
        wq = torch.empty(21504, 2688, dtype=torch.uint8, device="cuda")
        wsf = torch.empty(lib.mh3_nvfp4_scales_bytes(21504, 5376, 1), dtype=torch.uint8,
                          device="cuda")
        binding.mh3_nvfp4_quantize(None, b.qkv_weight.cuda(), gsw, wq, wsf, True)
        M, P = w.M, b.spec.P

        def call(out, stream):
            binding.mh3_nvfp4_preattn_run(h, stream, M, x, xw, sc, sc.stride(0), sh, sh.stride(0),
                                          sc.shape[0], idx, wq, wsf, w.weight_global_scale, gsa,
                                          None, qw, kw, cs, P, w.eps, None, None, None, out)

        ref = new_out(M, P)
        call(ref, None)  # grows the handle's activation codes and scales
        torch.cuda.synchronize()
        out = new_out(M, P)
        g = _capture_and_replay(lambda s: call(out, s))
        out.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert h.device_status() == 0
    finally:
        torch.cuda.synchronize()
        h.close()
