"""Failure detection without a GPU fault: the bounded waits of the CTA-pair
QKV GEMM.  A test hook makes the producer issue no loads, so the MMA thread's
wait on the first stage runs out (2 s); the kernel must record its code in
the device status word, drain and return (no hang, no fault), and the next
normal call on the same handle and stream must be correct."""
import time

import pytest
import torch

from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import make_workload

from parity_utils import check_outputs, new_out, oracle_tokens, run_norm_adaln, to_device

pytestmark = pytest.mark.gpu

# the first bounded wait to run out records its code: the MMA thread waiting
# for the first stage's operands (0x102) or an epilogue warp waiting for the
# first accumulator (0x104); both waits start together
STALL_CODES = (0x102, 0x104)


def _qkv(h, d, ws, out):
    qk = d.wl.spec.qk_eps if d.wl.spec.qk_eps is not None else d.wl.spec.eps
    binding.mh3_preattn_qkv(h, None, d.M, ws, d.W, d.qw, d.kw, d.cs, d.S, d.pos, d.P, qk, out)


def test_stalled_gemm_reports_a_status_code_and_the_next_call_is_correct(cuda_lib):
    h = binding.Handle(torch.cuda.current_device())
    try:
        wl = make_workload("c2", M=300)  # M > 128: the CTA-pair form
        d = to_device(wl)
        ws = torch.empty(d.M, 5376, dtype=torch.bfloat16, device="cuda")
        run_norm_adaln(h, d, ws)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        out = new_out(d.M, d.P, fill=7.0)
        h.set_test_stall(True)
        t0 = time.time()
        _qkv(h, d, ws, out)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        code = h.device_status()
        assert code in STALL_CODES, hex(code)
        assert 1.5 < elapsed < 30.0, elapsed          # the 2 s limit, not a hang
        assert bool((out == 7.0).all())               # nothing was stored
        # the flag cleared itself; the context and the handle still work
        _qkv(h, d, ws, out)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        ref = oracle_tokens(wl)
        from oracle import ulysses_unpack_rows
        st = check_outputs(ulysses_unpack_rows(out.cpu(), list(range(d.M))), ref.qkv, "after stall")
        assert st["exact"] > 0.99
    finally:
        torch.cuda.synchronize()
        h.close()


def test_stalled_nvfp4_gemm_reports_a_status_code_and_the_next_call_is_correct(cuda_lib):
    """The same for the NVFP4 GEMM (12 warps with a register split, scale-copy
    warps): every role gives up through a bounded wait and the CTA pair
    exits cleanly."""
    from norm_adaln_qkv_gb300.inputs import make_nvfp4_workload
    h = binding.Handle(torch.cuda.current_device())
    try:
        w = make_nvfp4_workload("c2", 300)
        b = w.base
        M, P = w.M, b.spec.P
        dev = "cuda"
        mod = b.adaln_mod.to(dev)
        sc, sh = b.table_views(mod)
        gsa = torch.tensor([w.act_global_scale], dtype=torch.float32, device=dev)
        gsw = torch.tensor([w.weight_global_scale], dtype=torch.float32, device=dev)
        lib = binding.load()
        wq = torch.empty(21504, 2688, dtype=torch.uint8, device=dev)
        wsf = torch.empty(lib.mh3_nvfp4_scales_bytes(21504, 5376, 1), dtype=torch.uint8, device=dev)
        binding.mh3_nvfp4_quantize(None, b.qkv_weight.to(dev), gsw, wq, wsf, True)
        aq = torch.empty(M, 2688, dtype=torch.uint8, device=dev)
        asf = torch.empty(lib.mh3_nvfp4_scales_bytes(M, 5376, 1), dtype=torch.uint8, device=dev)
        binding.mh3_nvfp4_norm_quant(h, None, M, b.x.to(dev), b.x_norm_weight.to(dev), sc,
                                     sc.stride(0), sh, sh.stride(0), sc.shape[0],
                                     w.adaln_index.to(dev), w.eps, gsa, aq, asf, True)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        qw, kw, cs = b.q_norm_weight.to(dev), b.k_norm_weight.to(dev), w.rope_cos_sin.to(dev)

        def gemm(o):
            binding.mh3_nvfp4_qkv(h, None, M, aq, asf, wq, wsf, w.weight_global_scale, gsa, None,
                                  qw, kw, cs, P, w.eps, None, o)
        good = torch.empty((P, M, 56 // P, 3, 128), dtype=torch.bfloat16, device=dev)
        gemm(good)  # a normal launch (its parity is covered by the NVFP4 tests)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        out = torch.full((P, M, 56 // P, 3, 128), 7.0, dtype=torch.bfloat16, device=dev)
        h.set_test_stall(True)
        t0 = time.time()
        gemm(out)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        code = h.device_status()
        assert code in STALL_CODES, hex(code)
        assert 1.5 < elapsed < 30.0, elapsed          # the 2 s limit, not a hang
        assert bool((out == 7.0).all())               # nothing was stored
        gemm(out)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        assert torch.equal(out.view(torch.int16), good.view(torch.int16))
    finally:
        torch.cuda.synchronize()
        h.close()
