"""The split tail of the CTA-pair QKV GEMM (mh3_preattn_run for M > 128):
when the last wave holds at most half as many 256 x 256 tiles as there are
resident CTA pairs, each of those tiles is computed by two pairs over the two
halves of K and the first hands its FP32 partial to the second through a
scratch of the handle.  The schedule is fixed by M and the device, so every
call of a size gives the same bits; these tests pin that the scratch carries
nothing from one call to the next (flags cleared, partials rewritten), that
kernel 2 alone (which clears the flags by a memset instead of kernel 1)
matches the whole stage, and that a split size stays inside the stage's
tolerance against the oracle at every token (the single-CTA and unsplit
sizes are covered by test_gpu_parity.py)."""
import pytest
import torch

from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import make_workload

from parity_utils import check_outputs, new_out, oracle_tokens, run_norm_adaln, run_stage, \
    to_device

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu()


def test_one_handle_across_sizes_equals_fresh_handles(cuda_lib):
    """M = 1024 and 300 split their last wave, 4096 does not (52 of 76 tiles
    left over) and 100 takes the single-CTA form: the sequence on one handle
    (growing and reusing the scratch) equals each size on a fresh handle."""
    sizes = [("c1", 1024), ("c2", 300), ("c2", 4096), ("c1", 1024), ("c2", 100), ("c2", 300)]
    work = {}
    for key, M in sizes:
        if (key, M) not in work:
            work[(key, M)] = to_device(make_workload(key, M=M))
    ref = {}
    for k, d in work.items():
        h = binding.Handle(torch.cuda.current_device())
        out = new_out(d.M, d.P)
        run_stage(h, d, out)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        ref[k] = _bits(out)
        h.close()
    h = binding.Handle(torch.cuda.current_device())
    for k in sizes:
        d = work[k]
        out = new_out(d.M, d.P, fill=float("nan"))
        run_stage(h, d, out)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        assert torch.equal(_bits(out), ref[k]), k
    h.close()


def test_kernel_two_alone_equals_the_stage(cuda_lib):
    """Kernel 1 then kernel 2 as two calls (kernel 2 clears the split flags
    with a memset) gives the stage's bits at a split size."""
    d = to_device(make_workload("c1"))
    h = binding.Handle(torch.cuda.current_device())
    ws = torch.empty((d.M, 5376), dtype=torch.bfloat16, device="cuda")
    ref = new_out(d.M, d.P)
    run_stage(h, d, ref, workspace=ws)
    ws2 = torch.empty_like(ws)
    run_norm_adaln(h, d, ws2)
    out = new_out(d.M, d.P, fill=float("nan"))
    qk = d.wl.spec.qk_eps if d.wl.spec.qk_eps is not None else d.wl.spec.eps
    for _ in range(2):  # twice: the second call starts from the first's flags
        binding.mh3_preattn_qkv(h, None, d.M, ws2, d.W, d.qw, d.kw, d.cs, d.S, d.pos, d.P, qk,
                                out)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        assert torch.equal(_bits(out), _bits(ref))
    h.close()


@pytest.mark.parametrize("key,M", [("c1", 1024), ("c2", 300)])
def test_split_sizes_against_the_oracle(cuda_lib, key, M):
    """Every token of a split size within the stage's tolerance."""
    wl = make_workload(key, M=M)
    d = to_device(wl)
    h = binding.Handle(torch.cuda.current_device())
    out = new_out(d.M, d.P)
    run_stage(h, d, out)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    got = out.permute(1, 0, 2, 3, 4).reshape(M, 56, 3, 128).cpu()
    ref = oracle_tokens(wl)
    st = check_outputs(got, ref.qkv, f"split {key} M={M}")
    assert st["exact"] > 0.98, st
    h.close()
