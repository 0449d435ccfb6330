"""GPU parity of the NVFP4 pre-attention stage against the oracle
(flashinfer.diffusion_ops.minimax_h3_nvfp4_pre_attention): the quantiser
and kernel 1's quantised activation bit for bit; the whole stage against the
oracle's GEMM and tail run on the GPU's own activation codes (same inputs to
the contraction, so only the FP32 summation order differs), and against the
oracle's whole pipeline within the bf16 stage's output bar."""
import pytest
import torch

from oracle import e4m3, nvfp4 as f
import oracle
from norm_adaln_qkv_gb300 import binding
from norm_adaln_qkv_gb300.inputs import make_nvfp4_workload

from parity_utils import check_outputs, untile

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


@pytest.fixture(scope="module")
def handle(cuda_lib):
    h = binding.Handle(torch.cuda.current_device())
    yield h
    torch.cuda.synchronize()
    h.close()


def gpu_quantize(x: torch.Tensor, gs: float, tiled=True):
    rows, cols = x.shape
    codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device="cuda")
    nsc = binding.load().mh3_nvfp4_scales_bytes(rows, cols, 1 if tiled else 0)
    scales = torch.full((nsc,), 0xEE, dtype=torch.uint8, device="cuda")
    g = torch.tensor([gs], dtype=torch.float32, device="cuda")
    binding.mh3_nvfp4_quantize(None, x, g, codes, scales, tiled)
    torch.cuda.synchronize()
    sc = scales.cpu()
    return codes.cpu(), (untile(sc, rows, cols) if tiled else sc.view(rows, cols // 16))


# ------------------------------------------------------------------ quantiser
def _quant_input(rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp2(torch.randint(-6, 6, (rows, 1), generator=g).float())
    x[0, :16] = 0.0                      # an all-zero block
    x[0, 16:32] = -0.0                   # signed zeros
    x[min(1, rows - 1), 32:64] = 1e-30   # scale underflows to 0 for small gs
    x[rows - 1, ::7] *= 1000             # saturation after the scale's rounding
    return x.to(BF16)


@pytest.mark.parametrize("rows,cols,gs,tiled", [(300, 5376, 336.0, True), (129, 64, 1.0, True),
                                                (300, 5376, 2.5e4, False), (1, 128, 7.0, False),
                                                (513, 256, 448.0 * 6, True)])
def test_quantiser_matches_oracle(cuda_lib, rows, cols, gs, tiled):
    x = _quant_input(rows, cols, rows + cols)
    codes, scales = gpu_quantize(x.cuda(), gs, tiled)
    ref_q, ref_s = f.fp4_quantize(x, gs)
    assert torch.equal(scales, ref_s), int((scales != ref_s).sum())
    bad = codes != ref_q
    assert not bool(bad.any()), (int(bad.sum()), torch.nonzero(bad)[:4].tolist())


def test_quantiser_e2m1_rounding_all_ties(cuda_lib):
    """Block amax 6 with gs 1 (scale 1.0, enc 1.0): every element is rounded
    by the e2m1 conversion itself; a sweep over [-7, 7] in steps of 1/64
    covers every tie and the saturation."""
    v = torch.arange(-7 * 64, 7 * 64 + 1, dtype=torch.float32) / 64
    n = (v.numel() + 14) // 15
    rows = torch.zeros(n, 16)
    rows[:, 0] = 6.0
    flat = rows[:, 1:].reshape(-1)
    flat[:v.numel()] = v
    x = rows.reshape(-1, 64 if (n * 16) % 64 == 0 else 16)
    if x.shape[1] != 64:
        pad = (-x.numel()) % 64
        x = torch.cat([x.reshape(-1), torch.full((pad,), 6.0)]).reshape(-1, 64)
    codes, _ = gpu_quantize(x.to(BF16).cuda(), 1.0, True)
    ref_q, _ = f.fp4_quantize(x.to(BF16), 1.0)
    assert torch.equal(codes, ref_q)


def test_quantiser_single_rounding_at_boundaries(cuda_lib):
    """Blocks whose exact amax * gs / 6, or x * gs / sf, lies within one FP32
    step of a UE4M3 or E2M1 rounding boundary (where rounding twice gives
    another code): the kernel's codes are the exact quotients' codes."""
    from test_oracle_nvfp4 import _element_cases, _scale_cases
    for amax, gs, exact, _ in _scale_cases():
        x = torch.zeros(1, 64)
        x[0, 0] = amax
        x[0, 16] = -amax
        _, scales = gpu_quantize(x.to(BF16).cuda(), gs, False)
        assert scales[0, :2].tolist() == [exact, exact], (amax, gs)
    for xv, amax, gs, sf_code, exact, _ in _element_cases():
        x = torch.zeros(1, 64)
        x[0, :3] = torch.tensor([xv, -xv, amax])
        x[0, 16 + 5] = xv                  # the same element at an odd position
        x[0, 16 + 9] = amax
        codes, scales = gpu_quantize(x.to(BF16).cuda(), gs, True)
        q = f.unpack_codes(codes)[0].tolist()
        assert scales[0, :2].tolist() == [sf_code, sf_code]
        assert (q[0], q[1], q[16 + 5]) == (exact, exact | 8, exact), (xv, gs)


# ------------------------------------------------------------- kernel 1 form
def _dev(w):
    b = w.base
    mod = b.adaln_mod.cuda()
    sc, sh = b.table_views(mod)
    return dict(x=b.x.cuda(), xw=b.x_norm_weight.cuda(), mod=mod, sc=sc, sh=sh,
                idx32=w.adaln_index.cuda(), idx64=w.adaln_index.long().cuda(),
                qw=b.q_norm_weight.cuda(), kw=b.k_norm_weight.cuda(), cs=w.rope_cos_sin.cuda(),
                gs=torch.tensor([w.act_global_scale], dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("key,M", [("c2", 300), ("c3", 257), ("c0", None)])
def test_kernel1_quantises_its_own_activation(handle, key, M):
    w = make_nvfp4_workload(key, M)
    d = _dev(w)
    M = w.M
    act_q = torch.empty(M, 2688, dtype=torch.uint8, device="cuda")
    act_sf = torch.empty(binding.load().mh3_nvfp4_scales_bytes(M, 5376, 1), dtype=torch.uint8,
                         device="cuda")
    binding.mh3_nvfp4_norm_quant(handle, None, M, d["x"], d["xw"], d["sc"], d["sc"].stride(0),
                                 d["sh"], d["sh"].stride(0), d["sc"].shape[0], d["idx32"],
                                 w.eps, d["gs"], act_q, act_sf, True)
    # the bf16 kernel 1 computes the same a (same code, int64 indices)
    ws = torch.empty(M, 5376, dtype=BF16, device="cuda")
    binding.mh3_preattn_norm_adaln(handle, None, M, d["x"], d["xw"], d["sc"], d["sc"].stride(0),
                                   d["sh"], d["sh"].stride(0), d["sc"].shape[0], d["idx64"],
                                   w.eps, ws)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    ref_q, ref_s = f.fp4_quantize(ws.cpu(), w.act_global_scale)
    assert torch.equal(untile(act_sf.cpu(), M, 5376), ref_s)
    assert torch.equal(act_q.cpu(), ref_q)
    bad = (w.adaln_index < 0) | (w.adaln_index >= w.base.spec.rows)
    if bool(bad.any()):
        assert int(act_q.cpu()[bad].sum()) == 0


# ----------------------------------------------------------------- the stage
@pytest.fixture(scope="module")
def weight(cuda_lib):
    w = make_nvfp4_workload("c2", 16)
    W = w.base.qkv_weight
    codes, scales = gpu_quantize(W.cuda(), w.weight_global_scale, True)
    ref_q, ref_s = f.fp4_quantize(W, w.weight_global_scale)
    assert torch.equal(codes, ref_q) and torch.equal(scales, ref_s)
    # device copies in the GEMM's (tiled) layout
    tiled = torch.empty(binding.load().mh3_nvfp4_scales_bytes(21504, 5376, 1), dtype=torch.uint8,
                        device="cuda")
    q_dev = torch.empty(21504, 2688, dtype=torch.uint8, device="cuda")
    g = torch.tensor([w.weight_global_scale], dtype=torch.float32, device="cuda")
    binding.mh3_nvfp4_quantize(None, W.cuda(), g, q_dev, tiled, True)
    torch.cuda.synchronize()
    return dict(q=ref_q, sf=ref_s, q_dev=q_dev, sf_dev=tiled, gs=w.weight_global_scale,
                products=f.block_products(ref_q, ref_s))


def run_stage(h, w, d, weight, out, alpha=None, descale=None, act_q=None, act_sf=None, P=None):
    P = w.base.spec.P if P is None else P
    binding.mh3_nvfp4_preattn_run(
        h, None, w.M, d["x"], d["xw"], d["sc"], d["sc"].stride(0), d["sh"], d["sh"].stride(0),
        d["sc"].shape[0], d["idx32"], weight["q_dev"], weight["sf_dev"], weight["gs"], d["gs"],
        alpha, d["qw"], d["kw"], d["cs"], P, w.eps, descale, act_q, act_sf, out)


def oracle_tail(w, weight, act_q, act_sf, tokens):
    """The oracle's GEMM, alpha, Q/K norm and RoPE on given activation codes."""
    al = f.alpha_from_scales(w.act_global_scale, weight["gs"])
    acc = f.block_products(act_q[tokens], act_sf[tokens]) @ weight["products"].T
    y = torch.mul(acc.to(torch.float32), torch.tensor(al, dtype=torch.float32)).to(BF16)
    T = len(tokens)
    y4 = y.view(T, 3, 56, 128)
    tok = torch.as_tensor(tokens)
    b = w.base
    q = oracle.rope_split_half(oracle.head_rmsnorm(y4[:, 0], b.q_norm_weight, w.eps), w.rope_cos_sin, tok)
    k = oracle.rope_split_half(oracle.head_rmsnorm(y4[:, 1], b.k_norm_weight, w.eps), w.rope_cos_sin, tok)
    return torch.stack([q, k, y4[:, 2]], dim=2)


def check_against_pipeline(got, full, aq, asf, tokens, what):
    """The oracle's whole pipeline on the tokens whose activation codes and
    scales equal the oracle's.  The bf16 activation may differ from the
    oracle's by one bf16 ulp, and near an E2M1 rounding or block-amax boundary
    that changes an FP4 code by a whole step; those few tokens are checked
    through the own-codes tail instead, and the quantiser's decisions are
    pinned bit for bit against the bf16 activation kernel 1 computes."""
    rows_eq = (aq[tokens] == full.act_q).all(1) & (asf[tokens] == full.act_sf).all(1)
    assert float(rows_eq.double().mean()) > 0.98, float(rows_eq.double().mean())
    return check_outputs(got[rows_eq], full.qkv[rows_eq], what)


@pytest.mark.parametrize("key,M", [("c2", 300), ("c3", 520), ("c0", None), ("c2", 1), ("c3", 257)])
def test_stage_parity(handle, weight, key, M):
    w = make_nvfp4_workload(key, M)
    d = _dev(w)
    M, P = w.M, w.base.spec.P
    act_q = torch.empty(M, 2688, dtype=torch.uint8, device="cuda")
    act_sf = torch.empty(binding.load().mh3_nvfp4_scales_bytes(M, 5376, 1), dtype=torch.uint8,
                         device="cuda")
    out = torch.full((P, M, 56 // P, 3, 128), float("nan"), dtype=BF16, device="cuda")
    run_stage(handle, w, d, weight, out, act_q=act_q, act_sf=act_sf)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    got = oracle.ulysses_unpack_rows(out.cpu(), list(range(M)))
    # 1. same activation codes: only the FP32 summation order differs
    aq, asf = act_q.cpu(), untile(act_sf.cpu(), M, 5376)
    ref = oracle_tail(w, weight, aq, asf, list(range(M)))
    st = check_outputs(got, ref, f"nvfp4 {key} M={M} (own codes)")
    assert st["exact"] > 0.99, st
    # 2. the oracle's whole pipeline
    b = w.base
    sc, sh = b.table_views()
    full = f.pre_attention_nvfp4_tokens(b.x, b.x_norm_weight, sc, sh, w.adaln_index,
                                        weight["q"], weight["sf"], weight["gs"],
                                        w.act_global_scale, b.q_norm_weight, b.k_norm_weight,
                                        w.rope_cos_sin, eps=w.eps)
    st2 = check_against_pipeline(got, full, aq, asf, list(range(M)),
                                 f"nvfp4 {key} M={M} (oracle pipeline)")
    print(key, M, st, st2)


def test_e4m3_output_and_alpha(handle, weight):
    w = make_nvfp4_workload("c2", 300)
    d = _dev(w)
    M, P = w.M, w.base.spec.P
    out = torch.empty((P, M, 56 // P, 3, 128), dtype=BF16, device="cuda")
    run_stage(handle, w, d, weight, out)                       # alpha derived on the device
    out2 = torch.empty_like(out)
    run_stage(handle, w, d, weight, out2, alpha=f.alpha_from_scales(w.act_global_scale, weight["gs"]))
    ds = (1 / 64, 1 / 48, 1 / 128)
    codes = torch.empty(out.shape, dtype=torch.uint8, device="cuda")
    run_stage(handle, w, d, weight, codes, descale=torch.tensor(ds, device="cuda"))
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(codes.cpu(), e4m3.quantize_packed(out.cpu(), ds))


# out_mode "nvfp4": q, k, v with their own global scales (calibration amax
# 8, 6 and 10: 448 * 6 / amax)
OUT_GS = (448.0 * 6 / 8, 448.0 * 6 / 6, 448.0 * 6 / 10)


def run_stage_nvfp4_out(h, w, d, weight, codes, sf, gs_dev, P):
    binding.mh3_nvfp4_preattn_run_nvfp4_out(
        h, None, w.M, d["x"], d["xw"], d["sc"], d["sc"].stride(0), d["sh"], d["sh"].stride(0),
        d["sc"].shape[0], d["idx32"], weight["q_dev"], weight["sf_dev"], weight["gs"], d["gs"],
        None, d["qw"], d["kw"], d["cs"], P, w.eps, gs_dev, None, None, codes, sf)


@pytest.mark.parametrize("key,M,P", [("c2", 300, 2), ("c2", 257, 8), ("c0", None, 1)])
def test_nvfp4_outputs_quantise_the_bf16_outputs(handle, weight, key, M, P):
    """Every code and scale of the NVFP4 output form equals the oracle's
    quantisation of the same call's bf16 outputs (guarded tokens included:
    their rows are zero, so are their codes and scales)."""
    w = make_nvfp4_workload(key, M)
    d = _dev(w)
    M = w.M
    out = torch.empty((P, M, 56 // P, 3, 128), dtype=BF16, device="cuda")
    run_stage(handle, w, d, weight, out, P=P)
    lib = binding.load()
    codes = torch.full((lib.mh3_preattn_out_nvfp4_bytes(M, 0),), 0xEE, dtype=torch.uint8,
                       device="cuda")
    sf = torch.full((lib.mh3_preattn_out_nvfp4_bytes(M, 1),), 0xEE, dtype=torch.uint8,
                    device="cuda")
    run_stage_nvfp4_out(handle, w, d, weight, codes, sf,
                        torch.tensor(OUT_GS, dtype=torch.float32, device="cuda"), P)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    toks = range(M)
    got_c = oracle.ulysses_unpack_rows(codes.cpu().view(P, M, 56 // P, 3, 64), toks)
    got_s = oracle.ulysses_unpack_rows(sf.cpu().view(P, M, 56 // P, 3, 8), toks)
    ref_c, ref_s = f.quantize_outputs(oracle.ulysses_unpack_rows(out.cpu(), toks), OUT_GS)
    assert torch.equal(got_s, ref_s), int((got_s != ref_s).sum())
    assert torch.equal(got_c, ref_c), int((got_c != ref_c).sum())


def test_invalid_arguments(handle, weight):
    w = make_nvfp4_workload("c2", 8)
    d = _dev(w)
    out = torch.empty((w.base.spec.P, 8, 56 // w.base.spec.P, 3, 128), dtype=BF16, device="cuda")
    with pytest.raises(RuntimeError, match="P"):
        run_stage(handle, w, d, weight, out, P=3)
    bad = dict(weight, gs=-1.0)
    with pytest.raises(RuntimeError, match="weight_global_scale"):
        run_stage(handle, w, d, bad, out)
    lib = binding.load()
    x = torch.zeros(4, 64, dtype=BF16, device="cuda")
    g = torch.ones(1, device="cuda")
    c = torch.empty(4, 32, dtype=torch.uint8, device="cuda")
    s = torch.empty(512, dtype=torch.uint8, device="cuda")
    assert lib.mh3_nvfp4_quantize(None, 4, 48, x.data_ptr(), g.data_ptr(), c.data_ptr(), s.data_ptr(), 1) == 1
    assert lib.mh3_nvfp4_quantize(None, 4, 64, x.data_ptr() + 2, g.data_ptr(), c.data_ptr(), s.data_ptr(), 1) == 2
    torch.cuda.synchronize()
    assert handle.device_status() == 0


@pytest.mark.parametrize("key", ["c3", "c4"])
def test_production_size_sampled_parity(handle, weight, key):
    """The production video sequence (M = 32760, P = 8) in the launch the
    bench times, and the upper-bound sequence (M = 149796, P = 4): sampled
    tokens against the oracle, every guarded token zero."""
    w = make_nvfp4_workload(key)
    d = _dev(w)
    M, P = w.M, w.base.spec.P
    act_q = torch.empty(M, 2688, dtype=torch.uint8, device="cuda")
    act_sf = torch.empty(binding.load().mh3_nvfp4_scales_bytes(M, 5376, 1), dtype=torch.uint8,
                         device="cuda")
    out = torch.full((P, M, 56 // P, 3, 128), float("nan"), dtype=BF16, device="cuda")
    run_stage(handle, w, d, weight, out, act_q=act_q, act_sf=act_sf)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    bad = (w.adaln_index < 0) | (w.adaln_index >= w.base.spec.rows)
    special = torch.nonzero(bad).flatten().tolist()
    every = 64 if key == "c3" else 256
    tokens = sorted(set(range(0, M, every)) | {M - 1} | set(special[:96]))
    got = oracle.ulysses_unpack_rows(out, tokens).cpu()  # the sampled rows only
    aq, asf = act_q.cpu(), untile(act_sf.cpu(), M, 5376)
    st = check_outputs(got, oracle_tail(w, weight, aq, asf, tokens), f"nvfp4 {key} sampled (own codes)")
    assert st["exact"] > 0.99, st
    b = w.base
    sc, sh = b.table_views()
    full = f.pre_attention_nvfp4_tokens(b.x, b.x_norm_weight, sc, sh, w.adaln_index,
                                        weight["q"], weight["sf"], weight["gs"],
                                        w.act_global_scale, b.q_norm_weight, b.k_norm_weight,
                                        w.rope_cos_sin, eps=w.eps, tokens=tokens)
    st2 = check_against_pipeline(got, full, aq, asf, tokens, f"nvfp4 {key} sampled (oracle pipeline)")
    code_eq = float((aq[tokens] == full.act_q).double().mean())
    sf_eq = float((asf[tokens] == full.act_sf).double().mean())
    assert code_eq > 0.999 and sf_eq > 0.999, (code_eq, sf_eq)
    # all guarded tokens (on the GPU): zero codes, zero scales, zero outputs
    assert int(bad.sum()) > 0
    bad_d = bad.cuda()
    assert bool((act_q[bad_d] == 0).all())
    assert bool((out.permute(1, 0, 2, 3, 4)[bad_d] == 0).all())
    assert bool(torch.isfinite(out).all())
    print(key, len(tokens), st, st2, code_eq, sf_eq)


def test_nvfp4_outputs_production_size_sampled(handle, weight):
    """out_mode "nvfp4" at the production size (M = 32760, P = 8) in the
    bench's launch configuration: the codes and scales of sampled tokens
    (every 64th, the last, guarded ones) against the oracle's quantisation of
    the same call's bf16 outputs, and every guarded token's codes and scales
    zero (by value)."""
    w = make_nvfp4_workload("c3")
    d = _dev(w)
    M, P = w.M, w.base.spec.P
    out = torch.empty((P, M, 56 // P, 3, 128), dtype=BF16, device="cuda")
    run_stage(handle, w, d, weight, out)
    lib = binding.load()
    codes = torch.full((lib.mh3_preattn_out_nvfp4_bytes(M, 0),), 0xEE, dtype=torch.uint8,
                       device="cuda")
    sf = torch.full((lib.mh3_preattn_out_nvfp4_bytes(M, 1),), 0xEE, dtype=torch.uint8,
                    device="cuda")
    run_stage_nvfp4_out(handle, w, d, weight, codes, sf,
                        torch.tensor(OUT_GS, dtype=torch.float32, device="cuda"), P)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    bad = (w.adaln_index < 0) | (w.adaln_index >= w.base.spec.rows)
    tokens = sorted(set(range(0, M, 64)) | {M - 1} | set(torch.nonzero(bad).flatten().tolist()[:48]))
    c5 = codes.view(P, M, 56 // P, 3, 64)
    s5 = sf.view(P, M, 56 // P, 3, 8)
    got_c = oracle.ulysses_unpack_rows(c5, tokens).cpu()
    got_s = oracle.ulysses_unpack_rows(s5, tokens).cpu()
    ref_c, ref_s = f.quantize_outputs(oracle.ulysses_unpack_rows(out, tokens).cpu(), OUT_GS)
    assert torch.equal(got_s, ref_s), int((got_s != ref_s).sum())
    assert torch.equal(got_c, ref_c), int((got_c != ref_c).sum())
    bad_d = bad.cuda()
    assert int(bad.sum()) > 0
    # zero by value: the bf16 outputs of a guarded token are +0 or -0, and a
    # -0 keeps its sign bit in the E2M1 code
    assert bool(((c5.permute(1, 0, 2, 3, 4)[bad_d] & 0x77) == 0).all())
    assert bool((s5.permute(1, 0, 2, 3, 4)[bad_d] == 0).all())


def test_repacking_is_bit_identical_across_P(handle, weight):
    """The pack is a pure relabelling: every P gives the same per-token values."""
    w = make_nvfp4_workload("c2", 300)
    d = _dev(w)
    M = w.M
    outs = {}
    for P in (1, 2, 4, 8):
        o = torch.empty((P, M, 56 // P, 3, 128), dtype=BF16, device="cuda")
        run_stage(handle, w, d, weight, o, P=P)
        outs[P] = o
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    base = outs[1][0]
    for P in (2, 4, 8):
        rep = outs[P].permute(1, 0, 2, 3, 4).reshape(M, 56, 3, 128)
        assert torch.equal(rep.view(torch.int16), base.view(torch.int16)), P


def test_guard_bands_untouched(handle, weight):
    """Nothing is written outside out, act_q and act_sf (M = 200: a ragged
    256-row tile and a ragged 128-row scale atom)."""
    w = make_nvfp4_workload("c3", 200)
    d = _dev(w)
    M, P = w.M, w.base.spec.P
    pad = 4096
    n_out = M * 21504
    nq = M * 2688
    ns = binding.load().mh3_nvfp4_scales_bytes(M, 5376, 1)
    obuf = torch.full((n_out + 2 * pad,), 7.0, dtype=BF16, device="cuda")
    qbuf = torch.full((nq + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda")
    sbuf = torch.full((ns + 2 * pad,), 0x5A, dtype=torch.uint8, device="cuda")
    out = obuf[pad:pad + n_out].view(P, M, 56 // P, 3, 128)
    act_q = qbuf[pad:pad + nq].view(M, 2688)
    act_sf = sbuf[pad:pad + ns]
    run_stage(handle, w, d, weight, out, act_q=act_q, act_sf=act_sf)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    for b, v in ((obuf, 7.0), (qbuf, 0xA5), (sbuf, 0x5A)):
        assert bool((b[:pad] == v).all()) and bool((b[-pad:] == v).all())
    tokens = list(range(M))
    got = oracle.ulysses_unpack_rows(out.cpu(), tokens)
    aq, asf = act_q.cpu(), untile(act_sf.cpu(), M, 5376)
    st = check_outputs(got, oracle_tail(w, weight, aq, asf, tokens), "nvfp4 guard-band case")
    assert st["exact"] > 0.99, st


def test_zero_tokens_is_a_no_op(handle, weight):
    w = make_nvfp4_workload("c0")
    d = _dev(w)
    empty = torch.empty(0, dtype=BF16, device="cuda")
    binding.mh3_nvfp4_preattn_run(
        handle, None, 0, None, d["xw"], d["sc"], d["sc"].stride(0), d["sh"], d["sh"].stride(0),
        d["sc"].shape[0], None, weight["q_dev"], weight["sf_dev"], weight["gs"], None, None,
        d["qw"], d["kw"], d["cs"], 1, w.eps, None, None, None, empty)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
