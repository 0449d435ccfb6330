"""Benchmark of the MiniMax-H3 BF16 pre-attention stage on GB300.

One step = one whole stage call (kernel 1 norm/AdaLN + kernel 2 QKV GEMM
with the fused epilogue) over the production video sequence workload
(M = 32760 tokens of a 21x30x52 grid, rows = 9 strided AdaLN chunks, P = 8,
explicit positions into an S = 40000 cache with 0.1% clamped, x ~ N(0, 2)
with 0.01% outliers, caller-provided workspace).  Inputs are seeded and
synthetic and are larger than L2 (x 352 MB, weight 231 MB), so no flush is
needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs N independent replicas (one per rank, launched by torchrun; the
stage has no cross-GPU step), timed with a barrier and the max over ranks.
``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("pre-attn µs/call & GEMM TFLOP/s at M=4096/32760; "
          "% of BF16 tensor/HBM roofline")
UNIT = "us/call"
WORKLOAD = "c3"
ALSO = "c2"
SMALL_CALLS = 50
E2E_PASSES = 5
FLOP_PER_TOKEN = 2 * 5376 * 21504
# kernel 2 at the bench size is the CTA-pair form; its traffic figure is tied
# to these sources
K2_SOURCES = ("norm_adaln_qkv_gb300/csrc/k2_qkv_gemm_pair.cu",
              "norm_adaln_qkv_gb300/csrc/gemm_pair.cuh",
              "norm_adaln_qkv_gb300/csrc/k2_common.cuh", "norm_adaln_qkv_gb300/csrc/ptx.cuh",
              "norm_adaln_qkv_gb300/csrc/common.cuh", "norm_adaln_qkv_gb300/csrc/e4m3.cuh",
              "norm_adaln_qkv_gb300/csrc/nvfp4.cuh")
OUT_PROJ_FLOP_PER_TOKEN = 2 * 7168 * 5376
MLP_FLOP_PER_TOKEN = 2 * 5376 * 28672 + 2 * 14336 * 5376
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "k2_traffic.json")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def _k2_source_hash() -> str:
    h = hashlib.sha256()
    for rel in K2_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _k2_traffic(M: int):
    """DRAM bytes per launch of kernel 2 from the committed ncu summary, or
    None when the kernel source changed since the counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("source_hash") != _k2_source_hash():
        return None
    per_token = t.get("dram_bytes_per_token")
    fixed = t.get("dram_bytes_fixed", 0)
    if per_token is None:
        return None
    return float(fixed + per_token * M)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.rows = []
        self.started = False

    def start(self):
        import tempfile
        self.started = True
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            os.unlink(self.path)
            return
        # polling is live before the caller's timed work starts (short runs
        # would otherwise end before the first sample): wait up to 3 s for it
        t0 = time.time()
        while time.time() - t0 < 3.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def pause(self):
        """Stop polling and keep the samples so far.  The polling slows the
        host<->device copies of the end-to-end passes (their times alternate
        by up to 40 % while it runs), so it is paused around them."""
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.proc = None
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    self.rows.append(parts)
        os.unlink(self.path)

    def resume(self):
        if self.started and self.proc is None:
            self.start()

    def stop(self):
        self.pause()
        rows = self.rows
        if not rows:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        pw = [num(r[3]) for r in rows if num(r[3]) is not None and num(r[1]) is not None
              and smax and num(r[1]) > 0.5 * max(smax)]
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w": statistics.median(pw) if pw else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(v: float, device=None) -> float:
    """Largest value over all ranks (the identity without a process group)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value_us(ms_total_max: float, steps: int, world: int) -> float:
    """Whole-job time per call: every rank runs one call per step, so the
    job completes steps * world calls in the slowest rank's time."""
    return ms_total_max * 1e3 / (steps * world)


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def bench_config(wl, world: int) -> dict:
    """The `config` object both arms print for the same workload."""
    return {"workload": wl.spec.name, "M": wl.M, "P": wl.spec.P, "S": wl.spec.S,
            "rows": wl.spec.rows,
            "l2": "inputs larger than L2 (x 352 MB, W 231 MB); no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    from norm_adaln_qkv_gb300.inputs import make_workload
    wl = make_workload(args.workload)
    sc, sh = wl.table_views()
    rows_per_step = args.ref_rows
    M = wl.M

    def step(i):
        t0 = (i * 997) % (M - rows_per_step)
        toks = list(range(t0, t0 + rows_per_step))
        oracle.pre_attention_tokens(
            wl.x, wl.x_norm_weight, sc, sh, wl.adaln_index, wl.qkv_weight, wl.q_norm_weight,
            wl.k_norm_weight, wl.rope_cos_sin, eps=wl.spec.eps, qk_eps=wl.spec.qk_eps,
            rope_positions=wl.rope_positions, tokens=toks)

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t
    us_per_call = el / args.steps * (M / rows_per_step) * 1e6
    cores = oracle.stage.threads()
    sample = (f"{rows_per_step} consecutive tokens of M={M} per step, time scaled "
              f"by M/{rows_per_step} (tokens are independent)")
    line = {
        "impl": "reference", "metric": METRIC, "value": us_per_call, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64-accumulate/f32/bf16", "data": "synthetic",
        "config": bench_config(wl, world),
        "cpu_baseline": {"value": us_per_call, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": us_per_call, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def cpu_baseline(wl, rows: int, chunk: int = 4096):
    """The oracle as it stands (plain C++, OpenMP over tokens), on the first
    ``rows`` tokens of the bench workload (in chunks of ``chunk`` tokens to
    bound host memory), scaled by M / rows: tokens are independent."""
    import oracle
    sc, sh = wl.table_views()
    rows = min(rows, wl.M)
    t = time.perf_counter()
    for t0 in range(0, rows, chunk):
        oracle.pre_attention_tokens(
            wl.x, wl.x_norm_weight, sc, sh, wl.adaln_index, wl.qkv_weight, wl.q_norm_weight,
            wl.k_norm_weight, wl.rope_cos_sin, eps=wl.spec.eps, qk_eps=wl.spec.qk_eps,
            rope_positions=wl.rope_positions, tokens=range(t0, min(rows, t0 + chunk)))
    el = time.perf_counter() - t
    what = (f"all {rows} tokens" if rows == wl.M else
            f"first {rows} tokens of M={wl.M}, scaled by M/{rows}")
    return {"value": el * (wl.M / rows) * 1e6, "unit": UNIT, "cores": oracle.stage.threads(),
            "kind": "oracle", "sample": f"{what}, {el:.1f} s of CPU time"}


def stage_roofline_us(wl, peaks) -> float:
    """max(FLOP / bf16 peak, compulsory bytes / HBM peak) for one stage call:
    x, W, out, indices, explicit positions, the cache rows used, both tables'
    rows and the norm weights."""
    M = wl.M
    flop_time = FLOP_PER_TOKEN * M / (peaks["bf16"] * 1e12)
    comp_bytes = (M * 10752 + 21504 * 5376 * 2 + M * 43008 + 8 * M +
                  (8 * M if wl.rope_positions is not None else 0) + min(wl.spec.S, M) * 192 +
                  wl.spec.rows * 2 * 5376 * 2 + 5376 * 2 + 2 * 128 * 2)
    return max(flop_time, comp_bytes / (peaks["hbm"] * 1e9)) * 1e6


def run_ours(args, world, rank, local):
    from norm_adaln_qkv_gb300 import binding, build
    from norm_adaln_qkv_gb300.inputs import make_workload

    # Oracle CPU baseline first (rank 0 only, N = 1 only), before any CUDA work.
    wl = make_workload(args.workload)
    cpu = cpu_baseline(wl, args.cpu_rows) if (rank == 0 and world == 1 and args.cpu_rows > 0) \
        else None

    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.lib:
        binding.load(os.path.abspath(args.lib))  # another build of the library
    else:
        build.build()
    h = binding.Handle(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks()

    def prepare(w):
        mod = w.adaln_mod.to(dev)
        sc, sh = w.table_views(mod)
        d = dict(x=w.x.to(dev), xw=w.x_norm_weight.to(dev), mod=mod, sc=sc, sh=sh,
                 idx=w.adaln_index.to(dev), W=w.qkv_weight.to(dev), qw=w.q_norm_weight.to(dev),
                 kw=w.k_norm_weight.to(dev), cs=w.rope_cos_sin.to(dev),
                 pos=None if w.rope_positions is None else w.rope_positions.to(dev))
        d["ws"] = torch.empty((w.M, 5376), dtype=torch.bfloat16, device=dev)
        d["out"] = torch.empty((w.spec.P, w.M, 56 // w.spec.P, 3, 128), dtype=torch.bfloat16,
                               device=dev)
        return d

    def stage(w, d):
        binding.mh3_preattn_run(h, stream, w.M, d["x"], d["xw"], d["sc"], d["sc"].stride(0),
                                d["sh"], d["sh"].stride(0), w.spec.rows, d["idx"], d["W"],
                                d["qw"], d["kw"], d["cs"], w.spec.S, d["pos"], w.spec.P,
                                w.spec.eps, w.spec.qk_eps, d["ws"], d["out"])

    def k1(w, d):
        binding.mh3_preattn_norm_adaln(h, stream, w.M, d["x"], d["xw"], d["sc"],
                                       d["sc"].stride(0), d["sh"], d["sh"].stride(0), w.spec.rows,
                                       d["idx"], w.spec.eps, d["ws"])

    def k2(w, d):
        qk = w.spec.qk_eps if w.spec.qk_eps is not None else w.spec.eps
        binding.mh3_preattn_qkv(h, stream, w.M, d["ws"], d["W"], d["qw"], d["kw"], d["cs"],
                                w.spec.S, d["pos"], w.spec.P, qk, d["out"])

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    d = prepare(wl)
    clocks = ClockSampler(local)
    clocks.start()
    # kernel 1 alone before any GEMM has run: the HBM-bound kernel timed on
    # its own, as the GEMM's burst peak is (later loops run at the clocks the
    # 1.4 kW cap leaves after seconds of GEMM work)
    for _ in range(3):
        k1(wl, d)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(args.steps):
        k1(wl, d)
    c1.record(stream)
    torch.cuda.synchronize()
    k1_first_ms = c0.elapsed_time(c1) / args.steps
    for _ in range(max(args.warmup, 3)):
        stage(wl, d)
    torch.cuda.synchronize()

    # ---- timed region: exactly K whole-stage steps
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        stage(wl, d)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), dev)
    gpu_launches = 2 * args.steps
    assert h.device_status(stream) == 0, "a kernel recorded a timeout"

    # ---- per-kernel breakdown, interleaved step by step with whole-stage
    # calls so that the stage and its two kernels are timed at the same
    # clock (the 1.4 kW cap lowers the SM clock as the run goes on): each
    # iteration times one stage call, then kernel 1 and kernel 2 launched
    # separately, with events on the launching stream.
    def breakdown(w, dd, n):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for i in range(n):
            ev[i][0].record(stream)
            stage(w, dd)
            ev[i][1].record(stream)
            k1(w, dd)
            ev[i][2].record(stream)
            k2(w, dd)
            ev[i][3].record(stream)
        torch.cuda.synchronize()
        ts = [e[0].elapsed_time(e[1]) for e in ev]
        t1 = [e[1].elapsed_time(e[2]) for e in ev]
        t2 = [e[2].elapsed_time(e[3]) for e in ev]
        breakdown.medians = (statistics.median(t1), statistics.median(t2),
                             statistics.median(a + b for a, b in zip(t1, t2)))
        breakdown.stage_ms = sum(ts) / n
        return sum(t1) / n, sum(t2) / n

    k1_ms, k2_ms = breakdown(wl, d, args.steps)
    k1_med, k2_med, pair_med = breakdown.medians
    stage_interleaved_ms = breakdown.stage_ms
    # kernel 2's share of a stage at one clock, applied to the timed region
    k2_share = k2_ms / (k1_ms + k2_ms)

    # kernel 1 alone, back to back (no GEMM between launches)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(args.steps):
        k1(wl, d)
    a1.record(stream)
    torch.cuda.synchronize()
    k1_alone_ms = a0.elapsed_time(a1) / args.steps

    clocks.pause()  # the polling would slow the copies of the passes below
    # ---- end to end through the public API: every step copies its inputs
    # (x, index, positions, AdaLN tensor) from pinned host memory and its
    # result (out) back.  Two buffer sets and three streams pipeline the
    # copies of neighbouring steps under the kernels of the current one.
    hx = wl.x.pin_memory()
    hidx = wl.adaln_index.pin_memory()
    hpos = wl.rope_positions.pin_memory() if wl.rope_positions is not None else None
    hmod = wl.adaln_mod.pin_memory()
    houts = [torch.empty(d["out"].shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = hx.numel() * 2 + hidx.numel() * 8 + hmod.numel() * 2 + \
        (hpos.numel() * 8 if hpos is not None else 0)
    d2h = houts[0].numel() * 2
    sets = []
    for _ in range(2):
        mod_in = torch.empty_like(d["mod"])
        sc_in, sh_in = wl.table_views(mod_in)
        sets.append(dict(d, x=torch.empty_like(d["x"]), idx=torch.empty_like(d["idx"]),
                         mod=mod_in, sc=sc_in, sh=sh_in, out=torch.empty_like(d["out"]),
                         pos=torch.empty_like(d["pos"]) if d["pos"] is not None else None))
    s_in = torch.cuda.Stream(dev)
    n_out = max(1, args.e2e_chunks)
    s_outs = [torch.cuda.Stream(dev) for _ in range(n_out)]
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    done_compute = [None, None]   # compute of the last step that used buffer set k
    done_d2h = [None, None]       # read-back of the last step that used buffer set k
    n_e2e = max(4, args.steps)  # the same step count as the device-timed value

    def e2e_step(i):
        k = i % 2
        bs = sets[k]
        with torch.cuda.stream(s_in):
            if done_compute[k] is not None:
                s_in.wait_event(done_compute[k])  # step i-2 no longer reads this set
            bs["x"].copy_(hx, non_blocking=True)
            bs["idx"].copy_(hidx, non_blocking=True)
            bs["mod"].copy_(hmod, non_blocking=True)
            if bs["pos"] is not None:
                bs["pos"].copy_(hpos, non_blocking=True)
            in_done = ev()
            in_done.record(s_in)
        stream.wait_event(in_done)
        if done_d2h[k] is not None:
            for e in done_d2h[k]:
                stream.wait_event(e)  # step i-2's result has left this set
        stage(wl, bs)
        done_compute[k] = ev()
        done_compute[k].record(stream)
        src, dst = bs["out"].view(-1), houts[k].view(-1)
        step = (src.numel() + n_out - 1) // n_out
        done_d2h[k] = []
        for c, so in enumerate(s_outs):  # contiguous pieces on parallel copy streams
            with torch.cuda.stream(so):
                so.wait_event(done_compute[k])
                dst[c * step:(c + 1) * step].copy_(src[c * step:(c + 1) * step], non_blocking=True)
                e = ev()
                e.record(so)
                done_d2h[k].append(e)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    # E2E_PASSES timed passes of n_e2e steps each; the median pass is the
    # number (the host link is shared with other tenants of the machine, so
    # single passes vary), all passes are reported beside it
    e2e_passes = []
    for _ in range(E2E_PASSES):
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(s_in)
        for i in range(n_e2e):
            e2e_step(i)
        for so in s_outs:
            s_in.wait_stream(so)
        s1.record(s_in)
        torch.cuda.synchronize()
        barrier()
        e2e_passes.append(max_over_ranks(s0.elapsed_time(s1), dev) / n_e2e)
    e2e_ms = statistics.median(e2e_passes)
    # the host link itself: one pinned copy each way of the step's bytes
    # (the e2e step moves h2d + d2h bytes; its floor is the slower direction)
    lk = torch.empty(d2h // 2, dtype=torch.bfloat16, device=dev)
    lh = torch.empty(d2h // 2, dtype=torch.bfloat16).pin_memory()
    torch.cuda.synchronize()
    l0, l1, l2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    l0.record(stream)
    lh.copy_(lk, non_blocking=True)
    l1.record(stream)
    lk.copy_(lh, non_blocking=True)
    l2.record(stream)
    torch.cuda.synchronize()
    d2h_gbs = d2h / (l0.elapsed_time(l1) * 1e-3) / 1e9
    h2d_gbs = d2h / (l1.elapsed_time(l2) * 1e-3) / 1e9
    del lk, lh
    # the result of the last step really came back
    assert torch.equal(houts[(n_e2e - 1) % 2].view(torch.int16)[0, :4],
                       sets[(n_e2e - 1) % 2]["out"].view(torch.int16)[0, :4].cpu())
    clocks.resume()

    # ---- the 4096-token block named by the metric (same stage, P = 2)
    also = None
    if not args.skip_also and args.workload != ALSO:
        wl2 = make_workload(ALSO)
        d2 = prepare(wl2)
        for _ in range(3):
            stage(wl2, d2)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(args.steps):
            stage(wl2, d2)
        a1.record(stream)
        torch.cuda.synchronize()
        st_ms = a0.elapsed_time(a1) / args.steps
        b1, b2 = breakdown(wl2, d2, args.steps)
        also = {"workload": wl2.spec.name, "stage_us": st_ms * 1e3, "k1_us": b1 * 1e3,
                "k2_us": b2 * 1e3,
                "k2_tflops": FLOP_PER_TOKEN * wl2.M / (b2 * 1e-3) / 1e12,
                "k2_frac_of_measured_bf16": FLOP_PER_TOKEN * wl2.M / (b2 * 1e-3) / 1e12 / peaks["bf16"]}
        del d2
    # ---- the stage with e4m3 outputs (per-tensor descales), same inputs
    e4m3_line = None
    if not args.skip_also:
        codes = torch.empty(d["out"].shape, dtype=torch.uint8, device=dev)
        descales = torch.tensor([1.0 / 64, 1.0 / 48, 1.0 / 128], dtype=torch.float32, device=dev)

        def e4m3_call():
            binding.mh3_preattn_run_e4m3(h, stream, wl.M, d["x"], d["xw"], d["sc"],
                                         d["sc"].stride(0), d["sh"], d["sh"].stride(0),
                                         wl.spec.rows, d["idx"], d["W"], d["qw"], d["kw"],
                                         d["cs"], wl.spec.S, d["pos"], wl.spec.P, wl.spec.eps,
                                         wl.spec.qk_eps, descales, d["ws"], codes)
        for _ in range(3):
            e4m3_call()
        torch.cuda.synchronize()
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        for _ in range(args.steps):
            e4m3_call()
        q1.record(stream)
        torch.cuda.synchronize()
        q_ms = q0.elapsed_time(q1) / args.steps
        e4m3_line = {"workload": f"{wl.spec.name}, out_mode e4m3 (descales q 1/64, k 1/48, "
                                 "v 1/128)", "stage_us": q_ms * 1e3,
                     "out_bytes": int(codes.numel()), "launches_per_call": 2}
        del codes
    # ---- the NVFP4 stage (FP4 operands, block-scaled tcgen05 GEMM), same x,
    # tables and weight; the weight is quantised once, outside the timing
    nvfp4_line = None
    if not args.skip_also:
        from norm_adaln_qkv_gb300.inputs import nvfp4_from_workload
        wf = nvfp4_from_workload(wl)
        lib = binding.load()
        Mf = wf.M
        idx32 = wf.adaln_index.to(dev)
        csf = wf.rope_cos_sin.to(dev)
        gsa = torch.tensor([wf.act_global_scale], dtype=torch.float32, device=dev)
        gsw = torch.tensor([wf.weight_global_scale], dtype=torch.float32, device=dev)
        wq = torch.empty(21504, 2688, dtype=torch.uint8, device=dev)
        wsf = torch.empty(lib.mh3_nvfp4_scales_bytes(21504, 5376, 1), dtype=torch.uint8, device=dev)
        binding.mh3_nvfp4_quantize(stream, d["W"], gsw, wq, wsf, True)
        aq = torch.empty(Mf, 2688, dtype=torch.uint8, device=dev)
        asf = torch.empty(lib.mh3_nvfp4_scales_bytes(Mf, 5376, 1), dtype=torch.uint8, device=dev)
        Pf = wl.spec.P

        def f_stage():
            binding.mh3_nvfp4_preattn_run(h, stream, Mf, d["x"], d["xw"], d["sc"], d["sc"].stride(0),
                                          d["sh"], d["sh"].stride(0), wl.spec.rows, idx32, wq, wsf,
                                          wf.weight_global_scale, gsa, None, d["qw"], d["kw"], csf,
                                          Pf, wl.spec.eps, None, aq, asf, d["out"])

        def f_k1():
            binding.mh3_nvfp4_norm_quant(h, stream, Mf, d["x"], d["xw"], d["sc"], d["sc"].stride(0),
                                         d["sh"], d["sh"].stride(0), wl.spec.rows, idx32,
                                         wl.spec.eps, gsa, aq, asf, True)

        def f_k2():
            binding.mh3_nvfp4_qkv(h, stream, Mf, aq, asf, wq, wsf, wf.weight_global_scale, gsa, None,
                                  d["qw"], d["kw"], csf, Pf, wl.spec.eps, None, d["out"])

        def timed(fn, n):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(n):
                fn()
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / n

        ocodes = torch.empty(lib.mh3_preattn_out_nvfp4_bytes(Mf, 0), dtype=torch.uint8, device=dev)
        osf = torch.empty(lib.mh3_preattn_out_nvfp4_bytes(Mf, 1), dtype=torch.uint8, device=dev)
        ogs = torch.tensor([336.0, 448.0, 268.8], dtype=torch.float32, device=dev)

        def f_stage_fp4out():
            binding.mh3_nvfp4_preattn_run_nvfp4_out(
                h, stream, Mf, d["x"], d["xw"], d["sc"], d["sc"].stride(0), d["sh"],
                d["sh"].stride(0), wl.spec.rows, idx32, wq, wsf, wf.weight_global_scale, gsa, None,
                d["qw"], d["kw"], csf, Pf, wl.spec.eps, ogs, aq, asf, ocodes, osf)

        st_ms = timed(f_stage, args.steps)
        k1f_ms = timed(f_k1, args.steps)
        k2f_ms = timed(f_k2, args.steps)
        st4_ms = timed(f_stage_fp4out, args.steps)
        del ocodes, osf
        tf4 = FLOP_PER_TOKEN * Mf / (k2f_ms * 1e-3) / 1e12
        k1f_bytes = Mf * 10752 + Mf * 4 + Mf * 2688 + Mf * 336
        nvfp4_line = {
            "workload": f"{wl.spec.name}, NVFP4 operands (W4A4, block 16, UE4M3 scales)",
            "stage_us": st_ms * 1e3, "k1_us": k1f_ms * 1e3, "k2_us": k2f_ms * 1e3,
            "stage_us_out_mode_nvfp4": st4_ms * 1e3,
            "k2_tflops": tf4,
            "k2_frac_of_bf16x4": tf4 / (4 * peaks["bf16"]),
            "k2_frac_of_bf16x6": tf4 / (6 * peaks["bf16"]),
            "fp4_peak_note": "FP4 peak = measured bf16 burst x 4 (the per-clock FP4/bf16 ratio "
                             "measured for this MMA shape) or x 6 (nominal 13.5/2.25)",
            "k1_gbs": k1f_bytes / (k1f_ms * 1e-3) / 1e9,
            "k1_frac_of_measured_hbm": k1f_bytes / (k1f_ms * 1e-3) / 1e9 / peaks["hbm"],
            "launches_per_call": 2}
        del wq, wsf, aq, asf, idx32, csf
    # ---- the attention output projection with the gated residual (the
    # step after attention, same GEMM machinery), at the bench's M
    out_proj = None
    out_proj_nvfp4 = None
    if not args.skip_also:
        from norm_adaln_qkv_gb300.inputs import make_out_proj_workload
        wo = make_out_proj_workload(wl.M)
        mod_o = wo.adaln_mod.to(dev)
        gate_o = wo.gate_view(mod_o)
        ao, Wo, gio, reso = (wo.attn_out.to(dev), wo.o_weight.to(dev), wo.gate_index.to(dev),
                             wo.residual.to(dev))
        outo = torch.empty_like(reso)

        def op_call():
            binding.mh3_out_proj_run(h, stream, wo.M, ao, Wo, gate_o, gate_o.stride(0),
                                     gate_o.shape[0], gio, reso, outo)
        for _ in range(3):
            op_call()
        torch.cuda.synchronize()
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        o0.record(stream)
        for _ in range(args.steps):
            op_call()
        o1.record(stream)
        torch.cuda.synchronize()
        op_ms = o0.elapsed_time(o1) / args.steps
        op_tf = OUT_PROJ_FLOP_PER_TOKEN * wo.M / (op_ms * 1e-3) / 1e12
        out_proj = {"workload": f"out-projection + gated residual, M={wo.M}, K=7168, N=5376",
                    "us": op_ms * 1e3, "tflops": op_tf, "frac_of_measured_bf16": op_tf / peaks["bf16"]}
        # the W4A4 (NVFP4) form: activation quantiser + block-scaled GEMM
        from norm_adaln_qkv_gb300.inputs import out_proj_nvfp4_global_scales
        ags, wgs = out_proj_nvfp4_global_scales()
        lib4 = binding.load()
        wq4 = torch.empty((5376, 3584), dtype=torch.uint8, device=dev)
        wsf4 = torch.empty(lib4.mh3_nvfp4_scales_bytes(5376, 7168, 1), dtype=torch.uint8,
                           device=dev)
        binding.mh3_nvfp4_quantize(stream, Wo, torch.tensor([wgs], device=dev), wq4, wsf4, True)
        ags_d = torch.tensor([ags], dtype=torch.float32, device=dev)
        aq4 = torch.empty((wo.M, 3584), dtype=torch.uint8, device=dev)
        asf4 = torch.empty(lib4.mh3_nvfp4_scales_bytes(wo.M, 7168, 1), dtype=torch.uint8,
                           device=dev)

        def op4_call():
            binding.mh3_nvfp4_out_proj_run(h, stream, wo.M, ao, wq4, wsf4, wgs, ags_d, gate_o,
                                           gate_o.stride(0), gate_o.shape[0], gio, reso, aq4,
                                           asf4, outo)

        def q4_call():
            binding.mh3_nvfp4_quantize(stream, ao, ags_d, aq4, asf4, True)
        res4 = {}
        for name, fn in (("call", op4_call), ("quantiser", q4_call)):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            res4[name] = e0.elapsed_time(e1) / args.steps
        op4_tf = OUT_PROJ_FLOP_PER_TOKEN * wo.M / (res4["call"] * 1e-3) / 1e12
        q4_bytes = wo.M * (7168 * 2 + 3584 + 448)  # bf16 in; codes and scales out
        gemm4_ms = res4["call"] - res4["quantiser"]
        out_proj_nvfp4 = {
            "workload": f"W4A4 (NVFP4) out-projection + gated residual, M={wo.M}, K=7168, N=5376",
            "us": res4["call"] * 1e3, "tflops": op4_tf,
            "frac_of_fp4_peak_bf16x4": op4_tf / (4 * peaks["bf16"]),
            "quantiser_us": res4["quantiser"] * 1e3,
            "quantiser_frac_of_measured_hbm":
                q4_bytes / (res4["quantiser"] * 1e-3) / 1e9 / peaks["hbm"],
            "gemm_us_by_difference": gemm4_ms * 1e3,
            "gemm_tflops_by_difference": OUT_PROJ_FLOP_PER_TOKEN * wo.M / (gemm4_ms * 1e-3) / 1e12,
            "fp4_peak_note": "FP4 peak = measured bf16 burst x 4 (the per-clock FP4/bf16 ratio "
                             "measured for this MMA shape)",
            "launches_per_call": 2}
        del ao, Wo, gio, reso, outo, mod_o, wq4, wsf4, aq4, asf4
    # ---- the MLP block (norm/AdaLN, fc1 + SwiGLU, fc2 + gated residual)
    mlp_line = None
    if not args.skip_also:
        from norm_adaln_qkv_gb300.inputs import make_mlp_workload
        wm = make_mlp_workload(wl.M)
        mod_m = wm.adaln_mod.to(dev)
        sc_m, sh_m, gt_m = wm.tables(mod_m)
        xm, xwm, im, rm = (wm.x.to(dev), wm.x_norm_weight.to(dev), wm.adaln_index.to(dev),
                           wm.residual.to(dev))
        f1, f2 = wm.fc1_weight.to(dev), wm.fc2_weight.to(dev)
        wam = torch.empty((wm.M, 5376), dtype=torch.bfloat16, device=dev)
        wym = torch.empty((wm.M, 14336), dtype=torch.bfloat16, device=dev)
        outm = torch.empty_like(rm)

        def mlp_call():
            binding.mh3_mlp_run(h, stream, wm.M, xm, xwm, sc_m, sc_m.stride(0), sh_m,
                                sh_m.stride(0), gt_m, gt_m.stride(0), sc_m.shape[0], im, rm, f1,
                                f2, wm.eps, wam, wym, outm)
        for _ in range(3):
            mlp_call()
        torch.cuda.synchronize()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for _ in range(args.steps):
            mlp_call()
        m1.record(stream)
        torch.cuda.synchronize()
        mlp_ms = m0.elapsed_time(m1) / args.steps
        mlp_tf = MLP_FLOP_PER_TOKEN * wm.M / (mlp_ms * 1e-3) / 1e12
        mlp_line = {"workload": f"MLP block (bf16), M={wm.M}, 5376 -> 2x14336 -> 5376",
                    "us": mlp_ms * 1e3, "tflops": mlp_tf,
                    "frac_of_measured_bf16": mlp_tf / peaks["bf16"], "launches_per_call": 3}
        del xm, f1, f2, wam, wym, outm, rm
    # ---- the FP8 (W8A8) MLP block (E4M3 weights and per-token activations)
    mlp_fp8_line = None
    if not args.skip_also:
        from norm_adaln_qkv_gb300.inputs import make_mlp_fp8_workload
        w8 = make_mlp_fp8_workload(wl.M)
        mod8 = w8.adaln_mod.to(dev)
        sc8, sh8, gt8 = w8.tables(mod8)
        x8, xw8, i8, r8 = (w8.x.to(dev), w8.x_norm_weight.to(dev), w8.adaln_index.to(dev),
                           w8.residual.to(dev))
        f1q, f1s, f2q, f2s = (w8.fc1_q.to(dev), w8.fc1_scale.to(dev), w8.fc2_q.to(dev),
                              w8.fc2_scale.to(dev))
        lib8 = binding.load()
        wsb = [torch.empty(lib8.mh3_mlp_fp8_workspace_bytes(wl.M, k), dtype=torch.uint8,
                           device=dev) for k in range(5)]
        out8 = torch.empty_like(r8)

        def mlp8_call():
            binding.mh3_mlp_fp8_run(h, stream, w8.M, x8, xw8, sc8, sc8.stride(0), sh8,
                                    sh8.stride(0), gt8, gt8.stride(0), sc8.shape[0], i8, r8, f1q,
                                    f1s, f2q, f2s, w8.eps, wsb[0], wsb[1], wsb[2], wsb[3], wsb[4],
                                    out8)
        for _ in range(3):
            mlp8_call()
        torch.cuda.synchronize()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for _ in range(args.steps):
            mlp8_call()
        m1.record(stream)
        torch.cuda.synchronize()
        mlp8_ms = m0.elapsed_time(m1) / args.steps
        mlp8_tf = MLP_FLOP_PER_TOKEN * w8.M / (mlp8_ms * 1e-3) / 1e12
        mlp_fp8_line = {"workload": f"MLP block (E4M3 W8A8), M={w8.M}, 5376 -> 2x14336 -> 5376",
                        "us": mlp8_ms * 1e3, "tflops": mlp8_tf,
                        "frac_of_fp8_peak": mlp8_tf / (2 * peaks["bf16"]),
                        "fp8_peak_note": "FP8 peak = measured bf16 burst x 2 (nominal 4.5/2.25)",
                        "launches_per_call": 4}
        del x8, r8, f1q, f2q, wsb, out8, mod8
    # ---- the small configurations (M = 16, 1024): per-call medians of the
    # whole stage, back to back (warm) and after writing 320 MB (> 2x L2)
    small = None
    if not args.skip_also:
        flush = torch.empty(80 * 2**20, dtype=torch.float32, device=dev)
        reread = torch.empty(80 * 2**20, dtype=torch.float32, device=dev).fill_(1.0)
        small = {}
        for key in ("c0", "c1"):
            ws_ = make_workload(key)
            ds_ = prepare(ws_)
            for _ in range(3):
                stage(ws_, ds_)
            per = {}
            for mode in ("warm", "cold", "cold_clean"):
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(SMALL_CALLS)]
                for i, (s0, s1) in enumerate(evs):
                    if mode != "warm":
                        flush.fill_(float(i))  # 320 MB written: nothing of the inputs stays in L2
                    if mode == "cold_clean":
                        reread.sum()  # 320 MB read: L2 left holding clean lines, no write-back due
                    s0.record(stream)
                    stage(ws_, ds_)
                    s1.record(stream)
                torch.cuda.synchronize()
                per[mode] = statistics.median(s0.elapsed_time(s1) for s0, s1 in evs) * 1e3
            roof = stage_roofline_us(ws_, peaks)
            small[key] = {"workload": ws_.spec.name, "stage_us_warm": per["warm"],
                          "stage_us_cold": per["cold"], "stage_us_cold_clean": per["cold_clean"],
                          "stage_roofline_us": roof,
                          "roofline_frac_warm": roof / per["warm"],
                          "roofline_frac_cold": roof / per["cold"],
                          "roofline_frac_cold_clean": roof / per["cold_clean"],
                          "timed": f"median of {SMALL_CALLS} calls, CUDA events around each; "
                                   "cold: after writing 320 MB (the write-backs of that buffer's "
                                   "dirty lines then fall in the timed call); cold_clean: after "
                                   "writing 320 MB and then reading another 320 MB"}
            del ds_
        del flush, reread
    clk = clocks.stop()
    assert h.device_status(stream) == 0, "a kernel recorded a timeout"

    if rank != 0:
        return
    M = wl.M
    ms_step = ms_total / args.steps
    value_us = job_value_us(ms_total, args.steps, world)
    # kernel 2's time inside the timed region: the timed step times its share
    k2_timed_ms = ms_step * k2_share
    k2_tflops = FLOP_PER_TOKEN * M / (k2_timed_ms * 1e-3) / 1e12
    k1_bytes = M * 5376 * 2 * 2 + M * 8
    k1_gbs = k1_bytes / (k1_first_ms * 1e-3) / 1e9
    k1_gbs_after = k1_bytes / (k1_alone_ms * 1e-3) / 1e9
    k1_gbs_stage = k1_bytes / (ms_step * (1 - k2_share) * 1e-3) / 1e9
    stage_roof_us = stage_roofline_us(wl, peaks)
    line = {
        "metric": METRIC, "value": value_us, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(wl, world),
        "gemm_tflops": k2_tflops,
        "stage_roofline_us": stage_roof_us,
        "stage_roofline_frac": stage_roof_us / (ms_step * 1e3),
        "k2_share": k2_share,
        "k2_us_in_timed_region": k2_timed_ms * 1e3,
        "kernels_us": {"k1_norm_adaln": k1_ms * 1e3, "k2_qkv_gemm": k2_ms * 1e3,
                       "stage_interleaved": stage_interleaved_ms * 1e3,
                       "k1_norm_adaln_alone": k1_first_ms * 1e3,
                       "k1_norm_adaln_alone_after_gemm": k1_alone_ms * 1e3,
                       "timed": f"{args.steps} iterations of (stage call, kernel 1, kernel 2) "
                                "after the timed region, CUDA events around each"},
        "kernels_us_median": {"k1_norm_adaln": k1_med * 1e3, "k2_qkv_gemm": k2_med * 1e3,
                              "k1_plus_k2": pair_med * 1e3,
                              "timed": f"median of {args.steps} calls, CUDA events around each "
                                       "kernel on the launching stream"},
        "roofline": {"bound": "tensor", "achieved": k2_tflops, "peak": peaks["bf16"],
                     "unit": "TFLOP/s", "frac": k2_tflops / peaks["bf16"],
                     "traffic": _k2_traffic(M),
                     "flop_per_launch": FLOP_PER_TOKEN * M,
                     "kernel_us": k2_timed_ms * 1e3,
                     "how": "achieved = flop_per_launch / kernel_us; kernel_us = ms_per_step x "
                            "k2_share, the share of kernel 2 in (kernel 1 + kernel 2) timed "
                            "step by step at the same clock",
                     "peak_source": f"{peaks['src']} bf16 burst (kernel timed alone)",
                     "frac_of_sustained": k2_tflops / peaks["bf16_sus"]},
        "k1_roofline": {"bound": "hbm", "achieved": k1_gbs, "peak": peaks["hbm"], "unit": "GB/s",
                        "frac": k1_gbs / peaks["hbm"], "bytes_per_launch": k1_bytes,
                        "timed": "kernel 1 alone, back to back, before any GEMM ran",
                        "after_gemm": {"achieved": k1_gbs_after,
                                       "frac": k1_gbs_after / peaks["hbm"],
                                       "timed": "kernel 1 alone, back to back, after the GEMM "
                                                "loops (power-capped clocks)"},
                        "in_stage": {"achieved": k1_gbs_stage,
                                     "frac": k1_gbs_stage / peaks["hbm"],
                                     "kernel_us": ms_step * (1 - k2_share) * 1e3,
                                     "timed": "ms_per_step x (1 - k2_share): kernel 1's part "
                                              "of the timed step"},
                        "frac_of_nominal_8tbs": k1_gbs / 8000.0},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_ms * 1e3 / world, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "link_gbs": {"d2h": d2h_gbs, "h2d": h2d_gbs},
                "link_floor_us": max(d2h / d2h_gbs, h2d / h2d_gbs) * 1e-3,
                "passes_us": [v * 1e3 / world for v in e2e_passes],
                "how": "pinned host inputs in and out back every step; copies of neighbouring "
                       "steps overlap the kernels (2 buffer sets; input, compute and "
                       f"{n_out} read-back streams); the clock sampling is paused during "
                       "these passes (its polling slows the host<->device copies)"},
        "gpu_launches": gpu_launches,
        "clocks": clk,
        "also": also,
        "e4m3": e4m3_line,
        "nvfp4": nvfp4_line,
        "out_proj": out_proj,
        "out_proj_nvfp4": out_proj_nvfp4,
        "mlp": mlp_line,
        "mlp_fp8": mlp_fp8_line,
        "small": small,
    }
    print(json.dumps(line), flush=True)


def run_out_proj_only(args, world, rank, local):
    """The attention output projection alone (small cases and profiling)."""
    from norm_adaln_qkv_gb300 import binding, build
    from norm_adaln_qkv_gb300.inputs import make_out_proj_workload
    torch.cuda.set_device(local)
    build.build()
    h = binding.Handle(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks()
    wo = make_out_proj_workload(args.op_tokens)
    mod = wo.adaln_mod.to(dev)
    gate = wo.gate_view(mod)
    a, W, gi, res = (wo.attn_out.to(dev), wo.o_weight.to(dev), wo.gate_index.to(dev),
                     wo.residual.to(dev))
    out = torch.empty_like(res)

    def call():
        binding.mh3_out_proj_run(h, stream, wo.M, a, W, gate, gate.stride(0), gate.shape[0], gi,
                                 res, out)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    assert h.device_status(stream) == 0, "a kernel recorded a timeout"
    ms = e0.elapsed_time(e1) / args.steps
    tf = OUT_PROJ_FLOP_PER_TOKEN * wo.M / (ms * 1e-3) / 1e12
    if rank == 0:
        print(json.dumps({"only": "out_proj", "M": wo.M, "us": ms * 1e3, "tflops": tf,
                          "frac_of_measured_bf16": tf / peaks["bf16"], "steps": args.steps}),
              flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=8192,
                    help="tokens of the oracle CPU-baseline sample (0 disables)")
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="tokens per step of the reference (oracle) arm")
    ap.add_argument("--skip-also", action="store_true", help="skip the M=4096 side measurement")
    ap.add_argument("--workload", default=WORKLOAD, choices=["c0", "c1", "c2", "c3", "c4"],
                    help="seeded workload (default: the M=32760 production sequence)")
    ap.add_argument("--e2e-chunks", type=int, default=1,
                    help="contiguous pieces (and streams) of the end-to-end read-back")
    ap.add_argument("--only", choices=["stage", "out_proj"], default="stage",
                    help="out_proj: time the output projection alone (no JSON bench line)")
    ap.add_argument("--op-tokens", type=int, default=4096,
                    help="tokens of the --only out_proj case")
    ap.add_argument("--lib", default=None,
                    help="time this build of the library instead of the package's own "
                         "(a variant from `python -m norm_adaln_qkv_gb300.build --out`)")
    args = ap.parse_args()
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.only == "out_proj":
        run_out_proj_only(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
