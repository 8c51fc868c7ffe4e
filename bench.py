"""Benchmark of the flash-attention backward over a raw q8_0 K/V cache on one GB300.

Workload (the long-context shape): N=2048 queries, M=75520 keys, H=24, Hkv=4 (GQA 6),
D=Dv=256, q8_0 K and V, causal tail, Q/dO/K/V ~ N(0,1) f32 before quantization (seeded,
synthetic).  One step = one fa_back() call: statistics and packing, the LSE/D pass, the dQ pass
and the dK/dV pass.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 4]

Prints one JSON line on rank 0.  Under torchrun each rank runs an independent replica on its
own GPU (the operation has no exchange step); value = work of all ranks / slowest rank's time.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "FA-back ms + TFLOP/s at N2048/M75520/H24/Hkv4/D256 q8_0; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_PRODUCTS = {  # contractions (of the five) each pass forms on every visible (i, j) pair
    "k_rows_lse": 2, "k_rows_dq": 3, "k_cols": 4, "k_cols_rowscale": 4, "k_dq_gemm": 1, "k_dq_raw": 1}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms while running; the summary
    keeps the samples taken inside the marked region (mark_start / mark_end)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 3.0 and os.path.getsize(self.file.name) == 0:  # wait for the first sample
                time.sleep(0.02)
        except Exception:
            self.proc = None
        self.t_start = self.t_end = None
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = [ln.strip().split(",") for ln in open(self.file.name) if ln.strip()]
        os.unlink(self.file.name)
        def when(r):
            try:
                return datetime.datetime.strptime(r[9].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except (ValueError, IndexError):
                return None
        if self.t_start is not None and self.t_end is not None:
            inside = [r for r in rows if when(r) is not None and self.t_start <= when(r) <= self.t_end + 0.01]
            if not inside:  # a region shorter than the sampling period: the first sample after it starts
                after = [r for r in rows if when(r) is not None and when(r) >= self.t_start]
                inside = after[:1]
            rows = inside
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _tail_problem(p, n):
    """The last n query positions (all heads) of p against its full cache."""
    return synth.gen.Problem(name=p.name + f"_last{n}", N=n, M=p.M, H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                             k_type=p.k_type, v_type=p.v_type, causal=p.causal, scale=p.scale,
                             q=p.q[p.N - n:], k=p.k, v=p.v, dO=p.dO[p.N - n:], mask=None, mask_heads=0)


def calibrate_oracle(p, target_s: float):
    """Rows of a bounded oracle sample that take about target_s seconds: time = a + b * n."""
    import oracle
    oracle.build()
    ts = {}
    for n in (2, 6):
        t0 = time.perf_counter()
        oracle.fa_back(_tail_problem(p, n))
        ts[n] = time.perf_counter() - t0
    b = max((ts[6] - ts[2]) / 4, 1e-4)
    a = max(ts[2] - 2 * b, 0.0)
    return int(max(2, min(p.N, (target_s - a) / b)))


def cpu_baseline(p, target_s: float = 12.0, n: int = 0):
    """The CPU oracle, as it stands, on a bounded sample of the workload: the last n query
    positions (all heads) against the full cache.  The causal tail of those rows is the same as
    in the full problem.  Returns TFLOP/s of the sample (10 * D * H * visible pairs / time)."""
    import oracle
    if n <= 0:
        n = calibrate_oracle(p, target_s)
    s = _tail_problem(p, n)
    t0 = time.perf_counter()
    oracle.fa_back(s)
    dt = time.perf_counter() - t0
    return {"value": s.flops() / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.default_threads(), "kind": "oracle",
            "sample": f"last {n} of {p.N} query positions x all {p.H} heads against all {p.M} keys "
                      f"(lse, delta, dQ and their dK/dV contributions), {dt:.1f} s"}


def workload(args):
    """The benchmarked problem and its config record (--keys shortens the cache for profiling)."""
    over = {"M": args.keys} if args.keys else {}
    p = synth.from_config(args.config, **over)
    name = f"N{p.N}/M{p.M}/H{p.H}/Hkv{p.Hkv}/D{p.D} {synth.TYPE_NAMES[p.k_type]}" + (
        " causal tail" if p.causal else "")
    in_mb = sum(a.nbytes for a in (p.q, p.dO, p.k, p.v, p.mask) if a is not None) / 1e6
    cfg = {"workload": name, "N": p.N, "M": p.M, "H": p.H, "Hkv": p.Hkv, "D": p.D, "Dv": p.Dv,
           "causal": bool(p.causal), "flops_per_step": p.flops(), "alg_bytes_per_step": p.alg_bytes(),
           "l2": (f"inputs ({in_mb:.0f} MB) larger than L2 (129 MB), no flush" if in_mb > 129 else
                  f"inputs ({in_mb:.0f} MB) fit in L2; no flush (profiling case, not a bench line)")}
    return p, cfg


def read_traffic(p) -> dict:
    """Per-launch DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) recorded under
    profiles/ for this workload, by kernel; empty when none was captured for it."""
    path = os.path.join(ROOT, "profiles", f"dram_traffic_N{p.N}_M{p.M}_H{p.H}_Hkv{p.Hkv}_D{p.D}_"
                                          f"{synth.TYPE_NAMES[p.k_type]}.md")
    out = {}
    if os.path.exists(path):
        for line in open(path):
            f = line.split()
            if len(f) == 3 and f[0] == "traffic":
                out[f[1]] = int(f[2])
    return out


def init_dist():
    """(dist, rank, world size) under torchrun, else (None, 0, 1).  NCCL where the GPUs are
    visible; gloo on host cores only (the reference arm on a machine without GPUs)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        return dist, dist.get_rank(), ws
    return None, 0, 1


def max_over_ranks(dist, values, device=None):
    """Each value's maximum over all ranks (the slowest rank's time); unchanged for one process."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    x = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return [float(v) for v in x.tolist()]


def job_tflops(world: int, flops_per_replica: float, ms: float) -> float:
    """Whole-job rate: every replica's work over the slowest rank's time per step."""
    return world * flops_per_replica / (ms * 1e-3) / 1e12


def run_reference(args):
    """--impl reference: the CPU oracle timed on the host cores (rank 0 only)."""
    dist, rank, world = init_dist()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    p, cfg = workload(args)
    # one calibration, then every step times the same bounded sample; the whole run stays
    # within a few minutes
    per_step = max(2.0, min(args.ref_seconds, 100.0 / max(1, args.steps + args.warmup)))
    n = calibrate_oracle(p, per_step)
    for _ in range(args.warmup):
        cpu_baseline(p, n=n)
    vals = []
    base = None
    t_all = time.perf_counter()
    for _ in range(args.steps):
        base = cpu_baseline(p, n=n)
        vals.append(base["value"])
    wall = time.perf_counter() - t_all
    value = float(np.median(vals))
    base["value"] = value
    cfg = dict(cfg, parallelism="host cores of rank 0", sample_per_step=base["sample"])
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1), q8_0 quantized)", "config": cfg,
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_ours(args):
    import torch

    import flash_attention_backward_gb300 as fb
    from flash_attention_backward_gb300 import build as fbuild

    dist, rank, world = init_dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fbuild.build()
    if dist is not None:
        dist.barrier()
    p, cfg = workload(args)
    t = synth.device.to_torch(p, dev)
    out = {
        "dQ": torch.empty((p.N, p.H, p.D), dtype=torch.float32, device=dev),
        "dK": torch.empty((p.M, p.Hkv, p.D), dtype=torch.float32, device=dev),
        "dV": torch.empty((p.M, p.Hkv, p.Dv), dtype=torch.float32, device=dev),
        "lse": torch.empty((p.N, p.H), dtype=torch.float32, device=dev),
        "delta": torch.empty((p.N, p.H), dtype=torch.float32, device=dev),
    }
    ws = fb.Workspace(dev)
    stream = torch.cuda.current_stream(dev)

    def step(tt=t):
        fb.backward(tt["q"], tt["k"], p.k_type, tt["v"], p.v_type, tt["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                    M=p.M, scale=p.scale, causal=p.causal, mask=tt["mask"], mask_heads=p.mask_heads, out=out,
                    workspace=ws, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    rc = fb.fa_back_get_error()
    assert rc == 0, fb.fa_back_status_string(rc)

    # ---- device-timed steps (inputs resident; the inputs exceed L2, so no flush is needed)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    fb.fa_back_profile(True)
    with ClockSampler(local) as clk:
        clk.mark_start()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    fb.fa_back_profile(False)
    kern = fb.fa_back_profile_read()
    ms, = max_over_ranks(dist, [ev0.elapsed_time(ev1) / args.steps], dev)
    clocks = clk.summary()
    launches = sum(c for _, c in kern.values())

    # ---- the other entry points on the same resident inputs (informative, not the metric): the
    # backward given the forward's statistics (lse and delta from the steps above), and the forward
    def timed(fn, n):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n
    lse_s, delta_s = out["lse"].clone(), out["delta"].clone()
    n_var = max(3, min(args.steps, 10))
    ws_ms = timed(lambda: fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D,
                                      Dv=p.Dv, M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"],
                                      mask_heads=p.mask_heads, workspace=ws, stream=stream, lse=lse_s,
                                      delta=delta_s), n_var)
    fw_ms = timed(lambda: fb.forward(t["q"], t["k"], p.k_type, t["v"], p.v_type, H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                                     M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"],
                                     mask_heads=p.mask_heads, workspace=ws, stream=stream), n_var)
    def timed_kernels(fn, n):
        # the same, plus each kernel's mean time from the library's profile record
        ms_ = timed(fn, n)
        fb.fa_back_profile(True)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        fb.fa_back_profile(False)
        return ms_, {k: v[0] / v[1] for k, v in fb.fa_back_profile_read().items() if v[1]}

    # the plans that keep no decoded copy of the cache: the stored dS with every pass decoding the
    # raw cache (fa_back_nocopy's default workspace), and the smallest workspace (level 0)
    wnc = fb.fa_back_workspace_size_nocopy(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    wsnc = fb.Workspace(dev)
    nc_ms, nc_kern = timed_kernels(lambda: fb.backward(
        t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M, scale=p.scale,
        causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads, out=out, workspace=wsnc, stream=stream,
        workspace_bytes=wnc, nocopy=True), n_var)
    del wsnc
    wmin = fb.fa_back_workspace_size_min(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    lvl_min = fb.fa_back_plan_info(p.N, p.M, p.H, p.Hkv, p.D, p.Dv, wmin)
    wsmin = fb.Workspace(dev)
    mn_ms, mn_kern = timed_kernels(lambda: fb.backward(
        t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M, scale=p.scale,
        causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads, out=out, workspace=wsmin, stream=stream,
        workspace_bytes=wmin), n_var)
    del wsmin
    assert fb.fa_back_get_error() == 0
    ws_ms, fw_ms, mn_ms, nc_ms = max_over_ranks(dist, [ws_ms, fw_ms, mn_ms, nc_ms], dev)
    pk_v, _ = peaks()
    peak_v = float(pk_v.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    variants = {
        "fa_back_with_stats": {"ms": ws_ms, "TFLOP/s": job_tflops(world, p.flops(), ws_ms),
                               "note": "lse and delta given; the LSE/D pass is skipped; same F_alg"},
        "fa_back_nocopy": {"ms": nc_ms, "TFLOP/s": job_tflops(world, p.flops(), nc_ms),
                           "path_roofline_frac": p.flops() / (peak_v * 1e12) / (nc_ms * 1e-3),
                           "workspace_bytes": wnc, "plan_level": 3 if "k_dq_raw" in nc_kern else 0,
                           "kernels_ms": nc_kern,
                           "note": "no decoded copy of the cache: raw K/V tiles decoded in shared memory by every "
                                   "pass, dS stored (plan level 3); fa_back_nocopy() with "
                                   "fa_back_workspace_size_nocopy() bytes"},
        "fa_back_min_workspace": {"ms": mn_ms, "TFLOP/s": job_tflops(world, p.flops(), mn_ms),
                                  "path_roofline_frac": p.flops() / (peak_v * 1e12) / (mn_ms * 1e-3),
                                  "workspace_bytes": wmin, "plan": lvl_min, "kernels_ms": mn_kern,
                                  "note": "fa_back given fa_back_workspace_size_min() bytes (level 0: no copy, "
                                          "dS recomputed in a dQ pass)"},
        "fa_forward": {"ms": fw_ms, "TFLOP/s": job_tflops(world, 4.0 * p.D * p.H * p.visible_pairs(), fw_ms),
                       "note": "O and lse; TFLOP/s of its two contractions (S, P V)"},
    }

    # ---- end to end: pinned host inputs -> device, fa_back, results -> pinned host, every step.
    # Pipelined: three streams and double buffers, so step i's compute overlaps step i+1's input
    # copy and step i-1's result copy.  The serial form (one stream) is reported beside it.
    hq = synth.device.to_torch(p, "cpu", pin=True)
    keys_in = [k for k, v in hq.items() if v is not None]
    hout = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()} for _ in range(2)]
    din = [dict({k: torch.empty_like(t[k]) for k in keys_in}, mask=None) for _ in range(2)]
    dout = [{k: torch.empty_like(v) for k, v in out.items()} for _ in range(2)]
    h2d = sum(hq[k].numel() * hq[k].element_size() for k in keys_in)
    d2h = sum(v.numel() * v.element_size() for v in out.values())
    # as many steps as the device-timed region: the first step's input copy and the last step's
    # result copy, which nothing overlaps, are spread over the same K steps
    e_steps = max(2, args.steps)

    host_ms = {}  # host time per step to enqueue the copies and the call
    phases = {}   # serial form: per step, ms of input copies, the call and result copies

    def run_e2e(pipelined: bool) -> float:
        s_c = stream
        s_in = torch.cuda.Stream(dev) if pipelined else s_c
        s_out = torch.cuda.Stream(dev) if pipelined else s_c
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_c = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tev = [] if not pipelined else None  # serial form: phase boundaries on the one stream
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        e0.record(s_in)
        for i in range(e_steps):
            b = i % 2 if pipelined else 0
            if tev is not None:
                tev.append([torch.cuda.Event(enable_timing=True) for _ in range(4)])
                tev[-1][0].record(s_c)
            if pipelined and i >= 2:
                s_in.wait_event(ev_c[b])  # inputs b are read by compute(i-2)
            with torch.cuda.stream(s_in):
                for k in keys_in:
                    din[b][k].copy_(hq[k], non_blocking=True)
            ev_in[b].record(s_in)
            if tev is not None:
                tev[-1][1].record(s_c)
            s_c.wait_event(ev_in[b])
            if pipelined and i >= 2:
                s_c.wait_event(ev_out[b])  # outputs b still being copied back for step i-2
            fb.backward(din[b]["q"], din[b]["k"], p.k_type, din[b]["v"], p.v_type, din[b]["dO"], H=p.H, Hkv=p.Hkv,
                        D=p.D, Dv=p.Dv, M=p.M, scale=p.scale, causal=p.causal, mask=din[b]["mask"],
                        mask_heads=p.mask_heads, out=dout[b], workspace=ws, stream=s_c)
            ev_c[b].record(s_c)
            if tev is not None:
                tev[-1][2].record(s_c)
            s_out.wait_event(ev_c[b])
            with torch.cuda.stream(s_out):
                for k, v in dout[b].items():
                    hout[b][k].copy_(v, non_blocking=True)
            ev_out[b].record(s_out)
            if tev is not None:
                tev[-1][3].record(s_c)
        e1.record(s_out)
        host_ms[pipelined] = (time.perf_counter() - h0) * 1e3 / e_steps  # enqueueing only: no wait inside
        torch.cuda.synchronize()
        if tev is not None:
            phases.update({k: sum(ev[a].elapsed_time(ev[a + 1]) for ev in tev) / e_steps
                           for a, k in enumerate(("h2d_ms", "call_ms", "d2h_ms"))})
        return e0.elapsed_time(e1) / e_steps

    def copy_ms(h2d_dir: bool) -> float:
        # one step's input copies (or result copies) alone on the compute stream: the copy rate
        # the pipelined form has to hide behind the backward
        best = float("inf")
        for _ in range(3):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            c0.record(stream)
            with torch.cuda.stream(stream):
                if h2d_dir:
                    for k in keys_in:
                        din[0][k].copy_(hq[k], non_blocking=True)
                else:
                    for k, v in dout[0].items():
                        hout[0][k].copy_(v, non_blocking=True)
            c1.record(stream)
            torch.cuda.synchronize()
            best = min(best, c0.elapsed_time(c1))
        return best

    run_e2e(True)  # warm: first use of the second buffer set and of the copy streams
    e2e_serial_ms = run_e2e(False)
    e2e_ms = min(run_e2e(True), run_e2e(True))
    h2d_ms, d2h_ms = copy_ms(True), copy_ms(False)
    rc = fb.fa_back_get_error()
    assert rc == 0, fb.fa_back_status_string(rc)
    e2e_ms, e2e_serial_ms, h2d_ms, d2h_ms = max_over_ranks(dist, [e2e_ms, e2e_serial_ms, h2d_ms, d2h_ms], dev)

    flops = p.flops()
    tflops = job_tflops(world, flops, ms)
    e2e_tflops = job_tflops(world, flops, e2e_ms)
    pk, pk_src = peaks()
    # binary16 runs at the bf16 rate.  One step lasts milliseconds and the timed region well
    # under a second, so the burst figure is the denominator (the sustained one, measured over
    # seconds under the power cap, is reported beside it)
    peak_tensor = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sust = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # dominant kernel and its algorithmic flops per launch
    dom = max(((n, v) for n, v in kern.items() if n in KERNEL_PRODUCTS), key=lambda kv: kv[1][0], default=None)
    roofline = None
    if dom is not None:
        name, (tot_ms, cnt) = dom
        per_ms = tot_ms / cnt
        alg = KERNEL_PRODUCTS[name] * 2.0 * p.D * p.H * p.visible_pairs()
        ach = alg / (per_ms * 1e-3) / 1e12
        traffic = read_traffic(p).get(name)
        roofline = {"bound": "tensor", "kernel": name, "achieved": ach, "peak": peak_tensor, "unit": "TFLOP/s",
                    "frac": ach / peak_tensor, "traffic": traffic,
                    "peak_source": f"{pk_src} bf16 dense, burst (sustained {peak_sust:g}: frac {ach / peak_sust:.3f})",
                    "avg_ms": per_ms}
    # the whole backward against its roofline: T_roof = max(F_alg / tensor peak, B_alg / HBM rate)
    t_flop_ms = flops / (peak_tensor * 1e12) * 1e3
    t_byte_ms = p.alg_bytes() / (peak_hbm * 1e9) * 1e3
    t_roof_ms = max(t_flop_ms, t_byte_ms)
    path_frac = t_roof_ms / ms
    path = {"bound": "tensor" if t_flop_ms >= t_byte_ms else "hbm", "t_roof_ms": t_roof_ms, "ms": ms,
            "frac": path_frac, "achieved": flops / (ms * 1e-3) / 1e12, "peak": peak_tensor, "unit": "TFLOP/s",
            "peak_source": f"{pk_src} bf16 dense, burst; HBM {peak_hbm:g} GB/s",
            "frac_sustained": (flops / (peak_sust * 1e12)) / (ms * 1e-3)}
    if roofline is not None:
        roofline["path"] = path
    line = {"metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16xf16->f32", "data": "synthetic (seeded N(0,1), q8_0 quantized)",
            "config": dict(cfg, path_roofline_frac=path_frac, parallelism=f"replicas x{world}"),
            "roofline": roofline, "kernels_ms": {k: v[0] / v[1] for k, v in kern.items()},
            "gpu_launches": launches, "clocks": clocks, "variants": variants,
            "e2e": {"value": e2e_tflops, "unit": "TFLOP/s", "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "pipelining": "input copy, backward and result copy on three streams, double-buffered",
                    "steps": e_steps,
                    # host time per step spent enqueueing (above ms_per_step, the GPU waits on the host)
                    "host_enqueue_ms_per_step": host_ms.get(True),
                    "serial": {"value": job_tflops(world, flops, e2e_serial_ms), "ms_per_step": e2e_serial_ms,
                               "phases": phases},
                    # what the overlap has to hide: each direction's copies alone, and the host
                    # setting that would serialise the three streams if set to 1
                    "copies": {"h2d_ms": h2d_ms, "d2h_ms": d2h_ms, "h2d_GBps": h2d / (h2d_ms * 1e6),
                               "d2h_GBps": d2h / (d2h_ms * 1e6),
                               "pipelined_bound_ms": max(ms, h2d_ms, d2h_ms),
                               "CUDA_DEVICE_MAX_CONNECTIONS": os.environ.get("CUDA_DEVICE_MAX_CONNECTIONS")}}}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="4")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=12.0)
    ap.add_argument("--keys", type=int, default=0, help="override M (shorter cache, for profiling runs)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
