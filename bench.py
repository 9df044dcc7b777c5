#!/usr/bin/env python3
"""LoRA-MLP forward + backward throughput on one GB300 (or N independent replicas).

One step = lora_mlp_forward + lora_mlp_backward over one batch of the 7B-shaped
workload (M = 8192 tokens = 4 x 2048, h = 4096, i = 14336, r = 16, alpha = 32,
SwiGLU, bf16), synthetic seeded inputs resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU with no
collective on the data path ("replicas only": the block's work has no exchange
step on one batch); value = tokens of all ranks / the slowest rank's time.

--impl reference times the CPU float64 oracle (the only other implementation of
this method here) on a bounded sample of the same workload, on the host's cores.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-MLP fwd+bwd tokens/s and TFLOP/s as % of GB300 dense-BF16 peak"
WORKLOAD = "llama7b"


# ---------------------------------------------------------------------------- ranks

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(backend: str, timeout_s: float = 600.0):
    """Joins the process group.  A rank that dies or never arrives makes the others'
    next barrier or reduction raise within timeout_s instead of waiting forever."""
    rank, world, _ = dist_env()
    if world > 1:
        import datetime
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend, timeout=datetime.timedelta(seconds=timeout_s))
    return rank, world


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value over all ranks (the slowest rank's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed_steps(step, steps: int, world: int, device=None, sync=None, timer=None):
    """Barrier + sync, run `steps` steps inside the timer, sync + barrier; returns the
    max over ranks of the elapsed seconds.  `timer` is a (start, stop) pair whose
    stop returns seconds (CUDA events on the GPU, perf_counter on the CPU)."""
    sync = sync or (lambda: None)
    barrier(world, device)
    sync()
    start, stop = timer
    start()
    for _ in range(steps):
        step()
    secs = stop()
    sync()
    barrier(world, device)
    return max_over_ranks(secs, world, device)


def cuda_timer(torch, stream):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def start():
        e0.record(stream)

    def stop():
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3

    return start, stop


# ---------------------------------------------------------------------------- clocks

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
CLOCK_PERIOD_MS = 20


class ClockSampler:
    """nvidia-smi samples every CLOCK_PERIOD_MS while the timed region runs.  start()
    returns once the first sample is written (so sampling covers the region from its
    first step); stop() keeps the samples stamped inside [start, stop]."""

    def __init__(self):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader",
                                          "-lms", str(CLOCK_PERIOD_MS), "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        deadline = time.time() + 10.0
        while time.time() < deadline and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.t1 = time.time()
        time.sleep(2e-3 * CLOCK_PERIOD_MS)     # the sample that covers the region's end
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        return parse_clock_rows(rows, self.t0, self.t1, CLOCK_PERIOD_MS * 1e-3)


def _stamp(s):
    import datetime
    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.datetime.strptime(s, fmt).timestamp()
        except ValueError:
            pass
    return None


def parse_clock_rows(rows, t0=None, t1=None, slack=0.0):
    """Clock summary of nvidia-smi rows (CLOCK_FIELDS order): the rows stamped within
    [t0 - slack, t1 + slack] when the stamps allow (else all rows); median SM clock
    under load (samples above half the peak power seen), the reasons seen active."""
    def num(s):
        try:
            return float(s.split()[0])
        except (ValueError, IndexError):
            return None
    window = "whole sampling"
    if t0 is not None and t1 is not None:
        inside = [r for r in rows if (lambda t: t is not None and t0 - slack <= t <= t1 + slack)(_stamp(r[0]))]
        if inside:
            rows, window = inside, "timed region"
    rows = [r[1:] for r in rows]
    sm = [num(r[1]) for r in rows if num(r[1]) is not None]
    mx = [num(r[2]) for r in rows if num(r[2]) is not None]
    pw = [num(r[3]) for r in rows if num(r[3]) is not None]
    if not sm:
        return None
    # under load: samples above half of the peak power seen in the region
    pmax = max(pw) if pw else 0.0
    loaded = [num(r[1]) for r in rows if pw and num(r[3]) is not None and num(r[3]) >= 0.5 * pmax] or sm
    reasons = sorted({REASONS[j] for r in rows for j in range(4) if r[5 + j].lower() == "active"})
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx) if mx else None,
            "sm_mhz_min": min(loaded), "reasons": reasons, "samples": len(rows), "power_w_max": pmax,
            "window": window, "period_ms": CLOCK_PERIOD_MS}


# ---------------------------------------------------------------------------- flops

def kernel_flops(cfg):
    """Algorithmic FLOPs per launch of each GEMM kind of one MLP step."""
    M, h, i, r = cfg.M, cfg.h, cfg.i, cfg.r
    return {"gate_up": 4.0 * M * i * (h + r), "proj": 2.0 * M * h * (i + r),
            "act_bwd": 2.0 * M * i * (h + r), "dgrad": 4.0 * M * h * (i + r)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# The sustained peak is a cuBLAS loop run back to back for about 4 s under the power
# cap; a shorter timed region runs at burst clocks and is held to the burst peak.
SUSTAINED_REGION_S = 4.0
# Nominal dense bf16 tensor rate of a GB300 (context only: the measured peaks are the
# denominators).
NOMINAL_BF16_TFLOPS = 2250.0


def choose_peak(region_s: float, peaks: dict):
    """(key, TFLOP/s) of the measured bf16 peak that applies to a timed region of
    region_s seconds: the burst peak unless the region is as long as the loop the
    sustained peak was measured over."""
    if region_s >= SUSTAINED_REGION_S and "bf16_tflops_sustained" in peaks:
        return "bf16_tflops_sustained", float(peaks["bf16_tflops_sustained"])
    return "bf16_tflops", float(peaks["bf16_tflops"])


def peak_fields(tflops: float, region_s: float):
    """The line's peak fields for a whole-step rate: the fraction against the peak
    that applies to the region, plus the other measured peak and the nominal rate,
    each labelled."""
    peaks, src = measured_peaks()
    key, peak = choose_peak(region_s, peaks)
    out = {"tflops": tflops, "pct_of_peak": 100.0 * tflops / peak, "peak_tflops": peak,
           "peak_source": f"{src} {key} (timed region {region_s:.3f} s; the sustained peak applies from "
                          f"{SUSTAINED_REGION_S:g} s)",
           "timed_region_s": region_s,
           "pct_of_nominal_dense_bf16": 100.0 * tflops / NOMINAL_BF16_TFLOPS}
    if "bf16_tflops_sustained" in peaks:
        out["pct_of_sustained_peak"] = 100.0 * tflops / float(peaks["bf16_tflops_sustained"])
    out["pct_of_burst_peak"] = 100.0 * tflops / float(peaks["bf16_tflops"])
    return out, peak, f"{src} {key}"


def kernel_source_sha() -> str:
    """sha256[:16] over the GEMM kernels' sources (ptx.cuh, gemm_tc.cuh, gemm_pair.cuh)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("ptx.cuh", "gemm_tc.cuh", "gemm_pair.cuh"):
        with open(os.path.join(ROOT, "rank_mlp_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_workload_key(cfg) -> str:
    """The workload column of profiles/traffic.md for an MLP config."""
    return f"{cfg.name} M={cfg.M} h={cfg.h} i={cfg.i} r={cfg.r}"


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` (traffic_workload_key) from
    profiles/traffic.md, if that capture was taken on the current kernel source; else
    None."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        sha = kernel_source_sha()
        for line in open(path):
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload and cells[2] == sha:
                return float(cells[3])
    except (OSError, ValueError):
        pass
    return None


def kernel_breakdown(lib, step, steps: int) -> dict:
    """{kind: [launches, total ms]} over `steps` traced steps (every launch bracketed by
    CUDA events; outside the timed region, since the events serialise the launches)."""
    import torch
    torch.cuda.synchronize()
    lib.trace_kinds(None)
    lib.trace_enable(64 * steps + 64)
    for _ in range(steps):
        step()
    trace = lib.trace_read(64 * steps + 64)
    lib.trace_enable(0)
    per_kind = {}
    for k, ms in trace:
        a = per_kind.setdefault(k, [0, 0.0])
        a[0] += 1
        a[1] += ms
    return per_kind


def timed_region(lib, step, steps, world, device, stream):
    """The timed region: `steps` untraced steps (no events between launches, so the
    kernels overlap as they do in use), clocks sampled meanwhile.  Returns (seconds,
    max over ranks; clocks; launches of the library's kernels)."""
    import torch
    n0 = lib.launch_count()
    rank = dist_env()[0]
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    secs = timed_steps(step, steps, world, device, torch.cuda.synchronize, cuda_timer(torch, stream))
    clk = clocks.stop() if rank == 0 else None
    return secs, clk, lib.launch_count() - n0


def kernel_launch_ms(lib, step, steps, kind):
    """A separate pass of `steps` steps with CUDA events around the launches of `kind`
    only (the dominant kernel); returns the duration of each of its launches (ms)."""
    import torch
    torch.cuda.synchronize()
    lib.trace_kinds([kind])
    lib.trace_enable(16 * steps + 16)
    for _ in range(steps):
        step()
    trace = lib.trace_read(16 * steps + 16)
    lib.trace_enable(0)
    lib.trace_kinds(None)
    return [ms for k, ms in trace if k == kind]


# ---------------------------------------------------------------------------- oracle

def oracle_step_fn(cfg, tokens: int, host):
    """One oracle fwd+bwd over the first `tokens` rows of the workload."""
    import oracle
    v = host
    x, dy = v["x"][:tokens], v["dy"][:tokens]

    def step():
        args = (x, v["W_gate"], v["A_gate"], v["B_gate"], v["W_up"], v["A_up"], v["B_up"],
                v["W_down"], v["A_down"], v["B_down"], cfg.s, cfg.act)
        f = oracle.mlp_forward(*args)
        b = oracle.mlp_backward(*args, dy)
        return f, b
    return step


def host_inputs(cfg, max_tokens: int, seed: int = 0):
    """Float64 copies of the workload's bf16 inputs (tokens truncated; the generator's
    streams do not depend on the token count, so these are the workload's first rows)."""
    import torch
    import synth
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    c = cfg.replace(M=max_tokens)
    t = synth.make_mlp_inputs(c, seed=seed, device=dev)
    return {k: synth.bf16_to_f64(x) for k, x in t.items()}


def parity_errors(got, ref) -> dict:
    """Relative Frobenius error and max-abs error / max |ref| of a GPU result (bf16
    tensor) against the float64 oracle."""
    import numpy as np
    import synth
    g = np.asarray(synth.bf16_to_f64(got), np.float64)
    ref = np.asarray(ref, np.float64)
    return {"rel_fro": float(np.linalg.norm(g - ref) / np.linalg.norm(ref)),
            "max_abs_over_max_ref": float(np.abs(g - ref).max() / np.abs(ref).max())}


def cpu_baseline(cfg, budget_s: float = 15.0, got=None, seed: int = 0):
    """Times the oracle as it stands on a sample of tokens sized for ~budget_s.  got:
    the GPU's results for the first tokens ({"y": ..., "dx": ...}, bf16 on the host):
    the sample's oracle results then also give the parity errors of those rows."""
    probe = 64
    host = host_inputs(cfg, 4096, seed)
    t0 = time.perf_counter()
    oracle_step_fn(cfg, probe, host)()
    per_tok = (time.perf_counter() - t0) / probe
    tokens = int(max(probe, min(4096, budget_s / max(per_tok, 1e-9))))
    step = oracle_step_fn(cfg, tokens, host)
    t0 = time.perf_counter()
    f, b = step()
    dt = time.perf_counter() - t0
    out = {"value": tokens / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
           "sample": f"fwd+bwd of the first {tokens} of {cfg.M} tokens (all weights full size), "
                     f"float64 numpy/BLAS, {dt:.1f} s"}
    if got:
        n = min(tokens, got["y"].shape[0])
        par = {"tokens": n, "tolerance": {"rel_fro": 1e-2, "max_abs_over_max_ref": 3e-2}}
        par["y"] = parity_errors(got["y"][:n], f["y"][:n])
        if "dx" in got:
            par["dx"] = parity_errors(got["dx"][:n], b["dx"][:n])
        out["parity"] = par
    return out


# ---------------------------------------------------------------------------- arms

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import synth
    cfg = mlp_config(args)
    host = host_inputs(cfg, 4096, args.seed)
    probe = 32
    t0 = time.perf_counter()
    oracle_step_fn(cfg, probe, host)()
    per_tok = (time.perf_counter() - t0) / probe
    budget = 150.0 / max(args.steps + args.warmup, 1)        # whole run within a few minutes
    tokens = int(max(16, min(4096, budget / max(per_tok, 1e-9))))
    step = oracle_step_fn(cfg, tokens, host)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    value = tokens * args.steps / secs
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator), bounded token sample",
        "config": {"workload": workload_name(cfg), "sample_tokens": tokens},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"fwd+bwd of {tokens} of {cfg.M} tokens per step, float64 numpy/BLAS"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def mlp_config(args):
    """The MLP workload with the command line's activation and rank overrides (a rank
    override keeps the scale s = alpha / r)."""
    import synth
    cfg = synth.MLP_CONFIGS[args.workload]
    if args.act:
        cfg = cfg.replace(act=args.act)
    if args.rank:
        cfg = cfg.replace(r=args.rank, alpha=cfg.s * args.rank)
    if getattr(args, "tokens", 0):
        cfg = cfg.replace(M=args.tokens)
    return cfg


def workload_name(cfg):
    return (f"{cfg.name}-shaped LoRA-MLP fwd+bwd: M={cfg.M} tokens ({cfg.batch}x{cfg.seq}), h={cfg.h}, "
            f"i={cfg.i}, r={cfg.r}, alpha={cfg.alpha:g}, {cfg.act}")


def mlp_workload(lib, cfg, device, seed, n_ex=0):
    """Device-resident inputs, outputs, saved blob and workspace of one MLP workload
    and its fwd+bwd step."""
    import torch
    import synth
    M, h, i, r = cfg.M, cfg.h, cfg.i, cfg.r
    t = synth.make_mlp_inputs(cfg, seed=seed, device=device)
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    gate, up, down = lin("gate"), lin("up"), lin("down")
    saved_b, ws_b = lib.mlp_sizes(M, h, i, r)
    if n_ex:
        ws_b = max(ws_b, lib.load().lora_mlp_per_example_workspace_bytes(M, h, i, r, n_ex))
    w = types.SimpleNamespace(cfg=cfg, t=t, gate=gate, up=up, down=down, n_ex=n_ex)
    w.saved = torch.empty(saved_b, dtype=torch.uint8, device=device)
    w.ws = torch.zeros(ws_b, dtype=torch.uint8, device=device)
    w.y = torch.empty(M, h, dtype=torch.bfloat16, device=device)
    w.dx = torch.empty(M, h, dtype=torch.bfloat16, device=device)
    e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device=device)  # noqa: E731
    w.grads = {"dA_gate": e(r, h), "dB_gate": e(i, r), "dA_up": e(r, h), "dB_up": e(i, r),
               "dA_down": e(r, i), "dB_down": e(h, r)}

    def step():
        lib.mlp_forward(t["x"], gate, up, down, cfg.s, cfg.act, y=w.y, saved=w.saved, ws=w.ws)
        if n_ex:
            lib.mlp_backward_per_example(t["x"], gate, up, down, cfg.s, cfg.act, w.saved, t["dy"], n_ex, ws=w.ws)
        else:
            lib.mlp_backward(t["x"], gate, up, down, cfg.s, cfg.act, w.saved, t["dy"], dx=w.dx, grads=w.grads,
                             ws=w.ws)
    w.step = step
    w.flops = kernel_flops(cfg)
    w.total_flops = cfg.flops()
    w.M = M
    return w


def qkvo_workload(lib, cfg, device, seed, rope=False):
    """The same for the Q/K/V + O projections (optionally with RoPE on q and k)."""
    import torch
    import synth
    t = synth.make_qkvo_inputs(cfg, seed=seed, device=device)
    lin = lambda n: (t["W_" + n], t["A_" + n], t["B_" + n])  # noqa: E731
    rp = None
    if rope:
        cos, sin = lib.rope_table(cfg.seq, cfg.head_dim, 10000.0, device=device)
        rp = {"cos": cos, "sin": sin, "pos": synth.positions(cfg.M, seq=cfg.seq, device=device),
              "head_dim": cfg.head_dim}
    M, h, r = cfg.M, cfg.h, cfg.r
    w = types.SimpleNamespace(cfg=cfg, t=t)
    w.ws = torch.zeros(lib.load().lora_qkvo_workspace_bytes(M, h, cfg.n_q, cfg.n_kv, r), dtype=torch.uint8,
                       device=device)
    w.saved = torch.empty(lib.load().lora_qkvo_saved_bytes(M, h, cfg.n_q, cfg.n_kv, r), dtype=torch.uint8,
                          device=device)

    def step():
        lib.qkvo_forward(t["x"], lin("q"), lin("k"), lin("v"), t["o_in"], lin("o"), cfg.s, rope=rp,
                         saved=w.saved, ws=w.ws)
        lib.qkvo_backward(t["x"], lin("q"), lin("k"), lin("v"), t["o_in"], lin("o"), cfg.s, w.saved,
                          t["dy_q"], t["dy_k"], t["dy_v"], t["dy_o"], rope=rp, ws=w.ws)
    w.step = step
    w.flops = qkvo_kernel_flops(cfg)
    w.total_flops = cfg.flops()
    w.M = M
    return w


def measure(lib, w, steps, warmup, world, device, stream, breakdown_steps):
    """Warm-up, the per-kernel breakdown (every launch traced), the untraced timed
    region and the dominant kernel's separate traced pass.  Raises if a kernel reports
    an asynchronous error."""
    import torch
    for _ in range(warmup):
        w.step()
    torch.cuda.synchronize()
    per_kind = kernel_breakdown(lib, w.step, breakdown_steps) if breakdown_steps else {}
    secs, clk, launches = timed_region(lib, w.step, steps, world, device, stream)
    status = lib.poll_status(w.ws)
    if status != 0:
        raise RuntimeError(f"kernel status {status} after the timed region")
    m = types.SimpleNamespace(secs=secs, clk=clk, launches=launches, per_kind=per_kind,
                              ms_step=secs / steps * 1e3)
    m.tflops = w.total_flops / (m.ms_step * 1e-3) / 1e12
    if per_kind:
        m.dom = max((k for k in per_kind if k in w.flops), key=lambda k: per_kind[k][1])
        m.dom_launch_ms = kernel_launch_ms(lib, w.step, steps, m.dom)
    return m


def roofline_obj(w, m, peak, peak_key, traffic):
    """The dominant kernel against the bf16 peak: algorithmic FLOPs per launch over its
    average launch duration from the separate traced pass."""
    launches_per_step = _launches_per_step(w, m)
    dom_ms = sum(m.dom_launch_ms) / len(m.dom_launch_ms)
    flops_launch = w.flops[m.dom] / launches_per_step
    achieved = flops_launch / (dom_ms * 1e-3) / 1e12
    peaks, _ = measured_peaks()
    out = {"bound": "tensor", "kernel": m.dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
           "frac": achieved / peak, "peak_key": peak_key, "traffic": traffic, "launch_ms": dom_ms,
           "flops_per_launch": flops_launch,
           "duration_source": "average launch of a separate pass of the same number of steps, CUDA events "
                              "around this kernel's launches only"}
    if "bf16_tflops_sustained" in peaks:
        out["frac_of_sustained"] = achieved / float(peaks["bf16_tflops_sustained"])
    out["frac_of_burst"] = achieved / float(peaks["bf16_tflops"])
    return out


def _launches_per_step(w, m):
    """Launches of the dominant kind per step (w.flops counts a kind's FLOPs per step)."""
    return max(1, round(m.per_kind[m.dom][0] / max(1, m.breakdown_steps)))


OTHER_WORKLOADS = (
    ("gemma7b_r8", "mlp", "gemma7b", {}),
    ("gemma7b_r64", "mlp", "gemma7b", {"r": 64}),
    ("gqa7b", "qkvo", "gqa7b", {}),
    ("gqa7b_rope", "qkvo", "gqa7b", {"rope": True}),
    ("qwen05b_m4096", "mlp", "qwen05b", {}),
    ("qwen05b_m4095", "mlp", "qwen05b", {"M": 4095}),
)


# Warm-up work before each other workload's timed region: at least 3 steps and about
# this many TFLOP, so that a small workload (a 0.5B-shaped step is ~0.22 TFLOP) runs
# at the clocks it settles at rather than those the larger workload before it left.
OTHER_WARMUP_TFLOP = 40.0


def other_warmup_steps(total_flops: float) -> int:
    return max(3, int(math.ceil(OTHER_WARMUP_TFLOP * 1e12 / total_flops)))


def other_workloads(lib, args, world, device, stream):
    """Device-timed fwd+bwd of the other workloads (no oracle, no end-to-end copies),
    each with its own untraced timed region, under one clock record."""
    import torch
    import synth
    steps = max(10, min(args.steps, 30))
    rank = dist_env()[0]
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    out = {}
    for label, kind, name, over in OTHER_WORKLOADS:
        if kind == "mlp":
            cfg = synth.MLP_CONFIGS[name]
            if "r" in over:
                cfg = cfg.replace(r=over["r"], alpha=cfg.s * over["r"])
            if "M" in over:
                cfg = cfg.replace(M=over["M"])
            w = mlp_workload(lib, cfg, device, args.seed)
            desc = workload_name(cfg)
        else:
            cfg = synth.QKVO_CONFIGS[name]
            w = qkvo_workload(lib, cfg, device, args.seed, rope=over.get("rope", False))
            desc = qkvo_name(cfg, over.get("rope", False))
        warm = other_warmup_steps(w.total_flops)
        m = measure(lib, w, steps, warm, world, device, stream, 0)
        pf, _, _ = peak_fields(m.tflops, m.secs)
        out[label] = {"workload": desc, "ms_per_step": m.ms_step, "tokens_per_s": world * w.M / (m.ms_step * 1e-3),
                      "tflops": m.tflops, "pct_of_peak": pf["pct_of_peak"], "peak_tflops": pf["peak_tflops"],
                      "steps": steps, "warmup": warm, "gpu_launches": m.launches}
        del w
        torch.cuda.empty_cache()
    out["clocks"] = clocks.stop() if rank == 0 else None
    out["note"] = (f"each: warm-up of at least 3 steps and {OTHER_WARMUP_TFLOP:g} TFLOP (its 'warmup'), then "
                   f"{steps} untraced timed steps on device-resident inputs; pct_of_peak against the measured "
                   "bf16 peak that applies to its timed region")
    return out


def run_ours(args):
    import torch
    from rank_mlp_gb300 import binding as lib

    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init("nccl")
    lib.load()
    cfg = mlp_config(args)
    M, h = cfg.M, cfg.h
    n_ex = args.per_example
    w = mlp_workload(lib, cfg, device, args.seed, n_ex)
    stream = torch.cuda.current_stream(device)

    # ---- warm-up, per-kernel breakdown (every launch traced), then the untraced timed
    # region, then a separate pass timing the dominant kernel's launches
    nb = max(1, min(args.steps, 20))
    m = measure(lib, w, args.steps, args.warmup, world, device, stream, nb)
    m.breakdown_steps = nb
    pf, peak, peak_key = peak_fields(m.tflops, m.secs)

    # ---- end to end through host buffers: every step copies its x, dy from pinned host
    # memory and its y, dx, dA, dB back.  Double-buffered, as a training loop would:
    # the copy stream moves step k+1's inputs in and step k's results out while the
    # compute stream runs step k.
    e2e = None
    if not args.no_e2e and not n_ex:
        e2e = run_e2e(lib, w, args, world, device, stream)

    others = None
    if not args.no_other and not n_ex:
        others = other_workloads(lib, args, world, device, stream)

    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        got = {"y": w.y[:4096].cpu()}
        if not n_ex:
            got["dx"] = w.dx[:4096].cpu()
        del w.t
        torch.cuda.empty_cache()
        cpu = cpu_baseline(cfg, got=got, seed=args.seed)
    traffic = ncu_traffic(m.dom, traffic_workload_key(cfg))
    line = {
        "metric": METRIC, "value": world * M * args.steps / m.secs, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": m.ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator: x, dy ~ N(0,1), W ~ N(0,1/fan_in), A ~ U(+-1/sqrt(fan_in)), "
                "B ~ N(0,0.02))",
        "config": {"seed": args.seed,
                   "workload": workload_name(cfg) + (f", per-example adapter gradients of {n_ex} examples"
                                                      if n_ex else ""),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (weights 352 MB + activations per step)"},
        **pf,
        "roofline": roofline_obj(w, m, peak, peak_key, traffic),
        "kernels_ms_per_step": {k: v[1] / nb for k, v in sorted(m.per_kind.items())},
        "kernels_ms_per_step_note": f"every launch traced over {nb} separate steps (serialised by the events)",
        "gpu_launches": m.launches,
        "clocks": m.clk,
        "e2e": e2e,
        "other_workloads": others,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(lib, w, args, world, device, stream):
    """fwd+bwd through pinned host buffers, double-buffered; returns the e2e object."""
    import torch
    cfg, t = w.cfg, w.t
    M, h = cfg.M, cfg.h
    x, dy, y, dx, grads = t["x"], t["dy"], w.y, w.dx, w.grads
    cs = torch.cuda.Stream(device)
    xh = x.cpu().pin_memory()
    dyh = dy.cpu().pin_memory()
    xd = [torch.empty_like(x) for _ in range(2)]
    dyd = [torch.empty_like(dy) for _ in range(2)]
    yd = [torch.empty_like(y) for _ in range(2)]
    dxd = [torch.empty_like(dx) for _ in range(2)]
    gd = [{k: torch.empty_like(v) for k, v in grads.items()} for _ in range(2)]
    yh = torch.empty(M, h, dtype=torch.bfloat16).pin_memory()
    dxh = torch.empty(M, h, dtype=torch.bfloat16).pin_memory()
    gh = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in grads.items()}
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(steps):
        """steps fwd+bwd through host buffers; returns seconds (CUDA events)."""
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(cs)
        with torch.cuda.stream(cs):
            xd[0].copy_(xh, non_blocking=True)
            dyd[0].copy_(dyh, non_blocking=True)
            ev_in[0].record(cs)
        for k in range(steps):
            b = k & 1
            stream.wait_event(ev_in[b])
            if k >= 2:
                stream.wait_event(ev_out[b])              # step k-2's results have left buffers b
            lib.mlp_forward(xd[b], w.gate, w.up, w.down, cfg.s, cfg.act, y=yd[b], saved=w.saved, ws=w.ws)
            lib.mlp_backward(xd[b], w.gate, w.up, w.down, cfg.s, cfg.act, w.saved, dyd[b], dx=dxd[b],
                             grads=gd[b], ws=w.ws)
            ev_done[b].record(stream)
            with torch.cuda.stream(cs):
                if k + 1 < steps:
                    if k >= 1:
                        cs.wait_event(ev_done[1 - b])     # step k-1 finished reading buffers 1-b
                    xd[1 - b].copy_(xh, non_blocking=True)
                    dyd[1 - b].copy_(dyh, non_blocking=True)
                    ev_in[1 - b].record(cs)
                cs.wait_event(ev_done[b])
                yh.copy_(yd[b], non_blocking=True)
                dxh.copy_(dxd[b], non_blocking=True)
                for n in grads:
                    gh[n].copy_(gd[b][n], non_blocking=True)
                ev_out[b].record(cs)
        t1.record(cs)
        t1.synchronize()
        return t0.elapsed_time(t1) / 1e3

    e2e_run(3)
    ke = max(1, min(args.steps, 50))
    barrier(world, device)
    torch.cuda.synchronize()
    esecs = max_over_ranks(e2e_run(ke), world, device)
    barrier(world, device)
    h2d = 2 * M * h * 2
    d2h = 2 * M * h * 2 + sum(v.numel() * 2 for v in grads.values())
    return {"value": world * M * ke / esecs, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": ke,
            "path": "pinned host x, dy -> device; lora_mlp_forward + lora_mlp_backward; y, dx, dA, dB -> "
                    "host; copies of step k+1 / k overlap step k's compute (copy stream, double buffers)"}


def qkvo_kernel_flops(cfg):
    """Algorithmic FLOPs per step of each GEMM kind of one Q/K/V + O fwd+bwd (two
    launches per kind: the q/k/v half and the O half)."""
    M, h, r, nq, nkv = cfg.M, cfg.h, cfg.r, cfg.n_q, cfg.n_kv
    return {"proj": 2.0 * M * ((nq + 2 * nkv) * (h + r) + h * (nq + r)),
            "dgrad": 2.0 * M * (h * (nq + 2 * nkv + 3 * r) + nq * (h + r))}


def qkvo_name(cfg, rope):
    return (f"{cfg.name}-shaped LoRA Q/K/V+O fwd+bwd: M={cfg.M} tokens ({cfg.batch}x{cfg.seq}), h={cfg.h}, "
            f"{cfg.heads_q}/{cfg.heads_kv} heads x {cfg.head_dim}, r={cfg.r}, alpha={cfg.alpha:g}"
            + (", RoPE on q and k (base 10000, positions restart per sequence)" if rope else ""))


def run_qkvo(args):
    """Q/K/V + O fwd+bwd (optionally with RoPE on q and k): device-resident timing."""
    import torch
    import synth
    from rank_mlp_gb300 import binding as lib

    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init("nccl")
    lib.load()
    cfg = synth.QKVO_CONFIGS[args.workload]
    if args.rank:
        cfg = cfg.replace(r=args.rank, alpha=cfg.s * args.rank)
    if args.tokens:
        cfg = cfg.replace(M=args.tokens)
    w = qkvo_workload(lib, cfg, device, args.seed, rope=args.rope)
    stream = torch.cuda.current_stream(device)
    nb = max(1, min(args.steps, 20))
    m = measure(lib, w, args.steps, args.warmup, world, device, stream, nb)
    m.breakdown_steps = nb
    if rank != 0:
        return 0
    pf, peak, peak_key = peak_fields(m.tflops, m.secs)
    line = {
        "metric": "LoRA Q/K/V+O fwd+bwd tokens/s", "value": world * cfg.M * args.steps / m.secs,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": m.ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded generator)",
        "config": {"workload": qkvo_name(cfg, args.rope), "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2"},
        **pf,
        "roofline": roofline_obj(w, m, peak, peak_key, None),
        "kernels_ms_per_step": {k: v[1] / nb for k, v in sorted(m.per_kind.items())},
        "kernels_ms_per_step_note": f"every launch traced over {nb} separate steps (serialised by the events)",
        "gpu_launches": m.launches, "clocks": m.clk, "e2e": None, "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--act", choices=("swiglu", "geglu_tanh", "geglu_erf"), default=None,
                    help="override the workload's activation")
    ap.add_argument("--rank", type=int, default=0, metavar="R",
                    help="override the workload's adapter rank (keeping s = alpha / r)")
    ap.add_argument("--tokens", type=int, default=0, metavar="M",
                    help="override the workload's token count (small cases for profiler captures)")
    ap.add_argument("--per-example", type=int, default=0, metavar="N",
                    help="backward with per-example adapter gradients of N examples (DP-SGD)")
    ap.add_argument("--rope", action="store_true", help="Q/K/V+O workloads: RoPE on q and k")
    ap.add_argument("--seed", type=int, default=0, help="seed of the synthetic inputs")
    ap.add_argument("--list", action="store_true", help="list the workloads and exit")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other", action="store_true", help="skip the other workloads' device-timed lines")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.rank < 0:
        ap.error("--rank must be positive")
    if args.tokens < 0:
        ap.error("--tokens must be positive")
    import synth
    if args.list:
        for name, c in synth.MLP_CONFIGS.items():
            print(f"{name:10s} LoRA-MLP fwd+bwd  M={c.M} h={c.h} i={c.i} r={c.r} alpha={c.alpha:g} {c.act}")
        for name, c in synth.QKVO_CONFIGS.items():
            print(f"{name:10s} LoRA Q/K/V+O fwd+bwd  M={c.M} h={c.h} heads {c.heads_q}/{c.heads_kv} x "
                  f"{c.head_dim} r={c.r} alpha={c.alpha:g}  (--rope: RoPE on q and k)")
        return 0
    if args.workload not in synth.MLP_CONFIGS and args.workload not in synth.QKVO_CONFIGS:
        ap.error(f"unknown workload {args.workload}")
    if args.impl == "reference":
        if args.workload not in synth.MLP_CONFIGS:
            ap.error("the reference arm times the MLP workloads")
        return run_reference(args)
    if args.workload in synth.QKVO_CONFIGS:
        return run_qkvo(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
