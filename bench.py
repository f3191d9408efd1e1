#!/usr/bin/env python3
"""Benchmark: fused RoPE + causal attention forward on GB300 (TFLOP/s, % of bf16 peak).

Default workload (one step = one pass of the forward hot path: the RoPE (cos, sin) table and
the fused forward kernel, through the C ABI): Llama-3-8B-shaped RoPE+causal forward,
B=4, Hq=32, Hkv=8, N=4096, d=128, rope_theta=5e5, fused RoPE, O and LSE, synthetic N(0,1)
bf16 inputs. Algorithmic work counts only the allowed (m, n) pairs: 4 d B Hq N(N+1)/2 FLOP.

Prints ONE JSON line (rank 0). Multi-GPU: one rank per GPU (torchrun), each rank runs the same
workload on its own GPU (weak scaling, no data-path collective); the time is the max over
ranks. ``--impl reference`` times the fp64 CPU oracle on a bounded sample instead.
Other measurements (``--workload``, ``--sweep``) print extra lines for the design notes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused RoPE+causal attn fwd TFLOP/s (bf16) and % of GB300 dense BF16 peak"
WORKLOADS = {
    # name: (B, Hq, Hkv, N, d, theta, rope_mode_name, mask)
    "llama8b_fused": (4, 32, 8, 4096, 128, 5e5, "fused", "causal"),
    "llama8b_prerotate": (4, 32, 8, 4096, 128, 5e5, "prerotate", "causal"),
    "llama8b_none": (4, 32, 8, 4096, 128, 5e5, "none", "causal"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b_fused", choices=sorted(WORKLOADS))
    ap.add_argument("--sweep", action="store_true", help="fused vs pre-rotated N sweep")
    ap.add_argument("--train", action="store_true",
                    help="forward + backward at B=8 Hq=32 Hkv=8 d=128, N=2048 and 4096")
    ap.add_argument("--variants", action="store_true",
                    help="mask-variant forwards and backwards at B=2 H=16 N=4096 d=64 (window, ALiBi, BigBird)")
    ap.add_argument("--tables", action="store_true",
                    help="the paper's GPT-2-small forwards and Llama-3-8B / Mistral-7B decodes")
    ap.add_argument("--decode", action="store_true",
                    help="split-KV decode at the Llama-3-70B head shape (B=1, 8; splits sweep)")
    ap.add_argument("--fp8", action="store_true",
                    help="e4m3 forward at the Llama-3-8B shape (causal, no RoPE) vs the bf16 one")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the nested records of the other workloads and the steady-state run")
    ap.add_argument("--profile", action="store_true",
                    help="one warm-up call and one call of the workload, then exit (for ncu)")
    ap.add_argument("--profile-target", default="fwd",
                    choices=["fwd", "decode", "decode-b1", "train", "train-prerotate", "d64-causal",
                             "fp8"],
                    help="--profile: forward workload, Llama-3-70B decode (B=8), fwd+bwd (N=2048) "
                         "or the head-dim-64 causal forward (B=2, H=16, N=4096, fused RoPE)")
    return ap.parse_args()


def causal_flops(B, Hq, N, d):
    return 4.0 * d * B * Hq * N * (N + 1) / 2.0


def max_over_ranks(value, device=None):
    """Max of a per-rank float over all ranks (identity without a process group)."""
    import torch

    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# ncu traffic figure committed under profiles/ (null when the kernel source changed since)
# ------------------------------------------------------------------------------------------
def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_attn_fwd_bwd_gb300", "csrc")
    for name in ("fwd_pp.cuh", "fwd_pp.cu", "ptx.cuh", "common.cuh", "launch.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload):
    path = os.path.join(ROOT, "profiles", f"fwd_kernel_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


# ------------------------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------
class OracleSampler:
    """The fp64 oracle as it stands, timed on sampled full query rows of the workload."""

    def __init__(self, B, Hq, Hkv, N, d, theta, rope_on, seed):
        import oracle
        from attention_attn_fwd_bwd_gb300 import inputs

        oracle.build()
        self.oracle, self.inputs = oracle, inputs
        x = inputs.prefill(B, Hq, Hkv, N, d, seed)
        self.q, self.k, self.v = (x[n].double().numpy() for n in ("q", "k", "v"))
        self.shape = (B, Hq, N, d)
        self.theta, self.rope_on = theta, rope_on
        self.var = oracle.Variant(mask=1)

    def run(self, nrows, seed):
        """One batch of nrows sampled rows: (flops, seconds)."""
        B, Hq, N, d = self.shape
        rows = self.inputs.sample_rows(B, Hq, N, nrows, seed=seed)
        t0 = time.perf_counter()
        self.oracle.forward_rows(self.q, self.k, self.v, d ** -0.5, self.theta, self.rope_on,
                                 self.var, rows)
        secs = time.perf_counter() - t0
        return sum(4.0 * d * (int(m) + 1) for _, _, m in rows), secs

    def timed(self, budget_s, batch):
        flops, secs, rows, it = 0.0, 0.0, 0, 0
        while secs < budget_s or rows == 0:
            f, s = self.run(batch, seed=7000 + it)
            flops, secs, rows, it = flops + f, secs + s, rows + batch, it + 1
        return flops / secs / 1e12, rows, secs


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def steady_state(step, stream, local, flops, ms_per_step):
    """The headline step repeated for at least ~1.2 s (clocks sampled throughout): a steadier
    number than the driver's short timed region, reported beside it."""
    import torch

    n = max(1000, int(1.2e3 / max(ms_per_step, 1e-3)))
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    return {"steps": n, "ms_per_step": ms, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "clocks": clocks.stop()}


def secondary_configs(args, local):
    """The other workloads of the target, each with its own clock record: the mask variants
    (B=2, H=16, N=4096, d=64: window 1024 + causal, ALiBi + causal, BigBird, causal), the
    training step (B=8, Hq=32, Hkv=8, d=128, N=2048 and 4096: forward, backward fused and
    pre-rotated), the Llama-3-70B-shaped split-KV decode (B=1 and 8, splits auto/1/8/32/128,
    cold and warm L2), the e4m3 forward at the Llama-3-8B shape and the fused / pre-rotated
    crossover sweep of the head-dim-128 forward (B*N = 16384, N = 256 .. 16384)."""
    out = {}
    for key, fn in (("mask_variants_d64", lambda: run_variants_bench(args, emit=False)),
                    ("training_fwd_bwd", lambda: run_train_bench(args, emit=False)),
                    ("decode_llama70b_head_shape", lambda: run_decode_bench(args, emit=False)),
                    ("fp8_e4m3_forward_d128", lambda: run_fp8_bench(args, emit=False)),
                    ("rotation_calculus_d128", lambda: run_sweep(args, quick=True, emit=False))):
        clk = ClockSampler(local)
        clk.start()
        time.sleep(0.2)
        t0 = time.perf_counter()
        rows = fn()
        out[key] = {"rows": rows, "clocks": clk.stop(), "wall_s": round(time.perf_counter() - t0, 1)}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    B, Hq, Hkv, N, d, theta, mode, _ = WORKLOADS[args.workload]
    smp = OracleSampler(B, Hq, Hkv, N, d, theta, mode != "none", seed=2000)
    batch = os.cpu_count() or 8
    per_step = []
    for i in range(args.warmup + args.steps):
        f, secs = smp.run(batch, seed=5000 + i)
        if i >= args.warmup:
            per_step.append((f, secs))
    tflops = sum(f for f, _ in per_step) / sum(t for _, t in per_step) / 1e12
    ms = 1e3 * sum(t for _, t in per_step) / len(per_step)
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(args.workload),
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": f"{batch} full query rows of the workload per step (fp64 "
                                   f"oracle, rows drawn uniformly over (b, h, m))"},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(name):
    B, Hq, Hkv, N, d, theta, mode, mask = WORKLOADS[name]
    return {"workload": f"Llama-3-8B-shaped RoPE+{mask} forward, {mode} RoPE "
                        f"(B={B}, Hq={Hq}, Hkv={Hkv}, N={N}, d={d})",
            "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "rope_theta": theta, "rope_mode": mode,
            "mask": mask, "outputs": "O bf16, LSE fp32",
            "l2": "inputs rotated over 3 resident sets (3 x 322 MiB > 126 MiB L2)"}


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------
def run_ours(args, rank, world):
    import torch

    import attention_attn_fwd_bwd_gb300 as af
    from attention_attn_fwd_bwd_gb300 import inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, Hq, Hkv, N, d, theta, mode, _ = WORKLOADS[args.workload]
    rope_mode = {"fused": af.ROPE_FUSED, "prerotate": af.ROPE_PREROTATE, "none": af.ROPE_NONE}[mode]
    scale = d ** -0.5
    flops = causal_flops(B, Hq, N, d)
    nsets = 3
    sets = []
    for i in range(nsets):
        x = inputs.prefill(B, Hq, Hkv, N, d, seed=2000 + i)
        sets.append({n: x[n].to(dev) for n in ("q", "k", "v")})
        sets[-1]["out"] = torch.empty_like(sets[-1]["q"])
        sets[-1]["lse"] = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    ws_n = af.fwd_workspace_size(B, Hq, Hkv, N, d, rope_mode)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    var = af.Variant(mask=af.MASK_CAUSAL)
    stream = torch.cuda.current_stream()

    def step(i, flags=0):
        s = sets[i % nsets]
        af.fwd(s["q"], s["k"], s["v"], scale=scale, rope_theta=theta, rope_mode=rope_mode | flags,
               variant=var, out=s["out"], lse=s["lse"], workspace=ws)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for i in range(max(3, args.warmup)):
        step(i)
    barrier()
    assert af.device_status() == 0

    # ---- timed region: K full steps (table + forward kernel) ----
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), dev)
    ms_per_step = elapsed_ms / args.steps
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    assert af.device_status() == 0

    # ---- the forward kernel alone (table reused): per-launch duration for the roofline ----
    # table + K rotation pass + forward (fused, head dim 128); table + forward (others)
    launches_per_step = (1 + (1 if rope_mode != af.ROPE_NONE else 0)
                         + (2 if rope_mode == af.ROPE_PREROTATE else 0)
                         + (1 if rope_mode == af.ROPE_FUSED and d == 128 else 0))
    kern_steps = min(args.steps, 200)
    barrier()
    ev0.record(stream)
    for i in range(kern_steps):
        step(i, af.ROPE_REUSE_TABLE if rope_mode == af.ROPE_FUSED else 0)
    ev1.record(stream)
    barrier()
    kern_ms = ev0.elapsed_time(ev1) / kern_steps
    kern_method = "CUDA events around the call with the table reused"
    if rope_mode == af.ROPE_FUSED and d == 128:
        kern_method += (" (the call's one-pass K rotation, ~17 us of 64 MB of K traffic, is "
                        "included: a conservative figure for the forward kernel)")
    if rope_mode == af.ROPE_PREROTATE:
        kern_ms = None  # pre-rotation launches three kernels per call; see the sweep lines

    # ---- end to end: host buffers, H2D + call + D2H inside the timed region ----
    e2e = None
    if rank == 0 or world > 1:
        pin = {n: sets[0][n].cpu().pin_memory() for n in ("q", "k", "v")}
        out_h = torch.empty(sets[0]["out"].shape, dtype=torch.bfloat16).pin_memory()
        lse_h = torch.empty(sets[0]["lse"].shape, dtype=torch.float32).pin_memory()
        e2e_steps = max(3, min(args.steps, 20))
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = out_h.numel() * 2 + lse_h.numel() * 4
        # attnfuse_fwd_host: copy-in, forward and copy-out pipelined over batch chunks
        chunk_b = 1
        ws_h = torch.empty(af.fwd_host_workspace_size(B, Hq, Hkv, N, d, rope_mode, chunk_b),
                           dtype=torch.uint8, device=dev)

        def e2e_step():
            af.fwd_host(pin["q"], pin["k"], pin["v"], scale=scale, rope_theta=theta,
                        rope_mode=rope_mode, variant=var, out=out_h, lse=lse_h, chunk_b=chunk_b,
                        workspace=ws_h, sync=False)

        e2e_step()
        barrier()
        ev0.record(stream)
        for i in range(e2e_steps):
            e2e_step()
        ev1.record(stream)
        barrier()
        e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / e2e_steps, dev)
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "api": f"attnfuse_fwd_host (pinned host buffers, chunk_b={chunk_b}: chunks of one "
                      f"batch element split into KV-head groups until there are 8; copy-in, "
                      f"forward and copy-out overlap)"}

    if rank != 0:
        return
    steady = configs = None
    if world == 1 and not args.no_configs:
        steady = steady_state(step, stream, local, flops, ms_per_step)
        configs = secondary_configs(args, local)
    peaks, src = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    roof = None
    if kern_ms is not None:
        ach = flops / (kern_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": committed_traffic(args.workload),
                "kernel": "fwd_pp_kernel<fused RoPE, no bias, softmax> (persistent 2-CTA clusters)", "kernel_ms": kern_ms,
                "kernel_ms_method": kern_method,
                "peak_source": f"{src} bf16 burst (MEASURED_PEAKS.json)" if src == "measured" else "fallback",
                "frac_of_sustained": ach / float(peaks.get("bf16_tflops_sustained", peak))}
    cpu = None
    if not args.no_cpu_baseline:
        smp = OracleSampler(B, Hq, Hkv, N, d, theta, mode != "none", seed=2000)
        tf, rows, secs = smp.timed(budget_s=12.0, batch=os.cpu_count() or 8)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": os.cpu_count(), "cpu_model": cpu_model(),
               "kind": "oracle",
               "sample": f"{rows} full query rows of the workload (fp64 oracle, {secs:.1f} s), "
                         f"rows drawn uniformly over (b, h, m); value = their causal FLOPs / time"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(args.workload),
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps, "clocks": clk,
        "steady_state": steady, "configs": configs,
    }
    print(json.dumps(line), flush=True)


def _median_ms(fn, reps=30, warm=5):
    import torch

    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    samples = []
    for _ in range(reps):
        evs[0].record()
        fn()
        evs[1].record()
        torch.cuda.synchronize()
        samples.append(evs[0].elapsed_time(evs[1]))
    return statistics.median(samples)


def _crossover(res, key):
    """N where res[key] (t_prerotate / t_fused) crosses 1, log-linear in N; None if it does not."""
    for a, b in zip(res, res[1:]):
        ra, rb = a[key] - 1, b[key] - 1
        if ra >= 0 > rb or ra <= 0 < rb:
            t = ra / (ra - rb)
            return math.exp(math.log(a["N"]) + t * (math.log(b["N"]) - math.log(a["N"])))
    return None


def run_sweep(args, quick=False, emit=True):
    """The Rotation Calculus on GB300: fused vs pre-rotated vs no RoPE over N at B*N = 16384
    tokens, forward for head dims 128 (Hq=32, Hkv=8) and 64 (H=16), and the d=128 backward.
    quick: the head-dim-128 forward only (the default run's nested record). Returns the rows
    and the crossover records."""
    import torch

    import attention_attn_fwd_bwd_gb300 as af
    from attention_attn_fwd_bwd_gb300 import inputs

    dev = torch.device("cuda")
    theta = 5e5
    rows_all = []
    for d, Hq, Hkv in ((128, 32, 8),) if quick else ((128, 32, 8), (64, 16, 16)):
        res = []
        for N in (256, 512, 1024, 2048, 4096, 8192, 16384):
            B = 16384 // N
            x = inputs.prefill(B, Hq, Hkv, N, d, seed=N, with_dout=(N <= 4096 and not quick))
            q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
            out = torch.empty_like(q)
            lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
            times = {}
            for name, mode in (("fused", af.ROPE_FUSED), ("prerotate", af.ROPE_PREROTATE),
                               ("none", af.ROPE_NONE)):
                ws = torch.empty(max(16, af.fwd_workspace_size(B, Hq, Hkv, N, d, mode)),
                                 dtype=torch.uint8, device=dev)
                times[name] = _median_ms(lambda: af.fwd(q, k, v, rope_theta=theta, rope_mode=mode,
                                                        out=out, lse=lse, workspace=ws))
            fl = causal_flops(B, Hq, N, d)
            row = {"d": d, "N": N, "B": B, **{f"{k}_ms": v for k, v in times.items()},
                   "fused_over_prerotate": times["prerotate"] / times["fused"],
                   "fused_tflops": fl / times["fused"] / 1e9,
                   "none_tflops": fl / times["none"] / 1e9}
            if "dout" in x:
                do = x["dout"].to(dev)
                dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                bt = {}
                for name, mode in (("fused", af.ROPE_FUSED), ("prerotate", af.ROPE_PREROTATE)):
                    af.fwd(q, k, v, rope_theta=theta, rope_mode=mode, out=out, lse=lse)
                    ws = torch.empty(af.bwd_workspace_size(B, Hq, Hkv, N, d, mode), dtype=torch.uint8, device=dev)
                    bt[name] = _median_ms(lambda: af.bwd(q, k, v, out, lse, do, rope_theta=theta, rope_mode=mode,
                                                         dq=dq, dk=dk, dv=dv, workspace=ws), reps=15)
                row.update({"bwd_fused_ms": bt["fused"], "bwd_prerotate_ms": bt["prerotate"],
                            "bwd_fused_over_prerotate": bt["prerotate"] / bt["fused"]})
            res.append(row)
            if emit:
                print(json.dumps({"sweep": "rotation_calculus", **row}), flush=True)
        bwd_rows = [r for r in res if "bwd_fused_over_prerotate" in r]
        cross = {"sweep": "rotation_calculus_crossover", "d": d,
                 "N_star_fwd": _crossover(res, "fused_over_prerotate"),
                 "N_star_bwd": _crossover(bwd_rows, "bwd_fused_over_prerotate") if bwd_rows else None,
                 "note": "speedup = t_prerotate / t_fused; >1 means fusion wins; "
                         "None: no crossing inside the measured N"}
        if emit:
            print(json.dumps(cross), flush=True)
        rows_all += res + [cross]
    return rows_all


def run_profile(args):
    """Warm-up call plus one call of a workload: a small, self-contained ncu target."""
    import torch

    import attention_attn_fwd_bwd_gb300 as af
    from attention_attn_fwd_bwd_gb300 import inputs

    if args.profile_target in ("decode", "decode-b1"):
        x = inputs.decode(8 if args.profile_target == "decode" else 1, 64, 8, 32768, 128, seed=5008)
        q, kc, vc = (x[n].cuda() for n in ("q", "k_cache", "v_cache"))
        for _ in range(2):
            af.decode(q, kc, vc, 32767, rope_theta=5e5)
    elif args.profile_target in ("train", "train-prerotate"):
        x = inputs.prefill(8, 32, 8, 2048, 128, seed=6048, with_dout=True)
        q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
        mode = af.ROPE_PREROTATE if args.profile_target == "train-prerotate" else af.ROPE_FUSED
        for _ in range(2):
            out, lse = af.fwd(q, k, v, rope_theta=5e5)
            af.bwd(q, k, v, out, lse, do, rope_theta=5e5, rope_mode=mode)
    elif args.profile_target == "fp8":
        x = inputs.prefill_e4m3(4, 32, 8, 4096, 128, seed=8000)
        q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
        for _ in range(2):
            af.fwd_fp8(q, k, v, x["q_scale"], x["k_scale"], x["v_scale"])
    elif args.profile_target == "d64-causal":
        x = inputs.prefill(2, 16, 16, 4096, 64, seed=3000)
        q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
        for _ in range(2):
            af.fwd(q, k, v, rope_theta=1e4, rope_mode=af.ROPE_FUSED,
                   variant=af.Variant(mask=af.MASK_CAUSAL))
    else:
        B, Hq, Hkv, N, d, theta, mode, _ = WORKLOADS[args.workload]
        rope_mode = {"fused": af.ROPE_FUSED, "prerotate": af.ROPE_PREROTATE, "none": af.ROPE_NONE}[mode]
        x = inputs.prefill(B, Hq, Hkv, N, d, seed=2000)
        q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
        for _ in range(2):
            af.fwd(q, k, v, rope_theta=theta, rope_mode=rope_mode)
    torch.cuda.synchronize()
    if af.device_status() != 0:
        raise SystemExit("device status reports a timeout")
    print(json.dumps({"profile": args.profile_target, "ok": True}))


def _time_ms(fn, reps=20, warm=3):
    """Median, min and p90 of fn() in ms (CUDA events on the current stream)."""
    import torch

    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    samples = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        samples.append(e0.elapsed_time(e1))
    samples.sort()
    return samples[len(samples) // 2], samples[0], samples[int(0.9 * len(samples))]


def run_train_bench(args, emit=True):
    """Training-step attention: fused-RoPE causal forward (O, LSE) and the 3-kernel backward."""
    import torch

    import attention_attn_fwd_bwd_gb300 as af
    from attention_attn_fwd_bwd_gb300 import inputs

    dev = torch.device("cuda")
    peaks, _ = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    B, Hq, Hkv, d, theta = 8, 32, 8, 128, 5e5
    rows = []
    for N in (2048, 4096):
        x = inputs.prefill(B, Hq, Hkv, N, d, seed=4000 + N, with_dout=True)
        q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
        out = torch.empty_like(q)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsf = torch.empty(af.fwd_workspace_size(B, Hq, Hkv, N, d, af.ROPE_FUSED), dtype=torch.uint8, device=dev)
        wsb = torch.empty(af.bwd_workspace_size(B, Hq, Hkv, N, d, af.ROPE_PREROTATE), dtype=torch.uint8, device=dev)
        fwd = lambda: af.fwd(q, k, v, rope_theta=theta, out=out, lse=lse, workspace=wsf)
        bwd = lambda: af.bwd(q, k, v, out, lse, do, rope_theta=theta, dq=dq, dk=dk, dv=dv, workspace=wsb)
        bwd_pre = lambda: af.bwd(q, k, v, out, lse, do, rope_theta=theta, rope_mode=af.ROPE_PREROTATE,
                                 dq=dq, dk=dk, dv=dv, workspace=wsb)
        tf, tf_min, tf_p90 = _time_ms(fwd)
        tb, tb_min, tb_p90 = _time_ms(bwd)
        tbp, _, _ = _time_ms(bwd_pre)
        fl = causal_flops(B, Hq, N, d)
        rows.append({"train": "fused_rope_causal", "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d,
                          "fwd_ms": tf, "bwd_ms": tb, "fwd_tflops": fl / tf / 1e9,
                          "bwd_tflops": 2.5 * fl / tb / 1e9,
                          "total_tflops": 3.5 * fl / (tf + tb) / 1e9,
                          "bwd_frac_of_peak": 2.5 * fl / tb / 1e9 / peak,
                          "total_frac_of_peak": 3.5 * fl / (tf + tb) / 1e9 / peak,
                          "fwd_min_p90_ms": [tf_min, tf_p90], "bwd_min_p90_ms": [tb_min, tb_p90],
                          "bwd_prerotate_ms": tbp, "bwd_prerotate_tflops": 2.5 * fl / tbp / 1e9,
                          "launches": {"fwd": 2, "bwd": 4, "bwd_prerotate": 6}})
        if emit:
            print(json.dumps(rows[-1]), flush=True)
    return rows


def allowed_pairs(N, mask, causal=False, window=0, row_ptr=None, col_idx=None, blk=64):
    """Allowed (m, n) pairs of one head, counted from the mask definitions (the algorithmic
    work of a masked forward): mask "full", "causal", "window" (|m - n| < W, n <= m if causal)
    or "block_sparse" (CSR of active blocks, n <= m if causal)."""
    import numpy as np

    m = np.arange(N, dtype=np.int64)
    if mask == "full":
        return N * N
    if mask == "causal":
        return int((m + 1).sum())
    if mask == "window":
        lo = np.maximum(0, m - window + 1)
        hi = m if causal else np.minimum(N - 1, m + window - 1)
        return int((hi - lo + 1).sum())
    total = 0
    nb = -(-N // blk)
    for br in range(nb):
        r0, r1 = br * blk, min(N, (br + 1) * blk)
        for bc in col_idx[row_ptr[br]:row_ptr[br + 1]]:
            c0, c1 = int(bc) * blk, min(N, (int(bc) + 1) * blk)
            if causal:
                rows = np.arange(r0, r1)
                total += int(np.clip(np.minimum(rows, c1 - 1) - c0 + 1, 0, None).sum())
            else:
                total += (r1 - r0) * (c1 - c0)
    return total


def run_variants_bench(args, emit=True):
    """Mask-variant forwards at B=2, H=16, N=4096, d=64, theta=1e4, fused RoPE."""
    import torch

    import attention_attn_fwd_bwd_gb300 as af
    from attention_attn_fwd_bwd_gb300 import inputs

    dev = torch.device("cuda")
    peaks, _ = measured_peaks()
    B, H, N, d = 2, 16, 4096, 64
    x = inputs.prefill(B, H, H, N, d, seed=3000)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    rp, ci = inputs.bigbird_csr(N // 64, seed=3003)
    cases = {
        "window1024_causal": (af.Variant(mask=af.MASK_WINDOW, window=1024, causal=True),
                              allowed_pairs(N, "window", causal=True, window=1024)),
        "alibi_causal": (af.Variant(mask=af.MASK_CAUSAL, bias=af.BIAS_ALIBI,
                                    alibi_slopes=torch.tensor(inputs.alibi_slopes(H), dtype=torch.float32, device=dev)),
                         allowed_pairs(N, "causal")),
        "bigbird_blocksparse": (af.Variant(mask=af.MASK_BLOCK_SPARSE, bs_block=64,
                                           bs_row_ptr=torch.tensor(rp, device=dev),
                                           bs_col_idx=torch.tensor(ci, device=dev)),
                                allowed_pairs(N, "block_sparse", row_ptr=rp, col_idx=ci)),
        "causal": (af.Variant(mask=af.MASK_CAUSAL), allowed_pairs(N, "causal")),
    }
    do = inputs.prefill(B, H, H, N, d, seed=3000, with_dout=True)["dout"].to(dev)
    rows = []
    for name, (gvar, pairs) in cases.items():
        ws = torch.empty(af.fwd_workspace_size(B, H, H, N, d, af.ROPE_FUSED), dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        t, tmin, tp90 = _time_ms(lambda: af.fwd(q, k, v, rope_theta=1e4, variant=gvar, out=out, lse=lse, workspace=ws))
        # backward of the same variant (paper §4.3: only active tiles), 2.5x the forward's FLOPs
        wsb = torch.empty(af.bwd_workspace_size(B, H, H, N, d, af.ROPE_FUSED), dtype=torch.uint8, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        tb, _, _ = _time_ms(lambda: af.bwd(q, k, v, out, lse, do, rope_theta=1e4, variant=gvar,
                                           dq=dq, dk=dk, dv=dv, workspace=wsb))
        fl = 4.0 * d * B * H * pairs
        rows.append({"variant": name, "B": B, "H": H, "N": N, "d": d, "ms": t, "min_ms": tmin,
                          "p90_ms": tp90, "allowed_pairs_per_head": pairs,
                          "algorithmic_tflops": fl / t / 1e9,
                          "frac_of_peak": fl / t / 1e9 / float(peaks["bf16_tflops"]),
                          "bwd_ms": tb, "bwd_algorithmic_tflops": 2.5 * fl / tb / 1e9,
                          **({"active_blocks": int(len(ci)), "active_fraction": len(ci) / (N // 64) ** 2}
                             if name.startswith("bigbird") else {})})
        if emit:
            print(json.dumps(rows[-1]), flush=True)
    return rows


def run_fp8_bench(args, emit=True):
    """e4m3 forward (per-tensor scales, no RoPE, causal) at B=4, Hq=32, Hkv=8, N=4096, d=128,
    beside the bf16 forward without RoPE on the same values; three input sets rotate so no call
    finds its operands in L2 from the call before. The fp8 peak is the measured bf16 GEMM peak
    times the nominal fp8/bf16 ratio (2); only the score half of the FLOPs runs at the fp8
    rate (P V is a bf16 MMA), so the mixed peak, 1 / (0.5 / fp8 + 0.5 / bf16), is reported
    too."""
    import torch

    import attention_attn_fwd_bwd_gb300 as af
    from attention_attn_fwd_bwd_gb300 import inputs

    dev = torch.device("cuda")
    peaks, _ = measured_peaks()
    bf16_peak = float(peaks["bf16_tflops"])
    fp8_peak = 2.0 * bf16_peak
    mixed_peak = 1.0 / (0.5 / fp8_peak + 0.5 / bf16_peak)
    B, Hq, Hkv, N, d = 4, 32, 8, 4096, 128
    sets = []
    for i in range(3):
        x = inputs.prefill_e4m3(B, Hq, Hkv, N, d, seed=8000 + i)
        sets.append(((x["q"].to(dev), x["k"].to(dev), x["v"].to(dev)),
                     (x["q_scale"], x["k_scale"], x["v_scale"])))
    ws = torch.empty(af.fwd_fp8_workspace_size(B, Hq, Hkv, N, d), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    it = [0]

    def call_fp8():
        (q, k, v), sc = sets[it[0] % 3]
        it[0] += 1
        af.fwd_fp8(q, k, v, *sc, out=out, lse=lse, workspace=ws)

    t, tmin, tp90 = _time_ms(call_fp8, reps=60, warm=5)
    # the bf16 forward (no RoPE) on bf16 copies of the same decoded values
    bsets = []
    for (q, k, v), (sq, sk, sv) in sets:
        bsets.append(tuple((t8.view(torch.float8_e4m3fn).float() * s).to(torch.bfloat16)
                           for t8, s in ((q, sq), (k, sk), (v, sv))))

    def call_bf16():
        q, k, v = bsets[it[0] % 3]
        it[0] += 1
        af.fwd(q, k, v, rope_mode=af.ROPE_NONE, out=out, lse=lse)

    tb, _, _ = _time_ms(call_bf16, reps=60, warm=5)
    fl = causal_flops(B, Hq, N, d)
    row = {"workload": "e4m3 forward, causal, no RoPE (B=4, Hq=32, Hkv=8, N=4096, d=128)",
           "ms": t, "min_ms": tmin, "p90_ms": tp90, "tflops": fl / t / 1e9,
           "fp8_peak_tflops": fp8_peak, "frac_of_fp8_peak": fl / t / 1e9 / fp8_peak,
           "mixed_peak_tflops": mixed_peak, "frac_of_mixed_peak": fl / t / 1e9 / mixed_peak,
           "bf16_none_ms": tb, "bf16_none_tflops": fl / tb / 1e9,
           "peak_source": "measured bf16 burst (MEASURED_PEAKS.json) x nominal fp8/bf16 ratio 2"}
    if emit:
        print(json.dumps(row), flush=True)
    return [row]


def _graph_of(fn):
    """Capture fn() (library calls on the current stream, buffers preallocated) in a CUDA
    graph, so small problems are timed without host-side launch latency."""
    import torch

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def run_tables_bench(args):
    """The paper's other workloads (§6.1-§6.3) on GB300, each one JSON line:
    GPT-2-small geometry forwards (B=4, H=12, d=64; N = 512..4096): dense, causal, causal
    sliding window 256, causal + ALiBi, and RoPE (fused, theta 1e4) + dense / causal /
    sliding window; decode at the Llama-3-8B (L=4096) and Mistral-7B (L=16384) head shapes
    (Hq=32, Hkv=8, d=128), B=1 and 8, q at L-1, cold L2."""
    import torch

    import attention_attn_fwd_bwd_gb300 as af
    from attention_attn_fwd_bwd_gb300 import inputs

    dev = torch.device("cuda")
    peaks, _ = measured_peaks()
    B, H, d = 4, 12, 64
    slopes = torch.tensor(inputs.alibi_slopes(H), dtype=torch.float32, device=dev)
    cells = [("dense", af.ROPE_NONE, dict(mask=af.MASK_FULL), ("full",)),
             ("causal", af.ROPE_NONE, dict(mask=af.MASK_CAUSAL), ("causal",)),
             ("sw256", af.ROPE_NONE, dict(mask=af.MASK_WINDOW, window=256, causal=True), ("window", True, 256)),
             ("causal_alibi", af.ROPE_NONE, dict(mask=af.MASK_CAUSAL, bias=af.BIAS_ALIBI, alibi_slopes=slopes), ("causal",)),
             ("rope_dense", af.ROPE_FUSED, dict(mask=af.MASK_FULL), ("full",)),
             ("rope_causal", af.ROPE_FUSED, dict(mask=af.MASK_CAUSAL), ("causal",)),
             ("rope_sw256", af.ROPE_FUSED, dict(mask=af.MASK_WINDOW, window=256, causal=True), ("window", True, 256))]
    for N in (512, 1024, 2048, 4096):
        x = inputs.prefill(B, H, H, N, d, seed=6000 + N)
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        out = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        for name, mode, vkw, pk in cells:
            var = af.Variant(**vkw)
            ws = torch.empty(max(16, af.fwd_workspace_size(B, H, H, N, d, mode)), dtype=torch.uint8, device=dev)
            call = lambda: af.fwd(q, k, v, rope_theta=1e4, rope_mode=mode, variant=var,
                                  out=out, lse=lse, workspace=ws)
            t, tmin, tp90 = _time_ms(call)
            g = _graph_of(call)
            tg, _, _ = _time_ms(g.replay)
            pairs = allowed_pairs(N, pk[0], causal=pk[1] if len(pk) > 1 else False,
                                  window=pk[2] if len(pk) > 2 else 0)
            fl = 4.0 * d * B * H * pairs
            print(json.dumps({"table": "gpt2_small_forward", "variant": name, "B": B, "H": H, "N": N, "d": d,
                              "ms": t, "min_ms": tmin, "p90_ms": tp90, "algorithmic_tflops": fl / t / 1e9,
                              "frac_of_peak": fl / t / 1e9 / float(peaks["bf16_tflops"]),
                              "ms_graph": tg, "algorithmic_tflops_graph": fl / tg / 1e9}), flush=True)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)  # 4x the L2
    Hq, Hkv, d = 32, 8, 128
    for geom, L in (("llama3_8b", 4096), ("mistral_7b", 16384)):
        for Bd in (1, 8):
            x = inputs.decode(Bd, Hq, Hkv, L, d, seed=7000 + L + Bd)
            q, kc, vc = (x[n].to(dev) for n in ("q", "k_cache", "v_cache"))
            out = torch.empty_like(q)
            lse = torch.empty((Bd, Hq), dtype=torch.float32, device=dev)
            ws = torch.empty(af.decode_workspace_size(Bd, Hq, Hkv, L, d, 0), dtype=torch.uint8, device=dev)
            call = lambda: af.decode(q, kc, vc, L - 1, rope_theta=5e5, out=out, lse=lse, workspace=ws)
            for _ in range(3):
                call()
            g = _graph_of(call)
            meds = []
            for fn in (call, g.replay):
                samples = []
                for _ in range(30):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    fn()
                    e1.record()
                    torch.cuda.synchronize()
                    samples.append(e0.elapsed_time(e1) * 1e3)
                samples.sort()
                meds.append(samples)
            samples = meds[0]
            med, medg = samples[len(samples) // 2], meds[1][len(meds[1]) // 2]
            nbytes = 2 * Bd * Hkv * L * d * 2
            print(json.dumps({"table": "decode", "geometry": geom, "B": Bd, "Hq": Hq, "Hkv": Hkv, "d": d,
                              "L": L, "splits_used": af.decode_auto_splits(Bd, Hkv, L),
                              "us_median_cold_l2": med, "us_min_cold_l2": samples[0],
                              "gbs_cold": nbytes / (med * 1e-6) / 1e9,
                              "frac_of_hbm": nbytes / (med * 1e-6) / 1e9 / float(peaks["hbm_gbs"]),
                              "us_graph_cold_l2": medg,
                              "frac_of_hbm_graph": nbytes / (medg * 1e-6) / 1e9 / float(peaks["hbm_gbs"])}), flush=True)


def run_decode_bench(args, emit=True):
    """Split-KV decode: Hq=64, Hkv=8, d=128, L=32768, q at 32767; K+V bytes / time (cold L2)."""
    import torch

    import attention_attn_fwd_bwd_gb300 as af
    from attention_attn_fwd_bwd_gb300 import inputs

    dev = torch.device("cuda")
    peaks, src = measured_peaks()
    Hq, Hkv, d, L = 64, 8, 128, 32768
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)  # 4x the L2
    # A write flush leaves up to a full L2 of dirty lines, written back to HBM while the timed
    # call reads: 126 MiB of write-back next to the 134 MB a B=1 decode reads. Reading another
    # buffer of 3x the L2 after the write leaves L2 clean (and still without the cache's lines).
    evict = torch.zeros(384 * 1024 * 1024, dtype=torch.uint8, device=dev)
    rows = []
    for B in (1, 8):
        x = inputs.decode(B, Hq, Hkv, L, d, seed=5000 + B)
        q, kc, vc = (x[n].to(dev) for n in ("q", "k_cache", "v_cache"))
        out = torch.empty_like(q)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        nbytes = 2 * B * Hkv * L * d * 2
        for splits in (0, 1, 8, 32, 128):
            ws = torch.empty(af.decode_workspace_size(B, Hq, Hkv, L, d, splits), dtype=torch.uint8,
                             device=dev)
            for _ in range(3):
                af.decode(q, kc, vc, L - 1, rope_theta=5e5, num_splits=splits, out=out, lse=lse,
                          workspace=ws)
            call = lambda: af.decode(q, kc, vc, L - 1, rope_theta=5e5, num_splits=splits,
                                     out=out, lse=lse, workspace=ws)
            res = {"cold": [], "cold_dirty": [], "warm": []}
            # cold L2 before each timed call: a write of 4x the L2, then (clean) a read of 3x
            for key in ("cold", "cold_dirty"):
                for _ in range(30):
                    flush.zero_()
                    if key == "cold":
                        evict.max()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    call()
                    e1.record()
                    torch.cuda.synchronize()
                    res[key].append(e0.elapsed_time(e1) * 1e3)
            # warm L2, device time: 20 back-to-back calls captured in one CUDA graph (the host's
            # per-call cost is measured separately below)
            g = _graph_of(lambda: [call() for _ in range(20)])
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                res["warm"].append(e0.elapsed_time(e1) * 1e3 / 20)
            del g
            # host cost of one eager call through the Python binding and the C entry point
            torch.cuda.synchronize()
            h0 = time.perf_counter()
            for _ in range(50):
                call()
            h1 = time.perf_counter()
            torch.cuda.synchronize()
            host_us = (h1 - h0) / 50 * 1e6
            for key in res:
                res[key].sort()
            med = res["cold"][len(res["cold"]) // 2]
            gbs = nbytes / (med * 1e-6) / 1e9
            used = splits if splits else af.decode_auto_splits(B, Hkv, L)
            rows.append({"decode": "llama70b_head_shape", "B": B, "splits": splits,
                              "splits_used": used, "us_median_cold_l2": med,
                              "us_min_cold_l2": res["cold"][0],
                              "us_p90_cold_l2": res["cold"][int(0.9 * len(res["cold"]))],
                              "cold_method": "512 MiB write, then 384 MiB read of another buffer",
                              "us_median_cold_l2_dirty": res["cold_dirty"][len(res["cold_dirty"]) // 2],
                              "frac_of_hbm_dirty": nbytes / (res["cold_dirty"][len(res["cold_dirty"]) // 2] * 1e-6) / 1e9 / float(peaks["hbm_gbs"]),
                              "us_median_warm_l2": res["warm"][len(res["warm"]) // 2],
                              "warm_method": "CUDA graph of 20 back-to-back calls, per call",
                              "us_host_per_eager_call": host_us,
                              "kv_bytes": nbytes, "gbs_cold": gbs,
                              "frac_of_hbm": gbs / float(peaks["hbm_gbs"]),
                              "launches": 2})
            if emit:
                print(json.dumps(rows[-1]), flush=True)
    return rows


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch

        torch.distributed.init_process_group("nccl")
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    if args.profile:
        run_profile(args)
        return
    if args.decode:
        if rank == 0:
            run_decode_bench(args)
        return
    if args.train:
        if rank == 0:
            run_train_bench(args)
        return
    if args.variants:
        if rank == 0:
            run_variants_bench(args)
        return
    if args.fp8:
        if rank == 0:
            run_fp8_bench(args)
        return
    if args.tables:
        if rank == 0:
            run_tables_bench(args)
        return
    run_ours(args, rank, world)
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
