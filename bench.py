#!/usr/bin/env python
"""Benchmark of the forget-gated causal attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
gate scan + fused forward (O, LSE), then (reading the forward's gate terms from
the shared workspace) backward rows + fused backward + dQ conversion + reverse
gate scan (dQ, dK, dV, dz). Throughput is nominal causal FLOPs (2 B H N^2 d
forward, 5 B H N^2 d backward) per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fox|reference]

Under torchrun each rank runs its own batch of independent (b, h) heads
(weak scaling, no data-path collective); rank 0 prints one JSON line.
--impl reference times the CPU fp64 oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "FoX causal attention fwd/bwd TFLOP/s (bf16) and % of GB300 tensor-core peak"
# Traced stream operations that are not this library's kernels (left out of gpu_launches).
NOT_OUR_KERNELS = ("dq_zero",)
WORKLOAD = wl.Workload(
    "long_bf16_B1H32N16384d128", 1, 16384, 32, 128, "bf16", 2, gate="head_linspace", lo=0.0, hi=8.0, sigma=0.5,
    backward=True,
)
# CPU sample of the same workload: all 32 heads of batch 0, each restricted to its first 4096 tokens
# (a causal prefix is a complete problem of its own), forward + backward.
CPU_SAMPLE_HEADS = 32
CPU_SAMPLE_TOKENS = 4096
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SUSTAINED_MIN_S = 3.0  # a timed region at least this long is compared with the sustained tensor peak


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(src: str) -> str:
    """C / CUDA source with comments removed and whitespace runs collapsed (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


# Sources that determine each traced kernel's code and launch (its own translation unit, the
# shared headers, and the host code that builds its tensor maps).
KERNEL_SOURCES = {
    "attn_fwd": ("fox_fwd.cu", "fox_api.cu", "fox_internal.h", "fox_ptx.cuh"),
    "attn_bwd": ("fox_bwd.cu", "fox_api.cu", "fox_internal.h", "fox_ptx.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (comments and layout ignored) of the sources behind `kernel`; an ncu
    traffic figure is only reported for the code it was taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "forget_gated_softmax_gb300", "csrc")
    for f in KERNEL_SOURCES.get(kernel, tuple(sorted(os.listdir(csrc)))):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:12]


def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes for `kernel` from profiles/ncu_traffic.md, if taken on this source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash(kernel)
    pat = re.compile(r"^\|\s*(\S+)\s*\|\s*(\S+)\s*\|\s*([0-9.eE+]+)\s*\|\s*([0-9a-f]+)\s*\|")
    with open(path) as f:
        for line in f:
            m = pat.match(line.strip())
            if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == src:
                return float(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fox_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def oracle_sample(arrays, heads: int, tokens: int):
    """Oracle forward + backward on heads (0, 0..heads-1) restricted to their first `tokens` tokens."""
    from oracle import fox_oracle as ora

    x = {n: (a[0, :tokens, :heads].astype(np.float64) if n == "z" else wl.as_f64(a[0, :tokens, :heads], "bf16"))
         for n, a in arrays.items()}
    t0 = time.perf_counter()
    for h in range(heads):
        ora.backward_head(x["q"][:, h], x["k"][:, h], x["v"][:, h], x["z"][:, h], x["dO"][:, h])
    dt = time.perf_counter() - t0
    flops = heads * 7.0 * tokens * tokens * WORKLOAD.d  # nominal fwd (2) + bwd (5) per head
    return flops / dt / 1e12, dt


def blas_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def sample_desc(heads: int = CPU_SAMPLE_HEADS):
    return (f"oracle forward+backward of heads (b=0, h=0..{heads - 1}) of {WORKLOAD.name}, each cut to "
            f"its first {CPU_SAMPLE_TOKENS} tokens (a causal prefix), fp64 numpy; TFLOP/s on nominal 7*N^2*d per head")


def oracle_one_thread_child():
    """(Run in a child process whose BLAS and OpenMP pools are held to one thread.) The oracle's
    forward on the whole tiny fp32 workload and the whole mid bf16 workload, each timed once."""
    from oracle import fox_oracle as ora

    out = {}
    for w in (wl.TINY_F32, wl.MID_BF16):
        a = wl.draw(w)
        x = {n: (v.astype(np.float64) if n == "z" else wl.as_f64(v, w.dtype)) for n, v in a.items()}
        t0 = time.perf_counter()
        ora.forward(x["q"], x["k"], x["v"], x["z"], bias_from_j=w.bias_from_j)
        dt = time.perf_counter() - t0
        out[w.name] = {"seconds": dt, "value": w.fwd_flops() / dt / 1e12, "unit": "TFLOP/s"}
    print(json.dumps(out), flush=True)


def oracle_one_thread():
    """The oracle's forward on the tiny and mid workloads with one host thread (a child process,
    BLAS / OpenMP pools held to 1 thread), for comparison with the all-cores figure."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-thread"], env=env,
                           capture_output=True, text=True, timeout=300)
        res = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, never fatal to the GPU measurement
        return {"error": f"{type(e).__name__}: {e}"[:200]}
    res["cores"] = 1
    res["kind"] = "oracle forward, whole workload, one thread"
    return res


REFERENCE_BUDGET_S = 120.0  # the whole --impl reference run (warm-up + timed steps) aims at about this


def run_reference(args, rank: int):
    """The oracle on the host cores: each step is forward + backward of a bounded sample of
    the workload's heads (each cut to its first CPU_SAMPLE_TOKENS tokens), with the number of
    heads per step chosen from a one-head calibration so that the run ends in a few minutes."""
    if rank != 0:
        return
    arrays = draw_inputs(WORKLOAD, rank, cut=CPU_SAMPLE_TOKENS)
    _, t_head = oracle_sample(arrays, 1, CPU_SAMPLE_TOKENS)  # calibration, not counted
    n_calls = max(1, args.steps + args.warmup)
    heads = int(max(1, min(CPU_SAMPLE_HEADS, REFERENCE_BUDGET_S / (n_calls * max(t_head, 1e-3)))))
    for _ in range(args.warmup):
        oracle_sample(arrays, heads, CPU_SAMPLE_TOKENS)
    vals, times = [], []
    for _ in range(args.steps):
        v, dt = oracle_sample(arrays, heads, CPU_SAMPLE_TOKENS)
        vals.append(v)
        times.append(dt)
    total_flops = args.steps * heads * 7.0 * CPU_SAMPLE_TOKENS**2 * WORKLOAD.d
    value = total_flops / sum(times) / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample_desc(heads)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(n_gpus: int):
    w = WORKLOAD
    return {
        "workload": f"{w.name}: forward+backward, causal, j+1 convention, q,k,v,dO ~ N(0,1) bf16, "
                    f"z = b_h + 0.5 N(0,1), b_h = linspace(0, 8, 32)",
        "B": w.B, "H": w.H, "N": w.N, "d": w.d,
        "flops_per_step": w.fwd_flops() + w.bwd_flops(),
        "l2": f"inputs larger than L2: q, k, v, dO are {w.tokens * w.d * 2 / 1e6:.0f} MB each",
        "parallelism": f"{n_gpus} rank(s), each an independent batch of heads (no collective)",
    }


def draw_inputs(w: wl.Workload, rank: int, cut: int = 0):
    """Seeded inputs; rank r draws the workload with seed + 1000 r (an independent batch of heads).
    With `cut`, only the first `cut` tokens of every tensor are kept."""
    import dataclasses

    if rank:
        w = dataclasses.replace(w, seed=w.seed + 1000 * rank)
    arrays = wl.draw(w, with_dO=True)
    if cut:
        arrays = {n: np.ascontiguousarray(a[:, :cut]) for n, a in arrays.items()}
    return arrays


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """Largest `value` over all ranks (the timing rule: the slowest rank sets the job's time)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed_variant(fox, torch, stream, fn, steps: int, flops: float) -> dict:
    """Warm up, then time `steps` calls of fn on `stream` with CUDA events and the
    library trace; returns ms per step, nominal TFLOP/s and per-kernel totals."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fox.trace_begin()
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    rec = fox.trace_end()
    ms = a.elapsed_time(b) / steps
    per = {}
    for name, t in rec:
        per[name] = per.get(name, 0.0) + t / steps
    return {"ms_per_step": ms, "tflops_nominal": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "kernel_ms_per_step": per, "launches_per_step": len(rec) // steps}


def run_fox(args, rank: int, world: int, local_rank: int):
    import torch

    import forget_gated_softmax_gb300 as fox

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    w = WORKLOAD
    t0 = time.time()
    arrays = draw_inputs(w, rank)
    log(f"[rank {rank}] inputs drawn in {time.time() - t0:.1f}s")

    def dev(name):
        a = arrays[name]
        if name == "z":
            return torch.from_numpy(a).cuda()
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v, z, dO = (dev(n) for n in ("q", "k", "v", "z", "dO"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.N, w.H), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dz = torch.empty_like(lse)
    pf = fox.make_params(w.B, w.N, w.H, w.d, 0, 0.0, False)
    # One workspace for the step: the backward reads the gate terms the forward left in it.
    ws_f = ws_b = fox.workspace(max(fox.fox_fwd_workspace_bytes(pf), fox.fox_bwd_workspace_bytes(pf)), "cuda")
    stream = torch.cuda.current_stream()

    def step():
        fox.fox_fwd(q, k, v, z, o=o, lse=lse, ws=ws_f, stream=stream)
        fox.fox_bwd(q, k, v, z, o, lse, dO, dq=dq, dk=dk, dv=dv, dz=dz, ws=ws_b, stream=stream, gate_ready=True)

    for i in range(args.warmup):
        step()
        if i == 0:
            assert fox.fox_check_error(ws_f) == 0, "device-side error"
    torch.cuda.synchronize()

    # ---------------- device-resident timed region
    # No events between the kernels of a step here: the kernels of each call are launched as
    # programmatic dependents of the one before, and an event between two launches would stop the
    # next one from starting early. The per-kernel breakdown comes from a second, traced region.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    with sampler:
        time.sleep(0.3)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            stops[i].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    clocks = sampler.summary()
    trace_steps = min(args.steps, 40)
    torch.cuda.synchronize()
    fox.trace_begin()
    for i in range(trace_steps):
        step()
    torch.cuda.synchronize()
    records = fox.trace_end()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, stops)]
    elapsed_ms = starts[0].elapsed_time(stops[-1])
    assert fox.fox_check_error(ws_f) == 0 and fox.fox_check_error(ws_b) == 0, "device-side error"
    elapsed_ms = max_over_ranks(elapsed_ms, dist, "cuda")
    flops_step = w.fwd_flops() + w.bwd_flops()
    value = world * flops_step * args.steps / (elapsed_ms * 1e-3) / 1e12

    # per-kernel breakdown from the trace (same timed region, events on the launching stream)
    per = {}
    for name, ms in records:
        per.setdefault(name, []).append(ms)
    peaks, peak_src = measured_peaks()
    # The tensor peak a fraction is taken against: the burst figure for a short timed region,
    # the sustained (power-capped) one only when the timed region runs for seconds.
    timed_s = elapsed_ms * 1e-3
    tensor_peak_key = "bf16_tflops_sustained" if timed_s >= SUSTAINED_MIN_S else "bf16_tflops"
    algo = {  # algorithmic work per launch
        "attn_fwd": ("tensor", w.fwd_flops()),
        "attn_bwd": ("tensor", w.bwd_flops()),
        "gate_tile_scan": ("hbm", w.tokens * (4 + 4 + 4 + 4)),   # z in; rowloc, colrec, tile totals out
        "gate_base_scan": ("hbm", w.B * w.H * ((w.N + 127) // 128) * (4 + 16)),
        # the base scan with the forward's fp16 copy of V: V (bf16) in, the copy out
        "gate_base_scan_v16": ("hbm", w.tokens * w.d * (2 + 2) + w.B * w.H * ((w.N + 127) // 128) * (4 + 16)),
        "dq_zero": ("hbm", w.tokens * 4 * w.d),  # the dQ accumulator cleared (a stream-ordered memset)
        "bwd_rows": ("hbm", w.tokens * (2 * w.d * 2 + 4 + 4 + 4 + 4 + 4)),  # O, dO, lse, rowloc in; delta, rho, R out
        "bwd_dq": ("hbm", w.tokens * w.d * (4 + 2)),
        "bwd_gate": ("hbm", w.tokens * (4 + 4 + 4 + 4)),  # R, C, z in; dz out (one pass)
    }
    kernels = {}
    for name, ms in per.items():  # (dq_zero is a cudaMemsetAsync, listed for its time)
        avg = sum(ms) / len(ms)
        kind, work = algo.get(name, ("hbm", 0))
        if kind == "tensor":
            ach = work / (avg * 1e-3) / 1e12
            peak = peaks[tensor_peak_key]
            unit = "TFLOP/s"
        else:
            ach = work / (avg * 1e-3) / 1e9
            peak = peaks["hbm_gbs"]
            unit = "GB/s"
        kernels[name] = {"launches": len(ms), "avg_ms": avg, "total_ms": sum(ms), "bound": kind,
                         "achieved": ach, "unit": unit, "frac": ach / peak}
    dominant = max(kernels, key=lambda n: kernels[n]["total_ms"])
    dk_ = kernels[dominant]
    peak_key = tensor_peak_key if dk_["bound"] == "tensor" else "hbm_gbs"
    roofline = {
        "kernel": dominant, "bound": dk_["bound"], "achieved": dk_["achieved"],
        "peak": peaks[peak_key], "unit": dk_["unit"], "frac": dk_["frac"],
        "traffic": ncu_traffic(dominant, w.name),
        "peak_source": f"{peak_src} ({peak_key}; timed region {timed_s:.2f} s)",
    }
    if dk_["bound"] == "tensor":
        roofline["frac_of_burst_peak"] = dk_["achieved"] / peaks["bf16_tflops"]
        roofline["frac_of_sustained_peak"] = dk_["achieved"] / peaks["bf16_tflops_sustained"]

    # ---------------- end to end through the public API with host buffers
    # Every step copies its inputs from pinned host memory and its results back to pinned
    # host memory, through the same fox_fwd / fox_bwd calls. The copies of one step overlap
    # the compute of its neighbours: inputs and outputs are double-buffered on the device,
    # with H2D on one stream, the step on another and D2H on a third (a prefetching data
    # loader's pattern). The timed region spans the first H2D to the last D2H.
    in_names = ("q", "k", "v", "z", "dO")
    out_names = ("o", "lse", "dq", "dk", "dv", "dz")
    dev_in0 = {"q": q, "k": k, "v": v, "z": z, "dO": dO}
    dev_out0 = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv, "dz": dz}
    pin = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in dev_in0.items()}
    for n, t in dev_in0.items():
        pin[n].copy_(t)
    outs = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in dev_out0.items()}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in outs.values())
    dev_in = [dev_in0, {n: torch.empty_like(t) for n, t in dev_in0.items()}]
    dev_out = [dev_out0, {n: torch.empty_like(t) for n, t in dev_out0.items()}]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(nsteps):
        ev_in = [None] * nsteps
        ev_comp = [None] * nsteps
        ev_out = [None] * nsteps
        for i in range(nsteps):
            slot = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])  # step i-2 is done reading this input slot
                for n in in_names:
                    dev_in[slot][n].copy_(pin[n], non_blocking=True)
                ev_in[i] = torch.cuda.Event()
                ev_in[i].record(s_in)
            s_comp.wait_event(ev_in[i])
            if i >= 2:
                s_comp.wait_event(ev_out[i - 2])  # this output slot has been copied out
            di, do_ = dev_in[slot], dev_out[slot]
            fox.fox_fwd(di["q"], di["k"], di["v"], di["z"], o=do_["o"], lse=do_["lse"], ws=ws_f, stream=s_comp)
            fox.fox_bwd(di["q"], di["k"], di["v"], di["z"], do_["o"], do_["lse"], di["dO"], dq=do_["dq"],
                        dk=do_["dk"], dv=do_["dv"], dz=do_["dz"], ws=ws_b, stream=s_comp, gate_ready=True)
            ev_comp[i] = torch.cuda.Event()
            ev_comp[i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                for n in out_names:
                    outs[n].copy_(do_[n], non_blocking=True)
                ev_out[i] = torch.cuda.Event()
                ev_out[i].record(s_out)
        torch.cuda.synchronize()  # the host reads the results

    e2e_run(2)
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    e2e_run(args.steps)
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, "cuda")
    e2e_value = world * flops_step * args.steps / e2e_s / 1e12
    assert fox.fox_check_error(ws_f) == 0 and fox.fox_check_error(ws_b) == 0, "device-side error"

    # ---------------- the widened rows (window, tile skipping, non-causal, gate projection, gate
    # steps at a large size): timed separately, not part of the step
    extra = {}
    ws_w = fox.workspace(fox.fox_window_workspace_bytes(pf), "cuda")
    win = torch.empty((w.B, w.N, w.H), dtype=torch.int32, device="cuda")
    for _ in range(3):
        fox.fox_window(z, 1e-3, window=win, ws=ws_w, stream=stream)
    torch.cuda.synchronize()
    fox.trace_begin()
    for _ in range(10):
        fox.fox_window(z, 1e-3, window=win, ws=ws_w, stream=stream)
    torch.cuda.synchronize()
    wrec = fox.trace_end()
    w_ms = sum(ms for _, ms in wrec) / 10
    w_bytes = w.tokens * (4 + 8 + 8 + 4)  # z read, fp64 local sums written and read, int32 window written
    extra["effective_window"] = {
        "eps": 1e-3, "ms": w_ms, "launches_per_call": len(wrec) // 10,
        "achieved": w_bytes / (w_ms * 1e-3) / 1e9, "unit": "GB/s", "bound": "hbm",
        "frac": w_bytes / (w_ms * 1e-3) / 1e9 / measured_peaks()[0]["hbm_gbs"],
        "rows_passing": int((win >= 0).sum().item()),
    }

    # Decay-aware tile skipping (causal, bit-identical outputs): the same step with
    # tile_skip = 1, on the same inputs; nominal FLOPs over its time is the effective rate.
    ps = fox.make_params(w.B, w.N, w.H, w.d, 0, 0.0, False, tile_skip=True)
    ws_sf = ws_sb = fox.workspace(max(fox.fox_fwd_workspace_bytes(ps), fox.fox_bwd_workspace_bytes(ps)), "cuda")

    def skip_step():
        fox.fox_fwd(q, k, v, z, o=o, lse=lse, ws=ws_sf, stream=stream, tile_skip=True)
        fox.fox_bwd(q, k, v, z, o, lse, dO, dq=dq, dk=dk, dv=dv, dz=dz, ws=ws_sb, stream=stream, tile_skip=True,
                    gate_ready=True)

    extra["tile_skip"] = timed_variant(fox, torch, stream, skip_step, 10, w.fwd_flops() + w.bwd_flops())
    assert fox.fox_check_error(ws_sf) == 0 and fox.fox_check_error(ws_sb) == 0, "device-side error"
    jmin, _ = fox.fox_tile_span(q, k, z, stream=stream)
    nT = jmin.shape[1]
    visited = (torch.arange(nT, device="cuda")[None, :] - jmin + 1).sum().item()
    extra["tile_skip"]["pairs_visited_frac"] = visited / (w.B * w.H * nT * (nT + 1) / 2)
    extra["tile_skip"]["speedup_vs_full_step"] = (elapsed_ms / args.steps) / extra["tile_skip"]["ms_per_step"]

    # Non-causal (encoder) mode on the same inputs: every key for every query.
    def nc_step():
        fox.fox_fwd(q, k, v, z, o=o, lse=lse, ws=ws_f, stream=stream, non_causal=True)
        fox.fox_bwd(q, k, v, z, o, lse, dO, dq=dq, dk=dk, dv=dv, dz=dz, ws=ws_b, stream=stream, non_causal=True,
                    gate_ready=True)

    nc_flops = 2 * (w.fwd_flops() + w.bwd_flops())  # the full N^2 score matrix instead of its causal half
    extra["non_causal"] = timed_variant(fox, torch, stream, nc_step, 5, nc_flops)
    extra["non_causal"]["note"] = ("flops: 4BHN^2d forward + 10BHN^2d backward; the backward first forms "
                                   "Delta = sum_j P dP from S = Q K^T and dP = dO V^T (one forward's worth of MMAs)")
    assert fox.fox_check_error(ws_f) == 0 and fox.fox_check_error(ws_b) == 0, "device-side error"

    # Gate projection fused with the gate scan (z = x W_f^T + b_f, hidden = H d): HBM-bound
    # on reading x; timed alone and as part of the forward from x.
    hidden = w.H * w.d
    gp = wl.draw_gate_projection(w, hidden)
    xg = torch.from_numpy(gp["x"].view(np.int16)).view(torch.bfloat16).cuda()
    wg = torch.from_numpy(gp["w_f"].view(np.int16)).view(torch.bfloat16).cuda()
    bg = torch.from_numpy(gp["b_f"]).cuda()
    zg = torch.empty_like(z)
    gp_res = timed_variant(fox, torch, stream, lambda: fox.fox_gate_proj(xg, wg, bg, z=zg, ws=ws_f, stream=stream),
                           20, 2.0 * w.tokens * hidden)
    gp_ms = gp_res["kernel_ms_per_step"].get("gate_proj_scan", gp_res["ms_per_step"])
    gp_bytes = w.B * w.N * hidden * 2 + w.H * hidden * 2 + w.tokens * (4 + 4 + 4 + 4)  # x, W in; z, gate terms out
    extra["gate_projection"] = {
        "hidden": hidden, "ms_per_call": gp_res["ms_per_step"], "kernel_ms": gp_ms,
        "achieved": gp_bytes / (gp_ms * 1e-3) / 1e9, "unit": "GB/s", "bound": "hbm",
        "frac": gp_bytes / (gp_ms * 1e-3) / 1e9 / measured_peaks()[0]["hbm_gbs"],
        "kernel_ms_per_call": gp_res["kernel_ms_per_step"],
    }
    assert fox.fox_check_error(ws_f) == 0, "device-side error"
    del xg

    # The gate steps alone on a large synthetic (B64 H32 N16384: 134 MB of z), where they are
    # not launch-bound: the scan (log-sigmoid, 128-token tile scans, fp64 tile bases) into the
    # workspace, and the gate gradient from the row and column sums of dS.
    GB, GN, GH = 64, 16384, 32
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    zl = 2.0 + torch.randn((GB, GN, GH), generator=gen, device="cuda", dtype=torch.float32)
    Rl = torch.randn((GB, GH, GN), generator=gen, device="cuda", dtype=torch.float32)
    Cl = torch.randn((GB, GH, GN), generator=gen, device="cuda", dtype=torch.float32)
    dzl = torch.empty_like(zl)
    pg = fox.make_params(GB, GN, GH, 64)
    ws_g = fox.workspace(fox.fox_gate_scan_workspace_bytes(pg), "cuda")
    big = GB * GN * GH
    peak_hbm = measured_peaks()[0]["hbm_gbs"]
    scan_res = timed_variant(fox, torch, stream, lambda: fox.fox_gate_scan(zl, want_c=False, ws=ws_g, stream=stream),
                             10, 0.0)
    scan_ms = sum(scan_res["kernel_ms_per_step"].values())
    scan_bytes = big * (4 + 4 + 4) + GB * GH * ((GN + 127) // 128) * 4 * 5  # z in; local and column terms out; tiles
    ws_gb = fox.workspace(fox.fox_gate_bwd_workspace_bytes(pg), "cuda")
    grad_res = timed_variant(fox, torch, stream, lambda: fox.fox_gate_bwd(zl, Rl, Cl, dz=dzl, ws=ws_gb, stream=stream),
                             10, 0.0)
    grad_ms = sum(grad_res["kernel_ms_per_step"].values())
    grad_bytes = big * (4 + 4 + 4 + 4)  # R, C, z in; dz out (one pass)
    extra["gate_steps_large"] = {
        "shape": f"B{GB} H{GH} N{GN} (z ~ N(2,1) fp32, R, C ~ N(0,1))",
        "scan": {"ms": scan_ms, "kernel_ms": scan_res["kernel_ms_per_step"],
                 "achieved": scan_bytes / (scan_ms * 1e-3) / 1e9, "unit": "GB/s", "bound": "hbm",
                 "frac": scan_bytes / (scan_ms * 1e-3) / 1e9 / peak_hbm},
        "gate_grad": {"ms": grad_ms, "kernel_ms": grad_res["kernel_ms_per_step"],
                      "achieved": grad_bytes / (grad_ms * 1e-3) / 1e9, "unit": "GB/s", "bound": "hbm",
                      "frac": grad_bytes / (grad_ms * 1e-3) / 1e9 / peak_hbm},
    }
    del zl, Rl, Cl, dzl, ws_g, ws_gb

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v_cpu, dt_cpu = oracle_sample(arrays, CPU_SAMPLE_HEADS, CPU_SAMPLE_TOKENS)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle", "sample": sample_desc(),
               "seconds": dt_cpu, "one_thread": oracle_one_thread()}

    if rank == 0:
        fwd_ms = sum(kernels[n]["total_ms"] for n in kernels if n in ("attn_fwd",)) / trace_steps
        bwd_ms = sum(kernels[n]["total_ms"] for n in kernels if n == "attn_bwd") / trace_steps
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(world),
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "copies": "pinned host <-> device every step, overlapped with the neighbouring steps' compute"},
            # this library's kernel launches in the timed region (per step, from the traced region)
            "gpu_launches": sum(1 for name, _ in records if name not in NOT_OUR_KERNELS) * args.steps // trace_steps,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "clock_normalised": {
                "timed_region_s": timed_s, "sm_mhz_median": clocks.get("sm_mhz"), "tensor_peak": tensor_peak_key,
                "ms_per_step_x_sm_ghz": (elapsed_ms / args.steps) * clocks["sm_mhz"] / 1e3 if clocks.get("sm_mhz")
                else None,
                "note": f"a timed region of at least {SUSTAINED_MIN_S:.0f} s (e.g. --steps 600) is compared with the "
                        "sustained tensor peak; a shorter one with the burst peak",
            },
            "next": extra,
            "breakdown": {
                "note": f"per-kernel times from a second, traced region of {trace_steps} steps",
                "step_ms_median": statistics.median(step_ms),
                "fwd_attn_ms": fwd_ms, "fwd_attn_tflops": w.fwd_flops() / (fwd_ms * 1e-3) / 1e12 if fwd_ms else None,
                "bwd_attn_ms": bwd_ms, "bwd_attn_tflops": w.bwd_flops() / (bwd_ms * 1e-3) / 1e12 if bwd_ms else None,
                "kernels": kernels,
            },
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_profile(args):
    """--profile: the forward+backward step alone on the workload (inputs, outputs and the two
    workspaces are all it holds on the device: about 1.5 GB at the default shape), warmup +
    steps calls, CUDA-event timed; for profiler captures of one kernel. Not a bench line."""
    import torch

    import forget_gated_softmax_gb300 as fox

    w = WORKLOAD
    arrays = draw_inputs(w, 0)
    dev = {n: (torch.from_numpy(a).cuda() if n == "z" else torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda())
           for n, a in arrays.items()}
    q, k, v, z, dO = (dev[n] for n in ("q", "k", "v", "z", "dO"))
    o, lse = torch.empty_like(q), torch.empty((w.B, w.N, w.H), dtype=torch.float32, device="cuda")
    dq, dk, dv, dz = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(lse)
    pf = fox.make_params(w.B, w.N, w.H, w.d)
    ws_f = ws_b = fox.workspace(max(fox.fox_fwd_workspace_bytes(pf), fox.fox_bwd_workspace_bytes(pf)), "cuda")
    stream = torch.cuda.current_stream()

    def step():
        fox.fox_fwd(q, k, v, z, o=o, lse=lse, ws=ws_f, stream=stream)
        fox.fox_bwd(q, k, v, z, o, lse, dO, dq=dq, dk=dk, dv=dv, dz=dz, ws=ws_b, stream=stream, gate_ready=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    fox.trace_begin()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    rec = fox.trace_end()
    assert fox.fox_check_error(ws_f) == 0 and fox.fox_check_error(ws_b) == 0, "device-side error"
    per = {}
    for name, ms in rec:
        per[name] = per.get(name, 0.0) + ms / max(1, args.steps)
    log(json.dumps({"workload": w.name, "profile_steps": args.steps, "kernel_ms_per_step": per,
                    "attn_fwd_tflops": w.fwd_flops() / (per.get("attn_fwd", 0) * 1e-3) / 1e12 if per.get("attn_fwd") else None,
                    "attn_bwd_tflops": w.bwd_flops() / (per.get("attn_bwd", 0) * 1e-3) / 1e12 if per.get("attn_bwd") else None}))


def run_profile_gate(args):
    """--profile-gate: the two gate steps alone on the large synthetic (B64 H32 N16384: z, R, C and dz
    are 134 MB each, about 0.6 GB on the device): warmup + steps calls of the gate scan and of the
    gate gradient, for profiler captures. Not a bench line."""
    import torch

    import forget_gated_softmax_gb300 as fox

    GB, GN, GH = 64, 16384, 32
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    zl = 2.0 + torch.randn((GB, GN, GH), generator=gen, device="cuda", dtype=torch.float32)
    Rl = torch.randn((GB, GH, GN), generator=gen, device="cuda", dtype=torch.float32)
    Cl = torch.randn((GB, GH, GN), generator=gen, device="cuda", dtype=torch.float32)
    dzl = torch.empty_like(zl)
    pg = fox.make_params(GB, GN, GH, 64)
    ws_g = fox.workspace(fox.fox_gate_scan_workspace_bytes(pg), "cuda")
    ws_gb = fox.workspace(fox.fox_gate_bwd_workspace_bytes(pg), "cuda")
    for _ in range(args.warmup + args.steps):
        fox.fox_gate_scan(zl, want_c=False, ws=ws_g)
        fox.fox_gate_bwd(zl, Rl, Cl, dz=dzl, ws=ws_gb)
    torch.cuda.synchronize()
    assert fox.fox_check_error(ws_g) == 0 and fox.fox_check_error(ws_gb) == 0, "device-side error"
    log(json.dumps({"profile_gate": f"B{GB} H{GH} N{GN}", "calls": args.warmup + args.steps}))


def run_configs(args):
    """--configs: forward (and backward where the workload has one) of each named input
    recipe on this GPU, CUDA-event timed; one JSON object per workload on stderr, and the
    oracle's fp64 rate on the host for comparison. Not a bench line."""
    import torch

    import forget_gated_softmax_gb300 as fox

    peaks, _ = measured_peaks()
    stream = torch.cuda.current_stream()
    for w in wl.ALL:
        arrays = wl.draw(w)
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

        def dev(name):
            a = arrays[name]
            if name == "z" or w.dtype == "f32":
                return torch.from_numpy(np.ascontiguousarray(a)).cuda()
            return torch.from_numpy(a.view(np.int16)).view(dt).cuda()

        q, k, v, z = (dev(n) for n in ("q", "k", "v", "z"))
        o, lse = torch.empty_like(q), torch.empty((w.B, w.N, w.H), dtype=torch.float32, device="cuda")
        pf = fox.make_params(w.B, w.N, w.H, w.d, 0 if w.dtype == "bf16" else 1, 0.0, w.bias_from_j)
        ws = fox.workspace(fox.fox_bwd_workspace_bytes(pf) if w.backward else fox.fox_fwd_workspace_bytes(pf), "cuda")
        fwd = lambda: fox.fox_fwd(q, k, v, z, o=o, lse=lse, ws=ws, stream=stream)  # noqa: E731
        res = {"workload": w.name, "dtype": w.dtype}
        reps = 20
        for _ in range(3):
            fwd()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fwd()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        res["fwd_ms"] = ms
        res["fwd_tflops"] = w.fwd_flops() / (ms * 1e-3) / 1e12
        if w.dtype == "bf16":
            res["fwd_frac_of_burst_peak"] = res["fwd_tflops"] / peaks["bf16_tflops"]
        if w.backward:
            dO = dev("dO")
            dq, dk, dv, dz = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(lse)
            bwd = lambda: fox.fox_bwd(q, k, v, z, o, lse, dO, dq=dq, dk=dk, dv=dv, dz=dz, ws=ws,  # noqa: E731
                                      stream=stream)
            for _ in range(3):
                bwd()
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(reps):
                bwd()
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / reps
            res["bwd_ms"] = ms
            res["bwd_tflops"] = w.bwd_flops() / (ms * 1e-3) / 1e12
            res["bwd_frac_of_burst_peak"] = res["bwd_tflops"] / peaks["bf16_tflops"]
        assert fox.fox_check_error(ws) == 0, "device-side error"
        log(json.dumps(res))
    if not args.no_cpu_baseline:
        v_cpu, dt_cpu = oracle_sample(draw_inputs(WORKLOAD, 0, CPU_SAMPLE_TOKENS), CPU_SAMPLE_HEADS, CPU_SAMPLE_TOKENS)
        log(json.dumps({"oracle": "fp64, all host cores", "tflops": v_cpu, "cores": blas_threads(),
                        "sample": sample_desc(), "seconds": dt_cpu}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("fox", "reference"), default="fox")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing on the host")
    ap.add_argument("--configs", action="store_true",
                    help="time every named workload recipe (fwd, and bwd where it has one); results on stderr")
    ap.add_argument("--oracle-one-thread", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--profile", action="store_true",
                    help="run only the forward+backward step (warmup + steps calls), for profiler captures; "
                         "prints timings on stderr, not a bench line")
    ap.add_argument("--profile-gate", action="store_true",
                    help="run only the gate scan and gate gradient on the large synthetic (profiler captures)")
    ap.add_argument("--shape", default=None,
                    help="B,N,H,d of a smaller case of the same workload recipe (profiling runs; not a bench line)")
    args = ap.parse_args()
    if args.shape:
        import dataclasses

        global WORKLOAD
        B, N, H, d = (int(x) for x in args.shape.split(","))
        WORKLOAD = dataclasses.replace(WORKLOAD, name=f"long_recipe_B{B}H{H}N{N}d{d}", B=B, N=N, H=H, d=d)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.oracle_one_thread:
        oracle_one_thread_child()
        return
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.profile:
        run_profile(args)
        return
    if args.profile_gate:
        run_profile_gate(args)
        return
    if args.configs:
        run_configs(args)
        return
    run_fox(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
