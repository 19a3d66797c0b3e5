#!/usr/bin/env python
"""Benchmark of the gated delta rule library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0.  A step is one gdn_prefill call over the
B=1, T=4096, Hk=16, Hv=32, Dk=Dv=128, bf16, chunk-64 workload with its
inputs resident in HBM; `value` is tokens/s (B*T per step).  The line also
carries the decode workload (B=64, Hk=16, Hv=32, 256 successive steps in one
CUDA graph, state updated in place) as `decode`, the roofline of each, the
end-to-end number through the C ABI from pinned host buffers (`e2e`) and the
fp64 oracle timed on the host cores (`cpu_baseline`).

Timing: W untimed warm-up steps; then exactly K steps, each bracketed by
CUDA events on the launching stream, with a 256 MiB write between steps to
flush the L2 (outside the events); barrier + synchronize on both sides; the
max over ranks.  N > 1 runs one independent replica per GPU (the heads of the
rule are independent; there is no exchange), so scaling is weak.

`--impl reference` times the fp64 oracle (the only reference this method has)
on the host cores on a bounded sample of the same workload, in the same metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import gdn_inputs  # noqa: E402

FLUSH_BYTES = 256 << 20

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per call from one
# ncu capture, summarised under profiles/, per workload.  Valid only for the
# kernel sources it was taken on (sha256 prefix of those files); otherwise
# reported as null.
_KDIR = os.path.join(ROOT, "gated_delta_rule_02_gb300", "csrc")
MEASURED_TRAFFIC = {
    "prefill_t4096": {"sources": ["prefill_tc.cu", "sm100_ptx.cuh"], "sha": "3230ab1f70e45acc",
                      "bytes": 157.1e6},
    "prefill_b4_t2048": {"sources": ["prefill_tc.cu", "sm100_ptx.cuh"],
                         "sha": "3230ab1f70e45acc", "bytes": 1049.7e6},
    "decode_b64": {"sources": ["decode.cu"], "sha": "48a64c9af36e1446", "bytes": 210.7e6},
    "prefill_b64_t16": {"sources": ["prefill_short_tc.cu", "warp_mma.cuh", "sm100_ptx.cuh"],
                        "sha": "aea52e59a7d765cc", "bytes": 238.1e6},
}


def measured_traffic(key):
    import hashlib
    entry = MEASURED_TRAFFIC.get(key)
    if entry is None:
        return None
    m = hashlib.sha256()
    try:
        for name in entry["sources"]:
            with open(os.path.join(_KDIR, name), "rb") as f:
                m.update(f.read())
    except OSError:
        return None
    return entry["bytes"] if m.hexdigest()[:16] == entry["sha"] else None


FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        # One process per GPU over NCCL; gloo on a host without GPUs (the
        # host-side logic of the replicas: barrier and max over ranks).
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

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
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def prefill_alg_bytes(w):
    """q, k, v, g, beta, y once each, plus the state in and out (fp32)."""
    eb = 4 if w.dtype == "f32" else 2
    tok = w.B * w.T
    return (tok * w.Hk * w.Dk * 2 * eb + tok * w.Hv * w.Dv * 2 * eb
            + tok * w.Hv * 2 * eb + 2 * w.B * w.Hv * w.Dv * w.Dk * 4)


def prefill_alg_flops(w):
    """6 D^2 + 8 C D per token per value head (chunk form, full C x C grams)."""
    D = w.Dk
    return w.B * w.T * w.Hv * (6 * D * D + 8 * w.chunk * D)


def decode_alg_bytes(w):
    eb = 4 if w.dtype == "f32" else 2
    return (2 * w.B * w.Hv * w.Dv * w.Dk * 4 + w.B * w.Hk * w.Dk * 2 * eb
            + w.B * w.Hv * w.Dv * 2 * eb + w.B * w.Hv * 2 * eb)


def roofline(alg_bytes, seconds, hbm_gbs, kind, traffic=None):
    achieved = alg_bytes / seconds / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_gbs,
            "unit": "GB/s", "frac": round(achieved / hbm_gbs, 4),
            "traffic": None if traffic is None else round(traffic),
            "algorithmic_bytes": alg_bytes, "peak_kind": kind}


def prefill_launches(w, dev):
    """Kernels one gdn_prefill call launches: T <= 32 one (a short-T
    kernel); bf16 or fp16 with 128-wide heads runs prep and scan as
    one cooperative kernel when B*Hv is at most a third of the SMs, else as
    two; the fp32 chunked path always two."""
    if w.T <= 32:
        return 1
    if w.dtype == "f32" or w.Dk != 128 or w.Dv != 128:
        return 2
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return 1 if 3 * w.B * w.Hv <= sms else 2


def event_ms(pairs):
    """Elapsed milliseconds of each (start, end) CUDA event pair."""
    return [a.elapsed_time(b) for a, b in pairs]


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def bench_prefill(gdn, w, dev, steps, warmup, world):
    """Median CUDA-event time (ms) of one gdn_prefill call over ``steps``
    timed calls, each preceded (outside the events) by a 256 MiB L2 flush."""
    ins = {n: t.to(dev) for n, t in gdn_inputs.workload_inputs(w).items()}
    y = torch.empty((w.B, w.T, w.Hv, w.Dv), dtype=w.torch_dtype, device=dev)
    s_out = torch.empty((w.B, w.Hv, w.Dv, w.Dk), dtype=torch.float32, device=dev)
    nbytes = gdn.gdn_prefill_workspace_bytes(w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv,
                                             w.chunk, w.torch_dtype)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        gdn.gdn_prefill(ins["q"], ins["k"], ins["v"], ins["g"], ins["beta"], ins["s0"],
                        s_out, y, w.chunk, workspace=ws, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    pairs = []
    t0 = time.perf_counter()
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - t0
    times = event_ms(pairs)
    return statistics.median(times), wall


def bench_prefill_e2e(gdn, w, dev, steps, warmup):
    """Through the C ABI from pinned host buffers: every step copies its inputs
    host -> device, runs gdn_prefill and copies y and the final state back, and
    the host waits for that result.  Measured two ways: one step at a time on
    one stream (``serial_ms_per_step``), and pipelined two steps deep on three
    streams (copies in, compute, copies out; double-buffered device and host
    buffers), the way a serving loop runs: step i + 1's inputs travel while step
    i computes and step i - 1's outputs come back.  ``value`` is the pipelined
    throughput."""
    host = {n: t.pin_memory() for n, t in gdn_inputs.workload_inputs(w).items()}
    dvs = [{n: torch.empty_like(t, device=dev) for n, t in host.items()} for _ in range(2)]
    ys = [torch.empty((w.B, w.T, w.Hv, w.Dv), dtype=w.torch_dtype, device=dev) for _ in range(2)]
    ss = [torch.empty((w.B, w.Hv, w.Dv, w.Dk), dtype=torch.float32, device=dev)
          for _ in range(2)]
    y_hs = [torch.empty(ys[0].shape, dtype=ys[0].dtype).pin_memory() for _ in range(2)]
    s_hs = [torch.empty(ss[0].shape, dtype=ss[0].dtype).pin_memory() for _ in range(2)]
    nbytes = gdn.gdn_prefill_workspace_bytes(w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv,
                                             w.chunk, w.torch_dtype)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = ys[0].numel() * ys[0].element_size() + ss[0].numel() * 4

    main = torch.cuda.current_stream(dev)

    def serial_step():
        dv, y, s_out = dvs[0], ys[0], ss[0]
        for n in host:
            dv[n].copy_(host[n], non_blocking=True)
        gdn.gdn_prefill(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["s0"], s_out,
                        y, w.chunk, workspace=ws, stream=main)
        y_hs[0].copy_(y, non_blocking=True)
        s_hs[0].copy_(s_out, non_blocking=True)
        torch.cuda.synchronize(dev)   # the host reads the step's result

    for _ in range(warmup):
        serial_step()
    t0 = time.perf_counter()
    for _ in range(steps):
        serial_step()
    serial = (time.perf_counter() - t0) / steps

    s_in, s_comp, s_out_st = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
    for j in range(2):   # every buffer starts free
        for k in ("comp", "out"):
            ev[k][j].record(main)

    def issue(i):
        j = i % 2
        dv, y, s_out = dvs[j], ys[j], ss[j]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev["comp"][j])          # step i - 2 has read these inputs
            for n in host:
                dv[n].copy_(host[n], non_blocking=True)
            ev["in"][j].record(s_in)
        s_comp.wait_event(ev["in"][j])
        s_comp.wait_event(ev["out"][j])             # step i - 2's outputs are copied out
        gdn.gdn_prefill(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["s0"], s_out,
                        y, w.chunk, workspace=ws, stream=s_comp)
        ev["comp"][j].record(s_comp)
        with torch.cuda.stream(s_out_st):
            s_out_st.wait_event(ev["comp"][j])
            y_hs[j].copy_(y, non_blocking=True)
            s_hs[j].copy_(s_out, non_blocking=True)
            ev["out"][j].record(s_out_st)

    def run(n):
        for i in range(n):
            issue(i)
            if i >= 1:
                ev["out"][(i - 1) % 2].synchronize()   # the host reads step i - 1's result
        ev["out"][(n - 1) % 2].synchronize()

    run(max(warmup, 2))
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    run(steps)
    sec = (time.perf_counter() - t0) / steps
    torch.cuda.synchronize(dev)
    return {"value": round(w.B * w.T / sec, 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(sec * 1e3, 4), "serial_ms_per_step": round(serial * 1e3, 4),
            "timing": "host wall clock; steps pipelined two deep on three streams (copies in, "
                      "compute, copies out), each step's copies inside the timed region"}


def bench_decode(gdn, w, dev, replays=5):
    """256 successive decode steps captured in one CUDA graph (state in place);
    the state (134 MB) is larger than the L2.  Before each timed replay the
    state is reset from a saved copy and the L2 is then flushed (256 MiB
    write), so no part of the state starts warm; the median replay is taken.
    Returns (us per step, cold), (us per step without the flush, warm)."""
    steps = w.steps
    s = gdn_inputs.workload_inputs(w, step=0)["s0"].to(dev)
    step_in = []
    for i in range(steps):
        ins = gdn_inputs.workload_inputs(w, step=i)
        step_in.append({n: ins[n].to(dev) for n in ("q", "k", "v", "g", "beta")})
    ys = torch.empty((steps, w.B, 1, w.Hv, w.Dv), dtype=w.torch_dtype, device=dev)
    side = torch.cuda.Stream(dev)
    s_work = s.clone()

    def run_all(stream):
        for i in range(steps):
            d = step_in[i]
            gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], s_work, s_work,
                                ys[i], stream=stream)

    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        run_all(side)          # warm-up outside capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run_all(side)
    torch.cuda.synchronize(dev)
    graph.replay()
    torch.cuda.synchronize(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed(cold):
        times = []
        for _ in range(replays):
            s_work.copy_(s)
            if cold:
                flush.zero_()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        return statistics.median(times) * 1e3 / steps

    return timed(True), timed(False)


def oracle_sample(w, n_kh):
    """The workload's first ``n_kh`` key heads and their value heads (every
    token, every batch row) as a stand-alone problem for the oracle."""
    ins = gdn_inputs.workload_inputs(w)
    grp = w.Hv // w.Hk
    n_kh = max(1, min(n_kh, w.Hk))
    hv = n_kh * grp
    sub = {"q": ins["q"][:, :, :n_kh], "k": ins["k"][:, :, :n_kh],
           "v": ins["v"][:, :, :hv], "g": ins["g"][:, :, :hv],
           "beta": ins["beta"][:, :, :hv], "s0": ins["s0"][:, :hv]}
    return {n: t.contiguous() for n, t in sub.items()}, hv


def time_oracle(sub, reps=1):
    import oracle
    names = ("q", "k", "v", "g", "beta")
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.gdn_sequential(*(sub[n] for n in names), sub["s0"])
    return (time.perf_counter() - t0) / reps


def oracle_threads(work_items):
    import oracle
    return max(1, min(oracle.num_threads(), work_items))


def cpu_baseline_prefill(w, min_seconds=10.0, max_reps=50):
    """The fp64 oracle, as it stands, on the host cores over the whole
    workload (every head, every token), repeated until about ten seconds of
    CPU work have been timed."""
    sub, hv = oracle_sample(w, w.Hk)
    time_oracle(sub)                       # first call builds / loads the oracle
    reps, total = 0, 0.0
    while total < min_seconds and reps < max_reps:
        total += time_oracle(sub)
        reps += 1
    dt = total / reps
    value = w.B * w.T * hv / w.Hv / dt
    return {"value": round(value, 2), "unit": "tokens/s",
            "cores": oracle_threads(w.B * hv), "kind": "oracle",
            "sample": f"the whole workload ({hv} value heads x B={w.B} x T={w.T}), fp64, "
                      f"{reps} runs, {total:.1f} s"}


def cpu_chunked_fp32(w, n_heads=2, chunk=32):
    """The fp32 host chunked form (the oracle package's Woodbury-Young form in
    float32, chunk 32: the host comparison of ferrox-core ``gdn_chunk.rs``),
    timed on ``n_heads`` value heads of the workload in a child process pinned
    to one BLAS/OpenMP thread, scaled to tokens/s of the whole workload."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
               MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-chunked-sample", w.name,
           "--sample-heads", str(n_heads), "--sample-chunk", str(chunk)]
    try:
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600,
                             check=True).stdout.strip().splitlines()[-1]
        sec, hv = json.loads(out)
    except (subprocess.SubprocessError, ValueError, IndexError, OSError) as e:
        return {"unavailable": f"{type(e).__name__}"}
    value = w.B * w.T * hv / w.Hv / sec
    return {"value": round(value, 2), "unit": "tokens/s", "cores": 1,
            "kind": "fp32 host chunked form (oracle package, chunk 32)",
            "sample": f"{hv} of {w.Hv} value heads x B={w.B} x T={w.T}, fp32, {sec:.1f} s; "
                      f"tokens/s scaled by {hv}/{w.Hv}"}


def _cpu_chunked_sample_main(name, n_heads, chunk):
    import numpy as np

    from oracle import forms
    w = gdn_inputs.WORKLOADS[name]
    grp = w.Hv // w.Hk
    sub, hv = oracle_sample(w, -(-n_heads // grp))
    t0 = time.perf_counter()
    forms.chunked_wy(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], sub["s0"],
                     chunk=chunk, dtype=np.float32)
    print(json.dumps([time.perf_counter() - t0, hv]), flush=True)
    return 0


def workload_config(w, world):
    """The ``config`` object of a line, identical on both arms."""
    return {"workload": w.name, "B": w.B, "T": w.T, "Hk": w.Hk, "Hv": w.Hv,
            "Dk": w.Dk, "Dv": w.Dv, "chunk": w.chunk, "input_dtype": w.dtype,
            "state": "fp32", "l2": "256 MiB flush write between timed steps",
            "parallelism": f"replicas x{world}"}


# ----------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ----------------------------------------------------------------------------
def run_reference(args, w):
    world, rank, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    grp = w.Hv // w.Hk
    sub, hv = oracle_sample(w, -(-cores // grp))
    for _ in range(args.warmup):
        time_oracle(sub)
    sec = time_oracle(sub, reps=args.steps)
    value = w.B * w.T * hv / w.Hv / sec
    sample = (f"{hv} of {w.Hv} value heads x B={w.B} x T={w.T} (every token) per step, "
              f"fp64; tokens/s scaled by {hv}/{w.Hv}")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2),
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.gpus),
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                         "cores": oracle_threads(w.B * hv), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = "GDN prefill tokens/s (B=1 T=4096 Hk=16 Hv=32 D=128 bf16 C=64) and decode steps/s"

# The other prefill workloads of the plan, timed after the headline one.
EXTRA_PREFILL = ["fp32_t64", "prefill_b4_t2048", "prefill_t65536", "prefill_b64_t16",
                 "prefill_t4096_f16", "prefill_t4096_d64", "prefill_t4096_d256"]


def prefill_entry(gdn, w, dev, steps, warmup, hbm, peak_kind, world):
    ms, _ = bench_prefill(gdn, w, dev, steps, warmup, world)
    ms = max_over_ranks(ms, world)
    r = roofline(prefill_alg_bytes(w), ms / 1e3, hbm, peak_kind, measured_traffic(w.name))
    r["scope"] = "whole gdn_prefill call (all its kernels)"
    r["tensor_tflops"] = round(prefill_alg_flops(w) / (ms / 1e3) / 1e12, 2)
    return {"ms_per_step": round(ms, 4), "steps": steps,
            "tokens_per_s": round(world * w.B * w.T / (ms / 1e3), 1),
            "launches_per_step": prefill_launches(w, dev), "dtype": w.dtype,
            "config": workload_config(w, world), "roofline": r}


def decode_entry(gdn, dev, hbm, peak_kind):
    dw = gdn_inputs.WORKLOADS["decode_b64"]
    us, us_warm = bench_decode(gdn, dw, dev)
    return {
        "workload": dw.name, "steps_per_s": round(1e6 / us, 1),
        "tokens_per_s": round(dw.B * 1e6 / us, 1), "us_per_step": round(us, 3),
        "us_per_step_warm_l2": round(us_warm, 3), "launches_per_step": 1,
        "timing": "256 steps in one CUDA graph, state in place (134 MB > L2); median of 5 "
                  "replays, each after a state reset and a 256 MiB L2 flush",
        "roofline": roofline(decode_alg_bytes(dw), us / 1e6, hbm, peak_kind,
                             measured_traffic("decode_b64"))}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill_t4096")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads, decode, e2e and cpu_baseline")
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode"],
                    help="profiling runs: time one path only (prints a partial line)")
    ap.add_argument("--cpu-chunked-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--sample-heads", type=int, default=2, help=argparse.SUPPRESS)
    ap.add_argument("--sample-chunk", type=int, default=32, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_chunked_sample:
        return _cpu_chunked_sample_main(args.cpu_chunked_sample, args.sample_heads,
                                        args.sample_chunk)
    args.warmup = max(args.warmup, 3)
    w = gdn_inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    import gated_delta_rule_02_gb300 as gdn
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gdn.lib()
    hbm, bf16, peak_kind = load_peaks()
    if args.only == "decode":
        d = decode_entry(gdn, dev, hbm, peak_kind)
        d["partial"] = "decode only"
        print(json.dumps(d), flush=True)
        return 0
    if args.only == "prefill":
        args.no_extras = True

    sampler = ClockSampler(local)
    sampler.start()
    ms, wall = bench_prefill(gdn, w, dev, args.steps, args.warmup, world)
    clocks = sampler.stop()
    ms = max_over_ranks(ms, world)
    tokens_per_s = world * w.B * w.T / (ms / 1e3)

    line = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, world),
        "roofline": roofline(prefill_alg_bytes(w), ms / 1e3, hbm, peak_kind,
                             measured_traffic(w.name)),
        "gpu_launches": prefill_launches(w, dev) * args.steps,
        "clocks": clocks,
    }
    line["roofline"]["scope"] = "whole gdn_prefill call (all its kernels)"
    line["roofline"]["tensor_tflops"] = round(prefill_alg_flops(w) / (ms / 1e3) / 1e12, 2)
    line["timing"] = "median of the timed steps (CUDA events on the launching stream)"

    if not args.no_extras:
        if rank == 0 or world > 1:
            line["e2e"] = bench_prefill_e2e(gdn, w, dev, max(10, args.steps // 2), 3)
        workloads = {}
        for name in EXTRA_PREFILL:
            ew = gdn_inputs.WORKLOADS[name]
            if ew.name == w.name:
                continue
            workloads[name] = prefill_entry(gdn, ew, dev, 20, 3, hbm, peak_kind, world)
        workloads["decode_b64"] = decode_entry(gdn, dev, hbm, peak_kind)
        line["workloads"] = workloads
        line["decode"] = workloads["decode_b64"]
        if rank == 0 and world == 1:
            line["cpu_baseline"] = cpu_baseline_prefill(w)
            line["cpu_baseline"]["chunked_fp32"] = cpu_chunked_fp32(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
