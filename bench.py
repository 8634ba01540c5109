#!/usr/bin/env python3
"""Benchmark of the MoE decode layer on one GB300 (or N independent replicas).

Workload (the metric's cache-defeating configuration): a stack of 48 MoE
layers with the Qwen-3-style shapes H=2048, I=768, E=128, K=8, each layer with
its own seeded MXFP8 weights (604 MB per layer, 29 GB in all, far above L2);
the BF16 output of layer l is the input of layer l+1; router outputs are the
seeded top-8 of N(0,1) logits per layer.  One step = one token-step of B
tokens through all 48 layers (96 kernel launches, replayed as a CUDA graph).

Reported metric: achieved HBM GB/s = exact algorithmic bytes of the step
(each distinct routed expert's weights and scales once per layer, plus x, the
intermediate h written and read, out, ids and weights) / step time; also
us/layer and the fraction of the copy-kernel bandwidth this bench measures
itself.  The headline line is B=32; the sweep B in {1,2,4,8,16,32} rides along.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = synth.WORKLOADS["qwen3_stack48"]
METRIC = "MoE decode layer HBM GB/s and us/layer at B=1-32, % of measured copy peak"
UNIT = "GB/s"
HEADLINE_B = 32
SWEEP_B = (1, 2, 4, 8, 16, 32)


# ------------------------------------------------------------------ helpers --

def algorithmic_bytes(ids_layers, B, H, I, E, K):
    """Exact bytes one step must move: per layer, every distinct routed expert's
    codes + scales once, x read, h written and read, out written, ids + w read."""
    per_layer_act = 2 * B * H + 2 * 2 * B * K * I + 2 * B * H + 8 * B * K
    wbytes = sum(synth.unique_expert_bytes(ids, E, H, I) for ids in ids_layers)
    return wbytes + per_layer_act * len(ids_layers)


def gate_up_bytes(ids, B, H, I, E, K):
    uniq = np.unique(ids[(ids >= 0) & (ids < E)]).size
    return uniq * (2 * I * H + 2 * I * H // 32) + 2 * B * H + 2 * B * K * I + 4 * B * K


def down_bytes(ids, B, H, I, E, K):
    uniq = np.unique(ids[(ids >= 0) & (ids < E)]).size
    return uniq * (H * I + H * I // 32) + 2 * B * K * I + 2 * B * H + 8 * B * K


def read_peaks_file():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_sources_sha():
    """sha256 prefix of the device-code sources (the C-ABI's host code and the
    bench's own copy/read kernels are left out)."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(os.path.join(ROOT, "moe_decode_gate_gb300", "csrc"))):
        if not f.endswith((".cu", ".cuh", ".h")) or f in ("wd_capi.cu", "wd_bench.cu"):
            continue
        with open(os.path.join(ROOT, "moe_decode_gate_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(kernel):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("sources_sha") != kernel_sources_sha():
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch_full")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- the GPU stack --

class Stack:
    """48 layers of device-resident MXFP8 weights plus per-B routing and buffers."""

    def __init__(self, torch, wd, dev, layers, max_batch, log):
        self.torch, self.wd, self.dev = torch, wd, dev
        wl = WORKLOAD
        self.H, self.I, self.E, self.K = wl.H, wl.I, wl.E, wl.K
        self.L = layers
        t0 = time.time()
        gu = np.empty((self.E, 2 * self.I, self.H), np.uint8)
        gus = np.empty((self.E, 2 * self.I, self.H // 32), np.uint8)
        dn = np.empty((self.E, self.H, self.I), np.uint8)
        dns = np.empty((self.E, self.H, self.I // 32), np.uint8)
        self.weights = []
        for l in range(layers):
            synth.gate_up(wl.seed, l, self.E, self.H, self.I, out=(gu, gus))
            synth.down(wl.seed, l, self.E, self.H, self.I, out=(dn, dns))
            self.weights.append(tuple(torch.from_numpy(a).to(dev) for a in (gu, gus, dn, dns)))
        torch.cuda.synchronize(dev)
        self.gen_seconds = time.time() - t0
        log(f"generated and uploaded {layers} layers in {self.gen_seconds:.1f} s")
        self.workspace = torch.empty(wd.wd_moe_workspace_size(max_batch, self.K, self.I),
                                     dtype=torch.uint8, device=dev)
        wd.wd_moe_workspace_init(self.workspace)

    def routing(self, B):
        wl = WORKLOAD
        ids, ws = [], []
        for l in range(self.L):
            i, w = synth.route(wl.seed, l, B, self.E, self.K)
            ids.append(i)
            ws.append(w)
        return np.stack(ids), np.stack(ws)

    def buffers(self, B):
        torch = self.torch
        ids, ws = self.routing(B)
        xs = synth.x(WORKLOAD.seed, 0, B, self.H)
        d = dict(B=B, ids_host=ids, w_host=ws, x_host=xs)
        d["ids"] = torch.from_numpy(ids).to(self.dev)
        d["w"] = torch.from_numpy(ws).to(self.dev)
        d["x0"] = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(self.dev)
        d["act"] = [torch.empty((B, self.H), dtype=torch.bfloat16, device=self.dev) for _ in range(2)]
        return d

    def layer_io(self, buf, l):
        x = buf["x0"] if l == 0 else buf["act"][(l - 1) % 2]
        return x, buf["act"][l % 2]

    def enqueue_step(self, buf, stream=None):
        wd = self.wd
        for l in range(self.L):
            gu, gus, dn, dns = self.weights[l]
            x, out = self.layer_io(buf, l)
            wd.wd_moe_decode(x, buf["ids"][l], buf["w"][l], gu, gus, dn, dns, out, self.workspace,
                             stream=stream)
        return buf["act"][(self.L - 1) % 2]

    def graph(self, buf):
        torch = self.torch
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            self.enqueue_step(buf, stream=s)  # warm the launch path outside capture
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.enqueue_step(buf, stream=s)
        return g, s


def time_graph(torch, dev, g, s, steps, warmup, barrier):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize(dev)
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        start.record(s)
        for _ in range(steps):
            g.replay()
        stop.record(s)
    torch.cuda.synchronize(dev)
    barrier()
    return start.elapsed_time(stop) / steps  # ms per step


def time_kernels_alone(torch, wd, dev, stack, buf, steps):
    """Per-launch device time of each kernel on its own (no overlap), events on
    the launching stream around every launch; weights are cold (48 layers)."""
    B, K, I, H = buf["B"], stack.K, stack.I, stack.H
    s = torch.cuda.Stream(device=dev)
    h = torch.empty((B, K, I), dtype=torch.bfloat16, device=dev)
    out = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
    n = stack.L * steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(2 * n)]
    x = buf["x0"]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(s):
        i = 0
        for _ in range(steps):
            for l in range(stack.L):
                gu, gus, dn, dns = stack.weights[l]
                a, b = ev[i]
                a.record(s)
                wd.wd_moe_gate_up(x, buf["ids"][l], gu, gus, h, stream=s)
                b.record(s)
                a, b = ev[i + 1]
                a.record(s)
                wd.wd_moe_down(h, buf["ids"][l], buf["w"][l], dn, dns, out, stream=s)
                b.record(s)
                i += 2
    torch.cuda.synchronize(dev)
    t_gu = [ev[2 * j][0].elapsed_time(ev[2 * j][1]) for j in range(n)]
    t_dn = [ev[2 * j + 1][0].elapsed_time(ev[2 * j + 1][1]) for j in range(n)]
    b_gu = [gate_up_bytes(buf["ids_host"][l], B, H, I, stack.E, K) for l in range(stack.L)] * steps
    b_dn = [down_bytes(buf["ids_host"][l], B, H, I, stack.E, K) for l in range(stack.L)] * steps
    return dict(gate_up_ms=float(np.mean(t_gu)), down_ms=float(np.mean(t_dn)),
                gate_up_bytes=float(np.mean(b_gu)), down_bytes=float(np.mean(b_dn)), launches=2 * n)


def measure_copy_peak(torch, wd, dev, reps=10):
    n = 2 << 30
    src = torch.empty(n, dtype=torch.uint8, device=dev)
    dst = torch.empty(n, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    wd.wd_bench_fill(src, 0x01020304)
    best_copy = best_read = 0.0
    for _ in range(reps):
        for kind in ("copy", "read"):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            if kind == "copy":
                wd.wd_bench_copy(dst, src)
            else:
                wd.wd_bench_read(src, sink)
            b.record()
            torch.cuda.synchronize(dev)
            ms = a.elapsed_time(b)
            if kind == "copy":
                best_copy = max(best_copy, 2 * n / ms / 1e6)
            else:
                best_read = max(best_read, n / ms / 1e6)
    del src, dst
    spec = wd.wd_bench_spec_gbs()
    return dict(copy_gbs=round(best_copy, 1), read_gbs=round(best_read, 1),
                spec_gbs=round(spec, 1) if spec > 0 else None)


def e2e_pass(torch, wd, dev, stack, buf, steps, warmup, barrier):
    """The same step through the public API with host buffers: every step copies
    x and all 48 layers' routing from pinned host memory to the device, runs
    the 48 wd_moe_decode calls and reads the result back."""
    B = buf["B"]
    x_h = torch.from_numpy(buf["x_host"].view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_h = torch.from_numpy(buf["ids_host"]).pin_memory()
    w_h = torch.from_numpy(buf["w_host"]).pin_memory()
    out_h = torch.empty((B, stack.H), dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.Stream(device=dev)

    def step():
        buf["x0"].copy_(x_h, non_blocking=True)
        buf["ids"].copy_(ids_h, non_blocking=True)
        buf["w"].copy_(w_h, non_blocking=True)
        out = stack.enqueue_step(buf, stream=s)
        out_h.copy_(out, non_blocking=True)

    with torch.cuda.stream(s):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(steps):
            step()
        b.record(s)
    torch.cuda.synchronize(dev)
    barrier()
    h2d = x_h.numel() * 2 + ids_h.numel() * 4 + w_h.numel() * 4
    return a.elapsed_time(b) / steps, h2d, out_h.numel() * 2


# ------------------------------------------------------------- CPU oracle --

_SAMPLE_CACHE = {}


def _sample_layer(l, tokens, B):
    """Routing and the routed experts' weights of layer l for the first `tokens`
    tokens (untimed; only the routed experts are generated)."""
    key = (l, tokens, B)
    if key not in _SAMPLE_CACHE:
        wl = WORKLOAD
        H, I, E, K = wl.H, wl.I, wl.E, wl.K
        ids, w = synth.route(wl.seed, l, B, E, K)
        ids, w = ids[:tokens], w[:tokens]
        gu = np.zeros((E, 2 * I, H), np.uint8)
        gus = np.zeros((E, 2 * I, H // 32), np.uint8)
        dn = np.zeros((E, H, I), np.uint8)
        dns = np.zeros((E, H, I // 32), np.uint8)
        for e in np.unique(ids):
            synth.gate_up(wl.seed, l, E, H, I, experts=(int(e), int(e) + 1), out=(gu, gus))
            synth.down(wl.seed, l, E, H, I, experts=(int(e), int(e) + 1), out=(dn, dns))
        _SAMPLE_CACHE.clear()
        _SAMPLE_CACHE[key] = (ids, w, gu, gus, dn, dns)
    return _SAMPLE_CACHE[key]


def oracle_sample(layers, tokens, B=HEADLINE_B):
    """Time the CPU oracle (as it stands, one thread) on `tokens` tokens of the
    stack's first `layers` layers at batch B; returns (seconds, bytes)."""
    import oracle

    wl = WORKLOAD
    H, I, E, K = wl.H, wl.I, wl.E, wl.K
    xs = synth.x(wl.seed, 0, B, H)[:tokens]
    secs, nbytes = 0.0, 0
    for l in range(layers):
        ids, w, gu, gus, dn, dns = _sample_layer(l, tokens, B)
        t0 = time.perf_counter()
        xs = oracle.moe_decode(xs, ids, w, gu, gus, dn, dns, I, E)
        secs += time.perf_counter() - t0
        nbytes += algorithmic_bytes([ids], tokens, H, I, E, K)
    return secs, nbytes


def run_reference(args, rank):
    """The oracle as the reference arm: same metric, unit and workload; each
    step is a bounded sample of the stack (token-layers) on one host core."""
    if rank != 0:
        return
    budget = float(os.environ.get("WD_REFERENCE_BUDGET_S", "150"))
    per_tl = 0.08  # approximate seconds per token-layer of the oracle
    tokens = max(1, min(HEADLINE_B, int(budget / (args.steps + args.warmup) / per_tl)))
    for _ in range(args.warmup):
        oracle_sample(1, tokens)
    secs, nbytes = 0.0, 0
    for _ in range(args.steps):
        s, b = oracle_sample(1, tokens)
        secs += s
        nbytes += b
    value = nbytes / secs / 1e9
    sample = f"layer 0 of the 48-layer stack, first {tokens} of {HEADLINE_B} tokens per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(HEADLINE_B),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(B):
    wl = WORKLOAD
    return {"workload": f"{wl.name}: 48 MoE layers, own MXFP8 weights each (29.2 GB), "
                        f"H={wl.H} I={wl.I} E={wl.E} K={wl.K}, B={B}, out of layer l feeds layer l+1",
            "global_batch": B, "layers": wl.layers, "H": wl.H, "I": wl.I, "E": wl.E, "K": wl.K,
            "weights": "MXFP8 (E4M3 + E8M0 per 32)", "activations": "BF16",
            "l2": "no flush: the 29.2 GB of weights cycle through a 126 MB L2 every step",
            "parallelism": "replicas"}


class RankOps:
    """Reductions over the bench's ranks (one process per GPU, replicas): a
    barrier, the max of a per-rank time and the sum of per-rank bytes.  With
    no process group (one GPU) they return the local value."""

    def __init__(self, torch, dist, device):
        self.torch, self.dist, self.device = torch, dist, device

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def _reduce(self, v, op):
        if self.dist is None:
            return v
        t = self.torch.tensor([v], dtype=self.torch.float64, device=self.device)
        self.dist.all_reduce(t, op=op)
        return float(t.item())

    def max(self, v):
        return self._reduce(v, None if self.dist is None else self.dist.ReduceOp.MAX)

    def sum(self, v):
        return self._reduce(v, None if self.dist is None else self.dist.ReduceOp.SUM)


def aggregate_gbps(local_bytes, local_ms, ranks):
    """Whole-job GB/s of N replicas: all ranks' bytes over the slowest rank's time."""
    return ranks.sum(float(local_bytes)) / ranks.max(local_ms) / 1e6


# ------------------------------------------------------------------- main --

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="wd", choices=["wd", "reference"])
    ap.add_argument("--layers", type=int, default=WORKLOAD.layers,
                    help="fewer layers for profiling runs (not a bench value)")
    ap.add_argument("--sweep", default=",".join(map(str, SWEEP_B)))
    ap.add_argument("--sweep-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="headline only (profiling runs)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3 and not args.quick:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch

    import moe_decode_gate_gb300 as wd

    def log(msg):
        if rank == 0:
            print(f"[bench] {msg}", file=sys.stderr, flush=True)

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    ranks = RankOps(torch, dist, dev)
    barrier, max_over_ranks, sum_over_ranks = ranks.barrier, ranks.max, ranks.sum

    peaks_file, peaks_kind = read_peaks_file()
    if args.quick:  # profiling runs keep the device footprint small
        peaks = dict(copy_gbs=float(peaks_file["hbm_gbs"]), read_gbs=None, spec_gbs=None)
    else:
        peaks = measure_copy_peak(torch, wd, dev)
        torch.cuda.empty_cache()
    log(f"copy peak {peaks['copy_gbs']} GB/s, read peak {peaks['read_gbs']} GB/s")

    sweep = [int(b) for b in args.sweep.split(",") if b] if not args.quick else []
    max_b = max([HEADLINE_B] + sweep)
    stack = Stack(torch, wd, dev, args.layers, max_b, log)
    H, I, E, K = stack.H, stack.I, stack.E, stack.K

    # ---- sweep over B (each B: its own routing and graph) ----
    sweep_rows = []
    for B in sweep:
        if B == HEADLINE_B:
            continue
        buf = stack.buffers(B)
        g, s = stack.graph(buf)
        ms = max_over_ranks(time_graph(torch, dev, g, s, args.sweep_steps, 3, barrier))
        nb = algorithmic_bytes(buf["ids_host"], B, H, I, E, K)
        sweep_rows.append({"B": B, "us_per_layer": round(ms * 1e3 / stack.L, 2),
                           "GBps": round(nb / ms / 1e6, 1),
                           "frac_copy_peak": round(nb / ms / 1e6 / peaks["copy_gbs"], 4),
                           "unique_MB_per_layer": round(nb / stack.L / 1e6, 2)})
        del g
        log(f"B={B}: {sweep_rows[-1]}")

    # ---- headline: B=32, graph replay, clocks sampled ----
    B = HEADLINE_B
    buf = stack.buffers(B)
    g, s = stack.graph(buf)
    nb = algorithmic_bytes(buf["ids_host"], B, H, I, E, K)
    with ClockSampler(local) as clocks:
        ms_local = time_graph(torch, dev, g, s, args.steps, args.warmup, barrier)
    ms = max_over_ranks(ms_local)
    total_bytes = sum_over_ranks(float(nb))
    value = aggregate_gbps(nb, ms_local, ranks)  # all ranks' bytes / the slowest rank's time
    per_rank_gbs = nb / ms / 1e6
    sweep_rows.append({"B": B, "us_per_layer": round(ms * 1e3 / stack.L, 2),
                       "GBps": round(per_rank_gbs, 1),
                       "frac_copy_peak": round(per_rank_gbs / peaks["copy_gbs"], 4),
                       "unique_MB_per_layer": round(nb / stack.L / 1e6, 2)})
    sweep_rows.sort(key=lambda r: r["B"])
    log(f"B=32 headline: {ms:.3f} ms/step, {per_rank_gbs:.1f} GB/s per GPU")

    # ---- roofline of the dominant kernel (each kernel timed alone, cold) ----
    kt = time_kernels_alone(torch, wd, dev, stack, buf, steps=max(2, min(10, args.steps // 20)))
    gu_gbs = kt["gate_up_bytes"] / kt["gate_up_ms"] / 1e6
    dn_gbs = kt["down_bytes"] / kt["down_ms"] / 1e6
    hbm_peak = float(peaks_file["hbm_gbs"])
    # the kernels the plan launches at this shape, e.g. "gate_up=moe_gate_up_persist<2,1> down=..."
    plan = dict(kv.split("=", 1) for kv in wd.wd_moe_describe_plan(B, H, I, E, K).split())
    gu_name, dn_name = plan["gate_up"], plan["down"]
    traffic = profile_traffic(gu_name.split("<")[0])
    roofline = {"kernel": gu_name, "bound": "hbm", "achieved": round(gu_gbs, 1),
                "peak": hbm_peak, "unit": "GB/s", "frac": round(gu_gbs / hbm_peak, 4),
                "traffic": traffic, "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peaks_kind})",
                "algorithmic_bytes_per_launch": round(kt["gate_up_bytes"]),
                "us_per_launch": round(kt["gate_up_ms"] * 1e3, 2),
                "second_kernel": {"kernel": dn_name, "achieved": round(dn_gbs, 1),
                                  "frac": round(dn_gbs / hbm_peak, 4),
                                  "algorithmic_bytes_per_launch": round(kt["down_bytes"]),
                                  "us_per_launch": round(kt["down_ms"] * 1e3, 2),
                                  "traffic": profile_traffic(dn_name.split("<")[0])}}

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.quick:
        e2e_steps = max(5, args.steps // 4)
        e2e_ms, h2d, d2h = e2e_pass(torch, wd, dev, stack, buf, e2e_steps, 3, barrier)
        e2e_ms = max_over_ranks(e2e_ms)
        e2e = {"value": round(total_bytes / e2e_ms / 1e6, 1), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
               "how": "pinned H2D of x and all layers' ids/w, one wd_moe_decode call per layer "
                      "(no graph), D2H of out, events on the launching stream"}

    # ---- CPU oracle on a bounded sample (rank 0) ----
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not args.quick:
        secs, sb = oracle_sample(layers=1, tokens=B)
        cpu = {"value": round(sb / secs / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"layer 0 of the stack, all {B} tokens ({secs:.1f} s, FP64 C, one thread)"}

    launches = args.steps * stack.L * wd.wd_moe_launches_per_call()
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded Philox; Qwen-3-style shapes, random-init MXFP8 weights)",
            "config": config_dict(B),
            "us_per_layer": round(ms * 1e3 / stack.L, 3),
            "frac_copy_peak": round(per_rank_gbs / peaks["copy_gbs"], 4),
            "peaks": {**peaks, "measured_peaks_json_hbm_gbs": hbm_peak},
            "sweep": sweep_rows, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks.summary(),
            "context": {"pages_b200": "3.95 TB/s at B=32 = 58% of a 6.8 TB/s copy peak (B200)"}}
    if args.quick or args.layers != WORKLOAD.layers:
        line["note"] = "profiling run: not a bench value"
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
