"""Benchmark of the causal Polar Attention hot path on GB300.

One step runs, inputs resident in HBM:
  * the headline prefill keyscale_16k (B2 H16 T16384 d128 bf16) and the
    split-KV decode decode_32k (B32 H16 Tkv32768 d128 bf16);
  * paged grouped-query decodes with 2, 4 and 8 query heads per KV head
    (paged_gqa2_32k, paged_gqa_32k, paged_gqa8_32k: B32, 16 query heads,
    32768 tokens in 64-token pages);
  * one in-place gated-delta memory step (memstep_256).
The other three configurations -- tiny_f32 (B1 H2 T256 d64 fp32),
needles_4k (B1 H8 T4096 d64 bf16) and needles_64k (B1 H16 T65536 d128
bf16) -- and the backward of keyscale_16k from the forward's saved row
statistics (backward_16k) are timed right after the step, each over as many
calls.
`value` is keyscale_16k's algorithmic TFLOP/s (causal pairs only: 4 d n(n+1)/2
flop per head); every workload's time, TFLOP/s, tokens/s, GB/s and roofline
fraction is reported under `configs`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own replica (independent problems, no
collective on the data path): weak scaling, value summed over ranks.
--impl reference times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PREFILL = "keyscale_16k"
DECODE = "decode_32k"
PAGED = "paged_gqa_32k"
MEMSTEP = "memstep_256"
BACKWARD = "backward_16k"  # keyscale_16k's gradients from the saved statistics
MEMORY_KERNEL_SRC = os.path.join(ROOT, "long_context_attention_causal_gb300", "csrc",
                                 "polar_memory.cu")
PREFILL_KERNEL_SRC = os.path.join(ROOT, "long_context_attention_causal_gb300",
                                  "csrc", "polar_prefill_tc.cu")
DECODE_KERNEL_SRC = os.path.join(ROOT, "long_context_attention_causal_gb300",
                                 "csrc", "polar_decode.cu")
PAGED_KERNEL_SRC = os.path.join(ROOT, "long_context_attention_causal_gb300",
                                "csrc", "polar_decode_paged_tc.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
METRIC = ("Polar-attn fwd TFLOP/s & % BF16 tensor peak at T=16K; "
          "decode GB/s at 32K KV")


def prefill_flops(wl) -> float:
    n = wl.T
    return float(wl.B * wl.H) * 4.0 * wl.d * n * (n + 1) / 2.0


def decode_bytes(wl) -> float:
    B, H, T, d = wl.B, wl.H, wl.T, wl.d
    return 2.0 * B * H * T * d * 2 + 3.0 * B * H * d * 2 + B * H * 4


def paged_bytes(wl) -> float:
    """K + V rows of the KV heads actually read, plus q, mem, out, n_eff and
    the block table (every sequence of paged_gqa_32k is full)."""
    keys = float(wl.B) * wl.T
    return (2.0 * keys * wl.Hkv * wl.d * 2 + 3.0 * wl.B * wl.Hq * wl.d * 2 +
            wl.B * wl.Hq * 4 + wl.B * ((wl.T + wl.page - 1) // wl.page) * 4)


def memory_bytes(wl) -> float:
    """The fp32 state read and written once, plus q, k, v, mem and the gates."""
    return (2.0 * wl.B * wl.H * wl.d * wl.d * 4 + 4.0 * wl.B * wl.H * wl.T * wl.d * 2 +
            2.0 * wl.B * wl.H * wl.T * 4)


def prefill_bytes(wl) -> float:
    B, H, T, d = wl.B, wl.H, wl.T, wl.d
    return 5.0 * B * H * T * d * 2 + B * H * T * 4


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sus": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "src": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "src": "fallback"}


DEVICE_HEADER = os.path.join(ROOT, "long_context_attention_causal_gb300", "csrc",
                             "polar_device.cuh")


def src_hash(path) -> str:
    """Hash of a kernel's source file and the device header it includes."""
    h = hashlib.sha256()
    for p in (path, DEVICE_HEADER):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, path: str):
    """Per-launch DRAM bytes from the committed ncu summary, valid only while
    the kernel source still has the hash recorded beside the number."""
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and parts[0] == kernel and parts[1] == src_hash(path):
                    return float(parts[2])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            # the timed region starts only once sampling has started
            self.first = self.proc.stdout.readline()
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
            self.out = (self.first or "") + (self.out or "")

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for nm, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x: float) -> float:
    """Largest value over the ranks (the slowest rank sets the job time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, work_per_rank: float, rank_seconds: float) -> float:
    """Whole-job rate of `world` replicas that each did `work_per_rank`: the
    total work over the max-over-ranks time (weak scaling)."""
    return world * work_per_rank / max_over_ranks(world, rank_seconds)


# ------------------------------------------------------------ CPU oracle --

def hold_stream(stream, cycles: int = 20_000_000):
    """Queue a spin of ~10 ms on `stream` before a timed region starts, so
    the host enqueues the timed calls while the device is still busy: a
    host-side pause (the machine's host is shared) then cannot open a gap
    inside the timed region.  The spin itself ends before the start
    event."""
    import torch
    spin = getattr(torch.cuda, "_sleep", None)  # torch's own spin kernel
    if spin is None:
        return
    with torch.cuda.stream(stream):
        spin(cycles)


def oracle_sample(budget_s: float, seed: int = 0):
    """Times the fp64 oracle on rows of the prefill workload (one head's
    q/k/v/mem, rows spread over [0, T)), on all host cores, for about
    budget_s seconds.  Returns (flop/s, seconds, rows, cores)."""
    import numpy as np
    import torch

    from long_context_attention_causal_gb300 import inputs
    from oracle import oracle_rows
    wl = inputs.WORKLOADS[PREFILL]
    g = torch.Generator().manual_seed(seed)
    T, d = wl.T, wl.d
    # same recipe as the workload (one head): N(0,1), key scale U[0.5, 2]
    q = torch.randn((T, d), generator=g).to(torch.bfloat16)
    k = (torch.randn((T, d), generator=g) * (torch.rand(1, generator=g) * 1.5 + 0.5)
         ).to(torch.bfloat16)
    v = torch.randn((T, d), generator=g).to(torch.bfloat16)
    mem = (torch.randn((T, d), generator=g) * 0.1).to(torch.bfloat16)
    w = torch.randn(d, generator=g) * 0.02
    rng = np.random.default_rng(seed)
    cores = os.cpu_count() or 1
    flops, done, rows_done = 0.0, 0.0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        rows = np.sort(rng.integers(0, T, 4 * cores))
        oracle_rows(q, k, v, mem, w, rows, nthreads=cores)
        flops += float(np.sum(4.0 * d * (rows + 1)))
        rows_done += len(rows)
    done = time.perf_counter() - t0
    return flops / done, done, rows_done, cores


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from long_context_attention_causal_gb300 import inputs
    wl = inputs.WORKLOADS[PREFILL]
    budget = max(0.2, min(args.cpu_budget, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(min(budget, 2.0), seed=1)
    args.steps = max(1, args.steps)
    vals, secs, rows = [], 0.0, 0
    cores = os.cpu_count() or 1
    for s in range(args.steps):
        r, t, n, cores = oracle_sample(budget, seed=2 + s)
        vals.append(r)
        secs += t
        rows += n
    tf = sum(vals) / len(vals) / 1e12
    sample = (f"{rows} random causal rows of one head of {PREFILL} "
              f"(T={wl.T}, d={wl.d}), fp64 definition form, "
              f"{args.steps} steps of ~{budget:.0f} s")
    line = {
        "impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{PREFILL} prefill rows (oracle)", "oracle": "fp64 plain C"},
        "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------- GPU --

PREFILL_LEGS = ("tiny_f32", "needles_4k", "keyscale_16k", "needles_64k")
PAGED_LEGS = ("paged_gqa_32k", "paged_gqa2_32k", "paged_gqa8_32k")
ALL_LEGS = PREFILL_LEGS + (DECODE,) + PAGED_LEGS + (MEMSTEP, BACKWARD)
# the timed step: the headline prefill and decode plus the NEXT legs; the
# other three configurations are timed in a phase of their own right after
# it (same warm-up and step count), so that needles_64k's 12 ms of dense
# products, and the power cap they bring, do not sit inside the headline's
# step
STEP_LEGS = (PREFILL, DECODE) + PAGED_LEGS + (MEMSTEP,)


def measure_copy_rates(host_in, dev_in, host_out, dev_out, stream, reps=3):
    """Plain pinned-memory copies of the e2e step's own bytes (one
    cudaMemcpyAsync per tensor, as torch issues them), best of `reps`: the
    inputs host -> device alone, the outputs device -> host alone, and both
    at once on two streams (the link's floor for the whole step)."""
    import torch
    nin = sum(t.numel() * t.element_size() for t in host_in)
    nout = sum(t.numel() * t.element_size() for t in host_out)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def h2d():
        with torch.cuda.stream(s_in):
            for h, d in zip(host_in, dev_in):
                d.copy_(h, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            for h, d in zip(host_out, dev_out):
                h.copy_(d, non_blocking=True)

    def timed(fns):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for f in fns:
            f()
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    best = {"h2d": 1e30, "d2h": 1e30, "both": 1e30}
    for _ in range(reps):
        best["h2d"] = min(best["h2d"], timed([h2d]))
        best["d2h"] = min(best["d2h"], timed([d2h]))
        best["both"] = min(best["both"], timed([h2d, d2h]))
    return {"h2d_gbs": nin / (best["h2d"] * 1e-3) / 1e9,
            "d2h_gbs": nout / (best["d2h"] * 1e-3) / 1e9,
            "both_ms": best["both"]}


def gpu_numa_node(index: int):
    """NUMA node of the GPU's PCI function and the host CPUs this process may
    run on (informational: where pinned buffers land)."""
    bus = None
    try:
        r = subprocess.run(["nvidia-smi", "-i", str(index), "--query-gpu=pci.bus_id",
                            "--format=csv,noheader"], capture_output=True, text=True,
                           timeout=20)
        bus = r.stdout.strip().splitlines()[0].strip() if r.stdout.strip() else None
    except (OSError, subprocess.TimeoutExpired, IndexError):
        bus = None
    node = None
    if bus:
        b = bus.lower()
        for cand in (b, b[4:], "0000" + b[8:] if len(b) > 12 else b):
            path = f"/sys/bus/pci/devices/{cand}/numa_node"
            if os.path.exists(path):
                try:
                    node = int(open(path).read().strip())
                except ValueError:
                    pass
                break
    try:
        cpus = sorted(os.sched_getaffinity(0))
    except AttributeError:
        cpus = []
    return {"gpu_pci": bus, "gpu_numa_node": node, "cpus": len(cpus)}


def run_gpu(args):
    import dataclasses

    import torch

    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs

    world, rank, local = dist_setup()
    dev = torch.device(f"cuda:{local}")
    legs = [x for x in ALL_LEGS if args.only is None or x in args.only.split(",")]
    if not legs:
        raise SystemExit(f"--only names none of {', '.join(ALL_LEGS)}")
    # legs outside the step (when the step has any) are timed in their own
    # phase after it
    step_names = [x for x in legs if x in STEP_LEGS] or legs
    stream = torch.cuda.current_stream()
    calls = []   # (name, fn, launches)
    info = {}    # name -> dict(workload description, work, unit, bound)
    keep = []    # tensors of every leg stay resident
    xp = None    # the headline prefill's inputs (the e2e leg copies them)
    for name in legs:
        if name in PREFILL_LEGS:
            wl = inputs.WORKLOADS[name]
            x = inputs.make_prefill(wl, dev)
            out = torch.empty_like(x["q"])
            ne = torch.empty((wl.B, wl.H, wl.T), device=dev, dtype=torch.float32)
            keep.append((x, out, ne))
            if name == PREFILL:
                xp = x
            fn = (lambda x=x, out=out, ne=ne: pa.fwd(x["q"], x["k"], x["v"], x["mem"],
                                                      x["w_count"], out=out, n_eff=ne))
            info[name] = {"wl": wl, "kind": "prefill",
                          "desc": f"{name} prefill B{wl.B} H{wl.H} T{wl.T} d{wl.d} {wl.dtype}"}
            calls.append((name, fn, 1))
        elif name == DECODE:
            wl = inputs.WORKLOADS[DECODE]
            if args.decode_batch:
                wl = dataclasses.replace(wl, B=args.decode_batch)
            x = inputs.make_decode(wl, dev)
            out = torch.empty_like(x["q"])
            ne = torch.empty((wl.B, wl.H), device=dev, dtype=torch.float32)
            ws = torch.empty(max(16, pa.decode_workspace_bytes(wl.B, wl.H, wl.T, wl.d)),
                             device=dev, dtype=torch.uint8)
            keep.append((x, out, ne, ws))
            fn = (lambda x=x, out=out, ne=ne, ws=ws: pa.decode(
                x["q"], x["k_cache"], x["v_cache"], x["mem"], x["w_count"], workspace=ws,
                out=out, n_eff=ne))
            info[name] = {"wl": wl, "kind": "decode",
                          "desc": f"{name} decode B{wl.B} H{wl.H} Tkv{wl.T} d{wl.d} bf16",
                          "splits": pa.decode_num_splits(wl.B, wl.H, wl.T, wl.d)}
            calls.append((name, fn, 2))
        elif name in PAGED_LEGS:
            wl = inputs.PAGED_WORKLOADS[name]
            if args.paged_batch:
                wl = dataclasses.replace(wl, B=args.paged_batch)
            x = inputs.make_paged_decode(wl, dev)
            out = torch.empty_like(x["q"])
            ne = torch.empty((wl.B, wl.Hq), device=dev, dtype=torch.float32)
            ws = torch.empty(max(16, pa.decode_paged_workspace_bytes(
                wl.B, wl.Hq, wl.Hkv, wl.T, wl.d, args.paged_splits)), device=dev,
                dtype=torch.uint8)
            keep.append((x, out, ne, ws))
            fn = (lambda x=x, out=out, ne=ne, ws=ws, wl=wl: pa.decode_paged(
                x["q"], x["k_pages"], x["v_pages"], x["block_table"], x["seq_lens"],
                x["mem"], x["w_count"], max_seq_len=wl.T, num_splits=args.paged_splits,
                workspace=ws, out=out, n_eff=ne))
            info[name] = {"wl": wl, "kind": "paged",
                          "desc": (f"{name} paged decode B{wl.B} Hq{wl.Hq} Hkv{wl.Hkv} "
                                   f"T{wl.T} d{wl.d} page{wl.page} bf16"),
                          "splits": args.paged_splits or
                          pa.lib().polar_attn_decode_paged_num_splits(wl.B, wl.Hkv, wl.T, wl.d)}
            calls.append((name, fn, 2))
        elif name == BACKWARD:
            # the training pair's backward on the headline prefill's shape
            # and inputs: the forward's outputs and row statistics are made
            # once, the timed call is polar_attn_bwd_stats
            wl = inputs.WORKLOADS[PREFILL]
            xb = xp if xp is not None else inputs.make_prefill(wl, dev)
            fo = pa.fwd_stats(xb["q"], xb["k"], xb["v"], xb["mem"], xb["w_count"])
            gen = torch.Generator(device=dev)
            gen.manual_seed(77)
            dout = torch.randn(xb["q"].shape, generator=gen, device=dev).to(torch.bfloat16)
            gr = [torch.empty(xb["q"].shape, device=dev, dtype=torch.float32) for _ in range(3)]
            dw = torch.empty((wl.H, wl.d), device=dev, dtype=torch.float32)
            ws = torch.empty(pa.bwd_workspace_bytes(wl.B, wl.H, wl.T, wl.d), device=dev,
                             dtype=torch.uint8)
            keep.append((xb, fo, dout, gr, dw, ws))
            fn = (lambda xb=xb, fo=fo, dout=dout, gr=gr, dw=dw, ws=ws: pa.bwd_stats(
                xb["q"], xb["k"], xb["v"], xb["mem"], xb["w_count"], *fo, dout, workspace=ws,
                dq=gr[0], dk=gr[1], dv=gr[2], dw=dw))
            info[name] = {"wl": wl, "kind": "backward",
                          "desc": (f"{name} backward from saved statistics B{wl.B} H{wl.H} "
                                   f"T{wl.T} d{wl.d} bf16")}
            calls.append((name, fn, 4))
        else:
            wl = inputs.MEMORY_WORKLOADS[MEMSTEP]
            x = inputs.make_memory(wl, dev)
            mem = torch.empty_like(x["q"])
            keep.append((x, mem))
            fn = (lambda x=x, mem=mem: pa.memory_step(
                x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], mem=mem))
            info[name] = {"wl": wl, "kind": "memory",
                          "desc": f"{name} memory step B{wl.B} H{wl.H} T{wl.T} d{wl.d} bf16"}
            calls.append((name, fn, 1))

    step_calls = [c for c in calls if c[0] in step_names]
    phase_calls = [c for c in calls if c[0] not in step_names]

    def step(evs=None):
        for i, (_n, fn, _l) in enumerate(step_calls):
            if evs is not None:
                evs[i].record(stream)
            fn()
        if evs is not None:
            evs[len(step_calls)].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert pa.device_status() == 0, "a kernel wait ran out during warm-up"

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(step_calls) + 1)]
           for _ in range(args.steps)]
    leg_ms, eager_ms, median_ms = {}, {}, {}
    barrier(world)
    torch.cuda.synchronize()
    gc.disable()  # no collector pause while the timed calls are enqueued
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        hold_stream(stream)
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        total_ms = max_over_ranks(world, t_start.elapsed_time(t_end))
        for i, (name, _fn, _l) in enumerate(step_calls):
            ms = [e[i].elapsed_time(e[i + 1]) for e in evs]
            leg_ms[name] = max_over_ranks(world, sum(ms) / len(ms))
            median_ms[name] = max_over_ranks(world, statistics.median(ms))
        # the other configurations: each warmed up and timed over as many
        # calls as the step count, CUDA events on the same stream.  The
        # calls are replayed from a CUDA graph, so the device time of the
        # short ones (tiny_f32 runs for microseconds) is not hidden behind
        # the host's per-call cost; that per-call time through the binding
        # is reported beside it (ms_eager)
        for name, fn, _l in phase_calls:
            for _ in range(max(3, args.warmup)):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(args.steps):
                    fn()
            graph.replay()
            torch.cuda.synchronize()
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize()
            leg_ms[name] = max_over_ranks(world, a.elapsed_time(b) / args.steps)
            del graph
            a.record(stream)
            for _ in range(args.steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            eager_ms[name] = max_over_ranks(world, a.elapsed_time(b) / args.steps)
        barrier(world)
    status = pa.device_status()
    pk = peaks()

    def leg_line(name):
        inf, ms = info[name], leg_ms[name]
        wl, sec = inf["wl"], leg_ms[name] * 1e-3
        d = {"workload": inf["desc"], "ms": ms}
        if name in median_ms:
            d["ms_median"] = median_ms[name]  # of the step's per-call events
        if name in eager_ms:
            d["ms_eager"] = eager_ms[name]
            d["timing"] = "CUDA-graph replay of the calls (ms_eager: the same calls from Python)"
        if inf["kind"] == "prefill":
            fl, by = prefill_flops(wl), prefill_bytes(wl) * (2 if wl.dtype == "f32" else 1)
            tf = fl / sec / 1e12
            d.update({"TFLOP/s": world * tf, "tokens/s": world * wl.B * wl.T / sec,
                      "GB/s": world * by / sec / 1e9})
            if wl.dtype == "bf16":
                d["roofline"] = {"bound": "tensor", "achieved": tf, "peak": pk["bf16"],
                                 "unit": "TFLOP/s", "frac": tf / pk["bf16"],
                                 "frac_sustained": tf / pk["bf16_sus"],
                                 "peak_source": f"{pk['src']} bf16 burst"}
            else:
                d["roofline"] = {"bound": "latency", "frac": None,
                                 "note": "fp32, 1.7e7 flop: one partial wave; absolute time"}
        elif inf["kind"] in ("decode", "paged"):
            by = decode_bytes(wl) if inf["kind"] == "decode" else paged_bytes(wl)
            gbs = by / sec / 1e9
            heads = wl.H if inf["kind"] == "decode" else wl.Hq
            d.update({"GB/s": world * gbs, "tokens/s": world * wl.B / sec,
                      "TFLOP/s": world * 4.0 * wl.d * wl.T * wl.B * heads / sec / 1e12,
                      "splits": inf["splits"],
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm"],
                                   "unit": "GB/s", "frac": gbs / pk["hbm"],
                                   "peak_source": f"{pk['src']} copy"}})
        elif inf["kind"] == "backward":
            tf = 2.5 * prefill_flops(wl) / sec / 1e12  # 10 d flop per causal pair
            d.update({"TFLOP/s": world * tf, "tokens/s": world * wl.B * wl.T / sec,
                      "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16"],
                                   "unit": "TFLOP/s", "frac": tf / pk["bf16"],
                                   "frac_sustained": tf / pk["bf16_sus"],
                                   "peak_source": f"{pk['src']} bf16 burst",
                                   "note": "algorithmic 10 d flop per causal pair (S, dP, dV, "
                                           "dK, dQ); the kernels execute 14 d"}})
        else:
            gbs = memory_bytes(wl) / sec / 1e9
            d.update({"GB/s": world * gbs, "tokens/s": world * wl.B * wl.T / sec,
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm"],
                                   "unit": "GB/s", "frac": gbs / pk["hbm"],
                                   "peak_source": f"{pk['src']} copy"}})
        return d

    legs_out = {name: leg_line(name) for name in leg_ms}
    # DRAM traffic of one launch, from the committed ncu summaries (valid
    # while the kernel source still has the recorded hash)
    if PREFILL in legs_out:
        legs_out[PREFILL]["roofline"].update({
            "kernel": "polar_fwd_tc_kernel<128>",
            "traffic": recorded_traffic("polar_fwd_tc_kernel", PREFILL_KERNEL_SRC),
            "algorithmic_bytes": prefill_bytes(inputs.WORKLOADS[PREFILL]),
            "launch_ms": leg_ms[PREFILL]})
    if DECODE in legs_out:
        legs_out[DECODE]["roofline"]["traffic"] = (
            None if args.decode_batch else
            recorded_traffic("polar_decode_split_kernel", DECODE_KERNEL_SRC))
        legs_out[DECODE]["kernels"] = ["polar_decode_split_kernel<128,bf16>",
                                       "polar_decode_combine_kernel<128,bf16>"]
    if PAGED in legs_out:
        legs_out[PAGED]["roofline"]["traffic"] = (
            None if args.paged_batch else
            recorded_traffic("polar_decode_paged_tc_kernel", PAGED_KERNEL_SRC))
    if MEMSTEP in legs_out:
        legs_out[MEMSTEP]["roofline"]["traffic"] = recorded_traffic(
            "polar_memory_step_kernel", MEMORY_KERNEL_SRC)
        legs_out[MEMSTEP]["roofline"]["traffic_note"] = (
            "ncu counts DRAM bytes inside the launch only: dirty state lines still in L2 "
            "at kernel end are written back later, so traffic undercounts the state write")

    # end to end through the public API with pinned HOST buffers: copy the
    # step's inputs in, run, read the result back, all inside the timed region
    e2e = None
    if PREFILL in legs and not args.no_e2e:
        wp = inputs.WORKLOADS[PREFILL]
        # polar_attn_fwd_host: the library cuts the (b, h) range into pieces
        # and overlaps each piece's copies with the other pieces' kernels
        hq = {k: xp[k].cpu().pin_memory() for k in ("q", "k", "v", "mem")}
        hw = xp["w_count"].cpu().pin_memory()
        ho = torch.empty(xp["q"].shape, dtype=xp["q"].dtype).pin_memory()
        hn = torch.empty((wp.B, wp.H, wp.T), dtype=torch.float32).pin_memory()
        ws_h = torch.empty(pa.fwd_host_workspace_bytes(wp.B, wp.H, wp.T, wp.d),
                           device=dev, dtype=torch.uint8)

        # consecutive steps alternate between two streams and two
        # workspaces, as a training or serving loop pipelines them: step
        # i + 1's inputs are copied in while step i's last pieces compute and
        # its outputs are copied out (the library orders each call after its
        # own stream's earlier work only)
        ws_h2 = torch.empty_like(ws_h)
        side = torch.cuda.Stream()

        def e2e_step(i=0):
            s, ws = (side, ws_h2) if i % 2 else (stream, ws_h)
            pa.fwd_host(hq["q"], hq["k"], hq["v"], hq["mem"], hw, out=ho, n_eff=hn,
                        workspace=ws, num_pieces=args.e2e_pieces, stream=s,
                        synchronize=False)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        ks = max(3, min(args.steps, 20))
        # serial: one step after another on one stream, an event after each;
        # the per-call spread shows what is left of host-side stalls (the
        # box's host is shared) separately from the pipeline's own time
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(ks + 1)]
        hold_stream(stream)
        ev[0].record(stream)
        for i in range(ks):
            e2e_step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        serial_ms = max_over_ranks(world, ev[0].elapsed_time(ev[ks]) / ks)
        per_call = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(ks))
        # pipelined: the same steps on alternating streams, timed as a whole
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_stream(stream)
        e0.record(stream)
        side.wait_stream(stream)
        for i in range(ks):
            e2e_step(i)
        stream.wait_stream(side)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(world, e0.elapsed_time(e1) / ks)
        h2d = sum(t.numel() * t.element_size() for t in hq.values()) + hw.numel() * 4
        d2h = ho.numel() * ho.element_size() + hn.numel() * 4
        # the link's own rates, measured on the same bytes: the copies
        # alone, then in and out at once (the whole step's floor)
        scratch_in = [torch.empty_like(xp[k]) for k in ("q", "k", "v", "mem")]
        scratch_out = [torch.empty(ho.shape, dtype=ho.dtype, device=dev),
                       torch.empty(hn.shape, dtype=hn.dtype, device=dev)]
        rates = measure_copy_rates(list(hq.values()), scratch_in, [ho, hn], scratch_out, stream)
        del scratch_in, scratch_out
        e2e = {"value": world * prefill_flops(wp) / (e2e_ms * 1e-3) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "steps_timed": ks,
               "pipelining": "steps alternate between two streams and two workspaces",
               "serial_ms_per_step": serial_ms, "serial_value": world * prefill_flops(wp)
               / (serial_ms * 1e-3) / 1e12,
               "ms_per_call_median": per_call[ks // 2],
               "ms_per_call_max": per_call[-1], "pieces": args.e2e_pieces or "auto",
               "h2d_gbs_measured": rates["h2d_gbs"], "d2h_gbs_measured": rates["d2h_gbs"],
               "copy_floor_ms": rates["both_ms"],
               "copy_floor_note": "the step's inputs in and outputs out at once on two streams, "
                                  "no kernel: the link's floor for the step",
               "host": gpu_numa_node(local)}
    gc.enable()
    clocks = clk.summary()
    if rank != 0:
        return 0

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        r, t, n, cores = oracle_sample(args.cpu_budget)
        wp = inputs.WORKLOADS[PREFILL]
        cpu = {"value": r / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} random causal rows of one head of {PREFILL} "
                         f"(T={wp.T}, d={wp.d}), fp64, {t:.1f} s"}
    head = PREFILL if PREFILL in legs_out else legs[0]
    hl = legs_out[head]
    line = {
        "metric": METRIC,
        "value": hl.get("TFLOP/s") if head == PREFILL else hl.get("GB/s"),
        "unit": "TFLOP/s" if head == PREFILL else "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": " + ".join(info[n]["desc"] for n in step_names),
            "also_timed": [info[n]["desc"] for n in legs if n not in step_names],
            "value_from": f"{head} (every workload under 'configs')",
            "l2": ("no flush; the large inputs exceed L2 (keyscale_16k 512 MiB, needles_64k "
                   "1 GiB, decode 8.6 GB, paged 1-4 GB, memory state 268 MB); tiny_f32 and "
                   "needles_4k (4 MiB per tensor) stay L2-resident between steps, as a "
                   "prefill's own K/V re-reads do"),
            "parallelism": f"replicas x{world}",
        },
        "roofline": dict(hl["roofline"]),
        "configs": legs_out,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (sum(l for (n, _f, l) in calls if n in step_names)
                         + 2 * sum(l for (n, _f, l) in calls if n not in step_names)) * args.steps,
        "gpu_launches_note": "the step's launches plus those of the configurations timed after "
                             "it (each timed twice: from Python and replayed from a CUDA graph)",
        "clocks": clocks,
        "device_status": status,
    }
    if DECODE in legs_out:
        line["decode"] = {"value": legs_out[DECODE]["GB/s"], "unit": "GB/s",
                          "ms": legs_out[DECODE]["ms"], "roofline": legs_out[DECODE]["roofline"]}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_configs(args):
    """One JSON line per workload (the five configurations plus the NEXT
    legs): time per call, TFLOP/s, tokens/s, GB/s and roofline fraction,
    CUDA events on the launching stream, after warm-up."""
    import torch

    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    pk = peaks()
    stream = torch.cuda.current_stream()

    def timed(fn, iters):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters

    for name, wl in inputs.WORKLOADS.items():
        if wl.kind == "prefill":
            x = inputs.make_prefill(wl, dev)
            out = torch.empty_like(x["q"])
            ne = torch.empty((wl.B, wl.H, wl.T), device=dev)
            ms = timed(lambda: pa.fwd(x["q"], x["k"], x["v"], x["mem"], x["w_count"],
                                      out=out, n_eff=ne), 5 if wl.T > 16384 else 20)
            fl = prefill_flops(wl)
            by = prefill_bytes(wl) * (2 if wl.dtype == "f32" else 1)
            tf = fl / (ms * 1e-3) / 1e12
            line = {"workload": name, "kind": "prefill", "dtype": wl.dtype, "ms": ms,
                    "TFLOP/s": tf, "tokens/s": wl.B * wl.T / (ms * 1e-3),
                    "GB/s": by / (ms * 1e-3) / 1e9,
                    "roofline": ({"bound": "tensor", "frac": tf / pk["bf16"]}
                                 if wl.dtype == "bf16" else
                                 {"bound": "latency", "note": "fp32, tiny: absolute time"})}
        else:
            x = inputs.make_decode(wl, dev)
            out = torch.empty_like(x["q"])
            ne = torch.empty((wl.B, wl.H), device=dev)
            ws = torch.empty(max(16, pa.decode_workspace_bytes(wl.B, wl.H, wl.T, wl.d)),
                             device=dev, dtype=torch.uint8)
            ms = timed(lambda: pa.decode(x["q"], x["k_cache"], x["v_cache"], x["mem"],
                                         x["w_count"], workspace=ws, out=out, n_eff=ne), 20)
            gbs = decode_bytes(wl) / (ms * 1e-3) / 1e9
            line = {"workload": name, "kind": "decode", "dtype": wl.dtype, "ms": ms,
                    "TFLOP/s": 4.0 * wl.d * wl.T * wl.B * wl.H / (ms * 1e-3) / 1e12,
                    "tokens/s": wl.B / (ms * 1e-3), "GB/s": gbs,
                    "roofline": {"bound": "hbm", "frac": gbs / pk["hbm"]}}
        print(json.dumps(line), flush=True)
        del x
        torch.cuda.empty_cache()
    # backward (NEXT-2, bf16 on the tensor cores): algorithmic 10 d flop per
    # causal pair (S, dP, dV, dK, dQ; the kernels also recompute the forward
    # and S, dP a second time, 18 d executed), against the bf16 peak
    for name in ("needles_4k", "keyscale_16k"):
        wl = inputs.WORKLOADS[name]
        x = inputs.make_prefill(wl, dev)
        dout = torch.randn_like(x["q"])
        ws = torch.empty(pa.bwd_workspace_bytes(wl.B, wl.H, wl.T, wl.d), device=dev,
                         dtype=torch.uint8)
        ms = timed(lambda: pa.bwd(x["q"], x["k"], x["v"], x["w_count"], dout, workspace=ws),
                   10 if wl.T <= 4096 else 5)
        fl = prefill_flops(wl) * 2.5
        tf = fl / (ms * 1e-3) / 1e12
        print(json.dumps({"workload": name, "kind": "backward", "dtype": wl.dtype, "ms": ms,
                          "TFLOP/s": tf, "tokens/s": wl.B * wl.T / (ms * 1e-3),
                          "roofline": {"bound": "tensor", "peak": pk["bf16"],
                                       "unit": "TFLOP/s", "frac": tf / pk["bf16"],
                                       "note": "algorithmic 10 d flop per causal pair"}}),
              flush=True)
        # the same gradients from the saved outputs of fwd_stats (no forward
        # recomputation; the training pair's backward half)
        out, ne, cf, st = pa.fwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"])
        ms = timed(lambda: pa.bwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"], out,
                                        ne, cf, st, dout, workspace=ws),
                   10 if wl.T <= 4096 else 5)
        tf = fl / (ms * 1e-3) / 1e12
        print(json.dumps({"workload": name, "kind": "backward_from_stats", "dtype": wl.dtype,
                          "ms": ms, "TFLOP/s": tf, "tokens/s": wl.B * wl.T / (ms * 1e-3),
                          "roofline": {"bound": "tensor", "peak": pk["bf16"],
                                       "unit": "TFLOP/s", "frac": tf / pk["bf16"],
                                       "note": "algorithmic 10 d flop per causal pair"}}),
              flush=True)
        del x, dout, ws, out, ne, cf, st
        torch.cuda.empty_cache()
    wg = inputs.PAGED_WORKLOADS[PAGED]
    x = inputs.make_paged_decode(wg, dev)
    ws = torch.empty(max(16, pa.decode_paged_workspace_bytes(wg.B, wg.Hq, wg.Hkv, wg.T, wg.d)),
                     device=dev, dtype=torch.uint8)
    ms = timed(lambda: pa.decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                                       x["seq_lens"], x["mem"], x["w_count"], max_seq_len=wg.T,
                                       workspace=ws), 20)
    gbs = paged_bytes(wg) / (ms * 1e-3) / 1e9
    print(json.dumps({"workload": PAGED, "kind": "paged decode", "dtype": wg.dtype, "ms": ms,
                      "tokens/s": wg.B / (ms * 1e-3), "GB/s": gbs,
                      "roofline": {"bound": "hbm", "frac": gbs / pk["hbm"]}}), flush=True)
    del x
    wm = inputs.MEMORY_WORKLOADS[MEMSTEP]
    x = inputs.make_memory(wm, dev)
    ms = timed(lambda: pa.memory_step(x["state"], x["q"], x["k"], x["v"], x["alpha"],
                                      x["beta"]), 20)
    gbs = memory_bytes(wm) / (ms * 1e-3) / 1e9
    print(json.dumps({"workload": MEMSTEP, "kind": "memory step", "dtype": wm.dtype, "ms": ms,
                      "tokens/s": wm.B / (ms * 1e-3), "GB/s": gbs,
                      "roofline": {"bound": "hbm", "frac": gbs / pk["hbm"]}}), flush=True)
    return 0


def run_backward(args):
    """Backward of one synthetic bf16 prefill of the given shape (the tile
    kernels' profiling target): W + K calls, K timed with CUDA events."""
    import torch

    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs
    B, H, T, d = (int(x) for x in args.backward.split(","))
    torch.cuda.set_device(0)
    wl = inputs.custom("prefill", B=B, H=H, T=T, d=d, dtype="bf16", seed=5, needles=1)
    x = inputs.make_prefill(wl, "cuda")
    dout = torch.randn_like(x["q"])
    ws = torch.empty(pa.bwd_workspace_bytes(B, H, T, d), device="cuda", dtype=torch.uint8)
    if args.from_stats:
        out, ne, cf, st = pa.fwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"])
        call = lambda: pa.bwd_stats(x["q"], x["k"], x["v"], x["mem"], x["w_count"], out,  # noqa: E731
                                    ne, cf, st, dout, workspace=ws)
    else:
        call = lambda: pa.bwd(x["q"], x["k"], x["v"], x["w_count"], dout, workspace=ws)  # noqa: E731
    for _ in range(args.warmup):
        call()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(args.steps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / max(1, args.steps)
    fl = 10.0 * d * B * H * T * (T + 1) / 2.0
    print(json.dumps({"kind": "backward_from_stats" if args.from_stats else "backward",
                      "shape": [B, H, T, d], "ms": ms, "TFLOP/s": fl / (ms * 1e-3) / 1e12,
                      "note": "algorithmic 10 d flop per causal pair",
                      "device_status": pa.device_status()}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--paged-splits", type=int, default=0,
                    help="split count of the paged decode (0: the library's choice)")
    ap.add_argument("--e2e-pieces", type=int, default=0,
                    help="pieces of the host-buffer prefill (0: the library's choice)")
    ap.add_argument("--only", default=None, metavar="LEG[,LEG]",
                    help="run these legs of the step only (smaller captures): "
                         + ", ".join(ALL_LEGS))
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="override the decode batch (smaller captures)")
    ap.add_argument("--paged-batch", type=int, default=0,
                    help="sequences of the paged workload (smaller cases for profiling)")
    ap.add_argument("--configs", action="store_true",
                    help="print one line per workload instead of the bench line")
    ap.add_argument("--backward", default=None, metavar="B,H,T,d",
                    help="time the backward of one bf16 prefill of this shape")
    ap.add_argument("--from-stats", action="store_true",
                    help="with --backward: the training pair's backward (saved statistics)")
    args = ap.parse_args()
    if args.backward:
        return run_backward(args)
    if args.configs:
        return run_configs(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
