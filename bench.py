"""Benchmark of the causal Polar Attention hot path on GB300.

One step = one causal prefill of keyscale_16k (B=2, H=16, T=16384, d=128,
bf16), one split-KV decode of decode_32k (B=32, H=16, Tkv=32768, d=128,
bf16), one paged grouped-query decode of paged_gqa_32k (B=32, 16 query
heads on 4 KV heads, 32768 tokens in 64-token pages) and one in-place
gated-delta memory step of memstep_256 (256 x 16 heads, 128 x 128 fp32
state), all inputs resident in HBM.  `value` is the prefill's
algorithmic TFLOP/s (causal pairs only: 4 d n(n+1)/2 flop per head); the
decode's GB/s (K + V + q + mem + out + n_eff bytes) is reported beside it.
Inputs are larger than the 129 MB L2 (512 MiB prefill, 8.6 GB decode), so
no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own replica (independent problems, no
collective on the data path): weak scaling, value summed over ranks.
--impl reference times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
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

def run_gpu(args):
    import torch

    import long_context_attention_causal_gb300 as pa
    from long_context_attention_causal_gb300 import inputs

    world, rank, local = dist_setup()
    dev = torch.device(f"cuda:{local}")
    wp = inputs.WORKLOADS[PREFILL]
    wd = inputs.WORKLOADS[DECODE]
    do_p = args.only in (None, "prefill")
    do_d = args.only in (None, "decode")
    do_g = args.only in (None, "paged")
    do_m = args.only in (None, "memory")
    wg = inputs.PAGED_WORKLOADS[PAGED]
    wm = inputs.MEMORY_WORKLOADS[MEMSTEP]
    if args.decode_batch:
        import dataclasses
        wd = dataclasses.replace(wd, B=args.decode_batch)
    if args.paged_batch:
        import dataclasses
        wg = dataclasses.replace(wg, B=args.paged_batch)
    xp = inputs.make_prefill(wp, dev) if do_p else None
    xd = inputs.make_decode(wd, dev) if do_d else None
    if do_p:
        out_p = torch.empty_like(xp["q"])
        neff_p = torch.empty((wp.B, wp.H, wp.T), device=dev, dtype=torch.float32)
    if do_d:
        out_d = torch.empty_like(xd["q"])
        neff_d = torch.empty((wd.B, wd.H), device=dev, dtype=torch.float32)
        ws = torch.empty(max(16, pa.decode_workspace_bytes(wd.B, wd.H, wd.T, wd.d)),
                         device=dev, dtype=torch.uint8)
    if do_g:
        xg = inputs.make_paged_decode(wg, dev)
        out_g = torch.empty_like(xg["q"])
        neff_g = torch.empty((wg.B, wg.Hq), device=dev, dtype=torch.float32)
        ws_g = torch.empty(max(16, pa.decode_paged_workspace_bytes(
            wg.B, wg.Hq, wg.Hkv, wg.T, wg.d, args.paged_splits)), device=dev, dtype=torch.uint8)
    if do_m:
        xm = inputs.make_memory(wm, dev)
        mem_m = torch.empty_like(xm["q"])
    splits = pa.decode_num_splits(wd.B, wd.H, wd.T, wd.d)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if do_p:
            pa.fwd(xp["q"], xp["k"], xp["v"], xp["mem"], xp["w_count"], out=out_p,
                   n_eff=neff_p)
        if ev is not None:
            ev[1].record(stream)
        if do_d:
            pa.decode(xd["q"], xd["k_cache"], xd["v_cache"], xd["mem"], xd["w_count"],
                      workspace=ws, out=out_d, n_eff=neff_d)
        if ev is not None:
            ev[2].record(stream)
        if do_g:
            pa.decode_paged(xg["q"], xg["k_pages"], xg["v_pages"], xg["block_table"],
                            xg["seq_lens"], xg["mem"], xg["w_count"], max_seq_len=wg.T,
                            num_splits=args.paged_splits, workspace=ws_g, out=out_g,
                            n_eff=neff_g)
        if ev is not None:
            ev[3].record(stream)
        if do_m:
            pa.memory_step(xm["state"], xm["q"], xm["k"], xm["v"], xm["alpha"], xm["beta"],
                           mem=mem_m)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert pa.device_status() == 0, "a kernel wait ran out during warm-up"

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)]
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    pag_ms = [e[2].elapsed_time(e[3]) for e in evs]
    mem_ms = [e[3].elapsed_time(e[4]) for e in evs]
    total_ms = max_over_ranks(world, total_ms)
    pre_avg = max_over_ranks(world, sum(pre_ms) / len(pre_ms))
    dec_avg = max_over_ranks(world, sum(dec_ms) / len(dec_ms))
    pag_avg = max_over_ranks(world, sum(pag_ms) / len(pag_ms))
    mem_avg = max_over_ranks(world, sum(mem_ms) / len(mem_ms))
    status = pa.device_status()

    # end to end through the public API with pinned HOST buffers: copy the
    # step's inputs in, run, read the result back, all inside the timed region
    e2e = None
    if do_p and not args.no_e2e:
        # polar_attn_fwd_host: the library cuts the (b, h) range into pieces
        # and overlaps each piece's copies with the other pieces' kernels
        hq = {k: xp[k].cpu().pin_memory() for k in ("q", "k", "v", "mem")}
        hw = xp["w_count"].cpu().pin_memory()
        ho = torch.empty(out_p.shape, dtype=out_p.dtype).pin_memory()
        hn = torch.empty(neff_p.shape, dtype=torch.float32).pin_memory()
        ws_h = torch.empty(pa.fwd_host_workspace_bytes(wp.B, wp.H, wp.T, wp.d),
                           device=dev, dtype=torch.uint8)

        def e2e_step():
            pa.fwd_host(hq["q"], hq["k"], hq["v"], hq["mem"], hw, out=ho, n_eff=hn,
                        workspace=ws_h, num_pieces=args.e2e_pieces, stream=stream,
                        synchronize=False)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        ks = max(3, min(args.steps, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(ks):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(world, a.elapsed_time(b) / ks)
        h2d = sum(t.numel() * t.element_size() for t in hq.values()) + hw.numel() * 4
        d2h = ho.numel() * ho.element_size() + hn.numel() * 4
        e2e = {"value": world * prefill_flops(wp) / (e2e_ms * 1e-3) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "pieces": args.e2e_pieces or "auto"}

    pk = peaks()
    pf = prefill_flops(wp)
    db = decode_bytes(wd)
    pre_tflops = pf / (pre_avg * 1e-3) / 1e12 if do_p else 0.0
    dec_gbs = db / (dec_avg * 1e-3) / 1e9 if do_d else 0.0
    gb = paged_bytes(wg)
    pag_gbs = gb / (pag_avg * 1e-3) / 1e9 if do_g else 0.0
    mb = memory_bytes(wm)
    mem_gbs = mb / (mem_avg * 1e-3) / 1e9 if do_m else 0.0
    clocks = clk.summary()
    if rank != 0:
        return 0

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        r, t, n, cores = oracle_sample(args.cpu_budget)
        cpu = {"value": r / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} random causal rows of one head of {PREFILL} "
                         f"(T={wp.T}, d={wp.d}), fp64, {t:.1f} s"}
    line = {
        "metric": METRIC,
        "value": world * pre_tflops,
        "unit": "TFLOP/s",
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
            "workload": (f"{PREFILL} prefill B{wp.B} H{wp.H} T{wp.T} d{wp.d} bf16 + "
                         f"{DECODE} decode B{wd.B} H{wd.H} Tkv{wd.T} d{wd.d} bf16 + "
                         f"{PAGED} paged GQA decode + {MEMSTEP} memory step"),
            "value_from": "prefill (decode reported under 'decode')",
            "l2": "inputs larger than L2 (prefill 512 MiB, decode 8.6 GB); no flush",
            "decode_splits": splits,
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "kernel": "polar_fwd_tc_kernel<128>",
            "bound": "tensor",
            "achieved": pre_tflops,
            "peak": pk["bf16"],
            "unit": "TFLOP/s",
            "frac": pre_tflops / pk["bf16"],
            "frac_sustained": pre_tflops / pk["bf16_sus"],
            "peak_source": f"{pk['src']} bf16 burst",
            "traffic": recorded_traffic("polar_fwd_tc_kernel", PREFILL_KERNEL_SRC),
            "algorithmic_bytes": prefill_bytes(wp),
            "launch_ms": pre_avg,
        },
        "decode": {
            "kernels": ["polar_decode_split_kernel<128,bf16>",
                        "polar_decode_combine_kernel<128,bf16>"],
            "value": world * dec_gbs,
            "unit": "GB/s",
            "ms": dec_avg,
            "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": pk["hbm"],
                         "unit": "GB/s", "frac": dec_gbs / pk["hbm"],
                         "peak_source": f"{pk['src']} copy",
                         "traffic": None if args.decode_batch else
                         recorded_traffic("polar_decode_split_kernel", DECODE_KERNEL_SRC)},
        },
        "decode_paged": {
            "workload": (f"{PAGED} B{wg.B} Hq{wg.Hq} Hkv{wg.Hkv} T{wg.T} d{wg.d} "
                         f"page{wg.page} bf16"),
            "kernels": ["polar_decode_paged_tc_kernel<128,4>",
                        "polar_decode_combine_kernel<128,bf16>"],
            "value": world * pag_gbs,
            "unit": "GB/s",
            "ms": pag_avg,
            "splits": args.paged_splits or
            pa.lib().polar_attn_decode_paged_num_splits(wg.B, wg.Hkv, wg.T, wg.d),
            "roofline": {"bound": "hbm", "achieved": pag_gbs, "peak": pk["hbm"],
                         "unit": "GB/s", "frac": pag_gbs / pk["hbm"],
                         "peak_source": f"{pk['src']} copy",
                         "traffic": None if args.paged_batch else
                         recorded_traffic("polar_decode_paged_tc_kernel", PAGED_KERNEL_SRC)},
        },
        "memory_step": {
            "workload": f"{MEMSTEP} B{wm.B} H{wm.H} T{wm.T} d{wm.d} bf16, fp32 state",
            "kernels": ["polar_memory_step_kernel<128,bf16>"],
            "value": world * mem_gbs,
            "unit": "GB/s",
            "ms": mem_avg,
            "roofline": {"bound": "hbm", "achieved": mem_gbs, "peak": pk["hbm"],
                         "unit": "GB/s", "frac": mem_gbs / pk["hbm"],
                         "peak_source": f"{pk['src']} copy",
                         "traffic": recorded_traffic("polar_memory_step_kernel",
                                                     MEMORY_KERNEL_SRC)},
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (int(do_p) + 2 * int(do_d) + 2 * int(do_g) + int(do_m)) * args.steps,
        "clocks": clocks,
        "device_status": status,
    }
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
    ap.add_argument("--only", choices=["prefill", "decode", "paged", "memory"], default=None,
                    help="run one half of the step (smaller captures)")
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
