#!/usr/bin/env python
"""Throughput of one low-rank (CoLA) bottleneck decoder block, forward + backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one forward and one backward pass of the whole block over one batch
of synthetic tokens (default: the 1B shape, T = 4 x 4096 tokens, d = 2048,
r = 512, d_ff = 5461, Online RMSNorm over S = 4 shards, bf16 with fp32
accumulation). Inputs are resident in HBM when the timed region starts; L2 is
flushed (a 256 MiB write) before every timed step, outside the step's events.
Under torchrun the ranks are data parallel over tokens: each holds the weights
and its own T tokens (weak scaling) and every step ends with one all-reduce of
the weight gradients (rank_bottleneck_gb300.dp), inside the timed region; the
time is the max over ranks.

Prints one JSON line (rank 0) with the throughput, the roofline of the dominant
kernel (the tcgen05 GEMM engine) against MEASURED_PEAKS.json, the end-to-end
number through the public API with host buffers, the clocks seen during the
timed region, and the fp64 CPU oracle timed on a bounded sample.
--impl reference times that oracle alone, as the reference arm.
"""
from __future__ import annotations

import argparse
import csv
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CoLA block fwd+bwd tokens/s and TFLOP/s as % of GB300 bf16 dense peak"
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# process group (one rank per GPU, data parallel over tokens)
# ---------------------------------------------------------------------------

def dist_init():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 0, 1
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist.get_rank(), int(os.environ.get("LOCAL_RANK", "0")), dist.get_world_size()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Seed of the rank's own tokens (every rank draws the weights with seed 0)."""
    return rank


# ---------------------------------------------------------------------------
# peaks, clocks
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        self.proc = None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        gpu_index = ids[local_rank] if local_rank < len(ids) and ids[local_rank].isdigit() \
            else str(local_rank)
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], None, set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for row in csv.reader(f):
                if len(row) < 9:
                    continue
                try:
                    sm.append(float(row[1]))
                    smax = float(row[2])
                    power.append(float(row[3]))
                except ValueError:
                    continue
                for name, val in zip(names, row[5:9]):
                    if val.strip().lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_step(cfg, inp):
    import numpy as np
    import oracle as O
    f = {k: v.astype(np.float64) for k, v in inp.items()}
    p = {k: f[k] for k in cfg.param_shapes()}
    oc = dict(kind=cfg.kind, dense=cfg.dense, sigma=cfg.sigma, eps=cfg.eps,
              checkpoint=cfg.checkpoint, attn=cfg.attn, seq_len=cfg.seq_len or None)
    out, saved = O.block_forward(p, f["x"], oc)
    dq, dk = (None, None) if cfg.attn else (f.get("dq"), f.get("dk"))
    O.block_backward(p, f["x"], saved, f["dy"], dq, dk, oc)


def oracle_sample_cfg(cfg, rows):
    """The workload on `rows` token rows; with the attention core inside, one
    sequence of `rows` tokens (the oracle's attention holds rows^2 scores per head)."""
    from rank_bottleneck_gb300.block import BlockConfig
    kw = {k: getattr(cfg, k) for k in ("d", "r", "d_ff", "S", "sigma", "dtype", "kind", "dense",
                                       "checkpoint", "eps", "attn")}
    return BlockConfig(T=rows, seq_len=rows if cfg.attn else 0, **kw)


def time_oracle(cfg, rows, seed=0):
    from rank_bottleneck_gb300.synth import make_block_inputs
    c = oracle_sample_cfg(cfg, rows)
    inp = make_block_inputs(c.T, c.d, c.r, c.d_ff, kind=c.kind, dense=c.dense, dtype=c.dtype,
                            seed=seed)
    t0 = time.perf_counter()
    oracle_step(c, inp)
    return time.perf_counter() - t0


def cpu_baseline(cfg, target_s=15.0):
    """Time the oracle on a bounded row sample (about target_s of CPU work)."""
    rows = 128
    t = time_oracle(cfg, rows)
    rows = int(min(max(rows * target_s / max(t, 1e-3), 128), cfg.T))
    rows = max(64, rows // 64 * 64)
    if cfg.attn:
        rows = min(rows, 1024)
    t = time_oracle(cfg, rows)
    return {"value": rows / t, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{rows} of the workload's {cfg.T} token rows, one fp64 forward+backward "
                      f"({t:.1f} s)" + (f"; attention over one sequence of {rows} tokens (the "
                                        f"workload's are {cfg.seq_len})" if cfg.attn else "")}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, local_rank, world):
    import numpy as np
    import torch
    from rank_bottleneck_gb300 import block as B
    from rank_bottleneck_gb300.configs import WORKLOADS, model_flops, recompute_flops
    from rank_bottleneck_gb300.dp import GradBuffer, allreduce_grads
    from rank_bottleneck_gb300.synth import make_block_inputs

    B.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = B.BlockConfig(**WORKLOADS[args.workload])
    dt = cfg.torch_dtype
    # every rank holds the same weights (seed 0) and its own tokens
    inp = make_block_inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, kind=cfg.kind, dense=cfg.dense,
                            dtype=cfg.dtype, seed=0, ranks=cfg.ranks)
    if rank > 0:
        own = make_block_inputs(cfg.T, cfg.d, cfg.r, cfg.d_ff, kind=cfg.kind, dense=cfg.dense,
                                dtype=cfg.dtype, seed=rank_seed(rank), ranks=cfg.ranks)
        for n in ("x", "dy", "dq", "dk"):
            if n in own:
                inp[n] = own[n]
    params = {}
    for n in cfg.param_shapes():
        t = torch.from_numpy(inp[n]).to(dev, dt)
        if n == "A_d":
            params[n] = B.empty_param(cfg, n, dev)
            params[n].copy_(t)
        else:
            params[n] = t
    # q and k leave the block (and dq, dk enter it) only when the attention core
    # runs outside it
    qk_io = cfg.kind == "full" and not cfg.attn
    act_names = ["x", "dy"] + (["dq", "dk"] if qk_io else [])
    acts = {n: torch.from_numpy(inp[n]).to(dev, dt) for n in act_names}
    ws = B.Workspace(cfg, dev)
    y = torch.empty_like(acts["x"])
    q = torch.empty_like(acts["x"]) if qk_io else None
    k = torch.empty_like(acts["x"]) if qk_io else None
    dx = torch.empty_like(acts["x"])
    # the weight gradients as views into one flat buffer: under torchrun one
    # all-reduce per step sums them over the ranks (token-sharded data parallelism)
    gbuf = GradBuffer(cfg, dev)
    grads = gbuf.grads
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    launches = [0, 0]

    def compute():
        B.forward(cfg, params, acts["x"], ws, y, q, k)
        launches[0] = B.last_launch_count()
        B.backward(cfg, params, acts["x"], ws, acts["dy"], acts.get("dq"), acts.get("dk"), dx, grads)
        launches[1] = B.last_launch_count()

    def step():
        compute()
        if world > 1:
            allreduce_grads(gbuf)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if B.device_status(ws) != 0:
        raise RuntimeError("device status reports a timeout during warm-up")

    # The step's library launches captured once into a CUDA graph and replayed:
    # the same kernels with the same arguments, without the host issuing each
    # launch through the C ABI every step (about 0.9 ms of host time a step at
    # the 1B shape). The gradient all-reduce of N > 1 runs after each replay.
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            compute()
        torch.cuda.synchronize()
        for _ in range(2):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize()
        if B.device_status(ws) != 0:
            raise RuntimeError("device status reports a timeout in the captured step")

    def timed_step():
        if graph is None:
            step()
            return
        graph.replay()
        if world > 1:
            allreduce_grads(gbuf)

    # ---- timed region: K steps, device time per step (L2 flushed between steps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        timed_step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    if B.device_status(ws) != 0:
        raise RuntimeError("device status reports a timeout in the timed region")

    tokens = world * args.steps * cfg.T
    value = tokens / (total_ms / 1e3)
    mflops = model_flops(cfg)
    hflops = mflops + recompute_flops(cfg)
    tflops = world * args.steps * mflops / (total_ms / 1e3) / 1e12
    peaks, peak_src = load_peaks()

    # ---- per-kernel device times (launch events) on a few more steps
    nprof = max(2, min(args.steps, 5))
    B.profile_start()
    prof_ms = []
    for _ in range(nprof):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        torch.cuda.synchronize()
        prof_ms.append(a.elapsed_time(b))
    recs = B.profile_stop()
    kernels = {}
    for r in recs:
        kk = kernels.setdefault(r["kernel"], dict(launches=0, ms=0.0, flops=0.0, bytes=0.0))
        kk["launches"] += 1
        kk["ms"] += r["ms"]
        kk["flops"] += r["flops"]
        kk["bytes"] += r["bytes"]
    tot_kernel_ms = sum(v["ms"] for v in kernels.values())
    breakdown = {}
    for name, v in sorted(kernels.items(), key=lambda kv: -kv[1]["ms"]):
        breakdown[name] = {
            "launches_per_step": v["launches"] / nprof, "ms_per_step": v["ms"] / nprof,
            "share": v["ms"] / tot_kernel_ms if tot_kernel_ms else None,
            "tflops": v["flops"] / (v["ms"] / 1e3) / 1e12 if v["ms"] > 0 else None,
            "gbs": v["bytes"] / (v["ms"] / 1e3) / 1e9 if v["ms"] > 0 else None}
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    dk = kernels[dom]
    if dom.startswith("gemm") or dom == "attention":
        # the engine's launches run inside a millisecond-scale step, not a
        # seconds-long loop under the power cap: the burst figure is the peak
        achieved = dk["flops"] / (dk["ms"] / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} bf16 burst",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    else:
        achieved = dk["bytes"] / (dk["ms"] / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} HBM copy"}
    roof.update(kernel=dom, launches_per_step=dk["launches"] / nprof,
                ms_per_launch=dk["ms"] / dk["launches"], traffic=traffic_for(dom, args.workload),
                flops_per_launch=dk["flops"] / dk["launches"],
                bytes_per_launch=dk["bytes"] / dk["launches"])

    # ---- end to end through the public API: host buffers, copies in the timed region
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, cfg, inp, params, ws, act_names, dev, stream, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg)

    # activation memory: what the forward keeps for the backward (`saved`), the
    # backward's temporaries (`scratch`), and the process's peak device allocation
    n_saved, n_scratch = B.workspace_size(cfg)
    act = {"saved_bytes": n_saved, "scratch_bytes": n_scratch,
           "peak_allocated_bytes": torch.cuda.max_memory_allocated(dev)}
    if cfg.checkpoint:
        import dataclasses
        act["saved_bytes_without_checkpoint"] = B.workspace_size(
            dataclasses.replace(cfg, checkpoint=False))[0]

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
            "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) factors)",
            "config": workload_config(args, cfg, world),
            "tflops": tflops, "model_tflop_per_step": mflops / 1e12,
            "hardware_tflop_per_step": hflops / 1e12,
            "pct_of_bf16_peak": {"measured_burst": 100 * tflops / peaks["bf16_tflops"],
                                 "measured_sustained": 100 * tflops / peaks["bf16_tflops_sustained"],
                                 "nominal_dense_2250": 100 * tflops / NOMINAL_BF16_TFLOPS,
                                 "source": peak_src},
            "roofline": roof,
            "activation_bytes": act,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": (launches[0] + launches[1]) * args.steps,
            "execution": ("CUDA graph replay of the step's library launches (captured once "
                          "through the C ABI)" if graph is not None else "eager launches"),
            "launches_per_step": {"forward": launches[0], "backward": launches[1]},
            "kernels": breakdown,
            "profiled_ms_per_step": statistics.median(prof_ms),
            "step_ms_median": statistics.median(step_ms),
            "wall_s_timed_region": wall,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)


def workload_config(args, cfg, world):
    """The `config` object of both arms' JSON lines (the same workload, the same keys)."""
    return {"workload": args.workload, "T": cfg.T, "d": cfg.d, "r": cfg.r, "d_ff": cfg.d_ff,
            "S": cfg.S, "sigma": cfg.sigma, "kind": cfg.kind, "dense": cfg.dense,
            "checkpoint": cfg.checkpoint, "btp": cfg.btp, "attn": cfg.attn,
            "seq_len": cfg.seq_len if cfg.attn else None,
            "l2": "GPU arm: flushed before every timed step (256 MiB write, outside the step "
                  "events)",
            "parallelism": (f"data parallel over tokens: {cfg.T} per GPU, one NCCL all-reduce "
                            f"of the weight gradients per step" if world > 1 else "single GPU")}


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload with the current kernel source (every file the entry names,
    hashed in order); None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    entry = t.get(kernel)
    if not entry or entry.get("workload") != workload:
        return None
    import hashlib
    srcs = entry["source"] if isinstance(entry["source"], list) else [entry["source"]]
    h = hashlib.sha256()
    try:
        for name in srcs:
            with open(os.path.join(ROOT, "rank_bottleneck_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return entry["dram_bytes_per_launch"] if h.hexdigest()[:16] == entry["source_sha256_16"] else None


def run_e2e(args, cfg, inp, params, ws, act_names, dev, stream, world):
    """The step through the public binding with host buffers: per step, the
    host-to-device copies of its inputs (x, dy, dq, dk) from pinned memory, the
    forward and backward, and the device-to-host copies of y, dx and every weight
    gradient. Copies run on two copy streams, double-buffered, so that step i's
    compute overlaps step i+1's inputs and step i-1's results in flight; the
    timed region runs from the first input copy to the last result copy."""
    import torch
    from rank_bottleneck_gb300 import block as B
    dt = cfg.torch_dtype
    NB = 2  # buffer sets
    host_in = [{n: torch.from_numpy(inp[n]).to(dt).pin_memory() for n in act_names}
               for _ in range(NB)]
    dev_in = [{n: torch.empty(host_in[0][n].shape, dtype=dt, device=dev) for n in act_names}
              for _ in range(NB)]
    full = cfg.kind == "full" and not cfg.attn
    dev_out = [{"y": torch.empty(cfg.T, cfg.d, dtype=dt, device=dev),
                "dx": torch.empty(cfg.T, cfg.d, dtype=dt, device=dev),
                "q": torch.empty(cfg.T, cfg.d, dtype=dt, device=dev) if full else None,
                "k": torch.empty(cfg.T, cfg.d, dtype=dt, device=dev) if full else None}
               for _ in range(NB)]
    from rank_bottleneck_gb300.dp import GradBuffer, allreduce_grads
    gbufs = [GradBuffer(cfg, dev) for _ in range(NB)]
    grads = [gb.grads for gb in gbufs]
    host_out = [{"y": torch.empty(cfg.T, cfg.d, dtype=dt).pin_memory(),
                 "dx": torch.empty(cfg.T, cfg.d, dtype=dt).pin_memory()} for _ in range(NB)]
    host_grads = [{n: torch.empty(g.shape, dtype=dt).pin_memory() for n, g in grads[0].items()}
                  for _ in range(NB)]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values()) + \
        sum(t.numel() * t.element_size() for t in host_grads[0].values())
    # enough steps that the pipeline's first input copy and last result copy,
    # which nothing overlaps, are a small part of the timed region
    steps = min(max(args.steps, 50), 200)
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    done = [torch.cuda.Event() for _ in range(NB)]     # compute of the slot's last step
    landed = [torch.cuda.Event() for _ in range(NB)]   # the slot's inputs are on the device
    read = [torch.cuda.Event() for _ in range(NB)]     # the slot's results are on the host
    for e in done + read:
        e.record(stream)

    def compute(s):
        o = dev_out[s]
        B.forward(cfg, params, dev_in[s]["x"], ws, o["y"], o["q"], o["k"])
        B.backward(cfg, params, dev_in[s]["x"], ws, dev_in[s]["dy"], dev_in[s].get("dq"),
                   dev_in[s].get("dk"), o["dx"], grads[s])

    run = [compute]  # eager; replaced by graph replays once they are captured

    def e2e_step(i):
        s = i % NB
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(done[s])  # the step before that used this slot is done
            for n in act_names:
                dev_in[s][n].copy_(host_in[s][n], non_blocking=True)
            landed[s].record(h2d_stream)
        stream.wait_event(landed[s])
        stream.wait_event(read[s])          # its previous results have left the slot
        run[0](s)
        if world > 1:
            allreduce_grads(gbufs[s])
        done[s].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(done[s])
            o = dev_out[s]
            host_out[s]["y"].copy_(o["y"], non_blocking=True)
            host_out[s]["dx"].copy_(o["dx"], non_blocking=True)
            for n in grads[s]:
                host_grads[s][n].copy_(grads[s][n], non_blocking=True)
            read[s].record(d2h_stream)

    for i in range(NB):
        e2e_step(i)
    torch.cuda.synchronize()
    if not args.no_graph:
        # each buffer set's forward + backward captured once, replayed per step
        graphs = []
        for s_ in range(NB):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                compute(s_)
            graphs.append(g)
        torch.cuda.synchronize()
        run[0] = lambda s_: graphs[s_].replay()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(h2d_stream)
    for i in range(steps):
        e2e_step(i)
    b.record(d2h_stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    return {"value": world * steps * cfg.T / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps,
            "compute": "CUDA graph replay per buffer set" if not args.no_graph else "eager",
            "overlap": "double-buffered: step i's compute overlaps step i+1's input copies "
                       "and step i-1's result copies (two copy streams)"}


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    from rank_bottleneck_gb300.block import BlockConfig
    from rank_bottleneck_gb300.configs import WORKLOADS
    from rank_bottleneck_gb300.synth import make_block_inputs
    cfg = BlockConfig(**WORKLOADS[args.workload])
    # size each step so that warm-up + timed steps take about two minutes
    t64 = time_oracle(cfg, 64)
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(8, min(cfg.T, 64 * budget / max(t64, 1e-3))))
    if cfg.attn:
        rows = min(rows, 1024)  # one sequence of `rows` tokens
    c = oracle_sample_cfg(cfg, rows)
    inp = make_block_inputs(c.T, c.d, c.r, c.d_ff, kind=c.kind, dense=c.dense, dtype=c.dtype, seed=0)
    for _ in range(args.warmup):
        oracle_step(c, inp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(c, inp)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    sample = (f"{rows} of the workload's {cfg.T} token rows per step, fp64 numpy forward+backward"
              + (f"; attention over one sequence of {rows} tokens (the workload's are "
                 f"{cfg.seq_len})" if cfg.attn else ""))
    # ms_per_step is the measured time of one sampled step (rows_per_step token
    # rows), so that steps x ms_per_step is the timed region's length
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "rows_per_step": rows,
            "wall_s_timed_region": dt, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args, cfg, 1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="issue every launch through the C ABI each step instead of replaying "
                         "a captured CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    from rank_bottleneck_gb300.configs import DEFAULT, WORKLOADS
    args.workload = args.workload or DEFAULT
    if args.workload not in WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; one of {sorted(WORKLOADS)}")
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    rank, local_rank, world = dist_init()
    if args.gpus != world:
        raise SystemExit(f"--gpus {args.gpus} but {world} process(es) were launched: run N > 1 "
                         f"under torchrun with --nproc-per-node N")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local_rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
