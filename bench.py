#!/usr/bin/env python3
"""Benchmark: MoE expert-parallel dispatch + combine on one GB300.

A step is one whole pass of the path over one batch of N simulated ranks' tokens:
routing layout (histogram, scans, placements) -> dispatch send (pack + per-peer write) ->
dispatch recv (grouped expert rows) -> identity expert -> combine send (reverse shuffle +
per-peer write back) -> combine recv (fp32 weighted sum -> bf16). The library runs each
phase as one kernel per token batch (dispatch: pack, write and shuffle; combine: reverse
shuffle, write back and sum), every buffer as the separate steps leave it; the same step
with the separate kernels is reported beside it (`separate_moves`). The bf16 step is one
moe_forward call, which runs the pass in the library's token micro-batches; the fp8 step
calls the layout, moe_dispatch, the identity expert and moe_combine (in token batches) so
that the expert can be timed apart and left out. The same step in one batch is reported
beside it (`one_batch`), as are the per-kernel times of whole-pass launches (roofline),
both with L2 carried over from kernel to kernel as in the step and cold (L2 evicted before
each kernel).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

With no --config the JSON line's top level is the largest workload (EP16, T=512, H=4096,
every token routed to rank 0's experts: 3.4 GB of algorithmic bytes per step) and
`per_config` carries the other three full-size workloads measured the same way in the same
run (EP8 bf16, EP32 zipf bf16, EP64 fp8), each checked against the CPU oracle; --config C
measures workload C alone.

Prints one JSON line (rank 0). `value` is tokens/s over all GPUs: (N*T tokens per
simulated group) x (GPUs) / (step time, max over ranks), timed with CUDA events on the
launching stream, inputs resident in HBM, L2 flushed (a write of 2x the L2 size, then a
read of another 2x, so no dirty flush lines are written back inside the step) before
every timed step. With --gpus G > 1 (torchrun, one process per GPU) the workload's N
simulated ranks are split over the G GPUs in rank windows of N/G ranks: the routing is
all-gathered, each GPU's kernels move the rows inside its window, and the slices between
windows go over NCCL point-to-point (strong scaling: the job processes N*T tokens per step);
--replicas runs an independent copy of the whole group on every GPU instead.
"""
from __future__ import annotations

import argparse
import ctypes
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
KERNELS = ["route_count", "layout_maps", "quant_fp8", "pack", "scatter", "unpack", "expert",
           "combine_pack", "combine_scatter", "combine_reduce", "route_scan", "pack_push", "combine_push",
           "combine_partial", "combine_sum", "dispatch_split", "quant_pack", "dispatch_dedicated", "dispatch_fused",
           "quant_dispatch_fused", "combine_fused"]
HEADLINE_CONFIG = 4          # the largest workload: the line's top level
OTHER_CONFIGS = (1, 2, 3)    # measured in the same run, reported under per_config
L2_NOTE = "flushed before every timed step (write of 2x L2, then read of 2x L2)"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--config", type=int, default=None,
                   help="measure this workload alone (default: workload 4 at the top level and 1, 2, 3 "
                        "under per_config)")
    p.add_argument("--shape", default="", help="custom workload N,T,H,E,R[,payload[,cap[,routing]]] (seed 11; "
                   "routing uniform, zipf or skew0, default uniform) instead of --config, e.g. for profiling "
                   "a smaller footprint")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--mover", choices=["auto", "tma", "ldg"], default="auto")
    p.add_argument("--tma-stages", type=int, default=0)
    p.add_argument("--ctas-per-sm", type=int, default=0)
    p.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    p.add_argument("--staged-quant", action="store_true",
                   help="fp8: quantise into a staging buffer, then pack (two kernels) instead of inside the pack")
    p.add_argument("--batches", type=int, default=0,
                   help="token batches of the batched passes (0: the library's automatic choice)")
    p.add_argument("--one-batch", action="store_true",
                   help="run moe_forward (and the host pass) as one token batch instead of micro-batches")
    p.add_argument("--separate-moves", action="store_true",
                   help="run each phase as separate kernels (pack, write, shuffle; combine pack, write, sum: "
                        "MOE_FLAG_SEPARATE_MOVES) instead of one kernel per phase and token batch")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="CPU work for the oracle baseline of the top-level workload (single thread, then "
                        "all cores)")
    p.add_argument("--other-cpu-seconds", type=float, default=3.0,
                   help="CPU work for the single-thread oracle baseline of each per_config workload")
    p.add_argument("--sharded", action="store_true",
                   help="the expert-parallel path of --gpus > 1 also on one GPU (one window holding every rank)")
    p.add_argument("--replicas", action="store_true",
                   help="with --gpus > 1: an independent replica of the whole group on every GPU instead of "
                        "expert parallelism over the GPUs")
    p.add_argument("--profile-step", choices=["pass", "split", "dedicated"], default=None,
                   help="run only W + K steps of one kind (L2 flushed before each) and print a short summary, "
                        "for the ncu captures in profiles/: 'pass' the whole pass in one batch (whole-pass "
                        "launches), 'split' and 'dedicated' the direct-push step with the split-phase dispatch "
                        "(without or with dedicated space)")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------- distributed helpers

def workload_of(args) -> workloads.Workload:
    if not args.shape:
        return workloads.config(HEADLINE_CONFIG if args.config is None else args.config)
    f = args.shape.split(",")
    N, T, H, E, R = (int(v) for v in f[:5])
    payload = f[5] if len(f) > 5 else "bf16"
    cap = int(f[6]) if len(f) > 6 else 0
    routing = f[7] if len(f) > 7 else "uniform"
    return workloads.Workload(f"custom-N{N}-T{T}-H{H}-E{E}-R{R}-{payload}-cap{cap}-{routing}", N, T, H, E, R,
                              payload, routing, 11, cap=cap)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(backend: str):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return dist if ws > 1 else None


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (identity on one rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 20 ms while running; summarised on stop()."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)  # let it emit its first sample
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        self.proc.wait()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [r for r in rows if r[2] > 0.25 * max(x[2] for x in rows)] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------- byte accounting

def algorithmic_bytes(wl: workloads.Workload, P: int, Pk: int) -> dict:
    """Bytes each kernel must move per launch: payload reads + writes (index, weight and layout
    traffic is under 1% for the data kernels and is counted only for the layout kernels).
    P = routed pairs, Pk = pairs kept in the grouped buffers (P unless capacity dropped some)."""
    N, T, H, E, R, L = wl.N, wl.T, wl.H, wl.E, wl.R, wl.L
    B, cap, RB = wl.row_bytes, wl.cap_eff, wl.RB
    tok = N * T
    P_all = tok * R
    return {
        "route_count": 8 * P_all + 4 * N * E * ((T * R + 255) // 256),
        "route_scan": 4 * N * E * (2 * ((T * R + 255) // 256) + 5) + 4 * 3 * N * N,
        "layout_maps": 36 * P_all + 4 * E * cap + 4 * N * RB,
        "quant_fp8": tok * 2 * H + tok * B,
        "pack": tok * B + P * B,
        "scatter": 2 * P * B,
        "unpack": 2 * P * B,
        "expert": Pk * (H + H // 32) + Pk * 2 * H if wl.payload == "fp8" else 2 * Pk * 2 * H,
        "combine_pack": 2 * Pk * 2 * H,
        "combine_scatter": 2 * Pk * 2 * H,
        "combine_reduce": Pk * 2 * H + tok * 2 * H,
        "pack_push": tok * B + P * B,
        "quant_pack": tok * 2 * H + P * B,
        "combine_push": 2 * Pk * 2 * H,
        "dispatch_split": tok * B + P * B + 2 * Pk * B,
        "dispatch_dedicated": tok * B + P * B + 2 * Pk * B,
        "dispatch_fused": tok * B + 2 * P * B + Pk * B,
        "quant_dispatch_fused": tok * 2 * H + 2 * P * B + Pk * B,
        "combine_fused": Pk * 2 * H + 2 * Pk * 2 * H + tok * 2 * H,
    }


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        if d.get("hbm_gbs"):
            return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_sha() -> str:
    """Hash of the files that define the kernels the traffic table measures and their launch
    configuration (device helpers, layout, movers, numerics); host-side changes elsewhere
    (entry points, streams) leave it unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_routing_count_gb300", "csrc")
    for f in ("common.cuh", "layout.cu", "movers.cu", "numerics.cu"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def dram_table(workload: str):
    """The committed ncu DRAM capture for this workload (profiles/ncu_traffic.json), if it was
    taken on these kernel sources: per kernel the DRAM bytes of one whole-pass launch on a
    smaller case of the same shape family ('cold': L2 flushed before the kernel; 'warm_l2': L2
    carried over from the previous kernel, as in the step) and the pairs of that case."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    if d.get("source_sha") != kernel_source_sha():
        return None
    return d.get("workloads", {}).get(workload)


def scaled_dram(table, mode: str, kernel: str, pairs: int):
    """DRAM bytes of one whole-pass launch of `kernel` at `pairs` routed pairs, scaled from the
    capture by the pairs processed (every data kernel's traffic is per pair or per token, and
    the captured case has the same R, H and payload); None without a capture."""
    if not table:
        return None
    v = table.get(mode, {}).get(kernel)
    if v is None or not table.get("pairs"):
        return None
    return int(round(v * pairs / table["pairs"]))


# ---------------------------------------------------------------------------- CPU oracle baseline

def cpu_baseline(wl, inp, seconds: float, all_cores: bool = True) -> dict:
    import oracle
    b = oracle.alloc_step(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload)
    oracle.run_step(b, inp["x"], inp["idx"], inp["w"])   # first touch of the buffers, untimed
    times = []
    t_end = time.perf_counter() + seconds
    while len(times) < 3 or time.perf_counter() < t_end:
        t0 = time.perf_counter()
        oracle.run_step(b, inp["x"], inp["idx"], inp["w"])
        times.append(time.perf_counter() - t0)
    med = statistics.median(times)
    out = {"value": wl.N * wl.T / med, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{len(times)} whole steps of {wl.name} (all {wl.N} simulated ranks), median "
                     f"{med * 1e3:.1f} ms, single-threaded C"}
    if all_cores:
        out["all_cores"] = cpu_baseline_all_cores(wl, inp, seconds, b)
    out["out"] = b["out"]
    return out


def step_resident_bytes(b: dict) -> int:
    """Bytes a step's buffers touch: the receive regions and the grouped rows are sized for the
    worst case but written only where the N*T*R pairs land."""
    N, T, H, E, R, cap, payload = b["dims"]
    sparse = ("recv", "csend", "ex", "exq", "exs", "ey")
    dense = sum(a.nbytes for k, a in b.items() if isinstance(a, np.ndarray) and k not in sparse)
    grouped = b["B"] if payload != "fp8" else H + H // 32 + 2 * H
    return dense + N * T * R * (b["B"] + 2 * H + grouped)


def cpu_baseline_all_cores(wl, inp, seconds: float, b0: dict) -> dict:
    """The same oracle on every host core: one thread per core, each running whole steps of the
    workload on its own buffers (the oracle's C calls release the GIL). Threads are capped so
    their buffers take at most a quarter of the free host memory."""
    import threading

    import oracle
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    nthr = max(1, min(cores, free // 4 // max(1, step_resident_bytes(b0))))
    bufs = [b0] + [oracle.alloc_step(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload) for _ in range(nthr - 1)]
    for b in bufs[1:]:
        oracle.run_step(b, inp["x"], inp["idx"], inp["w"])   # first touch, untimed
    done = [0] * nthr
    start = threading.Barrier(nthr + 1)
    t_end = [0.0]

    def work(i):
        start.wait()
        while time.perf_counter() < t_end[0]:
            oracle.run_step(bufs[i], inp["x"], inp["idx"], inp["w"])
            done[i] += 1

    th = [threading.Thread(target=work, args=(i,)) for i in range(nthr)]
    for t in th:
        t.start()
    t_end[0] = time.perf_counter() + seconds
    t0 = time.perf_counter()
    start.wait()
    for t in th:
        t.join()
    el = time.perf_counter() - t0
    steps = sum(done)
    return {"value": round(steps * wl.N * wl.T / el, 1), "unit": "tokens/s", "cores": nthr, "kind": "oracle",
            "sample": f"{nthr} threads, each running whole steps of {wl.name} on its own buffers for "
                      f"{seconds:.0f} s ({steps} steps in all, {el:.1f} s wall); tokens of all steps / wall time"}


# ---------------------------------------------------------------------------- our arm

def _kernel_entry(ab: dict, name: str, ts: list, peak: float, K: int) -> dict:
    us = statistics.fmean(ts) * 1e3
    gbs = ab[name] / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "us_median": round(statistics.median(ts) * 1e3, 2),
            "launches_per_step": len(ts) / K, "bytes": ab[name], "gbs": round(gbs, 1), "frac": round(gbs / peak, 3)}


def measure(wl, args, dist, device, peak: float, peak_kind: str, cpu_seconds: float, all_cores: bool) -> dict:
    """Times one workload in every mode (see the module docstring) and returns its JSON object."""
    import torch
    from combine_routing_count_gb300 import KERNEL_NAMES, MoeEP, MoeProf, lib
    ws, rank, local = dist_env()
    inp = workloads.make_inputs(wl)
    ep = MoeEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, alias_buffers=(wl.payload == "bf16"),
               flags={"auto": 0, "ldg": 1, "tma": 4}[args.mover] | (2 if args.no_pdl else 0) |
               (0x10 if args.staged_quant else 0) | (0x40 if args.one_batch else 0) |
               (0x80 if args.separate_moves else 0), tma_stages=args.tma_stages,
               ctas_per_sm=args.ctas_per_sm, batches=args.batches)
    x = torch.from_numpy(inp["x"]).view(torch.bfloat16).to(device)
    idx = torch.from_numpy(inp["idx"]).to(device)
    w = torch.from_numpy(inp["w"]).to(device)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=device)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
    flush_sum = torch.empty((), dtype=torch.float32, device=device)

    def flush_l2():
        """Evicts the step's data from L2: a write of 2x L2, then a read of another 2x L2,
        so that the write's dirty lines are written back here and not inside the timed step."""
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sum)

    fp8 = wl.payload == "fp8"
    K = args.steps

    def step():
        ep.forward(x, idx, w)

    step_default = step

    def quant_dispatch_send():
        """fp8 dispatch send as moe_forward does it: quantisation inside the pack, or staged."""
        if args.staged_quant:
            ep.quantize(x)
            ep.dispatch_send(ep.xq)
        else:
            ep.quantize_dispatch_send(x)

    def step_split(e0, e1, e2, e3):
        """One pass with events around the identity expert (the grouped-GEMM stand-in), so
        its time can be left out of the step as the scope's tokens/s definition asks: the
        layout, moe_dispatch (in its token batches), the expert, moe_combine."""
        e0.record(stream)
        ep.layout_step(idx)
        if args.staged_quant:
            quant_dispatch_send()
            ep.dispatch_recv()
        else:
            ep.dispatch(x)
        e1.record(stream)
        ep.expert_identity()
        e2.record(stream)
        ep.combine(w)
        e3.record(stream)

    if args.profile_step:
        # Only one kind of step, for ncu: W + K steps, L2 flushed before each.
        ep.layout.flags |= 0x40
        if args.profile_step != "pass":
            ep.layout.flags |= 8
        for _ in range(args.warmup + K):
            flush_l2()
            if args.profile_step == "pass":
                step()
                continue
            ep.layout_step(idx)
            xin = x
            if fp8:
                ep.quantize(x)
                xin = ep.xq
            if args.profile_step == "split":
                ep.dispatch_split(xin)
            else:
                ep.dispatch_dedicated(xin, idx, 16)
            ep.expert_identity()
            ep.combine_send()
            ep.combine_recv(w)
        code, bits = ep.status()
        return {"profile_step": args.profile_step, "workload": wl.name, "steps": args.warmup + K, "status": code}

    for _ in range(args.warmup):
        flush_l2()
        step()
    code, bits = ep.status()
    if code != 0:
        raise RuntimeError(f"device status {code} bits {bits:#x}")
    lay = ep.layout_arrays()
    P = int(lay["rtot"].sum().item())
    Pk = int((lay["slot"] >= 0).sum().item())

    # per-step, per-kernel events through the library's profiling hook
    profs = []
    for _ in range(K):
        pr = MoeProf()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(KERNEL_NAMES))]
        for i, e in enumerate(evs):
            e.record(stream)
            pr.events[i] = e.cuda_event
        profs.append((pr, evs))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()

    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(vis[local] if local < len(vis) else local)

    # The variant steps below differ from the default step in one phase only: the other phase
    # is the same whole-phase call (moe_dispatch / moe_combine).
    def step_partial():
        ep.layout_step(idx)
        ep.dispatch(x)
        ep.expert_identity()
        ep.combine_partial(w)

    def step_splitphase():
        ep.layout_step(idx)
        if fp8:
            ep.quantize(x)
            ep.dispatch_split(ep.xq)
        else:
            ep.dispatch_split(x)
        ep.expert_identity()
        ep.combine(w)

    DED_K = 16   # dedicated rows per (receiver, sender)

    def step_dedicated():
        ep.layout_step(idx)
        if fp8:
            ep.quantize(x)
            ep.dispatch_dedicated(ep.xq, idx, DED_K)
        else:
            ep.dispatch_dedicated(x, idx, DED_K)
        ep.expert_identity()
        ep.combine(w)

    def kernel_region(step=step, cold=False):
        """Timed region: per-kernel CUDA events (the library records one pair around each of
        its launches on this stream) give each kernel's duration for the roofline. The pass
        runs as one batch here (MOE_FLAG_ONE_BATCH), so every kernel is its whole-pass launch
        and no two of them overlap; the step region below times the default micro-batches.
        With cold, the library reads a 2x-L2 buffer before each bracketed launch, so every
        kernel starts with nothing of the pass in L2 (the profiling hook's flush option)."""
        barrier(dist, device)
        torch.cuda.synchronize()
        flags0 = ep.layout.flags
        ep.layout.flags = flags0 | 0x40
        for i in range(K):
            flush_l2()
            pr, _ = profs[i]
            pr.n = 0
            pr.flush = flush_r.data_ptr() if cold else None
            pr.flush_bytes = flush_r.numel() * 4 if cold else 0
            ep.layout.prof = ctypes.pointer(pr)
            step()
        torch.cuda.synchronize()
        ep.layout.prof = None
        ep.layout.flags = flags0
        per_kernel = {}
        for pr, evs in profs:
            for j in range(pr.n):
                name = KERNEL_NAMES[pr.kernel[j]]
                per_kernel.setdefault(name, []).append(evs[2 * j].elapsed_time(evs[2 * j + 1]))
        return per_kernel

    def step_region(step=step):
        """Timed region: whole steps only (no events between the kernels, so consecutive
        kernels overlap launch and drain as they do in use); gives the step time."""
        barrier(dist, device)
        torch.cuda.synchronize()
        n0 = lib().moe_launch_count()
        split = fp8 and step is step_default
        if split:
            mids = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
            for i in range(K):
                flush_l2()
                step_split(starts[i], mids[i][0], mids[i][1], ends[i])
        else:
            for i in range(K):
                flush_l2()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
        torch.cuda.synchronize()
        barrier(dist, device)
        launches = lib().moe_launch_count() - n0
        code, bits = ep.status()
        if code != 0:
            raise RuntimeError(f"device status {code} bits {bits:#x}")
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        expert_ms = None
        if split:
            ex = [m0.elapsed_time(m1) for m0, m1 in mids]
            step_ms = [t - x_ for t, x_ in zip(step_ms, ex)]
            expert_ms = statistics.fmean(ex)
        step_region.median_ms = statistics.median(step_ms)
        return statistics.fmean(step_ms), expert_ms, launches

    # token batches of the timed step: moe_forward's micro-batches for bf16; the fp8 step
    # (which times the identity expert apart) runs moe_dispatch and moe_combine in theirs
    step_batches = int(lib().moe_batches(ctypes.byref(ep.dims), ctypes.byref(ep.layout), 2 if fp8 else 0))
    sampler.start()
    per_kernel = kernel_region()
    per_kernel_cold = kernel_region(cold=True)
    mean_ms, expert_ms, launches = step_region()
    median_ms = step_region.median_ms
    # the same step in one token batch (MOE_FLAG_ONE_BATCH), reported beside the default
    flags0 = ep.layout.flags
    ep.layout.flags = flags0 | 0x40
    one_ms, _, _ = step_region()
    # the same step with the four moves apart (MOE_FLAG_SEPARATE_MOVES, or without it when
    # the run asked for separate moves), reported beside the default
    ep.layout.flags = flags0 ^ 0x80
    other_ms, _, _ = step_region()
    # and the separate kernels' whole-pass launches, each with its own roofline fraction
    ep.layout.flags = flags0 | 0x80
    pk_sep = kernel_region() if not args.separate_moves else {}
    ep.layout.flags = flags0
    one_ms_all = max_over_ranks(one_ms, dist, device)
    other_ms_all = max_over_ranks(other_ms, dist, device)
    mean_ms_all = max_over_ranks(mean_ms, dist, device)
    tokens = wl.N * wl.T * ws
    value = tokens / (mean_ms_all * 1e-3)

    ab = algorithmic_bytes(wl, P, Pk)
    table = dram_table(wl.name)
    kernels = {}
    for name, ts in per_kernel.items():
        if name == "expert":
            continue  # the identity expert stands in for the grouped GEMM; reported separately
        kernels[name] = _kernel_entry(ab, name, ts, peak, K)
        tc = per_kernel_cold.get(name)
        if tc:
            us_c = statistics.fmean(tc) * 1e3
            kernels[name]["us_cold"] = round(us_c, 2)
            kernels[name]["frac_cold"] = round(ab[name] / (us_c * 1e-6) / 1e9 / peak, 3)
            db = scaled_dram(table, "cold", name, P)
            kernels[name]["dram_bytes"] = db
            kernels[name]["dram_frac"] = None if db is None else round(db / (us_c * 1e-6) / 1e9 / peak, 3)
    dom = max(kernels, key=lambda k: kernels[k]["us"] * kernels[k]["launches_per_step"])
    step_bytes = sum(ab[k] * kernels[k]["launches_per_step"] for k in kernels)
    # DRAM bytes of the one-batch pass: its data kernels' captures (the layout kernels move
    # well under 1 MB and have none)
    captured = [k for k in kernels if table and k in table.get("warm_l2", {})]
    dram_step = sum(scaled_dram(table, "warm_l2", k, P) for k in captured) if captured else None

    # The same step in direct-push mode (the pack writes into the owners' receive rows and
    # the combine send into the sources' rows, fusing away both per-peer write steps).
    ep.layout.flags |= 8
    for _ in range(args.warmup):
        flush_l2()
        step()
    pk_push = kernel_region()
    push_ms, _, _ = step_region()
    ep.layout.flags &= ~8
    sep_kernels = {}
    for name, ts in pk_sep.items():
        if name == "expert":
            continue
        e = _kernel_entry(ab, name, ts, peak, K)
        sep_kernels[name] = {k: e[k] for k in ("us", "gbs", "frac")}
    push_kernels = {}
    # with direct push the one-kernel phases write no send and no receive-order rows
    tokB, H2 = wl.N * wl.T * wl.row_bytes, 2 * wl.H
    ab_push = dict(ab, dispatch_fused=tokB + P * wl.row_bytes + Pk * wl.row_bytes,
                   quant_dispatch_fused=wl.N * wl.T * H2 + P * wl.row_bytes + Pk * wl.row_bytes,
                   combine_fused=2 * Pk * H2 + wl.N * wl.T * H2)
    for name, ts in pk_push.items():
        if name == "expert":
            continue
        e = _kernel_entry(ab_push, name, ts, peak, K)
        push_kernels[name] = {k: e[k] for k in ("us", "gbs", "frac")}
    push_bytes = sum(ab_push[k] for k in push_kernels)
    push_ms_all = max_over_ranks(push_ms, dist, device)

    # The same step with the combine's weighted sum started on the expert side: one row per
    # (token, destination rank) group instead of one per (token, expert) pair.
    slot_np = lay["slot"].cpu().numpy().reshape(-1, wl.R)
    own = np.where(slot_np >= 0, inp["idx"].reshape(-1, wl.R) // wl.L, -1)
    G = int(sum(len(set(r[r >= 0].tolist())) for r in own))
    ab["combine_partial"] = Pk * 2 * wl.H + G * 2 * wl.H
    ab["combine_sum"] = G * 2 * wl.H + wl.N * wl.T * 2 * wl.H
    for _ in range(args.warmup):
        flush_l2()
        step_partial()
    pk_part = kernel_region(step_partial)
    part_ms, _, _ = step_region(step_partial)
    if fp8:   # the identity expert is inside this step; take it out as for the main step
        part_ms -= expert_ms
    part_kernels = {}
    for name, ts in pk_part.items():
        if name.startswith("combine_p") or name == "combine_sum":
            e = _kernel_entry(ab, name, ts, peak, K)
            part_kernels[name] = {k: e[k] for k in ("us", "gbs", "frac")}
    part_ms_all = max_over_ranks(part_ms, dist, device)

    # The direct-push step with dispatch as one split-phase launch: every CTA pushes its
    # share of rows and signals per slice, then waits for each pair's slice and shuffles it.
    ep.layout.flags |= 8
    for _ in range(args.warmup):
        flush_l2()
        step_splitphase()
    pk_sp = kernel_region(step_splitphase)
    sp_ms, _, _ = step_region(step_splitphase)
    ep.layout.flags &= ~8
    if fp8:
        sp_ms -= expert_ms
    sp_kernels = {}
    for name, ts in pk_sp.items():
        if name == "dispatch_split":
            e = _kernel_entry(ab, name, ts, peak, K)
            sp_kernels[name] = {k: e[k] for k in ("us", "gbs", "frac")}
    sp_ms_all = max_over_ranks(sp_ms, dist, device)

    # Split-phase dispatch with per-sender dedicated space and piggybacked routing counts.
    ep.layout.flags |= 8
    for _ in range(args.warmup):
        flush_l2()
        step_dedicated()
    pk_ded = kernel_region(step_dedicated)
    ded_ms, _, _ = step_region(step_dedicated)
    ep.layout.flags &= ~8
    if fp8:
        ded_ms -= expert_ms
    ded_kernels = {}
    for name, ts in pk_ded.items():
        if name == "dispatch_dedicated":
            e = _kernel_entry(ab, name, ts, peak, K)
            ded_kernels[name] = {k: e[k] for k in ("us", "gbs", "frac")}
    ded_ms_all = max_over_ranks(ded_ms, dist, device)

    # fp8: the whole pass through moe_forward in its micro-batches, the identity expert
    # included (the headline step above calls the entry points one by one to exclude it)
    fwd_ms, fwd_batches = None, None
    if fp8:
        def step_forward():
            ep.forward(x, idx, w)
        for _ in range(args.warmup):
            flush_l2()
            step_forward()
        fwd_ms, _, _ = step_region(step_forward)
        fwd_ms = max_over_ranks(fwd_ms, dist, device)
        fwd_batches = int(lib().moe_batches(ctypes.byref(ep.dims), ctypes.byref(ep.layout), 0))

    # end to end through the C ABI with host buffers: H2D inputs, the pass, D2H output
    h_x = torch.from_numpy(inp["x"]).view(torch.bfloat16).pin_memory()
    h_idx = torch.from_numpy(inp["idx"]).pin_memory()
    h_w = torch.from_numpy(inp["w"]).pin_memory()
    h_out = torch.empty((wl.N, wl.T, wl.H), dtype=torch.bfloat16).pin_memory()

    def e2e_region():
        for _ in range(3):
            ep.forward_host(h_x, h_idx, h_w, h_out, x, idx, w)
        torch.cuda.synchronize()
        e_start = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e_end = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for i in range(K):
            flush_l2()
            e_start[i].record(stream)
            ep.forward_host(h_x, h_idx, h_w, h_out, x, idx, w)
            e_end[i].record(stream)
        torch.cuda.synchronize()
        ok = bool(np.array_equal(h_out.view(torch.int16).numpy(), ep.out.cpu().view(torch.int16).numpy()))
        return max_over_ranks(statistics.fmean(s.elapsed_time(e) for s, e in zip(e_start, e_end)), dist, device), ok

    # Default: the copy-engine pipeline over token batches; then one batch (copies in, the
    # pass, copy out); then the kernels on the pinned host memory itself (NVLink-C2C).
    e2e_ms, e2e_same = e2e_region()
    e2e_nb = lib().moe_batches(ctypes.byref(ep.dims), ctypes.byref(ep.layout), 1)
    f0 = ep.layout.flags
    ep.layout.flags = f0 | 0x40
    e2e_one_ms, _ = e2e_region()
    ep.layout.flags = f0 | 0x20
    e2e_mapped_ms, _ = e2e_region()
    ep.layout.flags = f0
    clocks = sampler.stop()
    h2d = inp["x"].nbytes + inp["idx"].nbytes + inp["w"].nbytes
    d2h = wl.N * wl.T * wl.H * 2

    eff_gbs = step_bytes / (mean_ms * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(mean_ms_all, 4), "ms_per_step_median": round(median_ms, 4),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8+bf16" if wl.payload == "fp8" else "bf16",
        "data": "synthetic (seeded; DeepSeek-V3/Kimi-K2-shaped routing, identity experts)",
        "config": {"workload": wl.name, "N_ranks_simulated": wl.N, "T": wl.T, "H": wl.H, "E": wl.E, "R": wl.R,
                   "payload": wl.payload, "routing": wl.routing, "seed": wl.seed, "l2": L2_NOTE},
        "launch": {"mover": args.mover, "pdl": not args.no_pdl,
                   "fp8_quant": ("staged" if args.staged_quant else "inside the pack") if fp8 else None,
                   "micro_batches": step_batches,
                   "parallelism": f"{ws} independent replica(s) of the {wl.N}-rank group"},
        "effective_gbs": round(eff_gbs, 1),
        "effective_frac": round(eff_gbs / peak, 3),
        "effective_note": "step-level algorithmic bytes / step time: an effective rate, not HBM throughput; it "
                          "exceeds the copy bandwidth because consecutive moves read part of their input from "
                          "L2 (alternating unit order, token batches). HBM figures: dram_* and each kernel's "
                          "dram_frac",
        "dram_bytes_per_step": dram_step,
        "dram_gbs_one_batch": None if dram_step is None else round(dram_step / (one_ms * 1e-3) / 1e9, 1),
        "dram_note": "DRAM bytes of one whole pass in one batch (sum over its kernels, L2 carried over from "
                     "kernel to kernel; ncu on a smaller case of the same shape, scaled by pairs: "
                     "profiles/ncu_traffic.json) / the one-batch step time; the micro-batched step keeps "
                     "more rows in L2, so it moves at most these bytes",
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["gbs"], "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": kernels[dom]["frac"],
                     "achieved_cold": (round(ab[dom] / (kernels[dom]["us_cold"] * 1e-6) / 1e9, 1)
                                       if "us_cold" in kernels[dom] else None),
                     "frac_cold": kernels[dom].get("frac_cold"),
                     "dram_frac": kernels[dom].get("dram_frac"),
                     "bytes_per_launch": ab[dom],
                     "traffic": scaled_dram(table, "cold", dom, P),
                     "traffic_warm_l2": scaled_dram(table, "warm_l2", dom, P),
                     "traffic_source": (None if not table else
                                        f"ncu capture of {table.get('shape')} ({table.get('pairs')} pairs), "
                                        f"scaled by pairs x{P / table['pairs']:.3g}"),
                     "launch": "whole-pass launch, timed in the per-kernel region (one batch): frac with L2 "
                               "carried over as in the step, frac_cold with L2 evicted before the kernel, "
                               "dram_frac = DRAM bytes / cold time"},
        "kernels": kernels,
        "direct_push": {"value": round(tokens / (push_ms_all * 1e-3), 1), "unit": "tokens/s",
                        "ms_per_step": round(push_ms_all, 4),
                        "effective_gbs": round(push_bytes / (push_ms * 1e-3) / 1e9, 1),
                        "kernels": push_kernels,
                        "note": "same results; the dispatch writes straight into the owners' receive rows "
                                "and the combine into the sources' rows, so neither the send rows nor "
                                "the receive-order rows are written"},
        "sender_side_combine": {"value": round(tokens / (part_ms_all * 1e-3), 1), "unit": "tokens/s",
                                "ms_per_step": round(part_ms_all, 4), "groups": G, "pairs": Pk,
                                "kernels": part_kernels,
                                "note": "combine sums each token's experts per destination rank on the "
                                        "expert side (bf16 partial rows), then over ranks on the source"},
        "split_phase_dispatch": {"value": round(tokens / (sp_ms_all * 1e-3), 1), "unit": "tokens/s",
                                 "ms_per_step": round(sp_ms_all, 4), "kernels": sp_kernels,
                                 "note": "direct-push step whose dispatch is one cooperative launch: "
                                         "push rows, signal per (destination, source) slice, wait "
                                         "(bounded), shuffle into the grouped rows"},
        "split_phase_dedicated": {"value": round(tokens / (ded_ms_all * 1e-3), 1), "unit": "tokens/s",
                                  "ms_per_step": round(ded_ms_all, 4), "dedicated_rows": DED_K,
                                  "kernels": ded_kernels,
                                  "note": "direct-push step whose dispatch is one cooperative launch with "
                                          "per-sender dedicated rows and the routing counts piggybacked; "
                                          "receivers compute their offsets from the reported counts"},
        "e2e": {"value": round(tokens / (e2e_ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": f"moe_forward_host (C ABI): copy engines move each of {e2e_nb} token batches in and "
                        "out of pinned host memory while the device works on the other batches",
                "batches": e2e_nb,
                "one_batch": {"value": round(tokens / (e2e_one_ms * 1e-3), 1), "ms_per_step": round(e2e_one_ms, 4),
                              "path": "MOE_FLAG_ONE_BATCH: copies in, the pass, copy out on one stream"},
                "out_equals_device_path": e2e_same,
                "mapped": {"value": round(tokens / (e2e_mapped_ms * 1e-3), 1),
                           "ms_per_step": round(e2e_mapped_ms, 4),
                           "path": "MOE_FLAG_HOST_MAPPED: kernels read the pinned inputs and write the output "
                                   "over the host link (two token batches on two streams)"}},
        "identity_expert": None if expert_ms is None else {
            "ms_per_step": round(expert_ms, 4), "kernel_us": round(statistics.fmean(per_kernel["expert"]) * 1e3, 2),
            "note": "fp8 dequantisation standing in for the grouped GEMM; excluded from ms_per_step and value"},
        "one_batch": {"value": round(tokens / (one_ms_all * 1e-3), 1), "unit": "tokens/s",
                      "ms_per_step": round(one_ms_all, 4),
                      "note": "the same step as one token batch (MOE_FLAG_ONE_BATCH): identical results; "
                              "the default splits it into token batches over two streams"},
        ("fused_moves" if args.separate_moves else "separate_moves"): {
            "value": round(tokens / (other_ms_all * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(other_ms_all, 4),
            **({"kernels": sep_kernels} if sep_kernels else {}),
            "note": "the same step with each phase "
                    + ("in one kernel per token batch (the default)" if args.separate_moves else
                       "as separate kernels (MOE_FLAG_SEPARATE_MOVES: pack, write, shuffle; combine pack, "
                       "write, sum); identical results")},
        "forward_with_expert": None if fwd_ms is None else {
            "value": round(tokens / (fwd_ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(fwd_ms, 4),
            "micro_batches": fwd_batches,
            "note": "moe_forward in its micro-batches with the identity expert inside the step (not excluded)"},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(wl, inp, cpu_seconds, all_cores=all_cores)
        gpu_out = ep.out.cpu().view(torch.int16).numpy().view(np.uint16)
        out["parity"] = {"out_bit_exact_vs_oracle": bool(np.array_equal(gpu_out, cb.pop("out")))}
        out["cpu_baseline"] = cb
    return out


def compact(r: dict) -> dict:
    """A per_config entry: the workload's headline figures, its roofline, per-kernel table,
    end-to-end figure, CPU baseline and parity, without the long notes."""
    keep = ("value", "unit", "ms_per_step", "ms_per_step_median", "dtype", "config", "launch", "effective_gbs",
            "effective_frac", "dram_bytes_per_step", "dram_gbs_one_batch", "roofline", "kernels", "parity",
            "cpu_baseline", "gpu_launches", "clocks")
    c = {k: r[k] for k in keep if k in r}
    c["roofline"] = {k: v for k, v in r["roofline"].items() if k != "launch"}
    c["e2e"] = {k: r["e2e"][k] for k in ("value", "unit", "ms_per_step", "h2d_bytes_per_step",
                                         "d2h_bytes_per_step", "batches", "out_equals_device_path")}
    for k in ("one_batch", "separate_moves", "fused_moves", "direct_push", "sender_side_combine",
              "split_phase_dispatch", "split_phase_dedicated", "forward_with_expert", "identity_expert"):
        if r.get(k) is not None:
            c[k] = {kk: vv for kk, vv in r[k].items() if kk not in ("note", "path")}
    return c


def measure_sharded(wl, args, dist, device, peak: float, peak_kind: str) -> dict:
    """The workload's N simulated ranks split over the GPUs of the job, one rank window per
    process (combine_routing_count_gb300.sharded): a step gathers the routing, lays it out,
    plans the slices, dispatches (kernels inside the window, NCCL point-to-point slices
    between windows), runs the identity expert and combines back. Strong scaling: the whole
    job processes the workload's N*T tokens per step."""
    import torch
    from combine_routing_count_gb300 import KERNEL_NAMES, MoeProf, lib
    from combine_routing_count_gb300.sharded import DistTransport, ShardedEP, sharded_forward, window_bounds
    ws, rank, local = dist_env()
    if wl.N % ws:
        raise SystemExit(f"{wl.name}: {wl.N} simulated ranks do not split evenly over {ws} GPUs")
    b = window_bounds(wl.N, ws)
    lo, hi = b[rank], b[rank + 1]
    inp = workloads.make_inputs(wl)
    sh = ShardedEP(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, bounds=b, me=rank)
    x = torch.from_numpy(inp["x"][lo:hi].copy()).view(torch.bfloat16).to(device)
    idx = torch.from_numpy(inp["idx"][lo:hi].copy()).to(device)
    w = torch.from_numpy(inp["w"][lo:hi].copy()).to(device)
    tr = DistTransport()
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=device)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
    flush_sum = torch.empty((), dtype=torch.float32, device=device)

    def flush_l2():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sum)

    def step():
        sharded_forward([sh], tr, [x], [idx], [w])

    K = args.steps
    for _ in range(args.warmup):
        flush_l2()
        step()
    code, bits = sh.status()
    if code != 0:
        raise RuntimeError(f"device status {code} bits {bits:#x}")
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(vis[local] if local < len(vis) else local)
    sampler.start()
    # per-kernel events of this window's launches (one batch)
    profs = []
    for _ in range(K):
        pr = MoeProf()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(KERNEL_NAMES))]
        for i, e in enumerate(evs):
            e.record(stream)
            pr.events[i] = e.cuda_event
        profs.append((pr, evs))
    barrier(dist, device)
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2()
        pr, _ = profs[i]
        pr.n = 0
        sh.layout.prof = ctypes.pointer(pr)
        step()
    torch.cuda.synchronize()
    sh.layout.prof = None
    per_kernel = {}
    for pr, evs in profs:
        for j in range(pr.n):
            per_kernel.setdefault(KERNEL_NAMES[pr.kernel[j]], []).append(evs[2 * j].elapsed_time(evs[2 * j + 1]))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(dist, device)
    torch.cuda.synchronize()
    n0 = lib().moe_launch_count()
    for i in range(K):
        flush_l2()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(dist, device)
    launches = lib().moe_launch_count() - n0
    mean_ms = statistics.fmean(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms_all = max_over_ranks(mean_ms, dist, device)
    # end to end: this window's inputs from pinned host memory, its output back
    h_x = torch.from_numpy(inp["x"][lo:hi].copy()).view(torch.bfloat16).pin_memory()
    h_idx = torch.from_numpy(inp["idx"][lo:hi].copy()).pin_memory()
    h_w = torch.from_numpy(inp["w"][lo:hi].copy()).pin_memory()
    h_out = torch.empty(tuple(sh.out.shape), dtype=torch.bfloat16).pin_memory()
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(dist, device)
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2()
        e_s[i].record(stream)
        x.copy_(h_x, non_blocking=True)
        idx.copy_(h_idx, non_blocking=True)
        w.copy_(h_w, non_blocking=True)
        step()
        h_out.copy_(sh.out, non_blocking=True)
        e_e[i].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    e2e_ms = max_over_ranks(statistics.fmean(s.elapsed_time(e) for s, e in zip(e_s, e_e)), dist, device)
    code, bits = sh.status()
    # parity: every window checks its output against the oracle's rows of its ranks
    import oracle
    o = oracle.forward(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload, inp["x"], inp["idx"], inp["w"])
    ok = bool(np.array_equal(sh.out.cpu().view(torch.int16).numpy().view(np.uint16), o["out"][lo:hi])) and code == 0
    ok_all = max_over_ranks(0.0 if ok else 1.0, dist, device) == 0.0
    lay = sh.layout_arrays()
    P = int(lay["rtot"].sum().item())
    Pk = int((lay["slot"] >= 0).sum().item())
    ab = algorithmic_bytes(wl, P, Pk)
    n = hi - lo
    frac_w = n / wl.N   # the window's share of the source-side work
    # the window's algorithmic bytes per kernel (rows it moves; no pair of these workloads is
    # dropped for capacity, so routed rows are kept rows)
    C = lay["C"].cpu().numpy().astype(np.int64)
    B, H2 = wl.row_bytes, 2 * wl.H
    pw = int(C[lo:hi, :].sum())          # pairs the window's tokens route
    rw = int(C[:, lo:hi].sum())          # rows the window's ranks receive
    inner = int(C[lo:hi, lo:hi].sum())   # rows whose both ends are in the window
    tin = n * wl.T * (2 * wl.H)          # the window's token rows (bf16)
    wbytes = {"pack": n * wl.T * B + pw * B, "quant_pack": tin + pw * B, "scatter": 2 * inner * B,
              "unpack": 2 * rw * B, "combine_pack": 2 * rw * H2, "combine_scatter": 2 * inner * H2,
              "combine_reduce": pw * H2 + n * wl.T * H2}
    kernels = {}
    for name, ts in per_kernel.items():
        if name == "expert":
            continue
        us = statistics.fmean(ts) * 1e3
        kernels[name] = {"us": round(us, 2), "launches_per_step": len(ts) / K}
        if name in wbytes:
            gbs = wbytes[name] / (us * 1e-6) / 1e9
            kernels[name].update({"bytes": wbytes[name], "gbs": round(gbs, 1), "frac": round(gbs / peak, 3)})
    dom = max((k for k in kernels if "bytes" in kernels[k]), key=lambda k: kernels[k]["us"], default=None)
    tokens = wl.N * wl.T
    slices = {k: len(v) for k, v in sh.plans.items()}
    return {
        "metric": METRIC, "value": round(tokens / (ms_all * 1e-3), 1), "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_all, 4), "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "fp8+bf16" if wl.payload == "fp8" else "bf16",
        "data": "synthetic (seeded; DeepSeek-V3/Kimi-K2-shaped routing, identity experts)",
        "config": {"workload": wl.name, "N_ranks_simulated": wl.N, "T": wl.T, "H": wl.H, "E": wl.E, "R": wl.R,
                   "payload": wl.payload, "routing": wl.routing, "seed": wl.seed, "l2": L2_NOTE,
                   "parallelism": f"expert parallel: {ws} GPUs, {n} of the {wl.N} ranks each (rank windows), "
                                  "routing all-gathered, slices between windows over NCCL point-to-point"},
        "roofline": {"bound": "hbm", "kernel": dom, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "achieved": kernels[dom]["gbs"] if dom else None, "frac": kernels[dom]["frac"] if dom else None,
                     "bytes_per_launch": kernels[dom]["bytes"] if dom else None, "traffic": None,
                     "launch": "rank 0's window: the rows its kernels move in one step (one batch)"},
        "kernels_rank0": kernels,
        "window_share": frac_w,
        "slices": {"dispatch_send": slices[(0, 1)], "dispatch_recv": slices[(0, 0)],
                   "combine_send": slices[(1, 1)], "combine_recv": slices[(1, 0)]},
        "e2e": {"value": round(tokens / (e2e_ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": (x.numel() * 2 + idx.numel() * 4 + w.numel() * 4) * ws,
                "d2h_bytes_per_step": sh.out.numel() * 2 * ws,
                "path": "each window's inputs copied in from pinned host memory and its output back, inside the step"},
        "parity": {"out_bit_exact_vs_oracle": ok_all},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "bytes_per_step_algorithmic": sum(ab[k] for k in ("pack", "scatter", "unpack", "combine_pack",
                                                          "combine_scatter", "combine_reduce")),
    }


def run_ours(args):
    import torch
    from combine_routing_count_gb300 import build
    build.build()
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init("nccl")
    peak, peak_kind = measured_peak()

    wl = workload_of(args)
    if (ws > 1 and not args.replicas) or args.sharded:
        if dist is None:   # --sharded on one GPU: a one-process group, the same code path
            import socket

            import torch.distributed as tdist
            with socket.socket() as sk:
                sk.bind(("127.0.0.1", 0))
                port = sk.getsockname()[1]
            tdist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                                     device_id=device)
            dist = tdist
        out = measure_sharded(wl, args, dist, device, peak, peak_kind)
        if dist is not None:
            dist.destroy_process_group()
        if rank == 0:
            print(json.dumps(out), file=_OUT, flush=True)
        return
    if args.profile_step:
        r = measure(wl, args, dist, device, peak, peak_kind, 0.0, False)
        if rank == 0:
            print(json.dumps(r), file=_OUT, flush=True)
        return
    out = measure(wl, args, dist, device, peak, peak_kind, args.cpu_seconds, True)
    if args.config is None and not args.shape:
        out["per_config"] = {}
        for cfg in OTHER_CONFIGS:
            gc.collect()
            torch.cuda.empty_cache()
            wc = workloads.config(cfg)
            out["per_config"][wc.name] = compact(
                measure(wc, args, dist, device, peak, peak_kind, args.other_cpu_seconds, False))
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), file=_OUT, flush=True)


_OUT = sys.stdout   # where the JSON line goes (main() points it at the real stdout)

# ---------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle, as it stands, timed on the host cores: K whole steps of the same workload."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    wl = workload_of(args)
    inp = workloads.make_inputs(wl)
    b = oracle.alloc_step(wl.N, wl.T, wl.H, wl.E, wl.R, wl.cap, wl.payload)
    oracle.run_step(b, inp["x"], inp["idx"], inp["w"])   # first touch
    for _ in range(max(0, args.warmup - 1)):
        oracle.run_step(b, inp["x"], inp["idx"], inp["w"])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.run_step(b, inp["x"], inp["idx"], inp["w"])
        times.append(time.perf_counter() - t0)
    mean = statistics.fmean(times)
    value = wl.N * wl.T / mean
    sample = f"{args.steps} whole steps of {wl.name} (all {wl.N} simulated ranks), single-threaded C oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8+bf16" if wl.payload == "fp8" else "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "N_ranks_simulated": wl.N, "T": wl.T, "H": wl.H, "E": wl.E, "R": wl.R,
                   "payload": wl.payload, "routing": wl.routing, "seed": wl.seed},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def _stdout_for_the_json_line():
    """The process's stdout for the one JSON line; everything else that writes to file
    descriptor 1 (NCCL prints its version there, at exit) goes to stderr."""
    sys.stdout.flush()
    fd = os.dup(1)
    os.dup2(2, 1)
    return os.fdopen(fd, "w")


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        global _OUT
        _OUT = _stdout_for_the_json_line()
        run_ours(args)


if __name__ == "__main__":
    main()
