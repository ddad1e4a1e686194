#!/usr/bin/env python
"""Benchmark: DDTree verify attention (MLA absorbed, page_size=1) on one GB300.

Default workload: Long TP8-slice, 65,536-token prefix, 32-node random tree,
8 heads, scattered indices into a 262,144-row pool (the 65k-prefix headline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Per step: an L2 flush (a write of 2x the L2 size, outside the timed events),
then one verify call replayed from a CUDA graph captured on an explicit
stream.  The call's device time, and the split-KV partial kernel's own time
(events the library records between its kernels), are taken with CUDA
events.  Rank 0 prints one JSON line.  N > 1 runs independent replicas (the
call does not shard across GPUs here), each rank on its own GPU.

--impl reference times the float64 CPU oracle on the host cores for the same
workload and metric (it is the only reference implementation this repo has).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import threading
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-attn µs/call & achieved HBM GB/s at 65k prefix; % of roofline"
UNIT = "us/call"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_scattered")
    ap.add_argument("--kernel", choices=["auto", "simt", "tc", "tc2"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-contiguous", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--step", choices=["verify", "accept", "relocate", "mask"], default="verify",
                    help="verify: the verify-attention call (the headline); accept: greedy "
                         "acceptance + KV commit after it; relocate: Tier-1 KV relocation; "
                         "mask: flattened custom tree mask -> parents")
    args = ap.parse_args()
    if args.workload == "long_scattered" and args.step not in ("verify", "mask"):
        args.workload = {"accept": "accept_long", "relocate": "relocate_long", "mask": "long_scattered"}[args.step]
    return args


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _arena(tensors, device):
    """One buffer (pinned when on the host) holding `tensors` at 256-byte aligned
    offsets, and a view of each with its dtype and shape."""
    offs, n = [], 0
    for t in tensors:
        n = (n + 255) // 256 * 256
        offs.append(n)
        n += t.numel() * t.element_size()
    n = (n + 255) // 256 * 256
    if str(device) == "cpu":
        buf = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    else:
        buf = torch.empty(n, dtype=torch.uint8, device=device)
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def _max_over_ranks(world, x: float) -> float:
    """The slowest rank's value (the timing rule for replicas); a host-side
    scalar exchange, on the GPU for NCCL groups and on the CPU for gloo."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of each dominant kernel, tied to the sha1 of the kernel's source
# when it was taken (profiles/ has the summaries and commands).  Any other
# version of the source reports null.
TRAFFIC = {
    "k_partial_tc2.cu": ("53337ef9fab02683862ab9e5d5950e4d1e46ac7e", 76216064 + 2440704),
    "k_accept.cu": ("016411fbe872d42040beebcfdb04b0f2d27eef9e", 8556032),
    "k_mask.cu": ("35de2ba635e46a78af91ca088bc100827946414a", 2114000),
    # mark + check + copy of one relocate_long call
    "k_relocate.cu": ("da69118f77628fdfc09c46764f90ab939e28b300", 13677 + 290407 + 75807700 + 13497894),
}


def _traffic(source: str):
    import hashlib
    sha, byts = TRAFFIC.get(source, (None, None))
    path = os.path.join(ROOT, "speculative_decode_tree_gb300", "csrc", source)
    if sha is None or not os.path.exists(path):
        return None
    with open(path, "rb") as f:
        return byts if hashlib.sha1(f.read()).hexdigest() == sha else None


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while the timed region runs.

    Reads NVML through ctypes every 2 ms (read-only queries; nothing is set),
    so even a region of a few milliseconds gets samples; falls back to
    `nvidia-smi -lms 100` when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        self.idx = device_index
        self.samples = []
        self.max_mhz = None
        self.stop = threading.Event()
        self.thread = None
        self.nvml = None
        self.handle = None
        self.smi = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device_index)
            bus = getattr(props, "pci_bus_id", None)
            ok = False
            if bus is not None:
                pci = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus, getattr(props, "pci_device_id", 0))
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(h)) != 0:
                raise RuntimeError("no NVML handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nvml, self.handle, self.ct = nv, h, ctypes
        except Exception:
            self.nvml = None

    def sample(self):
        """One NVML sample (also called between timed steps by the caller)."""
        if self.nvml is None:
            return
        ct, nv, h = self.ct, self.nvml, self.handle
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, ct.c_int(1), ct.byref(clk)) == 0:
            r = rs.value if self.reason_fn(h, ct.byref(rs)) == 0 else 0
            self.samples.append((float(clk.value), int(r)))

    def _loop(self):
        while not self.stop.is_set():
            self.sample()
            time.sleep(0.002)

    def __enter__(self):
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        else:
            try:
                self.smi_out = os.path.join("/tmp", f"ddtree_clocks_{os.getpid()}.csv")
                self.f = open(self.smi_out, "w")
                self.smi = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-i", str(self.idx), "-lms", "100"],
                    stdout=self.f, stderr=subprocess.DEVNULL)
            except Exception:
                self.smi = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)
        if self.smi is not None:
            self.smi.terminate()
            try:
                self.smi.wait(timeout=5)
            except Exception:
                self.smi.kill()
            self.f.close()
            for line in open(self.smi_out):
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append((float(parts[0]), int(parts[2], 16)))
                    self.max_mhz = max(self.max_mhz or 0.0, float(parts[1]))
                except (ValueError, IndexError):
                    continue

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples),
                "source": "nvml" if self.nvml is not None else "nvidia-smi"}


def _pct(xs, q):
    xs = sorted(xs)
    k = (len(xs) - 1) * q
    lo, hi = math.floor(k), math.ceil(k)
    return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)


def run_reference(args, world, rank):
    """Float64 CPU oracle on the host cores, same workload/metric/unit."""
    if rank != 0:
        return
    from oracle import verify_batched
    from speculative_decode_tree_gb300.workloads import algorithmic_cost, workload
    inp = workload(args.workload)
    cost = algorithmic_cost(inp)
    cores = torch.get_num_threads()

    def step():
        t0 = time.perf_counter()
        verify_batched(inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices, inp.kv_indptr,
                       inp.prefix_lens, inp.tree_parent, inp.sm_scale)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step()
    ts = [step() for _ in range(args.steps)]
    us = statistics.median(ts) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(ts) * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "batch": inp.batch,
                                        "heads": inp.n_heads, "nodes": inp.n_nodes,
                                        "prefixes": inp.prefix_lens.tolist(), "pool_rows": inp.pool_rows},
        "gbs": cost["bytes"] / (us * 1e-6) / 1e9, "tflops": cost["flops"] / (us * 1e-6) / 1e12,
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"full {args.workload} call per step, {args.steps} steps"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    from speculative_decode_tree_gb300 import binding as B
    from speculative_decode_tree_gb300.build import build
    from speculative_decode_tree_gb300.runner import DeviceVerify
    from speculative_decode_tree_gb300.workloads import algorithmic_cost, workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build()
    _barrier(world)
    peaks = _peaks()
    inp = workload(args.workload)
    cost = algorithmic_cost(inp)
    kernel = {"auto": None, "simt": B.DDTREE_KERNEL_SIMT, "tc": B.DDTREE_KERNEL_TC, "tc2": B.DDTREE_KERNEL_TC2}[args.kernel]
    dv = DeviceVerify(inp, device=str(dev), kernel=kernel)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    stage = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in stage + [t0, t1]:  # torch creates the CUDA event on its first record
        e.record(stream)
    assert all(e.cuda_event for e in stage)

    with torch.cuda.stream(stream):
        dv.run_timed(stage)  # first call outside capture (kernel attributes)
    stream.synchronize()
    # The timed graph is the plain call; a second graph with event records
    # between the two kernels gives the per-kernel split, timed separately.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        dv.run()
    graph_split = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_split, stream=stream):
        dv.run_timed(stage)

    def one_step():
        with torch.cuda.stream(stream):
            flush.zero_()
            t0.record(stream)
            graph.replay()
            t1.record(stream)
        stream.synchronize()
        return t0.elapsed_time(t1) * 1e3

    for _ in range(args.warmup):
        one_step()
    _barrier(world)
    torch.cuda.synchronize()
    calls = []
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            calls.append(one_step())
            clk.sample()
        torch.cuda.synchronize()
        _barrier(world)
        wall = time.perf_counter() - wall0
    status = dv.status(stream)

    partials, combines = [], []
    for i in range(args.warmup + args.steps):
        with torch.cuda.stream(stream):
            flush.zero_()
            graph_split.replay()
        stream.synchronize()
        if i >= args.warmup:
            partials.append(stage[0].elapsed_time(stage[1]) * 1e3)
            combines.append(stage[1].elapsed_time(stage[2]) * 1e3)

    call_us = _max_over_ranks(world, statistics.median(calls))
    mean_call_us = _max_over_ranks(world, statistics.mean(calls))
    partial_us = _max_over_ranks(world, statistics.mean(partials))
    value = call_us / world  # replicas: calls of the whole job per unit time

    # The same call against the defragmented (contiguous) copy of the pool.
    contiguous_us = None
    if args.workload == "long_scattered" and not args.no_contiguous:
        dvc = DeviceVerify(workload("long_contiguous"), device=str(dev), kernel=kernel)
        gc = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            dvc.run()
        stream.synchronize()
        with torch.cuda.graph(gc, stream=stream):
            dvc.run()
        cs = []
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                flush.zero_()
                t0.record(stream)
                gc.replay()
                t1.record(stream)
            stream.synchronize()
            if i >= args.warmup:
                cs.append(t0.elapsed_time(t1) * 1e3)
        contiguous_us = statistics.median(cs)
        del dvc, gc

    # End to end through the C ABI with host buffers: pinned H2D of the step's
    # inputs (queries, indices, parents, lengths) and D2H of out + lse.  The
    # inputs sit in one pinned host arena and one device arena (one H2D copy),
    # out and lse side by side in one device arena (one D2H copy); the call
    # takes views into the arenas, bound once (the buffers stay the same from
    # step to step, as in a decode loop).
    e2e = None
    if not args.no_e2e:
        src = (inp.q_latent, inp.q_rope, inp.kv_indices, inp.kv_indptr, inp.prefix_lens, inp.tree_parent)
        host_in, h_views = _arena(src, "cpu")
        for v, t in zip(h_views, src):
            v.copy_(t)
        dev_in, d_views = _arena(src, dev)
        dev_out, (out_v, lse_v) = _arena((dv.out, dv.lse), dev)
        host_out = torch.empty(dev_out.numel(), dtype=torch.uint8, pin_memory=True)
        h2d = host_in.numel()
        d2h = host_out.numel()
        q_lat, q_rope, kv_idx, kv_ptr, p_lens, t_par = d_views
        call = B.BoundVerify(dv.plan, q_lat, q_rope, dv.kv_pool, kv_idx, kv_ptr, p_lens, t_par, inp.sm_scale,
                             out_v, lse_v, dv.workspace)
        es = []
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                flush.zero_()
                t0.record(stream)
                dev_in.copy_(host_in, non_blocking=True)
                call(stream)
                host_out.copy_(dev_out, non_blocking=True)
                t1.record(stream)
            stream.synchronize()
            if i >= args.warmup:
                es.append(t0.elapsed_time(t1) * 1e3)
        # The arena path computes what the device-resident runs did.
        if not (torch.equal(out_v, dv.out) and torch.equal(lse_v, dv.lse)):
            raise RuntimeError("end-to-end call through the arenas differs from the device-resident call")
        e2e_us = _max_over_ranks(world, statistics.median(es)) / world
        e2e = {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import verify_batched
        ts = []
        tstart = time.perf_counter()
        while not ts or time.perf_counter() - tstart < args.cpu_seconds:
            a = time.perf_counter()
            verify_batched(inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices, inp.kv_indptr,
                           inp.prefix_lens, inp.tree_parent, inp.sm_scale)
            ts.append(time.perf_counter() - a)
        cpu = {"value": statistics.median(ts) * 1e6, "unit": UNIT, "cores": torch.get_num_threads(),
               "kind": "oracle",
               "sample": f"{len(ts)} full {args.workload} calls (float64, torch CPU), median"}

    if rank != 0:
        return
    flops, byts = cost["flops"], cost["bytes"]
    fused = bool(dv.plan.fused_combine)
    tc_peak = peaks["bf16_tflops"]
    achieved = flops / (partial_us * 1e-6) / 1e12
    roof_us = max(byts / (peaks["hbm_gbs"] * 1e9), flops / (tc_peak * 1e12)) * 1e6
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_call_us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "batch": inp.batch, "heads": inp.n_heads,
                   "nodes": inp.n_nodes, "prefixes": inp.prefix_lens.tolist(),
                   "pool_rows": inp.pool_rows, "index_mode": inp.meta["index_mode"],
                   "l2": "flushed between steps (2x L2 write, outside the timed events)",
                   "timing": "CUDA graph replay on an explicit stream; CUDA events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "p10_us": _pct(calls, 0.1), "p90_us": _pct(calls, 0.9),
        "gbs": byts / (call_us * 1e-6) / 1e9,
        "tflops": flops / (call_us * 1e-6) / 1e12,
        "roofline_us": roof_us, "roofline_frac_call": roof_us / call_us,
        "partial_kernel_us": partial_us,
        # With the merge in the partial kernel there is no combine launch (the
        # event pair around the absent launch only measures event overhead).
        "combine_kernel_us": None if fused else statistics.mean(combines),
        "merge": "in the partial kernel (cooperative launch)" if fused else "combine_kernel",
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": achieved / tc_peak,
                     "traffic": _traffic({1: "k_partial_simt.cu", 2: "k_partial_tc.cu",
                                          3: "k_partial_tc2.cu"}[dv.plan.kernel])
                     if args.workload == "long_scattered" else None,
                     "peak_source": peaks["source"] + " bf16 burst (MEASURED_PEAKS.json)",
                     "kernel": "split-KV partial (%s)%s" % ({1: "simt", 2: "tcgen05 pair", 3: "tcgen05 cta_group::2 quad"}[dv.plan.kernel],
                                                            " incl. the split merge" if fused else "")},
        "alg_bytes": byts, "alg_flops": flops,
        "plan": dv.plan.as_dict(),
        "contiguous_us": contiguous_us,
        "scatter_over_contiguous": (call_us / contiguous_us) if contiguous_us else None,
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": (1 if fused else 2) * args.steps,
        "status_word": status, "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)


ACCEPT_METRIC = "greedy tree acceptance + KV commit µs/call (argmax over the target logits, walk, commit)"


def run_accept(args, world, rank, local):
    """Greedy acceptance + commit: device time of one call (CUDA graph, L2
    flushed between steps), its HBM roofline (one pass over the logits), the
    end-to-end call with host buffers, and the oracle on the host cores."""
    from speculative_decode_tree_gb300.build import build
    from speculative_decode_tree_gb300.runner import DeviceAccept
    from speculative_decode_tree_gb300.workloads import accept_workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build()
    _barrier(world)
    peaks = _peaks()
    inp = accept_workload(args.workload)
    da = DeviceAccept(inp, device=str(dev))
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        da.run(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        da.run(stream)

    def one_step():
        with torch.cuda.stream(stream):
            flush.zero_()
            t0.record(stream)
            graph.replay()
            t1.record(stream)
        stream.synchronize()
        return t0.elapsed_time(t1) * 1e3

    for _ in range(args.warmup):
        one_step()
    _barrier(world)
    calls = []
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            calls.append(one_step())
            clk.sample()
        torch.cuda.synchronize()
        _barrier(world)
        wall = time.perf_counter() - wall0
    status = da.status(stream)
    call_us = _max_over_ranks(world, statistics.median(calls))
    value = call_us / world

    # Algorithmic bytes: the logits once, drafts + parents + the tree rows'
    # indices read, the five outputs written.
    B_, T_, V_ = inp.batch, inp.n_nodes, inp.vocab
    byts = B_ * (T_ + 1) * V_ * 2 + B_ * T_ * 4 * 3 + B_ * 8 + B_ * 4 * 2 + B_ * T_ * 4 * 3
    hbm = peaks["hbm_gbs"]
    achieved = byts / (call_us * 1e-6) / 1e9

    e2e = None
    if not args.no_e2e:
        host_in = [t.pin_memory() for t in (inp.logits, inp.draft_tokens, inp.tree_parent)]
        dev_in = [da.logits, da.draft, da.parent]
        outs = [da.accept_len, da.next_token, da.accepted_nodes, da.commit_indices, da.freed_indices]
        host_out = [torch.empty_like(o, device="cpu").pin_memory() for o in outs]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        es = []
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                flush.zero_()
                t0.record(stream)
                for h, d in zip(host_in, dev_in):
                    d.copy_(h, non_blocking=True)
                da.run(stream)
                for h, d in zip(host_out, outs):
                    h.copy_(d, non_blocking=True)
                t1.record(stream)
            stream.synchronize()
            if i >= args.warmup:
                es.append(t0.elapsed_time(t1) * 1e3)
        e2e = {"value": _max_over_ranks(world, statistics.median(es)) / world, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import accept_batched
        ts = []
        tstart = time.perf_counter()
        while not ts or time.perf_counter() - tstart < min(args.cpu_seconds, 10.0):
            a = time.perf_counter()
            accept_batched(inp.logits, inp.draft_tokens, inp.tree_parent, inp.kv_indices, inp.kv_indptr,
                           inp.prefix_lens)
            ts.append(time.perf_counter() - a)
        cpu = {"value": statistics.median(ts) * 1e6, "unit": UNIT, "cores": torch.get_num_threads(),
               "kind": "oracle", "sample": f"{len(ts)} full {args.workload} calls (numpy/torch CPU), median"}
    if rank != 0:
        return
    line = {
        "metric": ACCEPT_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(calls) / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 logits, int32 indices", "data": "synthetic",
        "config": {"workload": args.workload, "batch": B_, "nodes": T_, "vocab": V_,
                   "prefixes": inp.prefix_lens.tolist(), "tree": inp.meta["tree"],
                   "l2": "flushed between steps (2x L2 write, outside the timed events)",
                   "timing": "CUDA graph replay on an explicit stream; CUDA events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "p10_us": _pct(calls, 0.1), "p90_us": _pct(calls, 0.9),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm,
                     "traffic": _traffic("k_accept.cu") if args.workload == "accept_long" else None,
                     "peak_source": peaks["source"] + " HBM copy (MEASURED_PEAKS.json)",
                     "kernel": "whole call (argmax pass + walk)"},
        "alg_bytes": byts, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk.summary(),
        "gpu_launches": 2 * args.steps, "status_word": status, "wall_s_timed_region": wall,
        "mean_accept_len": float(da.accept_len.float().mean().item()),
    }
    print(json.dumps(line), flush=True)


RELOCATE_METRIC = "Tier-1 KV relocation µs/call (scattered rows -> one contiguous region, indices rewritten)"


def run_relocate(args, world, rank, local):
    """Tier-1 relocation of one request's rows: device time of one call (its
    indices reset outside the timed events before every step), HBM roofline
    (each row read once and written once), e2e with host buffers, oracle."""
    from speculative_decode_tree_gb300 import binding as B
    from speculative_decode_tree_gb300.build import build
    from speculative_decode_tree_gb300.workloads import relocate_workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build()
    _barrier(world)
    peaks = _peaks()
    inp = relocate_workload(args.workload)
    pool = inp.kv_pool.to(dev)
    orig = inp.kv_indices.to(dev)
    idx = orig.clone()
    ptr = inp.kv_indptr.to(dev)
    dst = inp.dest_base.to(dev)
    old = torch.empty_like(idx)
    total = int(inp.kv_indptr[-1])
    ws = torch.empty(B.ddtree_relocate_kv_workspace_size(inp.pool_rows), dtype=torch.uint8, device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        B.ddtree_relocate_kv(pool, idx, ptr, dst, total, ws, old, stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        B.ddtree_relocate_kv(pool, idx, ptr, dst, total, ws, old, stream)

    def one_step():
        with torch.cuda.stream(stream):
            idx.copy_(orig)
            flush.zero_()
            t0.record(stream)
            graph.replay()
            t1.record(stream)
        stream.synchronize()
        return t0.elapsed_time(t1) * 1e3

    for _ in range(args.warmup):
        one_step()
    _barrier(world)
    calls = []
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            calls.append(one_step())
            clk.sample()
        torch.cuda.synchronize()
        _barrier(world)
        wall = time.perf_counter() - wall0
    status = B.ddtree_verify_mla_check(ws, stream)
    call_us = _max_over_ranks(world, statistics.median(calls))
    value = call_us / world
    byts = total * (2 * 1152 + 3 * 4) + inp.batch * 12
    hbm = peaks["hbm_gbs"]
    achieved = byts / (call_us * 1e-6) / 1e9

    e2e = None
    if not args.no_e2e:
        host_in = [inp.kv_indices.pin_memory(), inp.kv_indptr.pin_memory(), inp.dest_base.pin_memory()]
        dev_in = [idx, ptr, dst]
        host_out = [torch.empty_like(idx, device="cpu").pin_memory(), torch.empty_like(old, device="cpu").pin_memory()]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        es = []
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                flush.zero_()
                t0.record(stream)
                for h, d in zip(host_in, dev_in):
                    d.copy_(h, non_blocking=True)
                B.ddtree_relocate_kv(pool, idx, ptr, dst, total, ws, old, stream)
                host_out[0].copy_(idx, non_blocking=True)
                host_out[1].copy_(old, non_blocking=True)
                t1.record(stream)
            stream.synchronize()
            if i >= args.warmup:
                es.append(t0.elapsed_time(t1) * 1e3)
        e2e = {"value": _max_over_ranks(world, statistics.median(es)) / world, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import relocate
        ts = []
        tstart = time.perf_counter()
        while not ts or time.perf_counter() - tstart < min(args.cpu_seconds, 10.0):
            a = time.perf_counter()
            relocate(inp.kv_pool, inp.kv_indices, inp.kv_indptr, inp.dest_base)
            ts.append(time.perf_counter() - a)
        cpu = {"value": statistics.median(ts) * 1e6, "unit": UNIT, "cores": torch.get_num_threads(),
               "kind": "oracle", "sample": f"{len(ts)} full {args.workload} calls (torch CPU, row by row), median"}
    if rank != 0:
        return
    line = {
        "metric": RELOCATE_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(calls) / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 rows (copied bit for bit), int32 indices",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": inp.batch, "rows": total, "pool_rows": inp.pool_rows,
                   "l2": "flushed between steps (2x L2 write, outside the timed events)",
                   "timing": "CUDA graph replay on an explicit stream; CUDA events; indices reset before each step",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "p10_us": _pct(calls, 0.1), "p90_us": _pct(calls, 0.9),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm,
                     "traffic": _traffic("k_relocate.cu") if args.workload == "relocate_long" else None,
                     "peak_source": peaks["source"] + " HBM copy (MEASURED_PEAKS.json)",
                     "kernel": "whole call (mark + check + copy)"},
        "alg_bytes": byts, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk.summary(),
        "gpu_launches": 3 * args.steps, "status_word": status, "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)


MASK_METRIC = "flattened custom tree mask -> parent array µs/call (one pass over the mask)"


def run_mask(args, world, rank, local):
    """Mask reader on the trees and prefixes of a verify workload: device time
    of one call (graph, L2 flushed), HBM roofline over the mask bytes, e2e
    with the mask copied from host memory, oracle on the host cores."""
    from speculative_decode_tree_gb300 import binding as B
    from speculative_decode_tree_gb300.build import build
    from speculative_decode_tree_gb300.workloads import flat_tree_masks, workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build()
    _barrier(world)
    peaks = _peaks()
    inp = workload(args.workload)
    flat_h, indptr_h = flat_tree_masks(inp.tree_parent, inp.prefix_lens)
    flat, indptr = flat_h.to(dev), indptr_h.to(dev)
    plen = inp.prefix_lens.to(dev)
    Bn, T = inp.batch, inp.n_nodes
    parent = torch.empty(Bn, T, dtype=torch.int32, device=dev)
    anc = torch.empty(Bn, T, dtype=torch.int64, device=dev)
    ws = torch.empty(B.ddtree_tree_from_mask_workspace_size(Bn, T), dtype=torch.uint8, device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        B.ddtree_tree_from_mask(flat, indptr, plen, parent, ws, anc, stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        B.ddtree_tree_from_mask(flat, indptr, plen, parent, ws, anc, stream)

    def one_step():
        with torch.cuda.stream(stream):
            flush.zero_()
            t0.record(stream)
            graph.replay()
            t1.record(stream)
        stream.synchronize()
        return t0.elapsed_time(t1) * 1e3

    for _ in range(args.warmup):
        one_step()
    _barrier(world)
    calls = []
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            calls.append(one_step())
            clk.sample()
        torch.cuda.synchronize()
        _barrier(world)
        wall = time.perf_counter() - wall0
    status = B.ddtree_verify_mla_check(ws, stream)
    call_us = _max_over_ranks(world, statistics.median(calls))
    value = call_us / world
    byts = flat.numel() + (Bn + 1) * 8 + Bn * 4 + Bn * T * (4 + 8)
    hbm = peaks["hbm_gbs"]
    achieved = byts / (call_us * 1e-6) / 1e9

    e2e = None
    if not args.no_e2e:
        host_in = [flat_h.pin_memory(), indptr_h.pin_memory(), inp.prefix_lens.pin_memory()]
        dev_in = [flat, indptr, plen]
        host_out = [torch.empty_like(parent, device="cpu").pin_memory()]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        es = []
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                flush.zero_()
                t0.record(stream)
                for h, d in zip(host_in, dev_in):
                    d.copy_(h, non_blocking=True)
                B.ddtree_tree_from_mask(flat, indptr, plen, parent, ws, anc, stream)
                host_out[0].copy_(parent, non_blocking=True)
                t1.record(stream)
            stream.synchronize()
            if i >= args.warmup:
                es.append(t0.elapsed_time(t1) * 1e3)
        e2e = {"value": _max_over_ranks(world, statistics.median(es)) / world, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import trees_from_flat_mask
        flat_np, ind_l, pl_l = flat_h.numpy(), indptr_h.tolist(), inp.prefix_lens.tolist()
        ts = []
        tstart = time.perf_counter()
        while not ts or time.perf_counter() - tstart < min(args.cpu_seconds, 10.0):
            a = time.perf_counter()
            trees_from_flat_mask(flat_np, ind_l, pl_l, T)
            ts.append(time.perf_counter() - a)
        cpu = {"value": statistics.median(ts) * 1e6, "unit": UNIT, "cores": torch.get_num_threads(),
               "kind": "oracle", "sample": f"{len(ts)} full calls on {args.workload}'s trees (numpy), median"}
    if rank != 0:
        return
    line = {
        "metric": MASK_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(calls) / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8 mask, int32/u64 outputs", "data": "synthetic",
        "config": {"workload": args.workload, "batch": Bn, "nodes": T, "prefixes": inp.prefix_lens.tolist(),
                   "mask_bytes": int(flat.numel()),
                   "l2": "flushed between steps (2x L2 write, outside the timed events)",
                   "timing": "CUDA graph replay on an explicit stream; CUDA events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "p10_us": _pct(calls, 0.1), "p90_us": _pct(calls, 0.9),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": _traffic("k_mask.cu") if args.workload == "long_scattered" else None,
                     "peak_source": peaks["source"] + " HBM copy (MEASURED_PEAKS.json)",
                     "kernel": "mask_kernel"},
        "alg_bytes": byts, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk.summary(),
        "gpu_launches": args.steps, "status_word": status, "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)


def main():
    args = _args()
    world, rank, local = _dist()
    try:
        if args.step != "verify" and args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the verify step only"}))
        elif args.step == "accept":
            run_accept(args, world, rank, local)
        elif args.step == "relocate":
            run_relocate(args, world, rank, local)
        elif args.step == "mask":
            run_mask(args, world, rank, local)
        elif args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
