#!/usr/bin/env python
"""Benchmark of the triangle multiplicative update on B300 (one JSON line on rank 0).

A step is one pass of the whole path over one synthetic input: the projection,
contraction and finish kernels of the outgoing update and then of the incoming
update of the four-chain-complex workload (N = 3605 tokens, c_z = c_h = 128,
bf16, full mask), both on the same resident z. ``value`` is the algorithmic
FLOP rate of the whole job, 2 * (2 N^3 c_h + 2 (4 c_h c_z + c_z^2 + c_z c_h) N^2)
per step, over the device-timed region (CUDA events, max over ranks).

Under torchrun each rank runs an independent replica on its own GPU (the update
has no data-path exchange step), so per-GPU work is fixed and scaling is weak.

``--impl reference`` times the float64 CPU oracle instead (rank 0 only), each
step a bounded sample of the same workload.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ms per tri-mult update & TFLOP/s (frac of bf16 peak) at N=768/3605/6500"
FALLBACK_PEAKS = {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6400.0}
K2_SOURCE = os.path.join(ROOT, "pair_representation_boltz_b300", "csrc", "k2_contract.cu")
K2_PROFILE = os.path.join(ROOT, "profiles", "k2_contract_complex3605.md")


def flops_update(N: int, c_z: int, c_h: int) -> float:
    """Algorithmic FLOPs of one update: the contraction plus every projection (masked pairs counted)."""
    return 2.0 * N ** 3 * c_h + 2.0 * (4 * c_h * c_z + c_z * c_z + c_z * c_h) * N ** 2


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def profiled_traffic():
    """dram bytes per contraction launch from the committed ncu summary, if the kernel is unchanged."""
    if not os.path.exists(K2_PROFILE):
        return None
    text = open(K2_PROFILE).read()
    h = re.search(r"device_code_sha256:\s*([0-9a-f]{64})", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not h or not t:
        return None
    cur = device_code_sha256(K2_SOURCE)
    return float(t.group(1)) if cur == h.group(1) else None


def pcie_roofline(torch, host_src, host_dst, bytes_per_step, ms_per_step):
    """The host-buffer step's bound: its copies at the host link's measured rate, copies in and out at
    once on two streams (pinned buffers of one z each, best of four), as the step overlaps them."""
    dev_in = torch.empty_like(host_src, device="cuda")
    dev_out = torch.empty_like(host_dst, device="cuda")
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    best = None
    for _ in range(4):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        with torch.cuda.stream(s_in):
            dev_in.copy_(host_src, non_blocking=True)
        with torch.cuda.stream(s_out):
            host_dst.copy_(dev_out, non_blocking=True)
        torch.cuda.current_stream().wait_stream(s_in)
        torch.cuda.current_stream().wait_stream(s_out)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None or ms < best else best
    nbytes = host_src.numel() * host_src.element_size() + host_dst.numel() * host_dst.element_size()
    peak = nbytes / (best * 1e-3) / 1e9
    achieved = bytes_per_step / (ms_per_step * 1e-3) / 1e9
    del dev_in, dev_out
    return {"bound": "pcie", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": "host-to-device and device-to-host copies of one z each at once, measured here"}


def device_code_sha256(path: str) -> str:
    """sha256 of a kernel file's device code: the text before its first host launcher definition
    ("cudaError_t launch_"), so that edits to the host-side launcher alone keep a profile's counters
    attached to the kernel they were taken from."""
    text = open(path, "rb").read()
    cut = text.find(b"\ncudaError_t launch_")
    return hashlib.sha256(text if cut < 0 else text[:cut]).hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms, device):
    """The largest of ms over the ranks of the default process group (a job ends with its slowest rank);
    ms itself when there is no group or a single rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput: the units every rank processed, summed over the ranks, over the slowest
    rank's time in ms (each rank runs its own replica of the workload: weak scaling)."""
    return world * units_per_rank / (ms / 1e3)


# Algorithmic bytes per pair of the bandwidth-bound passes (c = 128): the projection reads z (256 B)
# and writes a and b (512 B); the finish reads x in its default fp16 storage (128 channels x 2 B) and z,
# and writes out (256 B each).
PROJECT_BYTES_PER_PAIR = 256 + 512
FINISH_BYTES_PER_PAIR = 128 * 2 + 256 + 256


# Tensor work the projection executes per pair: two 128 x 128 products (projection and gate) for each of
# a and b, each with bf16 hi and lo weight terms, 2 FLOP per multiply-add.
PROJECT_TENSOR_FLOP_PER_PAIR = 2 * 2 * 2 * 128 * 128 * 2


def add_kernel_bandwidth(kernels, ktime, peaks):
    """GB/s of the projection and finish kernels over their algorithmic bytes, and its fraction of the
    measured copy bandwidth; for the projection also its executed tensor rate against the bf16 peaks (the
    hi + lo weights make its tensor work, not its bytes, the larger bound)."""
    for name, per_pair in (("project", PROJECT_BYTES_PER_PAIR), ("finish", FINISH_BYTES_PER_PAIR)):
        v = ktime[name]
        if v["ms"] > 0 and name in kernels:
            gbs = v["units"] * per_pair / (v["ms"] / 1e3) / 1e9
            kernels[name]["gbs"] = gbs
            kernels[name]["frac_of_hbm"] = gbs / peaks["hbm_gbs"]
            kernels[name]["bytes_per_pair"] = per_pair
            if name == "project":
                tf = v["units"] * PROJECT_TENSOR_FLOP_PER_PAIR / (v["ms"] / 1e3) / 1e12
                kernels[name]["tensor_tflops"] = tf
                kernels[name]["frac_of_bf16_peak"] = tf / peaks["bf16_tflops"]
                kernels[name]["frac_of_bf16_sustained"] = tf / peaks["bf16_tflops_sustained"]
                kernels[name]["tensor_flop_per_pair"] = PROJECT_TENSOR_FLOP_PER_PAIR


def host_cores():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        blas = [i["num_threads"] for i in info if i.get("user_api") == "blas"]
        if blas:
            return max(blas)
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(z, m, W, w, n_rows, n_cols, seed):
    """Time the float64 oracle on an n_rows x n_cols grid of entries per direction; returns
    (seconds, effective TFLOP/s in the update's own FLOP count, description)."""
    import numpy as np

    import oracle
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.N, n_rows, replace=False))
    cols = np.sort(rng.choice(w.N, n_cols, replace=False))
    t0 = time.perf_counter()
    for d in w.directions:
        oracle.sampled(z, m, W, d, rows, cols)
    dt = time.perf_counter() - t0
    frac = n_rows * n_cols / float(w.N) ** 2
    flops = frac * len(w.directions) * flops_update(w.N, w.c_z, w.c_h)
    desc = (f"{n_rows}x{n_cols} (i,j) entries of each of {len(w.directions)} directions at N={w.N}, exact "
            f"float64 oracle (a/b rows or columns recomputed); value = their share of the update's FLOPs / time")
    return dt, flops / dt / 1e12, desc


# --------------------------------------------------------------------------- reference arm (CPU oracle)

def oracle_backward_sample(n):
    """The float64 backward oracle on the whole grid at N = n (bf16 z, c = 128): its gradient work
    (4 n^3 c + 12 per-pair 128 x 128 products) per second. Every dz entry depends on the whole grid, so the
    oracle has no sampled form of the backward; a small full case stands in."""
    import numpy as np
    import oracle
    import workloads as wl
    z = wl.make_z(n, 128, 3, "bf16")
    W = wl.make_weights(128, 128, 1)
    dout = wl.make_z(n, 128, 4, "bf16")
    t0 = time.perf_counter()
    oracle.full_backward(z, np.ones(n), W, "outgoing", dout, storage="bf16")
    dt = time.perf_counter() - t0
    f = 4.0 * n ** 3 * 128 + 12 * 2 * 128 * 128 * float(n) ** 2
    return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"full float64 backward at N={n}, outgoing", "seconds": dt}


def oracle_attention_sample(n):
    """The float64 triangle-attention oracle on the whole grid at N = n (starting node): algorithmic
    work per second."""
    import oracle.triangle_attention as TA
    import workloads as wl
    z = wl.make_z(n, 128, 3, "bf16")
    W = wl.make_attention_weights()
    m = wl.make_mask(n, "full")
    t0 = time.perf_counter()
    TA.full(z, m, W, "starting")
    dt = time.perf_counter() - t0
    f = 4.0 * n ** 3 * 128 + float(n) ** 2 * (2 * 128 * (4 * 128 + 4) + 2 * 128 * 128)
    return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"full float64 triangle attention at N={n}, starting node", "seconds": dt}


def measure_config(tm, torch, name, steps, warmup, peaks, barrier):
    """ms per update, per-kernel ms and the contraction's fraction of bf16 peak for another workload of
    the metric, in this run. z is drawn on the device (seeded normal values rounded to bf16), the mask
    and weights are the workload's own; every step runs the workload's directions once each."""
    import numpy as np
    import workloads as wl
    w = wl.WORKLOADS[name]
    gen = torch.Generator(device="cuda").manual_seed(w.seed_z)
    z = torch.randn((w.N, w.N, w.c_z), device="cuda", generator=gen).to(torch.bfloat16)
    mask = torch.from_numpy(np.ascontiguousarray(wl.make_mask(w.N, w.mask))).cuda()
    mod = tm.TriMul(w.c_z, w.c_h, wl.make_weights(w.c_z, w.c_h, w.seed_w))
    out = torch.empty_like(z)
    opts = {"block": w.block} if w.block else {}

    def step():
        for d in w.directions:
            tm.tm_forward_ex(mod.ctx, z, mask, d, out, **opts)

    for _ in range(warmup):
        step()
    barrier()
    tm.tm_set_timing(mod.ctx, True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = tm.tm_launch_count(mod.ctx)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    barrier()
    ms = e0.elapsed_time(e1)
    kt = tm.tm_get_timing(mod.ctx)
    tm.tm_set_timing(mod.ctx, False)
    if tm.tm_sync_status(mod.ctx) != tm.TM_OK:
        raise RuntimeError(f"device status after {name}: " + tm.tm_last_error(mod.ctx))
    launches = tm.tm_launch_count(mod.ctx) - l0
    updates = steps * len(w.directions)
    kernels = {k: {"launches": v["launches"], "ms_per_launch": v["ms"] / v["launches"]}
               for k, v in kt.items() if v["launches"]}
    add_kernel_bandwidth(kernels, kt, peaks)
    kc = kt["contract"]
    k2 = 2.0 * w.N * kc["units"] / (kc["ms"] / 1e3) / 1e12 if kc["ms"] > 0 else None
    res = {"workload": f"{name}: N={w.N} {w.mask} mask, {' + '.join(w.directions)}"
                       + (f", {w.block}x{w.block} output blocks" if w.block else ""),
           "N": w.N, "steps": steps, "warmup": warmup, "ms_per_update": ms / updates,
           "tflops": flops_update(w.N, w.c_z, w.c_h) * updates / (ms / 1e3) / 1e12, "gpu_launches": launches,
           "kernels": kernels, "contraction_tflops": k2,
           "contraction_frac_of_bf16_peak": k2 / peaks["bf16_tflops"] if k2 else None,
           "contraction_frac_of_sustained": k2 / peaks["bf16_tflops_sustained"] if k2 else None,
           "z": "torch.randn on the device (seeded), rounded to bf16"}
    mod.close()
    del z, out, mask
    torch.cuda.empty_cache()
    return res


def oracle_full_timing(name, directions):
    """The plain float64 oracle over a whole workload grid (every entry), timed on the host cores."""
    import oracle
    import workloads as wl
    w = wl.WORKLOADS[name]
    z, m, W = wl.make_inputs(w)
    storage = "bf16" if w.dtype == "bf16" else "exact"
    t0 = time.perf_counter()
    for d in directions:
        oracle.full(z, m, W, d, storage=storage)
    dt = time.perf_counter() - t0
    fl = len(directions) * flops_update(w.N, w.c_z, w.c_h)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"whole grid of {name} (N={w.N}, {w.dtype}), {' + '.join(directions)}, full float64 oracle",
            "seconds": dt, "ms_per_update": 1e3 * dt / len(directions)}


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401

    import workloads as wl
    z, m, W = wl.make_inputs(w)
    for s in range(args.warmup):
        oracle_sample(z, m, W, w, 2, 2, 1000 + s)
    total, tfs, desc = 0.0, [], ""
    for s in range(args.steps):
        dt, tf, desc = oracle_sample(z, m, W, w, 8, 8, 2000 + s)
        total += dt
        tfs.append(tf)
    value = sum(tfs) / len(tfs)
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": f"{w.name}: N={w.N} c_z={w.c_z} c_h={w.c_h} {w.dtype} {w.mask} mask, "
                        f"{' then '.join(w.directions)} per step",
            "N": w.N, "c_z": w.c_z, "c_h": w.c_h, "directions": list(w.directions),
            "block": w.block or None, "chains": list(w.chains) or None,
            "l2": "inputs larger than L2 (z alone is %.2f GB)" % (w.N * w.N * w.c_z * 2 / 1e9),
            "parallelism": "replicas"}


# --------------------------------------------------------------------------- our arm

def run_ours(args, w):
    import numpy as np
    import torch

    import workloads as wl
    from pair_representation_boltz_b300 import build, tm

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    tm.load_library()

    z_np, m_np, W = wl.make_inputs(w)
    zt = torch.from_numpy(z_np.view(np.int16)).view(torch.bfloat16)
    mt = torch.from_numpy(m_np)
    z = zt.cuda()
    mask = mt.cuda()
    mod = tm.TriMul(w.c_z, w.c_h, W)
    outs = [torch.empty_like(z) for _ in w.directions]
    opts = {"block": w.block} if w.block else {}

    def step():
        for d, o in zip(w.directions, outs):
            if opts:
                tm.tm_forward_ex(mod.ctx, z, mask, d, o, **opts)
            else:
                tm.tm_forward(mod.ctx, z, mask, d, o)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if tm.tm_sync_status(mod.ctx) != tm.TM_OK:
        raise RuntimeError("device status after warm-up: " + tm.tm_last_error(mod.ctx))

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    time.sleep(0.3)                         # let the sampler see the load from its first sample
    launches0 = tm.tm_launch_count(mod.ctx)
    tm.tm_set_timing(mod.ctx, True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev0.record()
    for k in range(args.steps):
        step()
        step_ev[k].record()             # one event per step: the distribution of step times
    ev1.record()
    barrier()
    clk = clocks.stop()
    ms_total = ev0.elapsed_time(ev1)
    per_step = sorted([ev0.elapsed_time(step_ev[0])] +
                      [step_ev[k - 1].elapsed_time(step_ev[k]) for k in range(1, args.steps)])
    def pct(q):
        return per_step[min(len(per_step) - 1, int(round(q * (len(per_step) - 1))))]
    step_stats = {"median": statistics.median(per_step), "p10": pct(0.1), "p90": pct(0.9), "n": len(per_step)}
    launches = tm.tm_launch_count(mod.ctx) - launches0
    ktime = tm.tm_get_timing(mod.ctx)
    tm.tm_set_timing(mod.ctx, False)
    if tm.tm_sync_status(mod.ctx) != tm.TM_OK:
        raise RuntimeError("device status after the timed region: " + tm.tm_last_error(mod.ctx))
    ms_total = max_over_ranks(ms_total, "cuda")

    flops_step = len(w.directions) * flops_update(w.N, w.c_z, w.c_h)
    value = job_rate(world, args.steps * flops_step, ms_total) / 1e12
    peaks, peak_src = read_peaks()

    # dominant kernel: the contraction. FLOPs per launch = 2 * N(k) * channels * output pairs.
    kc = ktime["contract"]
    k2_flops = 2.0 * w.N * kc["units"]
    k2_ms_per_launch = kc["ms"] / max(kc["launches"], 1)
    k2_tflops = k2_flops / (kc["ms"] / 1e3) / 1e12 if kc["ms"] > 0 else None
    # the committed summary is per whole-grid launch at N = 3605; other shapes get no figure
    traffic = profiled_traffic() if (w.N == 3605 and not w.block) else None
    roofline = {"bound": "tensor", "achieved": k2_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": (k2_tflops / peaks["bf16_tflops"]) if k2_tflops else None,
                "traffic": traffic, "kernel": "k2_contract", "peak_source": f"bf16 burst, {peak_src}",
                "frac_of_sustained": (k2_tflops / peaks["bf16_tflops_sustained"]) if k2_tflops else None,
                "ms_per_launch": k2_ms_per_launch,
                "flops_per_launch": k2_flops / max(kc["launches"], 1)}
    kernels = {}
    tot = sum(v["ms"] for v in ktime.values()) or 1.0
    for name in ("project", "contract", "finish", "f32"):
        v = ktime[name]
        if v["launches"]:
            kernels[name] = {"launches": v["launches"], "ms_per_launch": v["ms"] / v["launches"],
                             "share": v["ms"] / tot}
    add_kernel_bandwidth(kernels, ktime, peaks)

    # e2e: the same step through the C ABI on host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        zp = zt.pin_memory()
        mp = mt.pin_memory()
        outs_h = [torch.empty_like(zt).pin_memory() for _ in w.directions]

        def step_host():
            for d, o in zip(w.directions, outs_h):
                tm.tm_forward_host(mod.ctx, zp, mp, d, o)

        step_host()
        torch.cuda.synchronize()
        k_e2e = max(1, min(args.steps, 5))
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(k_e2e):
            step_host()
        e1.record()
        barrier()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1), "cuda")
        zbytes = z_np.nbytes
        e2e = {"value": job_rate(world, k_e2e * flops_step, ms_e2e) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": len(w.directions) * (zbytes + m_np.nbytes),
               "d2h_bytes_per_step": len(w.directions) * zbytes, "steps": k_e2e,
               "ms_per_step": ms_e2e / k_e2e}
        e2e["roofline"] = pcie_roofline(torch, zp, outs_h[0], e2e["h2d_bytes_per_step"] + e2e["d2h_bytes_per_step"],
                                        ms_e2e / k_e2e)
        del outs_h

    # reference point for the contraction: cuBLAS (torch.bmm) over the 128 channel planes, bf16 in, bf16 out.
    # Timed at N rounded up to a multiple of 64 (the row padding the library's own a and b use): at N = 3605 a
    # bf16 row is 7210 bytes, not a multiple of 16, which keeps cuBLAS off its fast paths. Rates compare.
    cublas = None
    if w.dtype == "bf16" and not w.block:
        nb = (w.N + 63) // 64 * 64
        gen = torch.Generator(device="cuda").manual_seed(9)
        A = torch.randn(w.c_h, nb, nb, device="cuda", generator=gen).to(torch.bfloat16)
        B = torch.randn(w.c_h, nb, nb, device="cuda", generator=gen).to(torch.bfloat16)
        C = torch.empty_like(A)
        for _ in range(2):
            torch.bmm(A, B.transpose(1, 2), out=C)
        barrier()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(5):
            torch.bmm(A, B.transpose(1, 2), out=C)
        c1.record()
        barrier()
        ms_c = c0.elapsed_time(c1) / 5
        tf_c = 2.0 * nb ** 3 * w.c_h / (ms_c / 1e3) / 1e12
        cublas = {"ms": ms_c, "N": nb, "tflops": tf_c, "k2_over_cublas": (k2_tflops / tf_c) if k2_tflops else None,
                  "op": f"torch.bmm(A, B^T), [{w.c_h}][{nb}][{nb}] bf16, outgoing form"}
        del A, B, C

    # the Pairformer's own chain: z <- z + outgoing(z); z <- z + incoming(z), in place (tm_pair_update,
    # the residual add fused into the finish kernel), on a copy of z
    pair = None
    if w.dtype == "bf16" and not w.block and len(w.directions) == 2:
        zc = z.clone()
        for _ in range(2):
            tm.tm_pair_update(mod.ctx, zc, mask)
        barrier()
        k_p = max(1, min(args.steps, 5))
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record()
        for _ in range(k_p):
            tm.tm_pair_update(mod.ctx, zc, mask)
        p1.record()
        barrier()
        if tm.tm_sync_status(mod.ctx) != tm.TM_OK:
            raise RuntimeError("device status after the pair update: " + tm.tm_last_error(mod.ctx))
        ms_p = p0.elapsed_time(p1) / k_p
        pair = {"ms_per_step": ms_p, "ms_per_update": ms_p / 2,
                "tflops": 2 * flops_update(w.N, w.c_z, w.c_h) / (ms_p / 1e3) / 1e12, "steps": k_p,
                "note": "outgoing then incoming on the updated z, residual adds fused, in place"}
        del zc

    # backward pass (training): tm_backward per direction on the same z, a seeded bf16 cotangent
    bwd = None
    if not args.no_backward and w.dtype == "bf16" and not w.block:
        gen = torch.Generator(device="cuda").manual_seed(5)
        dout = torch.randn(z.shape, device="cuda", generator=gen).to(torch.bfloat16)
        dz = torch.empty_like(z)
        shapes = {"ln_in_gamma": (w.c_z,), "ln_in_beta": (w.c_z,), "w_a": (w.c_h, w.c_z), "w_ga": (w.c_h, w.c_z),
                  "w_b": (w.c_h, w.c_z), "w_gb": (w.c_h, w.c_z), "w_g": (w.c_z, w.c_z),
                  "ln_out_gamma": (w.c_h,), "ln_out_beta": (w.c_h,), "w_o": (w.c_z, w.c_h)}
        grads = {n: torch.empty(sh, dtype=torch.float32, device="cuda") for n, sh in shapes.items()}

        def bstep():
            for d in w.directions:
                tm.tm_backward(mod.ctx, z, mask, d, dout, dz, grads)

        bstep()                             # sizes the workspace
        barrier()
        k_b = max(1, min(args.steps, 3))
        b_l0 = tm.tm_launch_count(mod.ctx)
        tm.tm_set_timing(mod.ctx, True)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record()
        for _ in range(k_b):
            bstep()
        b1.record()
        barrier()
        ms_b = b0.elapsed_time(b1) / (k_b * len(w.directions))
        bt = tm.tm_get_timing(mod.ctx)
        tm.tm_set_timing(mod.ctx, False)
        if tm.tm_sync_status(mod.ctx) != tm.TM_OK:
            raise RuntimeError("device status after the backward: " + tm.tm_last_error(mod.ctx))
        # the gradient's own work: the contractions dA = dX b-side and dB (2 x 2 N^3 c_h) and 12 per-pair
        # 128 x 128 products (W^T products and parameter sums of both per-pair stages); the recomputed
        # forward (projection, x) is not counted
        gflops = 4.0 * float(w.N) ** 3 * w.c_h + 12 * 2 * 128 * 128 * float(w.N) ** 2
        btot = sum(v["ms"] for v in bt.values()) or 1.0
        bwd = {"ms_per_update": ms_b, "grad_tflops": gflops / (ms_b / 1e3) / 1e12,
               "grad_flops_per_update": gflops, "gpu_launches": tm.tm_launch_count(mod.ctx) - b_l0,
               "kernels": {n: {"launches": v["launches"], "ms_per_update": v["ms"] / (k_b * len(w.directions)),
                               "share": v["ms"] / btot}
                           for n, v in bt.items() if v["launches"]}}
        # roofline of the dominant kernel (the contractions: recomputed x, dA, dB; 2 N FLOP per channel
        # and output pair), and the per-pair backward kernels' algorithmic bandwidth (1800 B per pair each)
        bc = bt["contract"]
        if bc["ms"] > 0:
            c_tf = 2.0 * w.N * bc["units"] / (bc["ms"] / 1e3) / 1e12
            bwd["roofline"] = {"bound": "tensor", "kernel": "k2_contract (x, dA, dB)", "achieved": c_tf,
                               "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": c_tf / peaks["bf16_tflops"],
                               "traffic": None, "peak_source": f"bf16 burst, {peak_src}"}
        for n in ("out_backward", "proj_backward"):
            v = bt[n]
            if v["ms"] > 0:
                bwd["kernels"][n]["gbs"] = v["units"] * 1800 / (v["ms"] / 1e3) / 1e9
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            bwd["cpu_baseline"] = oracle_backward_sample(192)
        del dout, dz, grads

    # triangle attention (starting and ending node) on the same z
    attn = None
    if not args.no_attention and w.dtype == "bf16" and not w.block:
        amod = tm.TriangleAttention(wl.make_attention_weights())
        aout = torch.empty_like(z)
        nodes = ("starting", "ending")
        for nd in nodes:
            amod(z, mask, nd, out=aout)
        barrier()
        k_a = max(1, min(args.steps, 2))
        a_l0 = tm.tm_launch_count(amod.ctx)
        tm.tm_set_timing(amod.ctx, True)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(k_a):
            for nd in nodes:
                amod(z, mask, nd, out=aout)
        a1.record()
        barrier()
        ms_a = a0.elapsed_time(a1) / (k_a * len(nodes))
        at = tm.tm_get_timing(amod.ctx)
        tm.tm_set_timing(amod.ctx, False)
        if tm.tm_sync_status(amod.ctx) != tm.TM_OK:
            raise RuntimeError("device status after the attention: " + tm.tm_last_error(amod.ctx))
        # algorithmic FLOPs: the two attention products 4 N^3 H c, and per pair the q, k, v, g, b
        # projections and the output (2 c_z (4 H c + H) + 2 H c c_z)
        hc = 128
        aflops = 4.0 * float(w.N) ** 3 * hc + float(w.N) ** 2 * (2 * 128 * (4 * hc + 4) + 2 * hc * 128)
        atot = sum(v["ms"] for v in at.values()) or 1.0
        attn = {"heads": 4, "head_dim": 32, "ms_per_node": ms_a, "tflops": aflops / (ms_a / 1e3) / 1e12,
                "flops_per_node": aflops, "gpu_launches": tm.tm_launch_count(amod.ctx) - a_l0,
                "kernels": {n: {"launches": v["launches"], "ms_per_node": v["ms"] / (k_a * len(nodes)),
                                "share": v["ms"] / atot}
                            for n, v in at.items() if v["launches"]}}
        # the attention kernel's arithmetic bound: one ex2 per logit (N^3 H per node) on the special-function
        # pipe, at the rate this device sustains (libtm's probe: independent ex2 chains on every SM); the
        # nominal unit count (16 per clock per SM at the maximum clock) beside it
        ta = at["attn_attend"]
        if ta["ms"] > 0:
            logits = float(w.N) ** 3 * 4 * ta["launches"]
            ach = logits / (ta["ms"] / 1e3) / 1e12
            pk = tm.tm_probe_ex2_rate(amod.ctx) / 1e12
            nominal = 16 * 148 * 2032e6 / 1e12
            attn["roofline"] = {"bound": "alu", "kernel": "k_ta_attend", "achieved": ach, "peak": pk,
                                "unit": "Tera-ex2/s", "frac": ach / pk, "traffic": None,
                                "peak_source": "measured: ex2.approx.ftz.f32 on independent chains, every SM",
                                "nominal_peak": nominal, "frac_of_nominal": ach / nominal}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            attn["cpu_baseline"] = oracle_attention_sample(256)
        amod.close()
        del aout

    # the metric's other workloads, measured in the same run (the step above is the four-chain complex)
    others = None
    if not args.no_other_configs and not args.N and w.name == "complex3605":
        del outs
        torch.cuda.empty_cache()
        others = {}
        for name, k in (("crop768", 50), ("ppi6500", 3), ("n10000", 2)):
            others[name] = measure_config(tm, torch, name, k, 3, peaks, barrier)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, tf, desc = oracle_sample(z_np, m_np, W, w, args.cpu_rows, args.cpu_rows, 7)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle", "sample": desc,
               "seconds": dt}
        # the full oracle on the workloads it finishes within minutes: the tiny fp32 case (both
        # directions) and the training crop (one direction, about half a minute on 16 cores)
        cpu["full_oracle"] = {"tiny48": oracle_full_timing("tiny48", ("outgoing", "incoming")),
                              "crop768": oracle_full_timing("crop768", ("outgoing",))}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w),
            "ms_per_update": ms_total / args.steps / len(w.directions),
            "frac_of_bf16_peak": value / world / peaks["bf16_tflops"],
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clk, "backward": bwd,
            "triangle_attention": attn, "pair_update": pair, "step_ms": step_stats,
            "cublas_bmm_reference": cublas, "other_configs": others,
        }
        print(json.dumps(line), flush=True)
    mod.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="complex3605")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward-pass measurement")
    ap.add_argument("--no-attention", action="store_true", help="skip the triangle-attention measurement")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the crop768, ppi6500 and n10000 measurements beside the step")
    ap.add_argument("--cpu-rows", type=int, default=48, help="side of the oracle's sampled grid")
    ap.add_argument("--N", type=int, default=0, help="override the workload's token count (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    import workloads as wl
    w = wl.WORKLOADS[args.workload]
    if args.N:
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}@N={args.N}", N=args.N, chains=())
    if w.dtype != "bf16":
        ap.error("the benchmark runs the bf16 workloads")
    return run_reference(args, w) if args.impl == "reference" else run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
