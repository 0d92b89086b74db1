"""Benchmark of the compressed Lion update step (Lion Cub / Distributed Lion)
with W simulated workers on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl lioncub|reference]

One step = one pass of the whole path over one batch of synthetic gradients:
update vectors, compression (packed signs or L1 codes, with the M1 pass),
the W-way vote or integer sum, the global sign and the theta update, the
momentum update and the selective momentum sync.  The default workload is
the largest one that fits one GPU: a GPT-2-XL-like layout with an untied
head (1,416,552,448 parameters), W = 8 workers, bf16 gradients
1e-3 * Student-t(3), 2-bit L1 codes with the integer sum (about 198 GB of
HBM traffic per step; theta and 8 momenta are 51 GB resident).

Metric: parameter-elements per second per step (d / step time), whole job.
Inputs are far larger than the 129 MB L2 for every GPT workload (11-200 GB
moved per step); the 1M-element workload flushes L2 between timed steps.

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (the path exchanges nothing between GPUs on one
box), the timed region is bracketed by barriers, and the step time is the
maximum over ranks.  `--impl reference` times the CPU oracle instead, on a
bounded sample of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
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

import synth  # noqa: E402

DEFAULT_CONFIG = 5
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
# GB300 HBM3e bandwidth as the vendor states it (8 TB/s per GPU), for context
# next to the measured copy bandwidth
NOMINAL_HBM_GBS = 8000.0

# DRAM bytes per parameter of each kernel in one step: dram__bytes_read.sum +
# dram__bytes_write.sum over the kernel's launches of one step, divided by the
# parameters of the case, from one ncu capture of a small case of each
# workload (a slice of its layout, a few GB on the device, inputs still far
# larger than L2).  Every kernel streams each parameter's bytes once, so its
# traffic grows in proportion to the parameters; the bench scales the figure
# by the full workload's parameter count.  Writes read a little low: up to an
# L2's worth of dirty lines are still in L2 when a launch ends (2-3.5 % of a
# 3 GB compress launch; about 18 % of the 0.3-0.4 GB reduce launches of the
# small cases, which makes their scaled figure a lower bound).  An entry
# holds for the kernel sources it was taken on: traffic is reported only
# while the fingerprint of those sources still matches.
KERNEL_SOURCES = {
    "compress": ("compress.cu", "compress_common.cuh", "device_common.cuh", "internal.h"),
    "m1_partial": ("m1.cu", "device_common.cuh", "internal.h"),
    "m1_finalize": ("m1.cu", "device_common.cuh", "internal.h"),
    "reduce_apply": ("reduce_apply.cu", "aggregate.cuh", "device_common.cuh", "internal.h"),
}
MEASURED_TRAFFIC_PER_PARAM = {
    "fingerprints": {"compress": "ea587c8f9a3ef666", "m1_partial": "407d4a46b6fa5cc1", "m1_finalize": "407d4a46b6fa5cc1", "reduce_apply": "1d62bcda443aa8a0"},
    "gpt2-small-124M-w8-sign": {"compress": 79.4851, "reduce_apply": 7.3486},
    "gpt2-medium-350M-w8-l1n4": {"m1_partial": 48.1083, "m1_finalize": 0.0317, "compress": 82.4089, "reduce_apply": 10.5165},
    "gpt2-medium-350M-w16-sign-wte-sync": {"compress": 154.9262, "reduce_apply": 6.3065},
    "gpt2-xl-like-1.3B-w8-l1n2": {"m1_partial": 48.0995, "m1_finalize": 0.0318, "compress": 80.2036, "reduce_apply": 8.1618},
}


def source_fingerprint(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "communication_compressed_sign_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(wl: synth.Workload, kernel: str):
    """DRAM bytes per step of `kernel` on workload `wl` (the small-case figure
    per parameter times wl.d), or None when no capture exists for the
    workload or the kernel's sources changed since it was taken."""
    base = wl.name.split("[", 1)[0]
    entry = MEASURED_TRAFFIC_PER_PARAM.get(base, {})
    if kernel not in entry or kernel not in KERNEL_SOURCES:
        return None
    if MEASURED_TRAFFIC_PER_PARAM["fingerprints"].get(kernel) != source_fingerprint(kernel):
        return None
    return int(round(entry[kernel] * wl.d))


# ---------------------------------------------------------------------------
# algorithmic bytes (every byte that must move, per parameter)
# ---------------------------------------------------------------------------

def kernel_bytes(wl: synth.Workload) -> dict:
    """Algorithmic bytes per step of each kernel for workload wl."""
    d, W = wl.d, wl.W
    G = 4 if wl.grad == "f32" else 2
    bits = wl.nbits if wl.mode == 1 else 1
    out = {"compress": d * W * (G + 4 + 4) + W * ((d * bits + 31) // 32) * 4,
           "reduce_apply": W * ((d * bits + 31) // 32) * 4 + 8 * d}
    if wl.mode == 1:
        out["m1_partial"] = d * W * (G + 4)
        out["m1_finalize"] = 0
    return out


def step_bytes(wl: synth.Workload) -> int:
    return sum(kernel_bytes(wl).values())


def mode_label(wl: synth.Workload) -> str:
    if wl.mode == 1:
        return f"L1 n={wl.nbits} + int sum"
    return "sign + D-Lion average" if wl.flags & 0x200 else "sign+majority"


def sync_label(wl: synth.Workload) -> str:
    flagged = [name for (name, _, _, fl) in wl.layout if fl]
    if not wl.sync_interval or not flagged:
        return "none"
    every = "every step" if wl.sync_interval == 1 else f"every {wl.sync_interval} steps"
    return f"{', '.join(flagged)} {every}"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; only the timing is reduced)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_min(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples every 50 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
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
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm),
                "reasons": sorted(reasons)}


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = json.load(f)
        return float(v["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_sample(wl: synth.Workload, target_elems: int):
    """A sample of the workload: its tensors in layout order (after the two
    embeddings, which would dominate), the last one cut so that the sample
    holds about target_elems elements."""
    body = [t for t in wl.layout if t[0] not in ("wte", "wpe", "head")] or wl.layout
    sub, names, dst = [], [], 0
    for (name, off, n, fl) in body:
        if dst >= target_elems:
            break
        take = min(n, target_elems - dst)
        if take < n:
            take = max(32, take // 32 * 32)
        sub.append((dst, take, fl))
        names.append(name)
        dst += take
    return sub, dst, names


def time_oracle_steps(wl: synth.Workload, target_elems: int, steps: int, warmup: int = 0):
    import oracle
    sub, dsub, names = oracle_sample(wl, target_elems)
    grads_pool = [synth.numpy_grad(wl, dsub, 0, i) for i in range(min(wl.W, 2))]
    grads = [np.roll(grads_pool[i % len(grads_pool)], 977 * i) for i in range(wl.W)]
    theta = synth.numpy_theta(wl, dsub)
    m = [np.zeros(dsub, np.float32) for _ in range(wl.W)]
    times = []
    for t in range(warmup + steps):
        t0 = time.perf_counter()
        oracle.step(d=dsub, W=wl.W, layout=sub, beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr, wd=wl.wd,
                    mode=wl.mode, nbits=wl.nbits, flags=wl.flags, sync_interval=wl.sync_interval, t=t,
                    grads=grads, theta=theta, m=m, want_outputs=False)
        if t >= warmup:
            times.append(time.perf_counter() - t0)
    return dsub, names, times


def oracle_rate_probe(wl: synth.Workload) -> float:
    """Seconds per parameter of one oracle step (small probe)."""
    dsub, _, times = time_oracle_steps(wl, 300_000, 1)
    return times[0] / dsub


# Arm CPU part numbers (/proc/cpuinfo "CPU part") of the hosts this runs on
ARM_PARTS = {"0xd4f": "Arm Neoverse V2 (NVIDIA Grace)", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1"}


def cpu_info():
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                low = line.lower()
                if low.startswith("model name") or low.startswith("cpu part"):
                    model = line.split(":", 1)[1].strip()
                    model = ARM_PARTS.get(model.lower(), model)
                    break
    except OSError:
        pass
    return {"host_cores": os.cpu_count(), "cpu": model}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, wl: synth.Workload):
    import torch
    import torch.distributed as dist
    import __graft_entry__
    from communication_compressed_sign_gb300 import lioncub as lc

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    if rank == 0:
        __graft_entry__.build()
    barrier(dev)
    lc.load()

    d, W = wl.d, wl.W
    gdt = synth.grad_dtype(wl)
    theta = torch.empty(d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta, wl)
    m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(W)]
    nsets = 2
    grads = [[torch.empty(d, dtype=gdt, device=dev) for _ in range(W)] for _ in range(nsets)]
    for s in range(nsets):
        for i in range(W):
            synth.fill_grad_(grads[s][i], wl, s, i)
    gptrs = [[g.data_ptr() for g in grads[s]] for s in range(nsets)]
    h = lc.lioncub_create(d, W, synth.abi_layout(wl.layout), wl.beta1, wl.beta2, wl.lr, wl.wd, wl.mode | wl.flags,
                          wl.nbits, lc.GRAD_F32 if wl.grad == "f32" else lc.GRAD_BF16, wl.sync_interval)
    lc.lioncub_bind_state(h, theta.data_ptr(), [x.data_ptr() for x in m])
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    ws_bytes = step_bytes(wl)
    flush = ws_bytes < 4 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    # warm-up
    for s in range(args.warmup):
        lc.lioncub_step(h, gptrs[s % nsets], sp)
    torch.cuda.synchronize(dev)

    # timed region: per-kernel events inside the library, step events here
    lc.lioncub_profile(h, args.steps)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(dev)
    torch.cuda.synchronize(dev)
    if flush:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for s in range(args.steps):
            flush_buf.fill_(float(s))
            ev[s][0].record(stream)
            lc.lioncub_step(h, gptrs[s % nsets], sp)
            ev[s][1].record(stream)
        torch.cuda.synchronize(dev)
        step_ms = [a.elapsed_time(b) for a, b in ev]
        total_ms = sum(step_ms)
    else:
        # back-to-back steps; an event between consecutive steps gives each
        # step's time without adding work to the stream
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        ev[0].record(stream)
        for s in range(args.steps):
            lc.lioncub_step(h, gptrs[s % nsets], sp)
            ev[s + 1].record(stream)
        torch.cuda.synchronize(dev)
        step_ms = [ev[s].elapsed_time(ev[s + 1]) for s in range(args.steps)]
        total_ms = ev[0].elapsed_time(ev[-1])
    barrier(dev)
    clk = clocks.stop()
    ms_local = total_ms / args.steps
    ms = reduce_max(ms_local, dev)
    ms_median = reduce_max(float(statistics.median(step_ms)), dev)

    kb = kernel_bytes(wl)
    per_kernel = {}
    recorded = 0
    for k, name in lc.KERNEL_NAMES.items():
        tot, n = lc.lioncub_profile_read(h, k)
        recorded += n
        if n:
            per_kernel[name] = {"ms_per_step": tot / args.steps, "launches_per_step": n / args.steps,
                                "share": None, "alg_bytes": kb.get(name, 0),
                                "traffic": measured_traffic(wl, name)}
    ksum = sum(v["ms_per_step"] for v in per_kernel.values()) or 1.0
    for v in per_kernel.values():
        v["share"] = v["ms_per_step"] / ksum
        v["gbs"] = v["alg_bytes"] / (v["ms_per_step"] * 1e-3) / 1e9
    lc.lioncub_profile(h, 0)
    top = max(per_kernel, key=lambda k: per_kernel[k]["ms_per_step"])
    peak, peak_kind = measured_hbm_peak()
    achieved = per_kernel[top]["alg_bytes"] / (per_kernel[top]["ms_per_step"] * 1e-3) / 1e9
    step_gbs = ws_bytes / (ms * 1e-3) / 1e9

    # diagnostics pass (not part of the step): timed separately when asked
    diag = run_diagnose(args, wl, h, dev, stream, gptrs[0]) if args.diagnose else None

    # end to end: host gradients in, host theta out, through lioncub_step_host.
    # The device-resident leg's gradient buffers are released first: that leg
    # is done, and the host step stages its own copies (45 GB of idle device
    # buffers on the 1.3B workload measured up to 1.6x slower host steps on
    # some boxes, with a periodic stall).
    gptrs = None
    grads = None
    torch.cuda.empty_cache()
    e2e = None if args.no_e2e else run_e2e(args, wl, h, dev, stream)

    # the device status word (bounded waits that gave up, guard bands around
    # the library's scratch), read after all timing: a run that tripped it is
    # not a valid measurement
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    lc.lioncub_debug_export(h, lc.EXPORT_STATUS, status.data_ptr(), stream.cuda_stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status word is {int(status.item())} after the timed steps")

    lc.lioncub_destroy(h)
    del m, theta, flush_buf
    torch.cuda.empty_cache()

    result = {
        "metric": "param-elements/s per Lion Cub step (W simulated workers)",
        "value": ws * d / (ms * 1e-3),
        "unit": "param-elements/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "ms_per_step_median": ms_median,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded counter-based Student-t / normal gradients, uniform theta)",
        "config": {
            "workload": wl.name,
            "workers": W,
            "params": d,
            "tensors": len(wl.layout),
            "mode": mode_label(wl),
            "grad_dtype": wl.grad,
            "arithmetic": "f32 update vector, momentum and theta (one rounding per operation); integer vote / code sums; u32 packed wire",
            "sync": sync_label(wl),
            "parallelism": f"replicas x{ws} (no inter-GPU exchange)",
            "l2": "flushed between timed steps" if flush else f"inputs larger than L2 ({ws_bytes / 1e9:.1f} GB moved per step)",
        },
        "hbm": {"alg_bytes_per_step": ws_bytes, "achieved_gbs": step_gbs, "peak_gbs": peak,
                "frac_of_measured" if peak_kind == "measured" else "frac_of_fallback": step_gbs / peak,
                "frac_of_nominal_8000": step_gbs / NOMINAL_HBM_GBS},
        "roofline": {"bound": "hbm", "kernel": top, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": measured_traffic(wl, top),
                     "alg_bytes": per_kernel[top]["alg_bytes"]},
        "kernels": per_kernel,
        "gpu_launches": recorded,
        "clocks": clk,
        "e2e": e2e,
    }
    if diag is not None:
        result["diagnose"] = diag
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl)
    if ws > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


def run_gpu_exchange(args, wl: synth.Workload):
    """The data-parallel exchange: the workload's W workers spread over the N
    ranks (W/N each, one GPU per rank), every rank with its own theta; a step
    is the library's three launches with NCCL collectives between them
    (all-to-all of packed words and allgather of directions in sign mode,
    allreduce of code sums in L1 mode, allgather of synchronized momenta on
    sync steps).  The whole job takes one step over d parameters, so value =
    d / step time and the scaling is strong.  With one process (no torchrun)
    it runs as a one-rank NCCL group on GPU 0."""
    import torch
    import torch.distributed as dist
    import __graft_entry__
    from communication_compressed_sign_gb300 import lioncub as lc
    from communication_compressed_sign_gb300.dist import DistLionCub

    ws, rank, local = dist_env()
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    if ws == 1:
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            os.environ.setdefault("MASTER_PORT", str(sk.getsockname()[1]))
        os.environ.setdefault("RANK", "0")
        os.environ.setdefault("WORLD_SIZE", "1")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        __graft_entry__.build()
    barrier(dev)
    lc.load()
    d, W = wl.d, wl.W
    if W % ws:
        raise SystemExit(f"--exchange needs W ({W}) divisible by the number of ranks ({ws})")
    gcode = lc.GRAD_F32 if wl.grad == "f32" else lc.GRAD_BF16
    opt = DistLionCub(d, W, synth.abi_layout(wl.layout), beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr, wd=wl.wd,
                      mode=wl.mode | wl.flags, nbits=wl.nbits, grad_dtype=gcode, sync_interval=wl.sync_interval,
                      device=dev)
    Wl, first = opt.plan.local_workers, opt.plan.first_worker
    theta = torch.empty(d, dtype=torch.float32, device=dev)
    synth.fill_theta_(theta, wl)
    m = [torch.zeros(d, dtype=torch.float32, device=dev) for _ in range(Wl)]
    opt.bind(theta, m)
    gdt = synth.grad_dtype(wl)
    grads = [[torch.empty(d, dtype=gdt, device=dev) for _ in range(Wl)] for _ in range(2)]
    for s in range(2):
        for i in range(Wl):
            synth.fill_grad_(grads[s][i], wl, s, first + i)
    stream = torch.cuda.current_stream(dev)
    for s in range(args.warmup):
        opt.step(grads[s % 2], stream)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(dev)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(args.steps):
        opt.step(grads[s % 2], stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dev)
    clk = clocks.stop()
    ms = reduce_max(e0.elapsed_time(e1) / args.steps, dev)
    moved = {lc.DIST_BUFFER_NAMES[b]: int(opt.plan.bytes[b]) for b in range(lc.DIST_BUFFERS)}
    # the library's launches in the timed steps: (M1 pass and combine,) compress, reduce, apply, and the
    # momentum average on sync steps
    from communication_compressed_sign_gb300.dist import is_sync_step
    t0 = args.warmup
    launches = sum((5 if wl.mode == 1 else 3) + (1 if is_sync_step(t0 + s, wl.sync_interval, opt.plan) else 0)
                   for s in range(args.steps))
    opt.close()
    dist.destroy_process_group()
    if rank != 0:
        return None
    return {
        "metric": "param-elements/s per Lion Cub step (W simulated workers)",
        "value": d / (ms * 1e-3),
        "unit": "param-elements/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded counter-based Student-t / normal gradients, uniform theta)",
        "config": {"workload": wl.name, "workers": W, "workers_per_rank": Wl, "params": d, "mode": mode_label(wl),
                   "sync": sync_label(wl), "grad_dtype": wl.grad,
                   "parallelism": f"data-parallel exchange over {ws} rank(s): "
                                  + ("all-to-all of packed signs + allgather of 2-bit directions" if wl.mode == 0
                                     else "allreduce of integer code sums"),
                   "exchange_buffer_bytes_per_rank": moved},
        "clocks": clk,
        "gpu_launches": launches,
    }


def run_diagnose(args, wl, h, dev, stream, grad_ptrs):
    """Time lioncub_diagnose (the pages' sign match/flip, tie and momentum
    spread measurements) over the whole workload; report its bandwidth and the
    totals over all tensors."""
    import torch
    from communication_compressed_sign_gb300 import lioncub as lc
    K = len(wl.layout)
    out = torch.zeros(K * lc.DIAG_BYTES, dtype=torch.uint8, device=dev)
    sp = stream.cuda_stream
    for _ in range(2):
        lc.lioncub_diagnose(h, grad_ptrs, out.data_ptr(), sp)
    n = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(n):
        lc.lioncub_diagnose(h, grad_ptrs, out.data_ptr(), sp)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / n
    recs = lc.decode_diag(out.cpu().numpy().tobytes(), K)
    tot = {f: sum(r[f] for r in recs) for f in ("match", "flip", "dropped", "spurious", "ties")}
    G = 4 if wl.grad == "f32" else 2
    alg = wl.d * wl.W * (G + 4) * (2 if wl.mode == 1 else 1)  # (+ the M1 pass in L1 mode)
    worst = max(range(K), key=lambda k: recs[k]["max_std_m"])
    # the max-norm comparator (stochastic rounding) at the workload's code
    # width, 4 bits for sign-mode workloads
    qbits = wl.nbits if wl.mode == 1 else 4
    qout = torch.zeros(K * lc.QINF_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(2):
        lc.lioncub_diagnose_qinf(h, grad_ptrs, qbits, 0, qout.data_ptr(), sp)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(n):
        lc.lioncub_diagnose_qinf(h, grad_ptrs, qbits, 0, qout.data_ptr(), sp)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    qms = e0.elapsed_time(e1) / n
    qrecs = lc.decode_qinf(qout.cpu().numpy().tobytes(), K)
    qtot = {f: sum(r[f] for r in qrecs) for f in lc.QINF_FIELDS}
    qalg = 2 * wl.d * wl.W * (G + 4)  # the max-norm pass and the counting pass
    return {"ms": ms, "alg_bytes": alg, "gbs": alg / (ms * 1e-3) / 1e9,
            "fractions": {f: v / wl.d for f, v in tot.items()},
            "max_std_m": {"tensor": wl.layout[worst][0], "value": recs[worst]["max_std_m"]},
            "qinf": {"nbits": qbits, "ms": qms, "alg_bytes": qalg, "gbs": qalg / (qms * 1e-3) / 1e9,
                     "fractions": {f: qtot[f] / wl.d for f in ("match", "flip", "dropped", "spurious")},
                     "zero_code_fraction": qtot["zero_codes"] / (wl.d * wl.W)},
            "state": "after the warm-up and timed steps"}


def gpu_local_cpus(index: int):
    """CPUs attached to GPU `index` (from its PCI device's local_cpulist), or None."""
    try:
        bus = subprocess.run(["nvidia-smi", f"--id={index}", "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip().lower()
        if not bus:
            return None
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{dom[-4:]}:{rest}/local_cpulist"
        with open(path) as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
        return cpus or None
    except (OSError, ValueError, subprocess.SubprocessError):
        return None


def host_memory_available() -> int:
    """Bytes this process may still allocate on the host: MemAvailable, or
    the cgroup's remaining limit when that is lower."""
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            lim = f.read().strip()
        with open("/sys/fs/cgroup/memory.current") as f:
            cur = int(f.read().strip())
        if lim != "max":
            left = int(lim) - cur
            avail = left if avail is None else min(avail, left)
    except (OSError, ValueError):
        pass
    return avail if avail is not None else 1 << 62


def e2e_host_layout(W: int, grad_bytes: int, theta_bytes: int, ranks_here: int, avail: int):
    """How the host gradients of the host-buffer leg are laid out, so that
    every rank on this node fits in 60 % of the available host memory:
    two sets of W buffers (steps alternate), one set, or one buffer that all W
    workers read (the bytes copied per step are the same in every case).
    Returns (sets, distinct buffers per set) or None when even that does not
    fit."""
    budget = 0.6 * avail
    for sets, per_set in ((2, W), (1, W), (1, 1)):
        if ranks_here * (sets * per_set * grad_bytes + theta_bytes) <= budget:
            return sets, per_set
    return None


def run_e2e(args, wl, h, dev, stream):
    """K steps through lioncub_step_host: every step copies the W gradient
    buffers from pinned host memory to the device and theta back."""
    import torch
    from communication_compressed_sign_gb300 import lioncub as lc
    d, W = wl.d, wl.W
    gdt = synth.grad_dtype(wl)
    G = 4 if wl.grad == "f32" else 2
    ws, _, _ = dist_env()
    ranks_here = int(os.environ.get("LOCAL_WORLD_SIZE", ws))
    # every rank reads the host memory before any of them allocates, and all
    # take the smallest reading, so they choose the same layout
    barrier(dev)
    avail = int(reduce_min(float(host_memory_available()), dev))
    layout = e2e_host_layout(W, d * G, 4 * d, ranks_here, avail)
    if layout is None:
        return {"value": None, "unit": "param-elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "skipped": f"host memory: {ranks_here} ranks x one gradient buffer and theta do not fit"}
    nsets, per_set = layout
    # page-locked buffers from the library's allocator (torch's caching pinned
    # allocator measured up to 40 % slower host-to-device at the 1.3B size),
    # on the GPU's own NUMA node: allocate (first touch) from a thread bound
    # to the GPU's local CPUs
    cpus = gpu_local_cpus(dev.index)
    saved = os.sched_getaffinity(0)
    if cpus and cpus & saved:
        os.sched_setaffinity(0, cpus & saved)
    host = [[lc.HostBuffer(d, gdt) for _ in range(per_set)] for _ in range(nsets)]
    tmp = torch.empty(d, dtype=gdt, device=dev)
    for s in range(nsets):
        for i in range(per_set):
            synth.fill_grad_(tmp, wl, s, i)
            host[s][i].tensor.copy_(tmp)
    del tmp
    theta_host = lc.HostBuffer(d, torch.float32)
    # worker i of step s reads host[s % nsets][i % per_set]
    ptrs = [[host[s % nsets][i % per_set].data_ptr() for i in range(W)] for s in range(2)]
    sp = stream.cuda_stream
    for s in range(max(1, args.warmup)):
        lc.lioncub_step_host(h, ptrs[s % 2], theta_host.data_ptr(), sp)
    torch.cuda.synchronize(dev)
    barrier(dev)
    t0 = time.perf_counter()
    # an event after each step (after its theta download) gives the spread
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for s in range(args.steps):
        lc.lioncub_step_host(h, ptrs[s % 2], theta_host.data_ptr(), sp)
        ev[s + 1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    ms = reduce_max(ev[0].elapsed_time(ev[-1]) / args.steps, dev)
    per = sorted(ev[s].elapsed_time(ev[s + 1]) for s in range(args.steps))
    spread = {"median": per[len(per) // 2], "p10": per[len(per) // 10], "p90": per[(9 * len(per)) // 10],
              "max": per[-1]}
    h2d = W * d * G
    os.sched_setaffinity(0, saved)
    for row in host:
        for x in row:
            x.close()
    theta_host.close()
    return {"value": ws * d / (ms * 1e-3), "unit": "param-elements/s", "ms_per_step": ms,
            "ms_per_step_spread": spread,
            "wall_ms_per_step": wall * 1e3 / args.steps,
            "host_cpus_bound": sorted(cpus & saved) if cpus and cpus & saved else None,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4 * d,
            "h2d_gbs": h2d / (ms * 1e-3) / 1e9,
            "host_gradient_buffers": f"{nsets} set(s) of {per_set} (steps alternate between sets; "
                                     f"worker i reads buffer i mod {per_set})",
            "api": "lioncub_step_host (page-locked host buffers from lioncub_host_alloc; uploads overlap "
                   "the previous step)"}


def cpu_baseline(wl: synth.Workload, seconds: float = 12.0):
    rate = oracle_rate_probe(wl)
    target = int(min(wl.d, max(100_000, seconds / max(rate, 1e-12))))
    dsub, names, times = time_oracle_steps(wl, target, 1)
    info = cpu_info()
    return {"value": dsub / times[0], "unit": "param-elements/s", "cores": 1, "kind": "oracle",
            "sample": f"one step of {wl.name} restricted to {len(names)} whole tensors "
                      f"({dsub} of {wl.d} params, all {wl.W} workers), numpy-generated inputs "
                      f"of the same distribution",
            "seconds": times[0], **info}


def run_reference(args, wl: synth.Workload):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    rate = oracle_rate_probe(wl)
    budget_s = args.ref_seconds
    per_step = budget_s / max(1, args.steps + args.warmup)
    target = int(min(wl.d, max(50_000, per_step / max(rate, 1e-12))))
    dsub, names, times = time_oracle_steps(wl, target, args.steps, args.warmup)
    ms = 1e3 * sum(times) / len(times)
    value = dsub / (ms * 1e-3)
    info = cpu_info()
    return {
        "impl": "reference",
        "metric": "param-elements/s per Lion Cub step (W simulated workers)",
        "value": value,
        "unit": "param-elements/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (numpy Student-t / normal gradients of the workload's distribution)",
        "config": {"workload": wl.name, "workers": wl.W, "params": wl.d,
                   "sample_params": dsub, "sample_tensors": len(names)},
        "cpu_baseline": {"value": value, "unit": "param-elements/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(names)} whole tensors, {dsub} of {wl.d} params, all workers",
                         **info},
        "e2e": {"value": value, "unit": "param-elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def truncated(wl: synth.Workload, limit: int, skip: int = 0) -> synth.Workload:
    """The workload restricted to consecutive tensors: after the first `skip`
    tensors, the leading ones (at least one) up to about `limit` parameters,
    re-based to offset 0; the name records the cut."""
    keep, total = [], 0
    for (name, _, n, fl) in wl.layout[skip:]:
        if keep and total + n > limit:
            break
        keep.append((name, total, n, fl))
        total += n
    import dataclasses
    cut = f"tensors {skip}..{skip + len(keep) - 1}, {total} params"
    return dataclasses.replace(wl, layout=keep, name=f"{wl.name}[{cut}]")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=sorted(synth.workloads()),
                    help="workload: " + "; ".join(f"{k} = {w.name}" for k, w in sorted(synth.workloads().items())))
    ap.add_argument("--impl", default="lioncub", choices=["lioncub", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="--impl reference: CPU seconds the whole run aims at (sets the sample size)")
    ap.add_argument("--diagnose", action="store_true",
                    help="also time lioncub_diagnose (sign match/flip, ties, momentum spread)")
    ap.add_argument("--mode", choices=["sign", "l1"], default=None,
                    help="run the workload's layout and gradients with another compression mode")
    ap.add_argument("--nbits", type=int, default=None, help="code width for --mode l1 (2, 4 or 8)")
    ap.add_argument("--layout-limit", type=int, default=0,
                    help="profiling aid: keep only the workload's leading tensors, about this many parameters")
    ap.add_argument("--exchange", action="store_true",
                    help="spread the W workers over the ranks and exchange with NCCL (the multi-GPU path) "
                         "instead of running one replica per GPU")
    ap.add_argument("--skip-tensors", type=int, default=0,
                    help="profiling aid: with --layout-limit, start after this many tensors")
    ap.add_argument("--sync-names", default="",
                    help="profiling aid: comma-separated tensors whose momentum is synchronized instead of the "
                         "workload's own (needs a workload with a sync interval)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "lioncub":
        print("note: warm-up raised to 3 steps", file=sys.stderr)
        args.warmup = 3
    wl = synth.workloads()[args.config]
    if args.layout_limit:
        wl = truncated(wl, args.layout_limit, args.skip_tensors)
    if args.sync_names:
        import dataclasses
        names = set(args.sync_names.split(","))
        lay = [(n, o, c, synth.SYNC_M if n in names else 0) for (n, o, c, _) in wl.layout]
        wl = dataclasses.replace(wl, layout=lay, name=f"{wl.name}[sync {args.sync_names}]")
    if args.mode is not None:
        import dataclasses
        mode = 0 if args.mode == "sign" else 1
        nbits = 1 if mode == 0 else (args.nbits or 4)
        wl = dataclasses.replace(wl, mode=mode, nbits=nbits,
                                 name=f"{wl.name}[{'sign' if mode == 0 else f'L1 n={nbits}'}]")
    if args.impl == "reference":
        res = run_reference(args, wl)
    elif args.exchange:
        res = run_gpu_exchange(args, wl)
    else:
        res = run_gpu(args, wl)
    if res is not None:
        # libraries that print through C stdio (NCCL's version and debug
        # lines) are flushed first, so the result is the last line
        try:
            import ctypes
            ctypes.CDLL(None).fflush(None)
        except (OSError, AttributeError):
            pass
        sys.stdout.flush()
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
