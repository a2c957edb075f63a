"""Benchmark: head-major vision attention on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl vattn|reference]
                    [--workload 5] [--no-extras]

A step is one call of the whole path (vattn_forward: f16 staging, Q.K^T,
online softmax, P.V, normalise, store) over one batch of the workload.
Metric: attention TFLOP/s = 4*B*H*N^2*D / time.  The default workload is the
largest seeded one (B=8, H=16, N=2304 patches, D=64, keys with a shared
per-head offset); its inputs and output (302 MB) exceed the 129 MB L2, so
consecutive steps stream from HBM.

Under torchrun (N > 1) every rank runs its own replica of the workload on
its own GPU (the heads are independent; there is no collective on the data
path), timing is the max over ranks and `value` counts the work of all ranks
(weak scaling).

--impl reference times the f64 CPU oracle on the host cores instead (rank 0
only), each step a bounded sample of query rows of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s (4·B·H·N²·D) on 1 GB300; % of dense f16 tensor peak"
KERNEL_SOURCES = ["vision_encoder_flash_gb300/csrc/attn_kernel.cuh",
                  "vision_encoder_flash_gb300/csrc/ptx.cuh",
                  "vision_encoder_flash_gb300/csrc/vattn_api.cu",
                  "vision_encoder_flash_gb300/csrc/stage_kernel.cuh"]
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "vattn_fwd_kernel_b8_h16_n2304_d64.md")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
F16_OVER_BF16_NOMINAL = 1.0  # 2.25 PFLOP/s dense for both on GB300


# ---------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: the work of all ranks over the slowest rank's time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            data = json.load(f)
        return data, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """Hash of the kernel sources with comments and blank space removed, so
    that a comment edit does not invalidate the recorded counters."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def traffic_from_profile():
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (same hash); else None."""
    try:
        with open(TRAFFIC_SUMMARY) as f:
            text = f.read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi sampling (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []  # (host_time, sm_mhz, max_mhz, power_w, {reason: active})
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
                pw = float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else float("nan")
            except ValueError:
                continue
            flags = {r: (p.lower() == "active") for r, p in zip(self.REASONS, parts[5:9])}
            self.samples.append((time.time(), sm, mx, pw, flags))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        window = [s for s in self.samples if t0 <= s[0] <= t1]
        note = None
        if not window:
            # timed region shorter than the sampling period: nearest samples
            window = sorted(self.samples, key=lambda s: abs(s[0] - 0.5 * (t0 + t1)))[:3]
            note = "timed region shorter than the 100 ms sampling period; nearest samples"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        reasons = sorted({r for s in window for r, on in s[4].items() if on})
        out = {"sm_mhz": statistics.median(s[1] for s in window),
               "sm_max_mhz": max(s[2] for s in window), "reasons": reasons,
               "samples": len(window),
               "power_w_median": statistics.median(s[3] for s in window)}
        if note:
            out["note"] = note
        return out


def gpu_smi_id(torch, dev) -> str:
    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    dom = getattr(props, "pci_domain_id", None)
    pdev = getattr(props, "pci_device_id", None)
    if bus is not None and dom is not None and pdev is not None:
        return f"{dom:08x}:{bus:02x}:{pdev:02x}.0"
    return str(dev.index)


def gpu_numa_node(torch, dev):
    """NUMA node of the GPU's PCI function (sysfs), or None."""
    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    dom = getattr(props, "pci_domain_id", None)
    pdev = getattr(props, "pci_device_id", None)
    if bus is None or dom is None or pdev is None:
        return None
    try:
        with open(f"/sys/bus/pci/devices/{dom:04x}:{bus:02x}:{pdev:02x}.0/numa_node") as f:
            node = int(f.read().strip())
    except (OSError, ValueError):
        return None
    return node if node >= 0 else None


def node_cpus(node):
    """CPUs of a NUMA node (sysfs cpulist), as a set; empty if unknown."""
    cpus = set()
    try:
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            text = f.read().strip()
    except OSError:
        return cpus
    for part in text.split(","):
        if not part:
            continue
        a, _, b = part.partition("-")
        cpus.update(range(int(a), int(b or a) + 1))
    return cpus


def copy_ceiling(torch, dev, nbytes=256 * 1024 * 1024, reps=5):
    """Pinned host <-> device copy rates (GB/s, best of `reps`): host to
    device alone, device to host alone, and both at once on two streams
    (one cudaMemcpyAsync each way)."""
    n = nbytes // 4
    h_in = torch.empty(n, dtype=torch.float32, pin_memory=True)
    h_out = torch.empty(n, dtype=torch.float32, pin_memory=True)
    h_in.fill_(1.0)
    d_a = torch.empty(n, dtype=torch.float32, device=dev)
    d_b = torch.empty(n, dtype=torch.float32, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            d_a.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_out.copy_(d_b, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_h2d, t_d2h, t_both = timed(h2d), timed(d2h), timed(both)
    del h_in, h_out, d_a, d_b
    return {"h2d_gbs": round(nbytes / t_h2d / 1e9, 1), "d2h_gbs": round(nbytes / t_d2h / 1e9, 1),
            "both_gbs": round(2 * nbytes / t_both / 1e9, 1), "bytes_each_way": nbytes}


# ---------------------------------------------------------------- oracle timing
def oracle_rate(workload, q, k, v, target_s: float, max_rows=None):
    """Time the oracle on a bounded sample of query rows; returns
    (tflops, seconds, rows, threads)."""
    import numpy as np

    import oracle
    threads = oracle.default_threads()
    total = q.shape[0] * q.shape[1] * q.shape[2]
    rng = np.random.Generator(np.random.PCG64(workload.seed))
    probe = min(total, max(threads, 64))
    t = time.perf_counter()
    oracle.rows(q, k, v, rng.integers(0, total, size=probe), threads=threads)
    per_row = (time.perf_counter() - t) / probe
    n_rows = int(max(threads, min(total, target_s / max(per_row, 1e-9))))
    if max_rows is not None:
        n_rows = min(n_rows, max_rows)
    rows = rng.integers(0, total, size=n_rows)
    t = time.perf_counter()
    oracle.rows(q, k, v, rows, threads=threads)
    dt = time.perf_counter() - t
    flops = 4.0 * n_rows * workload.n_patches * workload.head_dim
    return flops / dt / 1e12, dt, n_rows, threads


def oracle_seconds(w, q, k, v, threads, target_s=3.0):
    """Seconds the oracle takes for the whole workload w on `threads`
    threads: timed in full when that is short, else on a random sample of
    query rows (each over all keys) scaled to the full row count."""
    import numpy as np

    import oracle
    total = q.shape[0] * q.shape[1] * q.shape[2]
    rng = np.random.Generator(np.random.PCG64(w.seed + 7))
    probe = min(total, max(threads, 16))
    t = time.perf_counter()
    oracle.rows(q, k, v, rng.integers(0, total, size=probe), threads=threads)
    per_row = (time.perf_counter() - t) / probe
    if per_row * total <= target_s:
        t = time.perf_counter()
        oracle.forward(q, k, v, threads=threads)
        return time.perf_counter() - t, "whole workload"
    n_rows = int(max(threads, min(total, target_s / max(per_row, 1e-9))))
    t = time.perf_counter()
    oracle.rows(q, k, v, rng.integers(0, total, size=n_rows), threads=threads)
    dt = time.perf_counter() - t
    return dt * total / n_rows, f"{n_rows} random rows of {total}, scaled to all rows"


# ---------------------------------------------------------------- arms
def run_reference(args, workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from vattn_inputs import make_inputs
    q, k, v = make_inputs(workload.batch, workload.n_heads, workload.n_patches, workload.head_dim,
                          workload.seed, workload.peaked)
    threads = oracle.default_threads()
    total = q.shape[0] * q.shape[1] * q.shape[2]
    rng = np.random.Generator(np.random.PCG64(workload.seed + 1))
    # size one step so that warmup + steps take about 60 s of host time
    probe = max(threads, 64)
    t = time.perf_counter()
    oracle.rows(q, k, v, rng.integers(0, total, size=probe), threads=threads)
    per_row = (time.perf_counter() - t) / probe
    rows_per_step = int(max(threads, min(total, 60.0 / (args.steps + args.warmup) / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle.rows(q, k, v, rng.integers(0, total, size=rows_per_step), threads=threads)
    samples = [rng.integers(0, total, size=rows_per_step) for _ in range(args.steps)]
    t = time.perf_counter()
    for rows in samples:
        oracle.rows(q, k, v, rows, threads=threads)
    dt = time.perf_counter() - t
    flops = 4.0 * rows_per_step * workload.n_patches * workload.head_dim * args.steps
    value = flops / dt / 1e12
    sample = (f"{rows_per_step} random query rows of {total} per step (each row: all "
              f"{workload.n_patches} keys), f64 three-pass oracle in C, {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload.name, "batch": workload.batch, "n_heads": workload.n_heads,
                   "n_patches": workload.n_patches, "head_dim": workload.head_dim,
                   "seed": workload.seed, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_vattn(args, workload):
    import numpy as np
    import torch

    import vision_encoder_flash_gb300 as vef
    from vattn_inputs import WORKLOADS, make_inputs

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()

    vef.load_library()
    q, k, v = make_inputs(workload.batch, workload.n_heads, workload.n_patches, workload.head_dim,
                          workload.seed + 1000 * rank, workload.peaked)
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    B, H, N, D = q.shape
    ptrs = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), B, H, N, D, sp)

    sampler = ClockSampler(gpu_smi_id(torch, dev))
    sampler.start()
    time.sleep(0.3)

    # ---- warmup
    for _ in range(args.warmup):
        vef.forward_raw(*ptrs)
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)

    # ---- timed region: exactly K launches; per-launch events on the same stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_all0, t_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    host_t0 = time.time()
    t_all0.record(stream)
    for s, e in ev:
        s.record(stream)
        vef.forward_raw(*ptrs)
        e.record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize(dev)
    host_t1 = time.time()
    barrier()
    torch.cuda.synchronize(dev)
    if vef.device_status() != 0:
        raise RuntimeError("kernel reported a wait timeout during the timed region")
    total_ms = t_all0.elapsed_time(t_all1)
    launch_ms = [s.elapsed_time(e) for s, e in ev]
    sampler.stop()
    clocks = sampler.summary(host_t0, host_t1)

    ms_per_step = max_over_ranks(total_ms / args.steps, pg, dev)
    call_ms = max_over_ranks(sum(launch_ms) / len(launch_ms), pg, dev)
    flops = float(workload.flops)
    value = weak_scaling_value(flops, world, ms_per_step)

    # ---- the dominant kernel alone.  With head_dim <= 64 (a multiple of 4)
    # and more than 128 patches a step is one attention kernel (which rounds
    # q, k and v to f16 itself; in the single kernel's mode after clearing its key-tile
    # flags with a memset), so the step's own CUDA events time it.  Otherwise
    # a step is the staging kernel and then the attention kernel; that one is
    # timed alone through vattn_forward_f32q on k and v rounded to f16 once
    # beforehand (untimed), per-launch events on the same stream.
    d_pad = (D + 15) // 16 * 16
    from vision_encoder_flash_gb300 import _lib
    mode = _lib.forward_mode(*ptrs[:8])
    one_kernel = mode in (_lib.MODE_DIRECT, _lib.MODE_SINGLE_KERNEL)
    if one_kernel:
        attn_ms = launch_ms
        n_attn = len(launch_ms)
        single = mode == _lib.MODE_SINGLE_KERNEL
        kernel_what = (("vattn_fwd_kernel<2, 1, 0, 0, kInStageKV>" if single else
                        "vattn_fwd_kernel<2, 1, 0, 0, kInF32>") +
                       " (the whole call is this one kernel; its CUDA events also hold the "
                       "launch gap" + (" and the flag memset)" if single else ")"))
    else:
        # two kernels: the attention kernel timed alone, on the operands the
        # staging pass would give it (k and v rounded to f16 once beforehand,
        # untimed): through vattn_forward_f32q where it applies (f32 q), else
        # vattn_forward_f16 (q rounded too)
        use_f32q = N > 128 and D <= 64 and D % 8 == 0
        if use_f32q:
            k16, v16 = kd.half(), vd.half()
            aptrs = (qd.data_ptr(), k16.data_ptr(), v16.data_ptr(), out.data_ptr(), B, H, N, D, sp)
            afn = vef.forward_f32q_raw
            keep = (k16, v16)
        elif D % 8 == 0:
            q16, k16, v16 = qd.half(), kd.half(), vd.half()
            aptrs = (q16.data_ptr(), k16.data_ptr(), v16.data_ptr(), out.data_ptr(), B, H, N, D, sp)
            afn = vef.forward_f16_raw
            keep = (q16, k16, v16)
        else:
            afn = None
        if afn is None:
            attn_ms = launch_ms
            n_attn = len(launch_ms)
            kernel_what = "the whole call (staging + attention; head_dim % 8 != 0 has no f16 entry)"
        else:
            for _ in range(args.warmup):
                afn(*aptrs)
            torch.cuda.synchronize(dev)
            n_attn = max(3, min(args.steps, 1000))
            ev16 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(n_attn)]
            for s, e in ev16:
                s.record(stream)
                afn(*aptrs)
                e.record(stream)
            torch.cuda.synchronize(dev)
            if vef.device_status() != 0:
                raise RuntimeError("kernel reported a wait timeout")
            attn_ms = [s.elapsed_time(e) for s, e in ev16]
            del keep
            kernel_what = (("vattn_fwd_kernel<2, 1, 0, 0, kInF32Q> (attention with f32 q, f16 k and v; "
                            "timed alone through vattn_forward_f32q)") if use_f32q else
                           "vattn_fwd_kernel (attention on f16 q, k, v; timed alone through "
                           "vattn_forward_f16)")
    kernel_ms = max_over_ranks(sum(attn_ms) / len(attn_ms), pg, dev)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    # the staging kernel: the rest of a call; HBM bytes read (f32 k and v)
    # and written (f16 k and v, rows padded to 16 elements)
    stage_ms = max(call_ms - kernel_ms, 1e-6)
    # (the staging pass rounds q too unless the attention kernel does: head_dim
    # <= 64 with two query tiles)
    n_staged = 2 if (d_pad <= 64 and N > 128 and D % 4 == 0) else 3
    stage_bytes = 0 if one_kernel else n_staged * B * H * N * (4 * D + 2 * d_pad)

    pk, pk_src = peaks()
    peak_tf = float(pk["bf16_tflops"]) * F16_OVER_BF16_NOMINAL

    # ---- end to end through the public API: pinned host tensors in, host out.
    # The pinned buffers are allocated (and first touched) by this thread
    # while it runs on the CPUs of the GPU's own NUMA node, so their pages sit
    # in the host memory nearest the GPU; the plain copy rates of that memory
    # (one 256 MB cudaMemcpyAsync each way, alone and both at once) are the
    # ceiling the end-to-end leg is judged against.
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 30))
        numa = gpu_numa_node(torch, dev)
        cpus = node_cpus(numa) if numa is not None else set()
        old_aff = None
        bound_node = None
        if cpus and hasattr(os, "sched_setaffinity"):
            old_aff = os.sched_getaffinity(0)
            if cpus & old_aff:
                os.sched_setaffinity(0, cpus & old_aff)
                bound_node = numa
            else:
                old_aff = None
        qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (q, k, v))
        oh = torch.empty(q.shape, dtype=torch.float32, pin_memory=True)
        ceiling = copy_ceiling(torch, dev)
        if old_aff is not None:
            os.sched_setaffinity(0, old_aff)
        vef.forward(qh, kh, vh, out=oh)  # warm the allocator
        barrier()
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        for _ in range(e2e_steps):
            vef.forward(qh, kh, vh, out=oh)  # H2D copies, kernel, D2H copy, stream sync
        e2e_s = max_over_ranks((time.perf_counter() - t) / e2e_steps, pg, dev)
        e2e_value = weak_scaling_value(flops, world, e2e_s * 1e3)
        h2d = 3 * q.nbytes
        d2h = oh.numel() * 4
        # the copies alone at the measured concurrent rate bound a step from below
        link_s = max((h2d + d2h) / (ceiling["both_gbs"] * 1e9), h2d / (ceiling["h2d_gbs"] * 1e9))

        e2e = {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": e2e_s * 1e3,
               "copy_peak_gbs": ceiling,
               "copy_bound_ms": link_s * 1e3,
               "frac_of_link": link_s / e2e_s,
               "host_numa_node": bound_node,
               "gpu_numa_node": numa,
               "link_note": "copy_bound_ms: the step's bytes at the measured pinned copy rates "
                            "(max of in+out at the concurrent rate and in alone at the "
                            "host-to-device rate); frac_of_link = copy_bound_ms / ms_per_step",
               "path": "vision_encoder_flash_gb300.forward on pinned host tensors (vattn_forward_host: eight chunks of heads, copies overlapping the kernels)"}

    # ---- oracle on the host cores (rank 0, N = 1 only)
    cpu_baseline = None
    if world == 1 and not args.no_cpu_baseline:
        tf, dt, n_rows, threads = oracle_rate(workload, q, k, v, target_s=10.0)
        cpu_baseline = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                        "sample": f"{n_rows} random query rows of {B * H * N} (each over all {N} "
                                  f"keys) of the same workload, f64 three-pass C oracle, "
                                  f"{dt:.1f} s on {threads} threads"}

    # ---- the other seeded workloads (context; not the bench line)
    extras = {}
    launch_floor = None
    if not args.no_extras:
        for idx, w in sorted(WORKLOADS.items()):
            if w.name == workload.name:
                continue
            xq, xk, xv = make_inputs(w.batch, w.n_heads, w.n_patches, w.head_dim, w.seed, w.peaked)
            xs = [torch.from_numpy(x).to(dev) for x in (xq, xk, xv)]
            xo = torch.empty_like(xs[0])
            xp = (xs[0].data_ptr(), xs[1].data_ptr(), xs[2].data_ptr(), xo.data_ptr(),
                  w.batch, w.n_heads, w.n_patches, w.head_dim, sp)
            for _ in range(10):
                vef.forward_raw(*xp)
            reps = 200
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                vef.forward_raw(*xp)
            b.record(stream)
            torch.cuda.synchronize(dev)
            ms = a.elapsed_time(b) / reps
            qf_ms = queue_filled_ms(torch, stream, lambda: vef.forward_raw(*xp))
            cold = cold_call_ms(torch, dev, stream, lambda: vef.forward_raw(*xp))
            c10, c50, c90 = percentiles(cold)
            wbytes = 16 * w.batch * w.n_heads * w.n_patches * w.head_dim
            extras[w.name] = {"ms": round(ms, 5), "tflops": round(w.flops / ms / 1e9, 2),
                              "frac_of_peak": round(w.flops / ms / 1e9 / peak_tf, 4),
                              "bytes": wbytes,
                              "achieved_gbs": round(wbytes / (ms * 1e-3) / 1e9, 1),
                              "frac_of_hbm": round(wbytes / (ms * 1e-3) / 1e9 / float(pk["hbm_gbs"]), 4),
                              "l2": "hot (back-to-back, inputs may fit in L2)",
                              "ms_queue_filled": round(qf_ms, 5),
                              "tflops_queue_filled": round(w.flops / qf_ms / 1e9, 2),
                              "queue_filled": "200 calls enqueued behind a 20 ms spin kernel: "
                                              "device time per call without host gaps",
                              "cold_ms_p10_p50_p90": [round(c10, 5), round(c50, 5), round(c90, 5)],
                              "cold_tflops_p50": round(w.flops / c50 / 1e9, 2),
                              "cold": "L2 flushed (512 MB written) before each of 30 calls, "
                                      "outside the timed events"}
            extras[w.name]["cold_gbs_p50"] = round(wbytes / (c50 * 1e-3) / 1e9, 1)
            if idx <= 3 and world == 1 and not args.no_cpu_baseline:
                # the oracle on one core and on all host cores (context)
                import oracle
                one_s, one_how = oracle_seconds(w, xq, xk, xv, 1)
                all_t = oracle.default_threads()
                all_s, all_how = oracle_seconds(w, xq, xk, xv, all_t)
                extras[w.name].update({"oracle_1core_s": round(one_s, 4), "oracle_1core_how": one_how,
                                       f"oracle_{all_t}core_s": round(all_s, 4),
                                       "oracle_allcore_how": all_how})
            if w.head_dim % 8 == 0:  # the attention kernel alone (f16 inputs)
                x16 = [t.half() for t in xs]
                xp16 = (x16[0].data_ptr(), x16[1].data_ptr(), x16[2].data_ptr(), xo.data_ptr(),
                        w.batch, w.n_heads, w.n_patches, w.head_dim, sp)
                for _ in range(10):
                    vef.forward_f16_raw(*xp16)
                a.record(stream)
                for _ in range(reps):
                    vef.forward_f16_raw(*xp16)
                b.record(stream)
                torch.cuda.synchronize(dev)
                kms = a.elapsed_time(b) / reps
                extras[w.name].update({"kernel_ms": round(kms, 5),
                                       "kernel_tflops": round(w.flops / kms / 1e9, 2),
                                       "kernel_frac_of_peak": round(w.flops / kms / 1e9 / peak_tf, 4)})
                del x16
        if vef.device_status() != 0:
            raise RuntimeError("kernel reported a wait timeout")
        launch_floor = {"us": round(1e3 * queue_filled_ms(
            torch, stream, lambda: torch.cuda._sleep(0), reps=1000), 3),
                        "how": "an empty kernel (torch.cuda._sleep(0)) launched 1000 times behind "
                               "a spin kernel: device time per launch"}

    # ---- NeoX RoPE rows (context): the rotation fused into the staging pass
    # of a full call, and the standalone in-place rotation of q (HBM-bound:
    # every rotated f32 element read and written once)
    variants = {}
    if not args.no_extras:
        reps = 200
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(10):
            vef.forward_rope(qd, kd, vd, D, 0, 10000.0, out=out)
        a.record(stream)
        for _ in range(reps):
            vef.forward_rope(qd, kd, vd, D, 0, 10000.0, out=out)
        b2.record(stream)
        torch.cuda.synchronize(dev)
        fms = a.elapsed_time(b2) / reps
        xr = torch.cat([qd, kd, vd], dim=0)  # 226 MB > L2: every step streams from HBM
        for _ in range(10):
            vef.rope_neox(xr, D, 0, 10000.0)
        a.record(stream)
        for _ in range(reps):
            vef.rope_neox(xr, D, 0, 10000.0)
        b2.record(stream)
        torch.cuda.synchronize(dev)
        rms = a.elapsed_time(b2) / reps
        rbytes = 3 * B * H * N * (D // 2 * 2) * 4 * 2
        x16 = [t.half() for t in (qd, kd, vd)]
        o16 = torch.empty_like(x16[0])
        for _ in range(10):
            vef.forward_f16io(*x16, out=o16)
        a.record(stream)
        for _ in range(reps):
            vef.forward_f16io(*x16, out=o16)
        b2.record(stream)
        torch.cuda.synchronize(dev)
        f16io_ms = a.elapsed_time(b2) / reps
        del x16, o16
        for _ in range(5):
            vef.forward_accurate(qd, kd, vd, out=out)
        a.record(stream)
        for _ in range(reps // 4):
            vef.forward_accurate(qd, kd, vd, out=out)
        b2.record(stream)
        torch.cuda.synchronize(dev)
        acc_ms = a.elapsed_time(b2) / (reps // 4)
        if vef.device_status() != 0:
            raise RuntimeError("kernel reported a wait timeout")
        variants = {
            "accurate_call": {"ms": round(acc_ms, 5), "tflops": round(flops / acc_ms / 1e9, 2),
                              "tensor_tflops": round(3 * flops / acc_ms / 1e9, 2),
                              "vs_plain_call": round(acc_ms / ms_per_step, 4),
                              "what": "vattn_forward_accurate (split-f16, three products per "
                                      "matrix product; tflops counts the algorithmic flops once)"},
            "rope_fused_call": {"ms": round(fms, 5), "tflops": round(flops / fms / 1e9, 2),
                                "vs_plain_call": round(fms / ms_per_step, 4),
                                "what": "vattn_forward_rope, rope_dims = head_dim, pos0 0, base 1e4"},
            "f16io_kernel": {"ms": round(f16io_ms, 5), "tflops": round(flops / f16io_ms / 1e9, 2),
                             "frac_of_peak": round(flops / f16io_ms / 1e9 / peak_tf, 4),
                             "what": "vattn_forward_f16io: the attention kernel alone, f16 in and out"},
            "rope_inplace": {"ms": round(rms, 5), "bytes": rbytes,
                             "achieved_gbs": round(rbytes / (rms * 1e-3) / 1e9, 1),
                             "frac_of_hbm": round(rbytes / (rms * 1e-3) / 1e9 / float(pk["hbm_gbs"]), 4),
                             "what": "vattn_rope_neox on q, k, v stacked (f32, in place, 226 MB > L2), includes the angle-table kernel"},
        }
        del xr
        variants["conv1d_step"] = conv1d_variant(torch, dev, stream, float(pk["hbm_gbs"]))

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": workload.name, "batch": B, "n_heads": H, "n_patches": N,
                   "head_dim": D, "seed": workload.seed, "inputs": "f32 head-major, q pre-scaled",
                   "l2": f"inputs+output {(4 * q.nbytes) / 1e6:.0f} MB per step > 129 MB L2 (no flush)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": traffic_from_profile(),
                     "peak_source": f"{pk_src} bf16_tflops (burst) x {F16_OVER_BF16_NOMINAL} "
                                    f"(f16/bf16 nominal ratio)",
                     "kernel": kernel_what,
                     "kernel_ms": kernel_ms, "launches_timed": n_attn,
                     "kernel_ms_p10_p50_p90": [round(x, 5) for x in percentiles(attn_ms)],
                     "frac_of_sustained": achieved / (float(pk.get("bf16_tflops_sustained", peak_tf))
                                                      * F16_OVER_BF16_NOMINAL),
                     "stage_kernel": None if one_kernel else {
                         "bound": "hbm", "ms": stage_ms, "bytes": stage_bytes,
                         "achieved_gbs": stage_bytes / (stage_ms * 1e-3) / 1e9,
                         "peak_gbs": float(pk["hbm_gbs"]),
                         "frac": stage_bytes / (stage_ms * 1e-3) / 1e9 / float(pk["hbm_gbs"]),
                         "what": f"vattn_stage_kernel on {'k and v' if n_staged == 2 else 'q, k and v'} (f32 in, f16 out)",
                         "how": "per-call time minus the attention kernel's time"}},
        "cpu_baseline": cpu_baseline,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": (1 if one_kernel else 2) * args.steps,  # (staging +) attention per step
        "other_workloads": extras,
        "launch_floor": launch_floor,
        "variants": variants,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def percentiles(xs, qs=(10, 50, 90)):
    """Nearest-rank percentiles of a list of numbers."""
    ys = sorted(xs)
    return [ys[min(len(ys) - 1, max(0, math.ceil(q / 100 * len(ys)) - 1))] for q in qs]


def queue_filled_ms(torch, stream, call, reps=200):
    """Device time per call with the host far ahead of the device: a spin
    kernel (about 20 ms) holds the stream while the host enqueues every call,
    so the events see back-to-back calls and no host-side gaps."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(40_000_000)
    a.record(stream)
    for _ in range(reps):
        call()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / reps


def cold_call_ms(torch, dev, stream, call, reps=30):
    """Per-call times with L2 flushed before each call: a 512 MB buffer (four
    times the 129 MB L2) is written between calls, outside the timed events."""
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    times = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    del flush
    return times


def conv1d_variant(torch, dev, stream, hbm_gbs):
    """The depthwise conv1d rolling-buffer step on its workload: two input
    sets used in turn (each 268 MB, so a step never finds the previous
    step's data in the 129 MB L2), CUDA events around 200 launches."""
    import vision_encoder_flash_gb300 as vef
    from vattn_inputs import CONV1D_WORKLOAD as wl, conv1d_inputs, conv1d_workload_name

    B, H, K, DC = wl["batch"], wl["hidden"], wl["kernel_size"], wl["d_conv"]
    sets = []
    for i in range(2):
        x, buf, w = conv1d_inputs(B, H, K, DC, wl["seed"] + i)
        sets.append(tuple(torch.from_numpy(a).to(dev) for a in (x, buf, w)) +
                    (torch.empty(B, H, device=dev),))
    reps = 200
    for i in range(10):
        x, buf, w, o = sets[i & 1]
        vef.conv1d_step(x, buf, w, out=o, stream=stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for i in range(reps):
        x, buf, w, o = sets[i & 1]
        vef.conv1d_step(x, buf, w, out=o, stream=stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / reps
    nbytes = B * H * (2 * DC + 2) * 4 + H * K * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    del sets
    return {"workload": conv1d_workload_name(), "ms": round(ms, 5), "bytes": nbytes,
            "achieved_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_gbs, 4),
            "bound": "hbm", "launches_timed": reps,
            "what": "vattn_conv1d_step: (2 d_conv + 2) * 4 algorithmic bytes per (sequence, channel) "
                    "(buffer read and rewritten, input read, output written) + the weights once; "
                    "two input sets in turn, larger than L2"}


def main(argv=None):
    from vattn_inputs import WORKLOADS
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["vattn", "reference"], default="vattn")
    ap.add_argument("--workload", type=int, default=5, choices=sorted(WORKLOADS))
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (host buffers); for profiling the device steps")
    ap.add_argument("--conv1d-only", action="store_true",
                    help="time only the conv1d rolling-buffer step and print its line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, _, _ = dist_env()
    if world != args.gpus:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}; using WORLD_SIZE",
              file=sys.stderr)
    workload = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, workload)
    if args.conv1d_only:
        import torch
        import vision_encoder_flash_gb300 as vef
        from vision_encoder_flash_gb300 import build
        build.build()
        vef.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        line = conv1d_variant(torch, dev, torch.cuda.current_stream(dev), float(peaks()[0]["hbm_gbs"]))
        print(json.dumps(line))
        return 0
    return run_vattn(args, workload)


if __name__ == "__main__":
    sys.exit(main())
