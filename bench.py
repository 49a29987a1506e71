#!/usr/bin/env python3
"""Benchmark: fused large-vocabulary cross-entropy forward + backward on GB300.

One "step" is one ce_fwd_bwd call (label census, row kernel, finalize) over
one batch of seeded synthetic logits already resident in HBM.  The default
workload is bf16 logits [N=2048, V=131072] (sequence 2048 x batch 1, the
128K vocabulary) with label smoothing 0.1, argmax and token accuracy.  The
same run times every other cross-entropy configuration the same way (the
line's "configs" object: fp32 [256, 4096], bf16 [8192, 32000], bf16
[8192, 151936] with a padded row stride and softcap 30, and 32 rows of
151936 on both the V-split and the row kernel), the fused linear
cross-entropy (flce_fwd_bwd: hidden [4096, 6656] x weight [202048, 6656],
softcap 30) against the dense bf16 tensor roofline ("flce"), and companion
legs (forward only, one vocabulary shard's rank step, SwiGLU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--no-flce]
                    [--no-configs]
    python bench.py --workload flce-bf16-4096x6656x202048-softcap30   # FLCE as the headline
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the rows of different batches never interact): weak scaling, no collective
on the data path; the elapsed time is the max over ranks.  A multi-GPU run
times the headline (and its host-buffer e2e) only; the other configurations
and legs run on one GPU.

Prints ONE JSON line on rank 0.
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

METRIC = "CE fwd+bwd ms & HBM GB/s (N=2048,V=128K bf16); % of HBM roofline"
FLCE_METRIC = "fused linear CE fwd+bwd TFLOP/s (6NVH, N=4096,H=6656,V=202048 bf16); % of dense bf16"
FLCE_DEFAULT = "flce-bf16-4096x6656x202048-softcap30"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
# The pages' fastest prior art on this exact workload (context, another machine):
# Transformer Engine CE fwd+bwd 0.711 ms on H100, BF16, seq 2048, batch 1, 128K vocab
# = 2*2048*131072*2 bytes / 0.711 ms = 1510 GB/s.
CONTEXT_GBS = 2 * 2048 * 131072 * 2 / 0.711e-3 / 1e9


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_tensor_peak(sustained: bool):
    """Dense bf16 TFLOP/s: the burst figure for a kernel timed alone, the
    sustained one (a seconds-long loop under the power cap) otherwise."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), f"measured ({key})"
    except Exception:
        return (FALLBACK_BF16_TFLOPS_SUSTAINED if sustained else FALLBACK_BF16_TFLOPS), "fallback"


# The CUDA sources each profiled kernel is built from (its launch code included):
# a change to any of them invalidates that kernel's recorded ncu traffic.
KERNEL_SOURCES = {
    "ce_rows_kernel": ["ce_rows.cuh", "ce_rows_bf16.cu", "ce_rows_f32.cu", "ce_common.cuh",
                       "ce_census.cuh", "ptx.cuh", "host_util.h", "ce.cu"],
    "ce_split_kernel": ["ce_split.cuh", "ce_split_bf16.cu", "ce_split_f32.cu", "ce_common.cuh",
                        "ce_census.cuh", "ptx.cuh", "host_util.h", "ce.cu"],
    "vlmce_gemm_kernel": ["gemm.cuh", "gemm_types.h", "gemm_launch.h", "gemm.cu", "tcgen05.cuh",
                          "ce_common.cuh", "ptx.cuh", "host_util.h", "flce.cu"],
}


def kernel_sources_sha(kernel: str) -> str:
    """sha256 over the CUDA sources of one kernel (file names and contents)."""
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kernel]):
        path = os.path.join(ROOT, "vocabulary_lm_cross_gb300", "csrc", name)
        h.update(name.encode())
        h.update(open(path, "rb").read() if os.path.exists(path) else b"<missing>")
    return h.hexdigest()


def recorded_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if the kernel
    source has not changed since the capture (else None)."""
    sha = kernel_sources_sha(kernel)
    path = os.path.join(ROOT, "profiles", f"ncu_{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            if ts < t0 or ts > t1 + 0.15:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        if self.uuid:
            mine = [r for r in rows if self.uuid in r[0]]
            rows = mine or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def oracle_gbs(w, x_host_bits, labels_host, rows, threads=0):
    """Time the fp64 oracle (forward + backward with gradient) on the given rows."""
    from oracle import ce as oc
    xs = x_host_bits[rows]
    ls = labels_host[rows]
    n_valid, _ = oc.count(labels_host, w.V, -100)
    scale = oc.scale(w.reduction, w.grad_scale, n_valid)
    t0 = time.perf_counter()
    oc.rows(xs, w.dtype, w.V, ls, label_smoothing=w.label_smoothing, softcap=w.softcap,
            row_scale=scale, want_grad=True, threads=threads)
    dt = time.perf_counter() - t0
    nbytes = 2 * len(rows) * w.V * w.elt_bytes
    return nbytes / dt / 1e9, dt


def host_inputs(w):
    """Pristine inputs on the host (seeded generator on the CPU)."""
    import numpy as np
    import torch
    from vocabulary_lm_cross_gb300.workloads import make_ce_inputs
    x, lab = make_ce_inputs(w, device="cpu")
    if w.dtype == "bf16":
        bits = x.view(torch.int16).numpy().view(np.uint16)
    else:
        bits = x.numpy()
    return x, lab, bits, lab.numpy()


def cpu_baseline_sample(w, budget_s=10.0):
    """Oracle throughput on a bounded sample of the workload's rows."""
    from oracle import ce as oc
    w_small = w.resized(N=min(w.N, 2048))
    _, _, bits, lab = host_inputs(w_small)
    threads = oc.default_threads()
    n0 = min(w_small.N, threads)
    _, dt0 = oracle_gbs(w_small, bits, lab, list(range(n0)), threads)
    per_row = dt0 / n0
    n = int(max(n0, min(w_small.N, budget_s / max(per_row, 1e-9))))
    # whole passes over the sample until the budget is spent
    reps, dt = 0, 0.0
    while reps == 0 or dt < budget_s:
        _, dti = oracle_gbs(w_small, bits, lab, list(range(n)), threads)
        reps += 1
        dt += dti
    gbs = 2 * n * w.V * w.elt_bytes * reps / dt / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle forward+backward (with gradient) on {n} rows of the same "
                      f"workload recipe (rows of V={w.V}), {reps} passes in {dt:.1f} s"}


def run_reference(args, w):
    """The oracle timed on the host cores: each step is a bounded sample of rows."""
    from oracle import ce as oc
    rank = env_int("RANK", 0)
    if rank != 0:
        return
    threads = oc.default_threads()
    rows_per_step = max(1, min(w.N, 2 * threads))
    w_small = w.resized(N=rows_per_step)
    _, _, bits, lab = host_inputs(w_small)
    rows = list(range(rows_per_step))
    for _ in range(args.warmup):
        oracle_gbs(w_small, bits, lab, rows, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_gbs(w_small, bits, lab, rows, threads)
    dt = time.perf_counter() - t0
    nbytes = 2 * rows_per_step * w.V * w.elt_bytes
    value = nbytes * args.steps / dt / 1e9
    sample = (f"fp64 oracle forward+backward on {rows_per_step} rows (of {w.N}) of the "
              f"workload per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "N": w.N, "V": w.V, "rows_per_step": rows_per_step},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# The other cross-entropy configurations timed beside the headline (one line
# each in the "configs" object), and the few-wide-rows case on both kernels.
CONFIG_WORKLOADS = ("ce-f32-256x4096", "ce-bf16-8192x32000",
                    "ce-bf16-8192x151936-stride152064-softcap30-sum")
WIDE_ROWS_WORKLOAD = "ce-bf16-32x151936-ls0.1-argmax"


def time_ce(w, dev, steps, warmup, *, rank=0, world=1, barrier=lambda: None, sampler=None,
            path=None, soak_s=0.0):
    """Time ce_fwd_bwd on one workload with inputs resident in HBM.

    Inputs larger than L2: a ring of copies, each timed step on a pristine one,
    K steps back to back between two CUDA events.  Inputs that fit in L2: each
    step on a pristine copy, a buffer twice the L2 size written before each
    step (outside the events), one event pair per step.  Then a second pass
    records the dominant kernel's duration per step (vlmce_profile_events).
    ``path`` ("rows" | "split") forces the kernel through VLMCE_CE_PATH."""
    import torch
    import torch.distributed as dist

    import vocabulary_lm_cross_gb300 as v
    from vocabulary_lm_cross_gb300 import capi
    from vocabulary_lm_cross_gb300.workloads import make_ce_inputs

    lib = capi.lib()
    old_path = os.environ.get("VLMCE_CE_PATH")
    if path:
        os.environ["VLMCE_CE_PATH"] = path
    try:
        x0, lab = make_ce_inputs(w.resized(seed=w.seed + 1000 * rank), device=dev)
        V = w.V
        buf_bytes = x0.numel() * x0.element_size()
        l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 132e6)
        big = buf_bytes > l2
        n_buf = min(warmup + steps, max(2, int(64e9 // buf_bytes)))
        bufs = [x0.clone() for _ in range(n_buf)]
        fresh = n_buf >= warmup + steps
        steps = min(steps, n_buf)  # every timed step on its own pristine copy
        flush = None if big else torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
        out = v.CEResult(loss=torch.empty(w.N, dtype=torch.float32, device=dev),
                         argmax=torch.empty(w.N, dtype=torch.int64, device=dev),
                         reduced=torch.empty(2, dtype=torch.float32, device=dev),
                         counts=torch.empty(4, dtype=torch.int64, device=dev))
        ws_bytes = v.workspace_bytes(w.N, V, x0.dtype)
        ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev)
        plan = v.describe_plan(w.N, V, x0.dtype, w.softcap)

        def step(i):
            v.ce_fwd_bwd(bufs[i % n_buf][:, :V], lab, ignore_index=-100,
                         label_smoothing=w.label_smoothing, softcap=w.softcap,
                         reduction=w.reduction, grad_scale=w.grad_scale, out=out, workspace=ws)

        def restore():
            for b in bufs:
                b.copy_(x0)
            torch.cuda.synchronize()

        def timed(i, kernel_events=None):
            """One step; returns its event pair when the steps are timed one by one."""
            if kernel_events is not None:
                lib.vlmce_profile_events(ctypes_handle(kernel_events[0], stream),
                                         ctypes_handle(kernel_events[1], stream))
            if big:
                step(i)
                return None
            flush.zero_()  # evict the previous step's lines from L2
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step(i)
            e1.record(stream)
            return e0, e1

        for i in range(warmup):
            step(i)
        torch.cuda.synchronize()
        t_soak0 = time.time()
        # soak: keep the GPU busy before the timed region so the clock samples
        # describe the loaded state (untimed; the buffers then hold gradients)
        j = 0
        while time.time() < t_soak0 + soak_s:
            for _ in range(10):
                step(j)
                j += 1
            torch.cuda.synchronize()
        restore()

        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        ev0.record(stream)
        pairs = [timed(warmup + i) for i in range(steps)]
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        t1 = time.time()
        ms = ev0.elapsed_time(ev1) / steps if big else \
            statistics.fmean(e0.elapsed_time(e1) for e0, e1 in pairs)
        if world > 1:
            t = torch.tensor([ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms = float(t.item())
        counts = out.counts.cpu().tolist()

        # the dominant kernel's duration, events recorded by the library on the stream
        restore()
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            timed(warmup + i, kev[i])
        torch.cuda.synchronize()
        kern_ms = statistics.fmean(b.elapsed_time(e) for b, e in kev)
        del bufs, flush
    finally:
        if path:
            if old_path is None:
                os.environ.pop("VLMCE_CE_PATH", None)
            else:
                os.environ["VLMCE_CE_PATH"] = old_path
    bytes_step = w.algorithmic_bytes
    kernel = "ce_rows_kernel" if plan["kernel"] == "rows" else "ce_split_kernel"
    peak, peak_src = load_peaks()
    if big:
        l2_note = (("inputs larger than L2: each timed step consumes its own fresh copy "
                    f"of the {buf_bytes / 1e6:.0f} MB logits ({buf_bytes * n_buf / 1e9:.1f} GB)")
                   if fresh else f"ring of {n_buf} buffers of {buf_bytes / 1e6:.0f} MB (> L2), "
                   "restored before the timed steps, one pristine copy per timed step")
    else:
        l2_note = (f"{buf_bytes / 1e6:.1f} MB of logits fit in L2: a {2 * l2 / 1e6:.0f} MB buffer "
                   "is written before every step (outside the events), each step on a pristine "
                   "copy, one event pair per step")
    return {"ms": ms, "kern_ms": kern_ms, "steps": steps, "bytes": bytes_step, "kernel": kernel,
            "plan": plan,
            "peak": peak, "peak_src": peak_src, "counts": counts, "ok": counts[3] == 0,
            "workspace_bytes": ws_bytes, "l2": l2_note, "t0": t0, "t1": t1,
            "t_soak0": t_soak0, "x0": x0, "lab": lab, "buf_bytes": buf_bytes,
            "clocks": sampler.summary(t0, t1) if sampler else None}


def config_entry(w, r):
    """The per-configuration object of the bench line."""
    gbs = r["bytes"] / (r["ms"] * 1e-3) / 1e9
    kgbs = r["bytes"] / (r["kern_ms"] * 1e-3) / 1e9
    return {"N": w.N, "V": w.V, "row_stride": w.stride, "dtype": w.dtype,
            "label_smoothing": w.label_smoothing, "softcap": w.softcap, "reduction": w.reduction,
            "ms": r["ms"], "steps": r["steps"], "GB/s": gbs, "step_frac": gbs / r["peak"],
            "roofline": {"bound": "hbm", "kernel": r["kernel"], "kernel_ms": r["kern_ms"],
                         "achieved": kgbs, "peak": r["peak"],
                         "peak_source": f"{r['peak_src']} (copy GB/s)", "unit": "GB/s",
                         "frac": kgbs / r["peak"], "bytes_per_launch": r["bytes"],
                         "traffic": recorded_traffic(r["kernel"], w.name)},
            "workspace_bytes": r["workspace_bytes"], "plan": r["plan"],
            "device_status_ok": r["ok"], "l2": r["l2"], "clocks": r["clocks"]}


def run_configs(args, head_name, dev, sampler):
    """Every other CE configuration, timed as the headline is (1 GPU)."""
    import torch

    from vocabulary_lm_cross_gb300.workloads import CE_WORKLOADS
    steps = max(5, min(args.steps, 30))
    out = {}
    for name in CONFIG_WORKLOADS:
        if name == head_name:
            continue
        w = CE_WORKLOADS[name]
        out[name] = config_entry(w, time_ce(w, dev, steps, args.warmup, sampler=sampler))
        torch.cuda.empty_cache()
    w = CE_WORKLOADS[WIDE_ROWS_WORKLOAD]
    out[w.name] = {path: config_entry(w, time_ce(w, dev, steps, args.warmup, sampler=sampler,
                                                 path=path))
                   for path in ("split", "rows")}
    out[w.name]["note"] = ("few wide rows: the V-split kernel (a cluster of CTAs per row, "
                           "TMA-staged slices, DSMEM merge) is the default; the row kernel "
                           "timed on the same inputs")
    torch.cuda.empty_cache()
    return out


def bind_to_gpu_local_cpus(dev) -> str:
    """Run this process on the CPUs local to the GPU (its NUMA node), so that
    page-locked host buffers allocated afterwards sit next to the GPU's host
    link; returns what was done (for the bench line).  The caller restores
    the previous affinity (os.sched_setaffinity) when it is done."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev)
        bdf = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        path = f"/sys/bus/pci/devices/{bdf}/local_cpulist"
        text = open(path).read().strip()
        cpus = set()
        for part in text.split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0) or cpus
        if not cpus or cpus == os.sched_getaffinity(0):
            return f"unchanged ({path}: {text})"
        os.sched_setaffinity(0, cpus)
        return f"bound to the GPU's local CPUs {text}"
    except Exception as e:  # no sysfs entry, or an older torch without PCI ids
        return f"unchanged ({type(e).__name__})"


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import vocabulary_lm_cross_gb300 as v

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local = env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cpus0 = os.sched_getaffinity(0)
    affinity = bind_to_gpu_local_cpus(dev)
    if world > 1:
        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            dist.barrier()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    head = time_ce(w, dev, args.steps, args.warmup, rank=rank, world=world, barrier=barrier,
                   sampler=sampler, soak_s=args.soak)
    x0, lab = head["x0"], head["lab"]
    ms = head["ms"] * args.steps
    kern_ms = head["kern_ms"]
    ok_status = head["ok"]
    V = w.V
    stream = torch.cuda.current_stream(dev)
    out = v.CEResult(loss=torch.empty(w.N, dtype=torch.float32, device=dev),
                     argmax=torch.empty(w.N, dtype=torch.int64, device=dev),
                     reduced=torch.empty(2, dtype=torch.float32, device=dev),
                     counts=torch.empty(4, dtype=torch.int64, device=dev))
    ws = torch.empty(v.workspace_bytes(w.N, V, x0.dtype), dtype=torch.uint8, device=dev)

    # forward only (compute_grad=False): one read of the logits per step; the
    # logits are not modified, so a ring of copies larger than L2 serves
    fw_steps = min(args.steps, 20)
    n_fw = max(2, min(fw_steps, int(2 * 129e6 // head["buf_bytes"]) + 2))
    fbufs = [x0.clone() for _ in range(n_fw)]
    fe0 = torch.cuda.Event(enable_timing=True)
    fe1 = torch.cuda.Event(enable_timing=True)

    def fw_step(i):
        v.ce_fwd_bwd(fbufs[i % n_fw][:, :V], lab, label_smoothing=w.label_smoothing,
                     softcap=w.softcap, reduction=w.reduction, grad_scale=w.grad_scale,
                     compute_grad=False, out=out, workspace=ws)

    for i in range(3):
        fw_step(i)
    torch.cuda.synchronize()
    fe0.record(stream)
    for i in range(fw_steps):
        fw_step(i)
    fe1.record(stream)
    torch.cuda.synchronize()
    del fbufs
    fw_ms = fe0.elapsed_time(fe1) / fw_steps
    fw_bytes = w.N * V * x0.element_size()
    peak_fw, peak_fw_src = load_peaks()
    forward_only = {"metric": "CE forward only (no gradient, logits kept) GB/s",
                    "value": world * fw_bytes / (fw_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "ms_per_step": fw_ms, "steps": fw_steps, "bytes_per_step": fw_bytes,
                    "roofline": {"bound": "hbm", "achieved": fw_bytes / (fw_ms * 1e-3) / 1e9,
                                 "peak": peak_fw, "peak_source": f"{peak_fw_src} (copy GB/s)",
                                 "unit": "GB/s",
                                 "frac": fw_bytes / (fw_ms * 1e-3) / 1e9 / peak_fw,
                                 "measured_over": "whole step (census, row kernel, finalize)"},
                    "l2": f"ring of {n_fw} copies of the logits (together > 2 x L2), round robin"}

    # end to end through the public API with host buffers: ce_fwd_bwd_host on
    # page-locked host logits (streamed through the GPU in chunks of rows, the
    # gradient copied back in place), labels and outputs in host memory.  Each
    # timed call gets a pristine host copy of the logits (restored untimed).
    x_pristine = x0.cpu()
    x_host = x_pristine.pin_memory()
    lab_host = lab.cpu().pin_memory()
    out_h = v.CEResult(loss=torch.empty(w.N, dtype=torch.float32).pin_memory(),
                       argmax=torch.empty(w.N, dtype=torch.int64).pin_memory(),
                       reduced=torch.empty(2, dtype=torch.float32).pin_memory(),
                       counts=torch.empty(4, dtype=torch.int64).pin_memory())
    ws_h = torch.empty(v.host_workspace_bytes(w.N, V, x_host.stride(0), x_host.dtype),
                       dtype=torch.uint8, device=dev)

    def e2e_call():
        v.ce_fwd_bwd_host(x_host[:, :V], lab_host, device=dev, ignore_index=-100,
                          label_smoothing=w.label_smoothing, softcap=w.softcap,
                          reduction=w.reduction, grad_scale=w.grad_scale, out=out_h,
                          workspace=ws_h)

    for _ in range(max(1, min(args.warmup, 3))):
        x_host.copy_(x_pristine)
        e2e_call()
        torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, 10))
    barrier()
    e2e_ms = 0.0
    for _ in range(e2e_steps):
        x_host.copy_(x_pristine)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        e2e_call()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= e2e_steps
    e2e_ok = int(out_h.counts[3]) == 0
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    row_bytes = V * x_host.element_size()
    h2d = w.N * row_bytes + lab_host.numel() * 8
    d2h = w.N * row_bytes + w.N * 4 + w.N * 8 + 8 + 32
    del x_host, x_pristine, ws_h
    os.sched_setaffinity(0, cpus0)  # the CPU baseline below uses every host core
    head.pop("x0")
    head.pop("lab")
    del x0, lab
    torch.cuda.empty_cache()

    # the other configurations and the companion legs run on one GPU only: a
    # multi-GPU run times the replicated headline alone
    single = world == 1
    configs = run_configs(args, w.name, dev, sampler) if single and not args.no_configs else None
    shard = run_shard(args, w, dev, world, barrier, sampler) \
        if single and w.V % 8 == 0 else None
    torch.cuda.empty_cache()
    swiglu = run_swiglu(args, dev, sampler) if single and not args.no_flce else None
    torch.cuda.empty_cache()

    flce = None
    if single and not args.no_flce:
        from vocabulary_lm_cross_gb300.workloads import FLCE_WORKLOADS
        fw = FLCE_WORKLOADS[FLCE_DEFAULT]
        f = run_flce(args, fw, min(args.steps, 10), dev, world, barrier, sampler)
        flce = {"metric": FLCE_METRIC, "value": f["value"], "unit": "TFLOP/s",
                "ms_per_step": f["ms"], "steps": f["steps"], "roofline": f["roofline"],
                "e2e": f["e2e"], "gpu_launches": f["gpu_launches"], "clocks": f["clocks"],
                "config": f["config"], "device_status_ok": f["ok_status"]}
        torch.cuda.empty_cache()
        flce["row_chunked"] = run_flce_rows(fw, dev)
    sampler.stop()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    bytes_step = w.algorithmic_bytes
    plan = head["plan"]
    kernel_name = head["kernel"]
    value = world * bytes_step * args.steps / (ms * 1e-3) / 1e9
    peak, peak_src = load_peaks()
    achieved = bytes_step / (kern_ms * 1e-3) / 1e9
    clocks = sampler.summary(head["t_soak0"], head["t1"])
    cpu = cpu_baseline_sample(w) if world == 1 else None
    headline = w.name == "ce-bf16-2048x131072-ls0.1-argmax"
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": (value / world / CONTEXT_GBS) if headline else None,
        "dtype": w.dtype, "data": "synthetic (seeded normal logits, uniform labels)",
        "config": {"workload": w.name, "N": w.N, "V": V, "row_stride": w.stride,
                   "label_smoothing": w.label_smoothing, "softcap": w.softcap,
                   "reduction": w.reduction, "parallelism": f"replicas x{world}",
                   "l2": head["l2"],
                   "vs_baseline_is": "value per GPU / 1510 GB/s = TE CE 0.711 ms on H100 "
                                     "(the pages' number, another machine: context)",
                   "device_status_ok": ok_status,
                   "workspace_bytes": head["workspace_bytes"],
                   "plan": plan},
        "roofline": {"bound": "hbm", "kernel": kernel_name, "achieved": achieved,
                     "peak": peak, "peak_source": f"{peak_src} (copy GB/s)", "unit": "GB/s",
                     "frac": achieved / peak, "kernel_ms": kern_ms,
                     "bytes_per_launch": bytes_step,
                     "traffic": recorded_traffic(kernel_name, w.name)},
        "cpu_baseline": cpu,
        "e2e": {"value": bytes_step / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "call": "ce_fwd_bwd_host on page-locked host logits, labels and outputs",
                "host_memory": affinity, "device_status_ok": e2e_ok},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "configs": configs,
        "forward_only": forward_only,
        "swiglu": swiglu,
        "shard": shard,
        "flce": flce,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_shard(args, w, dev, world, barrier, sampler, tp=8):
    """One rank's step of the vocabulary-sharded CE in a TP = `tp` layout of
    the workload: statistics of its shard, then loss and in-place gradient of
    its shard from the `tp` gathered records (merged inside the gradient
    kernel: ce_shard_fwd_bwd_gathered).  The other ranks' records are
    formed beforehand (on a real group they arrive by an all-gather of
    N x 32 bytes each).  Each timed step works on a fresh copy of the shard."""
    import torch

    from vocabulary_lm_cross_gb300 import shard as sh
    from vocabulary_lm_cross_gb300.ce import workspace_bytes as v_ws_bytes
    from vocabulary_lm_cross_gb300.workloads import make_ce_inputs

    x0, lab = make_ce_inputs(w, device=dev)
    V = w.V
    vl = V // tp
    shards = [x0[:, i * vl:(i + 1) * vl].contiguous() for i in range(tp)]
    del x0
    others = torch.stack([sh.shard_stats(s_, lab, i * vl, V, softcap=w.softcap)
                          for i, s_ in enumerate(shards)]).contiguous()
    mine0 = shards[0]
    del shards
    nb = max(2, int(2 * 129e6 // (mine0.numel() * mine0.element_size())) + 2)
    steps = min(args.steps, 30)
    bufs = [mine0.clone() for _ in range(nb)]
    from vocabulary_lm_cross_gb300.ce import CEResult
    out = CEResult(loss=torch.empty(w.N, dtype=torch.float32, device=dev),
                   argmax=torch.empty(w.N, dtype=torch.int64, device=dev),
                   reduced=torch.empty(2, dtype=torch.float32, device=dev),
                   counts=torch.empty(4, dtype=torch.int64, device=dev))
    gathered = others.clone()
    ws = torch.empty(v_ws_bytes(w.N, V, mine0.dtype), dtype=torch.uint8, device=dev)

    def step(b):
        sh.shard_stats(b, lab, 0, V, softcap=w.softcap, out=gathered[0])
        sh.shard_fwd_bwd(b, lab, 0, V, gathered, label_smoothing=w.label_smoothing,
                         softcap=w.softcap, reduction=w.reduction, grad_scale=w.grad_scale,
                         out=out, workspace=ws)

    # the rank step is four short launches: replay it as a CUDA graph, one per
    # buffer of the ring, so that host-side launch overhead is not timed
    for i in range(args.warmup):
        step(bufs[i % nb])
    torch.cuda.synchronize()
    graphs = []
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for b in bufs:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=side):
                step(b)
            graphs.append(gr)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    for b in bufs:
        b.copy_(mine0)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    t0 = time.time()
    ms = 0.0
    done = 0
    while done < steps:
        k = min(nb, steps - done)  # each timed step on a pristine buffer
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(k):
            graphs[i].replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms += ev0.elapsed_time(ev1)
        done += k
        for b in bufs[:k]:
            b.copy_(mine0)
    t1 = time.time()
    ms /= steps
    ok = int(out.counts[3]) == 0
    bytes_step = 2 * w.N * vl * mine0.element_size()
    peak, peak_src = load_peaks()
    return {"workload": f"{w.name}, vocabulary shard 0 of {tp} ([{w.N}, {vl}])",
            "metric": "vocab-sharded CE rank step GB/s (shard read + gradient write)",
            "value": bytes_step / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "steps": steps, "bytes_per_step": bytes_step,
            "roofline": {"bound": "hbm", "achieved": bytes_step / (ms * 1e-3) / 1e9,
                         "peak": peak, "peak_source": f"{peak_src} (copy GB/s)", "unit": "GB/s",
                         "frac": bytes_step / (ms * 1e-3) / 1e9 / peak,
                         "measured_over": "the whole rank step (stats, count, gradient with the "
                                          "records' merge, finalize: 4 launches), replayed as "
                                          "a CUDA graph"},
            "gpu_launches": 4 * steps, "device_status_ok": ok,
            "clocks": sampler.summary(t0, t1),
            "l2": f"ring of {nb} shard copies ({nb * bytes_step / 2 / 1e6:.0f} MB > 2 x L2); the "
                  "gradient pass re-reads the shard from L2"}


def run_swiglu(args, dev, sampler, T=8192, ns=(32768, 4096)):
    """The fused gate-up SwiGLU at the Megatron training shape of its page
    (S = 2048 x B = 4 tokens, bf16): forward and out-of-place backward per
    ffn width n, against the HBM roofline (bytes = what must move: x in and
    y out for the forward; x and dy in, dx out for the backward)."""
    import torch

    from vocabulary_lm_cross_gb300.swiglu import swiglu_bwd, swiglu_fwd

    peak, peak_src = load_peaks()
    out = {}
    for n in ns:
        g = torch.Generator(device=dev)
        g.manual_seed(n)
        x = (torch.randn((T, 2 * n), generator=g, device=dev) * 2).to(torch.bfloat16)
        dy = torch.randn((T, n), generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty((T, n), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((T, 2 * n), dtype=torch.bfloat16, device=dev)
        flush = torch.empty(int(2 * 129e6) // 4, dtype=torch.float32, device=dev)
        res = {}
        for name, fn, nbytes in (("forward", lambda: swiglu_fwd(x, out=y), 3 * T * n * 2),
                                 ("backward", lambda: swiglu_bwd(x, dy, out=dx), 5 * T * n * 2)):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            times = []
            t0 = time.time()
            for _ in range(min(args.steps, 20)):
                flush.zero_()  # evict the previous step's lines from L2
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.fmean(times)
            res[name] = {"ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9,
                         "frac": nbytes / (ms * 1e-3) / 1e9 / peak, "bytes": nbytes,
                         "clocks": sampler.summary(t0, time.time())}
        out[f"T{T}_n{n}"] = res
        del x, dy, y, dx, flush
        torch.cuda.empty_cache()
    return {"metric": "fused gate-up SwiGLU GB/s (bf16, [tokens, 2n] layout)", "unit": "GB/s",
            "peak": peak, "peak_source": f"{peak_src} (copy GB/s)", "bound": "hbm",
            "l2": "a 258 MB buffer is written between timed launches (flushes L2)",
            "gpu_launches_per_step": 1, "results": out}


def flce_oracle_sample(w, budget_s=10.0):
    """Oracle throughput (TFLOP/s of 6 n v H) on a bounded sub-problem: the
    workload's recipe at n rows and v vocabulary rows, H unchanged."""
    import numpy as np
    from oracle import flce as of
    from vocabulary_lm_cross_gb300.workloads import bf16_bits, make_flce_inputs

    def one(n, v):
        ws = w.resized(N=n, V=v)
        h, W, lab = make_flce_inputs(ws, device="cpu")
        h64 = of.widen_bf16(bf16_bits(h))
        W64 = of.widen_bf16(bf16_bits(W))
        labh = lab.numpy().astype(np.int64)
        t0 = time.perf_counter()
        of.flce_fwd_bwd(h64, W64, labh, label_smoothing=w.label_smoothing, softcap=w.softcap,
                        reduction=w.reduction, grad_scale=w.grad_scale)
        dt = time.perf_counter() - t0
        return ws.algorithmic_flops / dt / 1e12, dt, ws

    n = min(w.N, 256)
    _, dt0, _ = one(n, 1024)
    v = int(min(w.V, 32768, max(1024, 1024 * budget_s / max(dt0, 1e-6))))
    tf, dt, ws = one(n, v)
    return {"value": tf, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"fp64 oracle (numpy BLAS on all host cores + the C CE oracle) on the "
                      f"workload's recipe at N={ws.N}, V={ws.V}, H={ws.H}: "
                      f"{ws.algorithmic_flops / 1e9:.1f} GFLOP (6NVH) in {dt:.2f} s"}


def run_flce(args, w, steps, dev, world, barrier, sampler):
    """Time flce_fwd_bwd on resident inputs; returns the measurements (rank-local)."""
    import torch

    import vocabulary_lm_cross_gb300 as v
    from vocabulary_lm_cross_gb300 import capi
    from vocabulary_lm_cross_gb300.workloads import make_flce_inputs

    rank = env_int("RANK", 0)
    lib = capi.lib()
    h, W, lab = make_flce_inputs(w.resized(seed=w.seed + 1000 * rank), device=dev)
    gw = torch.empty((w.V, w.H), dtype=torch.float32, device=dev)
    ws = torch.empty(v.flce.workspace_bytes(w.N, w.H, w.V), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    kw = dict(label_smoothing=w.label_smoothing, softcap=w.softcap, reduction=w.reduction,
              grad_scale=w.grad_scale, grad_weight=gw, workspace=ws)

    def step():
        return v.flce_fwd_bwd(h, W, lab, **kw)

    t_w0 = time.time()
    for _ in range(args.warmup):
        res = step()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        res = step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_w1 = time.time()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    ok_status = int(res.counts[3].item()) == 0

    # the tensor-core region of each call (statistics GEMM, row merge, every
    # chunk's three GEMMs), events recorded by the library on its stream
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        lib.vlmce_flce_profile_events(ctypes_handle(kb[i], stream), ctypes_handle(ke[i], stream))
        step()
    torch.cuda.synchronize()
    kern_ms = statistics.fmean(kb[i].elapsed_time(ke[i]) for i in range(steps))

    # end to end through the public API with host buffers: page-locked buffers
    # (allocated on the GPU's local CPUs); every step copies its inputs in and its results
    # (grad_hidden, grad_weight, loss, reduced) out.  Two sets of device
    # buffers let step i's results go out (on one copy stream) and step i+1's
    # inputs come in (on another) while a call computes, as a caller streaming
    # host-resident weights would run it.
    cpus0 = os.sched_getaffinity(0)
    bind_to_gpu_local_cpus(dev)
    try:
        h_host = h.cpu().pin_memory()
        W_host = W.cpu().pin_memory()
        lab_host = lab.cpu().pin_memory()
        gh_host = torch.empty((w.N, w.H), dtype=torch.bfloat16).pin_memory()
        gw_host = torch.empty((w.V, w.H), dtype=torch.float32).pin_memory()
        loss_host = torch.empty(w.N, dtype=torch.float32).pin_memory()
        red_host = torch.empty(2, dtype=torch.float32).pin_memory()
    finally:
        os.sched_setaffinity(0, cpus0)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    hb, Wb, lb = [h, torch.empty_like(h)], [W, torch.empty_like(W)], [lab, torch.empty_like(lab)]
    gwb = [gw, torch.empty_like(gw)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    keep = [None, None]

    def e2e_step(i):
        b = i & 1
        if i >= 2:  # set b's inputs were read by step i - 2
            s_in.wait_event(ev_comp[b])
        with torch.cuda.stream(s_in):
            hb[b].copy_(h_host, non_blocking=True)
            Wb[b].copy_(W_host, non_blocking=True)
            lb[b].copy_(lab_host, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:  # set b's results of step i - 2 are out
            stream.wait_event(ev_out[b])
        r = v.flce_fwd_bwd(hb[b], Wb[b], lb[b], **dict(kw, grad_weight=gwb[b]))
        ev_comp[b].record(stream)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            gh_host.copy_(r.grad_hidden, non_blocking=True)
            gw_host.copy_(gwb[b], non_blocking=True)
            loss_host.copy_(r.loss, non_blocking=True)
            red_host.copy_(r.reduced, non_blocking=True)
        ev_out[b].record(s_out)
        keep[b] = r  # the result tensors stay allocated until copied out

    e2e_step(0)
    torch.cuda.synchronize()
    e2e_steps = 6
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(ev_out[(e2e_steps - 1) & 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    h2d = (h_host.numel() + W_host.numel()) * 2 + lab_host.numel() * 8
    d2h = gh_host.numel() * 2 + gw_host.numel() * 4 + w.N * 4 + 8
    nchunks = (w.V + 8191) // 8192
    flops = w.algorithmic_flops
    # the dominant region is the whole call less the census, merge and
    # finalize kernels (about 50 us of ~30 ms): achieved is taken over the
    # whole call as timed above (a lower bound for the GEMM region), against
    # the burst bf16 peak; the tensor region's own event time (a separate
    # pass, perturbed by the events it records) is reported beside it
    peak, peak_src = load_tensor_peak(sustained=False)
    peak_s, _ = load_tensor_peak(sustained=True)
    achieved = flops / (ms / steps * 1e-3) / 1e12
    return {
        "ms": ms / steps, "value": world * flops * steps / (ms * 1e-3) / 1e12,
        "roofline": {"bound": "tensor", "kernel": "vlmce_gemm_kernel",
                     "achieved": achieved, "peak": peak, "peak_source": peak_src,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "frac_of_sustained": achieved / peak_s,
                     "measured_over": "the whole call (1 statistics GEMM, the row merge, "
                                      f"{nchunks + 1} grouped chunk GEMM launches, census and "
                                      "finalize), CUDA events around K calls",
                     "tensor_region_ms": kern_ms, "flops_per_launch": flops,
                     "executed_flops": 8 * w.N * w.V * w.H,
                     "executed_frac": 8 * w.N * w.V * w.H / (ms / steps * 1e-3) / 1e12 / peak,
                     "traffic": recorded_traffic("vlmce_gemm_kernel", w.name)},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": (4 + 3 * nchunks) * steps, "ok_status": ok_status,
        "clocks": sampler.summary(t_w0, t_w1),
        "config": {"workload": w.name, "N": w.N, "H": w.H, "V": w.V, "softcap": w.softcap,
                   "label_smoothing": w.label_smoothing, "reduction": w.reduction,
                   "grad_weight": "fp32, overwritten", "chunk": 8192,
                   "l2": "inputs larger than L2 (weight 2.69 GB streamed three times a step)"},
        "steps": steps,
    }


def run_flce_rows(w, dev, steps=5, warmup=2, chunks=(1024, 4096)):
    """The row-chunked schedule (flce_fwd_bwd_rows) on the same workload, timed
    beside the vocabulary-chunked one: per block of rows the fp32 logits are
    written once, so the executed tensor work is 6 N V H (no recompute)."""
    import torch

    import vocabulary_lm_cross_gb300 as v
    from vocabulary_lm_cross_gb300.workloads import make_flce_inputs

    h, W, lab = make_flce_inputs(w, device=dev)
    gw = torch.empty((w.V, w.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_src = load_tensor_peak(sustained=True)
    flops = w.algorithmic_flops
    out = {}
    for c in chunks:
        ws = torch.empty(v.flce.workspace_bytes(w.N, w.H, w.V, c), dtype=torch.uint8, device=dev)

        def step():
            return v.flce_fwd_bwd(h, W, lab, label_smoothing=w.label_smoothing, softcap=w.softcap,
                                  reduction=w.reduction, grad_scale=w.grad_scale, grad_weight=gw,
                                  workspace=ws, chunk_rows=c)

        for _ in range(warmup):
            res = step()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            res = step()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / steps
        tf = flops / (ms * 1e-3) / 1e12
        out[f"chunk_rows_{c}"] = {
            "ms": ms, "TFLOP/s": tf, "frac": tf / peak, "blocks": -(-w.N // c),
            "workspace_bytes": ws.numel(), "device_status_ok": int(res.counts[3].item()) == 0}
        del ws
        torch.cuda.empty_cache()
    return {"metric": "row-chunked FLCE (flce_fwd_bwd_rows) TFLOP/s of 6NVH, whole call",
            "peak": peak, "peak_source": peak_src, "executed_flops": 6 * w.N * w.V * w.H,
            "steps": steps, "results": out}


def run_ours_flce(args, w):
    """The fused linear cross-entropy as the line's headline (--workload flce-...)."""
    import torch
    import torch.distributed as dist

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local = env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            dist.barrier()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    f = run_flce(args, w, args.steps, dev, world, barrier, sampler)
    sampler.stop()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    cfg = dict(f["config"])
    cfg["parallelism"] = f"replicas x{world}"
    cfg["device_status_ok"] = f["ok_status"]
    line = {"metric": FLCE_METRIC, "value": f["value"], "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": f["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded normal hidden states and weight, uniform labels)",
            "config": cfg, "roofline": f["roofline"],
            "cpu_baseline": flce_oracle_sample(w) if world == 1 else None,
            "e2e": f["e2e"], "gpu_launches": f["gpu_launches"], "clocks": f["clocks"]}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_flce(args, w):
    """The FLCE oracle on the host cores: each step a bounded sub-problem."""
    import numpy as np
    from oracle import flce as of
    from vocabulary_lm_cross_gb300.workloads import bf16_bits, make_flce_inputs
    if env_int("RANK", 0) != 0:
        return
    ws = w.resized(N=min(w.N, 128), V=min(w.V, 2048))
    h, W, lab = make_flce_inputs(ws, device="cpu")
    h64 = of.widen_bf16(bf16_bits(h))
    W64 = of.widen_bf16(bf16_bits(W))
    labh = lab.numpy().astype(np.int64)

    def one():
        of.flce_fwd_bwd(h64, W64, labh, label_smoothing=w.label_smoothing, softcap=w.softcap,
                        reduction=w.reduction, grad_scale=w.grad_scale)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    value = ws.algorithmic_flops * args.steps / dt / 1e12
    sample = (f"fp64 FLCE oracle on the workload's recipe at N={ws.N}, V={ws.V}, H={ws.H} "
              "per step")
    line = {"impl": "reference", "metric": FLCE_METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "N": w.N, "H": w.H, "V": w.V,
                       "sample_N": ws.N, "sample_V": ws.V},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def ctypes_handle(ev, stream):
    """The cudaEvent_t behind a torch.cuda.Event (created lazily on first record)."""
    if ev.cuda_event == 0:
        ev.record(stream)
    return ev.cuda_event


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ce-bf16-2048x131072-ls0.1-argmax")
    ap.add_argument("--no-flce", action="store_true",
                    help="skip the fused linear cross-entropy and SwiGLU legs of a "
                         "cross-entropy run")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other cross-entropy configurations of a cross-entropy run")
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of untimed steps before the headline's timed steps (so the "
                         "clock samples describe a loaded GPU); 0 for profiling commands, whose "
                         "launch counts must not depend on time")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from vocabulary_lm_cross_gb300.workloads import CE_WORKLOADS, FLCE_WORKLOADS
    if args.workload in FLCE_WORKLOADS:
        w = FLCE_WORKLOADS[args.workload]
        (run_reference_flce if args.impl == "reference" else run_ours_flce)(args, w)
        return
    w = CE_WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
