"""Benchmark of the per-token normalization hot path on GB300.

One step = one pass of every hot-path kernel over the prefill workloads:
  * layerwise QK-RMSNorm of Q and of K, each [8192, 5120] bf16, 1% outlier
    channels, N = 4 cluster shards (13B-like prefill), both tensors in one
    launch;
  * RMSNorm + MXFP8 cast, MXNorm p = 1 and MXNorm p = 2 (+ MXFP8 cast) of
    X [65536, 4096] bf16, B = 32, E4M3 values + E8M0 scales.

value = algorithmic HBM bytes of the step / step time (GB/s, 1e9 B/s); the
per-kernel tokens/s, GB/s and roofline fractions ride along.  Inputs are
resident in HBM; the step's working set (2.8 GB) is far above the L2, so no
flush is needed between steps.  `e2e` runs the same step through the C ABI's
host-buffer entry points (pinned host memory, copies inside the timed
region).  `cpu_baseline` times the CPU oracle on a bounded row sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl nts|reference]

Under torchrun (N > 1) every rank runs the same step on its own GPU
(replicas: the path needs no exchange between GPUs); value sums the ranks'
bytes over the slowest rank's time.
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

METRIC = ("tokens/s and achieved HBM GB/s vs ~8 TB/s peak (QK-RMSNorm, MXNorm) on 1 GB300")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

QK_T, QK_H, QK_N = 8192, 5120, 4
MX_T, MX_D, MX_B = 65536, 4096, 32
EPS = 1e-6

KERNELS = ["qknorm_rms_qk[Q+K]", "rmsnorm_mxcast", "mxnorm_cast[p=1]", "mxnorm_cast[p=2]"]
KERNEL_SOURCES = {   # files whose content the committed ncu traffic figures belong to
    "qknorm_rms_qk[Q+K]": ["normalization_token_split_gb300/csrc/qk_kernel.cuh",
                           "normalization_token_split_gb300/csrc/qk_launch.cu",
                           "normalization_token_split_gb300/csrc/nts_device.cuh",
                           "normalization_token_split_gb300/csrc/nts_internal.h"],
    "rmsnorm_mxcast": ["normalization_token_split_gb300/csrc/mx_kernel.cuh",
                       "normalization_token_split_gb300/csrc/mx_launch.cu",
                       "normalization_token_split_gb300/csrc/nts_device.cuh"],
}
KERNEL_SOURCES["mxnorm_cast[p=1]"] = KERNEL_SOURCES["rmsnorm_mxcast"]
KERNEL_SOURCES["mxnorm_cast[p=2]"] = KERNEL_SOURCES["rmsnorm_mxcast"]


def qk_bytes(T, H):
    return 4 * T * H                       # bf16 in + bf16 out


def mx_bytes(T, D, B):
    return T * (2 * D + D + D // B)        # bf16 in + E4M3 codes + E8M0 scales


def step_bytes():
    per = {"qknorm_rms_qk[Q+K]": 2 * qk_bytes(QK_T, QK_H)}
    for k in KERNELS[1:]:
        per[k] = mx_bytes(MX_T, MX_D, MX_B)
    return per


def step_tokens():
    return {k: (QK_T if k.startswith("qk") else MX_T) for k in KERNELS}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def workload_config():
    return {
        "workload": ("prefill layer norms: QK-RMSNorm Q,K [8192,5120] N=4 (one launch) + "
                     "RMSNorm+MXFP8, MXNorm p=1, MXNorm p=2 of [65536,4096] B=32 E4M3"),
        "qk": {"T": QK_T, "H": QK_H, "N": QK_N, "tensors": ["Q", "K"], "eps": EPS,
               "x": "bf16 N(0,1), 1% of channels x20", "gamma": "fp32 N(1,0.1)"},
        "mx": {"T": MX_T, "D": MX_D, "B": MX_B, "fmt": "E4M3", "scales": "E8M0",
               "kinds": ["rmsnorm_mxcast", "mxnorm p=1", "mxnorm p=2"], "gamma": None,
               "x": "bf16 N(0,1)", "eps": EPS},
        "l2": "no flush: each step touches 2.78 GB, far above the 126 MB L2",
        "io_dtypes": "bf16 in; bf16 / E4M3+E8M0 out",
    }


# --------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [l for (t, l) in self.lines if t0 <= t <= t1 + 0.15] or [l for _, l in self.lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Max of a per-rank scalar across the process group (host aggregation)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def kernel_traffic():
    """dram read + write bytes per launch from the committed ncu summaries
    (profiles/*.md lines "traffic_per_launch NAME BYTES source_sha256 H"),
    kept only where H matches the kernel's current source files."""
    prof = os.path.join(ROOT, "profiles")
    found = {}
    if os.path.isdir(prof):
        for fn in sorted(os.listdir(prof)):
            if fn.endswith(".md"):
                text = open(os.path.join(prof, fn)).read()
                for m in re.finditer(r"traffic_per_launch\s+(\S+)\s+(\d+)\s+source_sha256\s+(\w+)",
                                     text):
                    found[m.group(1)] = (int(m.group(2)), m.group(3))
    out = {}
    for name, files in KERNEL_SOURCES.items():
        try:
            digest = source_digest(files)
        except OSError:
            continue
        if name in found and found[name][1] == digest:
            out[name] = found[name][0]
    return out


def source_digest(files):
    """sha256 (16 hex digits) of the files' code with comments and blank
    lines removed, so that an edit of comments alone keeps the digest."""
    h = hashlib.sha256()
    for f in files:
        text = open(os.path.join(ROOT, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


# ------------------------------------------------------------ GPU arm

def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"

    import workloads
    import normalization_token_split_gb300 as nts

    per_bytes = step_bytes()
    tokens = step_tokens()
    total_bytes = sum(per_bytes.values())

    Q, gq = workloads.qk_inputs(QK_T, QK_H, seed=3000, outlier_frac=0.01, device=dev)
    K, gk = workloads.qk_inputs(QK_T, QK_H, seed=3001, outlier_frac=0.01, device=dev)
    X, _ = workloads.mx_inputs(MX_T, MX_D, seed=4000 + MX_T, device=dev)
    Yq, Yk = torch.empty_like(Q), torch.empty_like(K)
    outs = {}
    for name in KERNELS[1:]:
        outs[name] = (torch.empty(MX_T, MX_D, dtype=torch.uint8, device=dev),
                      torch.empty(MX_T, MX_D // MX_B, dtype=torch.uint8, device=dev))
    stream = torch.cuda.current_stream()

    launches = [
        ("qknorm_rms_qk[Q+K]", lambda: nts.qknorm_rms_qk(Q, gq, K, gk, eps=EPS, N=QK_N,
                                                         out_q=Yq, out_k=Yk)),
        ("rmsnorm_mxcast", lambda: nts.rmsnorm_mxcast(
            X, None, eps=EPS, B=MX_B, fmt="e4m3", codes=outs["rmsnorm_mxcast"][0],
            scales=outs["rmsnorm_mxcast"][1])),
        ("mxnorm_cast[p=1]", lambda: nts.mxnorm_cast(
            X, None, eps=EPS, B=MX_B, fmt="e4m3", p=1, codes=outs["mxnorm_cast[p=1]"][0],
            scales=outs["mxnorm_cast[p=1]"][1])),
        ("mxnorm_cast[p=2]", lambda: nts.mxnorm_cast(
            X, None, eps=EPS, B=MX_B, fmt="e4m3", p=2, codes=outs["mxnorm_cast[p=2]"][0],
            scales=outs["mxnorm_cast[p=2]"][1])),
    ]

    def step(events=None):
        # one event before each launch: launch i of step k runs between
        # marks[k*n + i] and marks[k*n + i + 1] (the next launch's mark, or
        # the closing mark), so no two event records sit between launches
        for i, (name, fn) in enumerate(launches):
            if events is not None:
                events[i].record(stream)
            fn()

    for _ in range(args.warmup):
        step()
    nts.check_status()

    # ---- timed region: K steps between two events on the launching stream.
    # Then K more steps with an event before every launch, for the per-kernel
    # durations: an event record between two launches costs ~2 us, so these
    # marks stay out of the region that gives the step time.
    n = len(launches)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps * n + 1)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    t_start.record(stream)
    for k in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    w1 = time.time()
    for k in range(args.steps):
        step(marks[k * n:(k + 1) * n])
    marks[-1].record(stream)
    torch.cuda.synchronize()
    w2 = time.time()
    time.sleep(0.25)
    clocks.stop()
    nts.check_status()

    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    marked_ms = marks[0].elapsed_time(marks[-1]) / args.steps
    per_kernel_ms = {name: statistics.mean(marks[k * n + i].elapsed_time(marks[k * n + i + 1])
                                           for k in range(args.steps))
                     for i, (name, _) in enumerate(launches)}
    ms_per_step = elapsed_ms / args.steps
    value = world * total_bytes * args.steps / (elapsed_ms * 1e-3) / 1e9

    peak, peak_kind = measured_peaks()
    kernels = {}   # rates between the marks of the second pass (each launch inside the step)
    for name in KERNELS:
        gbs = per_bytes[name] / (per_kernel_ms[name] * 1e-3) / 1e9
        kernels[name] = {"ms": round(per_kernel_ms[name], 5), "bytes": per_bytes[name],
                         "gbs": round(gbs, 1), "tokens_per_s": round(tokens[name] / (per_kernel_ms[name] * 1e-3)),
                         "frac_of_measured": round(gbs / peak, 4),
                         "frac_of_8TBs": round(gbs / NOMINAL_HBM_GBS, 4)}
    # each launch's marginal cost inside the step, with no marks: the time of
    # the unmarked step minus that of the step without it (the same
    # programmatic dependent launches between the others)
    for i, (name, _) in enumerate(launches):
        rest = [fn for j, (_, fn) in enumerate(launches) if j != i]
        ms_rest = time_launches(torch, rest, args.steps * len(rest), warmup=3)
        marginal = ms_per_step - ms_rest * len(rest)
        gbs = per_bytes[name] / (marginal * 1e-3) / 1e9
        kernels[name]["marginal_in_step"] = {"ms": round(marginal, 5), "gbs": round(gbs, 1),
                                             "frac_of_measured": round(gbs / peak, 4)}
    # each launch of the step alone, back to back (so every launch follows
    # one of its own kind): the kernel's steady-state rate, without the
    # write-back of the previous kernel's dirty L2 lines or the marks' gaps
    for name, fn in launches:
        ms = time_launches(torch, [fn], 20)
        gbs = per_bytes[name] / (ms * 1e-3) / 1e9
        kernels[name]["alone"] = {"ms": round(ms, 5), "gbs": round(gbs, 1),
                                  "frac_of_measured": round(gbs / peak, 4)}
    dominant = max(KERNELS, key=lambda n: per_kernel_ms[n])
    traffic = kernel_traffic()
    roofline = {"bound": "hbm", "kernel": dominant,
                "achieved": kernels[dominant]["gbs"], "peak": peak, "unit": "GB/s",
                "frac": round(kernels[dominant]["gbs"] / peak, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "traffic": traffic.get(dominant),
                "traffic_note": "ncu dram read+write bytes of one launch (profiles/); writes still "
                                "dirty in L2 at kernel end are not counted"}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(),
        "tokens_per_s": {n: kernels[n]["tokens_per_s"] for n in KERNELS},
        "frac_of_8TBs": round(value / world / NOMINAL_HBM_GBS, 4),
        "gpu_launches": len(launches) * args.steps,
        "clocks": clocks.summary(w0, w2),
        "wall_s_timed": round(w1 - w0, 4),
        "ms_per_step_with_kernel_marks": round(marked_ms, 5),
    }

    # the long tables first, the per-kernel figures and the roofline last
    # (a reader of the line's tail sees those)
    if not args.no_sweep:
        result["mxnorm_sweep_gbs"] = mxnorm_sweep(nts, torch, dev, peak)
        result["mx_vs_rms_by_block"] = mx_vs_rms_by_block(nts, torch, dev, peak)
        result["mx_config_by_T"] = mx_config_by_T(nts, torch, dev, peak)
    if not args.no_decode:
        result["decode_qk"] = decode_latency(nts, torch, dev)
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, nts, torch, dev, Q, K, X, gq, gk, world)
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if not args.no_variants:
        result["variants"] = variant_rates(nts, torch, dev, Q, gq, X, peak, K, gk)
        # the split-H paths again at T = 32768 rows (inputs and outputs of
        # every launch well above L2; launch ramp and tail a smaller share)
        Q4, gq4 = workloads.qk_inputs(4 * QK_T, QK_H, seed=3002, outlier_frac=0.01, device=dev)
        K4, gk4 = workloads.qk_inputs(4 * QK_T, QK_H, seed=3003, outlier_frac=0.01, device=dev)
        result["variants_T32768"] = variant_rates(nts, torch, dev, Q4, gq4, X, peak, K4, gk4,
                                                  with_mx=False)
        del Q4, K4
    result["kernels"] = kernels
    result["roofline"] = roofline
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, nts, torch, dev, Q, K, X, gq, gk, world):
    """Same step through the host-buffer C ABI forms, copies timed."""
    pin = lambda t: t.cpu().pin_memory()
    Qh, Kh, Xh = pin(Q), pin(K), pin(X)
    Yqh = torch.empty_like(Qh).pin_memory()
    Ykh = torch.empty_like(Kh).pin_memory()
    Xd = torch.empty_like(X)
    Qd, Kd = torch.empty_like(Q), torch.empty_like(K)
    Yqd, Ykd = torch.empty_like(Q), torch.empty_like(K)
    codes_h = {n: torch.empty(MX_T, MX_D, dtype=torch.uint8).pin_memory() for n in KERNELS[1:]}
    scales_h = {n: torch.empty(MX_T, MX_D // MX_B, dtype=torch.uint8).pin_memory()
                for n in KERNELS[1:]}
    codes_d = torch.empty(MX_T, MX_D, dtype=torch.uint8, device=dev)
    scales_d = torch.empty(MX_T, MX_D // MX_B, dtype=torch.uint8, device=dev)

    def step():
        nts.qknorm_rms_qk_host(Qh, gq, Yqh, Kh, gk, Ykh, Qd, Yqd, Kd, Ykd, eps=EPS, N=QK_N)
        nts.rmsnorm_mxcast_host(Xh, None, codes_h["rmsnorm_mxcast"], scales_h["rmsnorm_mxcast"],
                                Xd, codes_d, scales_d, eps=EPS, B=MX_B, fmt="e4m3")
        for p in (1, 2):
            n = f"mxnorm_cast[p={p}]"
            nts.mxnorm_cast_host(Xh, None, codes_h[n], scales_h[n], Xd, codes_d, scales_d,
                                 eps=EPS, B=MX_B, fmt="e4m3", p=p)

    steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(2):
        step()
    nts.check_status()
    # three timed runs of `steps` steps; the median one is reported (a host
    # copy over C2C now and then runs at a fraction of its rate for a while)
    runs = []
    for _ in range(3):
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            step()
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        barrier(world)
        runs.append(t1 - t0)
    nts.check_status()
    elapsed = max_over_ranks(statistics.median(runs), world)
    total = sum(step_bytes().values())
    h2d = 2 * QK_T * QK_H * 2 + 3 * MX_T * MX_D * 2
    d2h = 2 * QK_T * QK_H * 2 + 3 * (MX_T * MX_D + MX_T * (MX_D // MX_B))
    return {"value": round(world * total * steps / elapsed / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "runs_ms_per_step": [round(r / steps * 1e3, 3) for r in runs], "reported": "median run",
            "ms_per_step": round(elapsed / steps * 1e3, 4),
            "path": "nts_*_host C ABI entry points (Q and K in one nts_qknorm_rms_qk_host "
                    "call, as the device step launches them), pinned host buffers",
            "copy_only_gbs": copy_ceiling(
                torch,
                [(Qd, Qh), (Kd, Kh)] + [(Xd, Xh)] * 3,
                [(Yqh, Yqd), (Ykh, Ykd)] + [(codes_h[n], codes_d) for n in KERNELS[1:]]
                + [(scales_h[n], scales_d) for n in KERNELS[1:]], total)}


def copy_ceiling(torch, ins, outs, total, reps=5):
    """The step's bytes moved by plain copies alone, between the very host
    and device buffers the e2e step uses (so the same pinned pages): every
    (device, host) pair of `ins` host->device on one stream, every (host,
    device) pair of `outs` device->host on another, in 32 MiB pieces.  The
    ceiling for e2e on this link, in the step's GB/s."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    piece = 32 << 20

    def flat(t):
        return t.view(-1).view(torch.uint8)

    def copies():
        with torch.cuda.stream(s_in):
            for d, h in ins:
                d, h = flat(d), flat(h)
                for o in range(0, h.numel(), piece):
                    d[o:o + piece].copy_(h[o:o + piece], non_blocking=True)
        with torch.cuda.stream(s_out):
            for h, d in outs:
                h, d = flat(h), flat(d)
                for o in range(0, d.numel(), piece):
                    h[o:o + piece].copy_(d[o:o + piece], non_blocking=True)

    copies()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        copies()
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
    return round(total / statistics.median(times) / 1e9, 1)


def mxnorm_sweep(nts, torch, dev, peak, reps=20):
    """MXNorm p=2 over the sweep grid: T = 65536, D in {1024, 3072, 5120,
    7168, 16384}, B in {16, 32, 64}, E4M3 and E2M1, rows N(0,1) with 5 %
    Student-t(3).  Device time per launch over `reps` back-to-back launches
    (3 warm-up), algorithmic GB/s; plus the fraction of measured and of
    8 TB/s for each."""
    import workloads
    T = 65536
    out = {}
    for D in (1024, 3072, 5120, 7168, 16384):
        X, _ = workloads.mx_inputs(T, D, seed=5000 + D, t_frac=0.05, device=dev)
        codes = torch.empty(T * D, dtype=torch.uint8, device=dev)
        scales = torch.empty(T * D // 16, dtype=torch.uint8, device=dev)
        for fmt in ("e4m3", "e2m1"):
            for B in (16, 32, 64):
                cb = D if fmt == "e4m3" else D // 2
                c = codes[:T * cb].view(T, cb)
                sc = scales[:T * D // B].view(T, D // B)
                fn = lambda: nts.mxnorm_cast(X, None, eps=EPS, B=B, fmt=fmt, p=2, codes=c, scales=sc)
                for _ in range(3):
                    fn()
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record()
                for _ in range(reps):
                    fn()
                s1.record()
                torch.cuda.synchronize()
                ms = s0.elapsed_time(s1) / reps
                gbs = T * (2 * D + cb + D // B) / (ms * 1e-3) / 1e9
                out[f"D={D},B={B},{fmt}"] = {"us": round(ms * 1e3, 1), "gbs": round(gbs, 1),
                                             "frac_of_measured": round(gbs / peak, 4),
                                             "frac_of_8TBs": round(gbs / NOMINAL_HBM_GBS, 4)}
        del X, codes, scales
    nts.check_status()
    return out


def mx_vs_rms_by_block(nts, torch, dev, peak, reps=20):
    """The isolated-kernel comparison of the MXNorm card's Fig. 8 on this
    GPU: RMSNorm + MX cast against MXNorm (p = 1 and 2) + the same cast at
    [65536, 4096], for B in {16, 32, 64} and E4M3 / E2M1 elements (rows
    N(0,1)).  Device time per launch; speedup = RMSNorm time / MXNorm time."""
    out = {}
    for fmt in ("e4m3", "e2m1"):
        for B in (16, 32, 64):
            t = {}
            for name, spec in (("rmsnorm_mxcast", f"rmsnorm_mxcast:T=65536,D=4096,B={B},fmt={fmt}"),
                               ("mxnorm_p1", f"mxnorm_cast:T=65536,D=4096,B={B},fmt={fmt},p=1"),
                               ("mxnorm_p2", f"mxnorm_cast:T=65536,D=4096,B={B},fmt={fmt},p=2")):
                cname, q = parse_case(spec)
                fns = make_case(nts, torch, dev, cname, q, 1)
                ms = time_launches(torch, fns, reps)
                gbs = case_bytes(cname, q) / (ms * 1e-3) / 1e9
                t[name] = {"us": round(ms * 1e3, 1), "gbs": round(gbs, 1),
                           "frac_of_measured": round(gbs / peak, 4)}
                del fns
            for p in ("p1", "p2"):
                t[f"speedup_mxnorm_{p}"] = round(t["rmsnorm_mxcast"]["us"] / t[f"mxnorm_{p}"]["us"], 3)
            out[f"B={B},{fmt}"] = t
    nts.check_status()
    return out


def mx_config_by_T(nts, torch, dev, peak, reps=30):
    """RMSNorm + MXFP8 and MXNorm p = 1, 2 of X [T, 4096] (B = 32, E4M3) at
    T in {4096, 16384, 65536}.  Launches rotate through enough independent
    input/output sets that the data touched between two uses of a set is at
    least twice the L2 (and at least 3 sets below that size); configurations
    whose one-launch working set fits in L2 are flagged."""
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    out = {}
    for T in (4096, 16384, 65536):
        nbytes = mx_bytes(T, MX_D, MX_B)
        sets = 1 if nbytes > 2 * l2 else max(3, -(-2 * l2 // nbytes) + 1)
        row = {"bytes": nbytes, "input_sets": sets, "l2_resident": nbytes <= l2}
        for name, spec in (("rmsnorm_mxcast", f"rmsnorm_mxcast:T={T},D={MX_D},B={MX_B}"),
                           ("mxnorm_p1", f"mxnorm_cast:T={T},D={MX_D},B={MX_B},p=1"),
                           ("mxnorm_p2", f"mxnorm_cast:T={T},D={MX_D},B={MX_B},p=2")):
            cname, q = parse_case(spec)
            fns = make_case(nts, torch, dev, cname, q, sets)
            ms = time_launches(torch, fns, reps)
            gbs = nbytes / (ms * 1e-3) / 1e9
            row[name] = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                         "tokens_per_s": round(T / (ms * 1e-3)),
                         "frac_of_measured": round(gbs / peak, 4)}
            del fns
        out[f"T={T}"] = row
        torch.cuda.empty_cache()
    nts.check_status()
    return {"by_T": out, "l2_bytes": l2}


def variant_rates(nts, torch, dev, Q, gq, X, peak, K, gk, reps=20, with_mx=True):
    """The widened paths outside the step, each at the step's sizes: device
    time per launch (CUDA events around `reps` back-to-back launches on the
    launching stream, after 3 warm-up launches) and algorithmic GB/s.
    with_mx=False: only the split-H (QK) paths, at the size of Q."""
    import workloads
    T, H = Q.shape
    Tm, D = X.shape
    codes8, scale8, g8 = workloads.qk_inputs_fp8(T, H, seed=3000, outlier_frac=0.01, device=dev)
    beta = workloads.beta_vector(H, seed=3000, device=dev)
    ghd = workloads.gamma_vector(128, seed=128, device=dev)
    Y = torch.empty_like(Q)
    codes = torch.empty(Tm, D, dtype=torch.uint8, device=dev)
    codes4 = torch.empty(Tm, D // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(Tm, D // MX_B, dtype=torch.uint8, device=dev)
    scales16 = torch.empty(Tm, D // 16, dtype=torch.uint8, device=dev)
    qcodes = torch.empty(T, H, dtype=torch.uint8, device=dev)
    qcodes4 = torch.empty(T, H // 2, dtype=torch.uint8, device=dev)
    qscales = torch.empty(T, H // 32, dtype=torch.uint8, device=dev)
    qscales16 = torch.empty(T, H // 16, dtype=torch.uint8, device=dev)
    outq = nts.MxOut(qcodes, qscales, None, None)
    outk = nts.MxOut(torch.empty_like(qcodes), torch.empty_like(qscales), None, None)
    cases = {
        f"qknorm_rms_heads[{T}x{H},head_dim=128,N=1]": (
            4 * T * H, lambda: nts.qknorm_rms_heads(Q, ghd, 128, eps=EPS, N=1, out=Y)),
        f"qknorm_rms_fp8[{T}x{H},N={QK_N}]": (
            3 * T * H, lambda: nts.qknorm_rms_fp8(codes8, scale8, g8, eps=EPS, N=QK_N, out=Y)),
        f"qknorm_rms[{T}x{H},N={QK_N}]": (
            4 * T * H, lambda: nts.qknorm_rms(Q, gq, eps=EPS, N=QK_N, out=Y)),
        f"qknorm_rms_mxcast[{T}x{H},N={QK_N},B=32,e4m3]": (
            T * H * 3 + T * (H // 32), lambda: nts.qknorm_rms_mxcast(
                Q, gq, eps=EPS, N=QK_N, B=32, fmt="e4m3", codes=qcodes, scales=qscales)),
        f"qknorm_rms_mxcast[{T}x{H},N={QK_N},B=16,nvfp4]": (
            T * H * 2 + T * H // 2 + T * (H // 16), lambda: nts.qknorm_rms_mxcast(
                Q, gq, eps=EPS, N=QK_N, B=16, fmt="nvfp4", codes=qcodes4, scales=qscales16)),
        f"qknorm_rms_qk_mxcast[Q+K {T}x{H},N={QK_N},B=32,e4m3]": (
            2 * (T * H * 3 + T * (H // 32)), lambda: nts.qknorm_rms_qk_mxcast(
                Q, gq, K, gk, eps=EPS, N=QK_N, B=32, fmt="e4m3", out_q=outq, out_k=outk)),
        f"layernorm_split[{T}x{H},N={QK_N},beta]": (
            4 * T * H, lambda: nts.layernorm_split(Q, gq, beta, eps=1e-5, N=QK_N, out=Y)),
        f"mxnorm_postround_cast[{Tm}x{D},B={MX_B},p=2,e4m3]": (
            mx_bytes(Tm, D, MX_B), lambda: nts.mxnorm_postround_cast(
                X, None, eps=EPS, B=MX_B, fmt="e4m3", p=2, codes=codes, scales=scales)),
        f"mxnorm_cast[{Tm}x{D},B=16,p=2,nvfp4]": (
            Tm * (2 * D + D // 2 + D // 16), lambda: nts.mxnorm_cast(
                X, None, eps=EPS, B=16, fmt="nvfp4", p=2, codes=codes4, scales=scales16)),
        f"rmsnorm_mxcast[{Tm}x{D},B=16,nvfp4]": (
            Tm * (2 * D + D // 2 + D // 16), lambda: nts.rmsnorm_mxcast(
                X, None, eps=EPS, B=16, fmt="nvfp4", codes=codes4, scales=scales16)),
        f"rmsnorm_mxcast[{Tm}x{D},B={MX_B},e2m1]": (
            Tm * (2 * D + D // 2 + D // MX_B), lambda: nts.rmsnorm_mxcast(
                X, None, eps=EPS, B=MX_B, fmt="e2m1", codes=codes4, scales=scales)),
    }
    if not with_mx:
        cases = {k: v for k, v in cases.items() if not k.startswith(("mxnorm", "rmsnorm"))}
    stream = torch.cuda.current_stream()
    out = {}
    for name, (nbytes, fn) in cases.items():
        for _ in range(3):
            fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s.record(stream)
        for _ in range(reps):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        ms = s.elapsed_time(e) / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 5), "bytes": nbytes, "gbs": round(gbs, 1),
                     "frac_of_measured": round(gbs / peak, 4)}
    nts.check_status()
    return out


def decode_latency(nts, torch, dev):
    """Decode-shaped QK-Norm (Q and K each [T, 4096], 7B-like): GPU time per
    fused Q+K call, from CUDA-graph replays of 20 back-to-back calls (the
    host's launch cost is outside the graph)."""
    import workloads
    out = {}
    for N in (1, 2, 4, 8):
        for T in (1, 8, 64, 256):
            Q, gq = workloads.qk_inputs(T, 4096, seed=T, device=dev)
            K, gk = workloads.qk_inputs(T, 4096, seed=T + 1, device=dev)
            Yq, Yk = torch.empty_like(Q), torch.empty_like(K)
            call = lambda: nts.qknorm_rms_qk(Q, gq, K, gk, eps=EPS, N=N, out_q=Yq, out_k=Yk)
            call()                                  # fills the launch-shape caches
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(20):
                    call()
            graph.replay()
            torch.cuda.synchronize()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(10):
                graph.replay()
            e.record()
            torch.cuda.synchronize()
            us = s.elapsed_time(e) * 1e3 / 200
            gbs = 2 * qk_bytes(T, 4096) / (us * 1e-6) / 1e9
            out[f"N={N},T={T}"] = {"us_per_call": round(us, 2), "gbs": round(gbs, 1)}
    nts.check_status()
    return {"per_call": out, "note": "Q and K [T, 4096] each, one fused launch per call; "
            "CUDA-graph replays of 20 calls (host launch cost excluded); working set in L2 "
            "(latency-bound sizes: GB/s for information)"}


# ------------------------------------------------------- single cases

CASE_DEFAULTS = {
    "qknorm_rms": dict(T=8192, H=5120, N=4),
    "qknorm_rms_qk": dict(T=8192, H=5120, N=4),
    "qknorm_rms_fp8": dict(T=8192, H=5120, N=4),
    "qknorm_rms_heads": dict(T=8192, H=5120, N=1, hd=128),
    "layernorm_split": dict(T=8192, H=5120, N=4, beta=1),
    "qknorm_rms_mxcast": dict(T=8192, H=5120, N=4, B=32, fmt="e4m3"),
    "qknorm_rms_qk_mxcast": dict(T=8192, H=5120, N=4, B=32, fmt="e4m3"),
    "rmsnorm_mxcast": dict(T=65536, D=4096, B=32, fmt="e4m3", gamma=0),
    "mxnorm_cast": dict(T=65536, D=4096, B=32, fmt="e4m3", p=2, gamma=0),
    "mxnorm_postround_cast": dict(T=65536, D=4096, B=32, fmt="e4m3", p=2, gamma=0),
}


def parse_case(spec: str):
    """"name" or "name:key=value,key=value" -> (name, parameters)."""
    name, _, rest = spec.partition(":")
    if name not in CASE_DEFAULTS:
        raise SystemExit(f"unknown case {name!r}; known: {', '.join(CASE_DEFAULTS)}")
    params = dict(CASE_DEFAULTS[name])
    for item in filter(None, rest.split(",")):
        k, _, v = item.partition("=")
        if k not in params:
            raise SystemExit(f"case {name} has no parameter {k!r}")
        params[k] = type(params[k])(v)
    return name, params


TUNE_KEYS = ("vpt", "rows", "stages", "grid", "smem_budget")


def parse_tune(spec):
    """"key=value,..." over TUNE_KEYS (launch-shape overrides, 0 = automatic)
    -> keyword arguments of nts.set_tuning."""
    out = {}
    for item in filter(None, (spec or "").split(",")):
        k, _, v = item.partition("=")
        if k not in TUNE_KEYS:
            raise SystemExit(f"unknown tuning key {k!r}; known: {', '.join(TUNE_KEYS)}")
        out[k] = int(v)
    return out


def case_bytes(name, q):
    """Algorithmic HBM bytes of one launch (gamma and beta excluded)."""
    if name in ("rmsnorm_mxcast", "mxnorm_cast", "mxnorm_postround_cast"):
        cb = q["D"] if q["fmt"] == "e4m3" else q["D"] // 2
        return q["T"] * (2 * q["D"] + cb + q["D"] // q["B"])
    T, H = q["T"], q["H"]
    if name in ("qknorm_rms_mxcast", "qknorm_rms_qk_mxcast"):
        cb = H if q["fmt"] == "e4m3" else H // 2
        n = 2 if name == "qknorm_rms_qk_mxcast" else 1
        return n * T * (2 * H + cb + H // q["B"])
    if name == "qknorm_rms_fp8":
        return 3 * T * H
    return (2 if name == "qknorm_rms_qk" else 1) * 4 * T * H


def make_case(nts, torch, dev, name, q, sets):
    """`sets` independent input/output sets of the case (rotated between
    launches, so that small working sets do not stay in L2) and one launch
    function per set."""
    import workloads
    fns = []
    for k in range(sets):
        seed = 7000 + 13 * k
        if name in ("rmsnorm_mxcast", "mxnorm_cast", "mxnorm_postround_cast"):
            T, D, B, fmt = q["T"], q["D"], q["B"], q["fmt"]
            X, gam = workloads.mx_inputs(T, D, seed=seed, t_frac=0.05, with_gamma=bool(q["gamma"]),
                                         device=dev)
            codes = torch.empty(T, D if fmt == "e4m3" else D // 2, dtype=torch.uint8, device=dev)
            scales = torch.empty(T, D // B, dtype=torch.uint8, device=dev)
            kw = dict(eps=EPS, B=B, fmt=fmt, codes=codes, scales=scales)
            if name != "rmsnorm_mxcast":
                kw["p"] = q["p"]
            f = getattr(nts, name)
            fns.append(lambda X=X, gam=gam, f=f, kw=kw: f(X, gam, **kw))
            continue
        T, H, N = q["T"], q["H"], q["N"]
        X, g = workloads.qk_inputs(T, H, seed=seed, outlier_frac=0.01, device=dev)
        Y = torch.empty_like(X)
        if name == "qknorm_rms":
            fns.append(lambda X=X, g=g, Y=Y: nts.qknorm_rms(X, g, eps=EPS, N=N, out=Y))
        elif name == "qknorm_rms_qk":
            K, gk = workloads.qk_inputs(T, H, seed=seed + 1, outlier_frac=0.01, device=dev)
            Yk = torch.empty_like(K)
            fns.append(lambda X=X, g=g, Y=Y, K=K, gk=gk, Yk=Yk: nts.qknorm_rms_qk(
                X, g, K, gk, eps=EPS, N=N, out_q=Y, out_k=Yk))
        elif name == "qknorm_rms_fp8":
            c8, s8, g8 = workloads.qk_inputs_fp8(T, H, seed=seed, outlier_frac=0.01, device=dev)
            fns.append(lambda c8=c8, s8=s8, g8=g8, Y=Y: nts.qknorm_rms_fp8(
                c8, s8, g8, eps=EPS, N=N, out=Y))
        elif name == "qknorm_rms_heads":
            gh = workloads.gamma_vector(q["hd"], seed=seed, device=dev)
            fns.append(lambda X=X, gh=gh, Y=Y: nts.qknorm_rms_heads(
                X, gh, q["hd"], eps=EPS, N=N, out=Y))
        elif name == "layernorm_split":
            beta = workloads.beta_vector(H, seed=seed, device=dev) if q["beta"] else None
            fns.append(lambda X=X, g=g, Y=Y, beta=beta: nts.layernorm_split(
                X, g, beta, eps=1e-5, N=N, out=Y))
        else:
            B, fmt = q["B"], q["fmt"]
            cb = H if fmt == "e4m3" else H // 2
            mk = lambda: nts.MxOut(torch.empty(T, cb, dtype=torch.uint8, device=dev),
                                   torch.empty(T, H // B, dtype=torch.uint8, device=dev),
                                   None, None)
            oq = mk()
            if name == "qknorm_rms_mxcast":
                fns.append(lambda X=X, g=g, oq=oq: nts.qknorm_rms_mxcast(
                    X, g, eps=EPS, N=N, B=B, fmt=fmt, codes=oq.codes, scales=oq.scales))
            else:
                K, gk = workloads.qk_inputs(T, H, seed=seed + 1, outlier_frac=0.01, device=dev)
                ok = mk()
                fns.append(lambda X=X, g=g, oq=oq, K=K, gk=gk, ok=ok: nts.qknorm_rms_qk_mxcast(
                    X, g, K, gk, eps=EPS, N=N, B=B, fmt=fmt, out_q=oq, out_k=ok))
    return fns


def time_launches(torch, fns, reps, warmup=3):
    """Mean device time of one launch (ms): `reps` back-to-back launches
    cycling through `fns`, between two CUDA events on the launching stream,
    after `warmup` rounds."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for f in fns:
            f()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record(stream)
    for i in range(reps):
        fns[i % len(fns)]()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


def run_case(args):
    """--case: one kernel alone, for profiling and per-kernel figures."""
    import torch
    import normalization_token_split_gb300 as nts
    dev = "cuda:0"
    torch.cuda.set_device(0)
    name, q = parse_case(args.case)
    tune = parse_tune(args.tune)
    fns = make_case(nts, torch, dev, name, q, args.sets)
    if tune:
        nts.set_tuning(**tune)
    try:
        ms = time_launches(torch, fns, args.steps, warmup=args.warmup)
        nts.check_status()
    finally:
        nts.set_tuning()
    peak, peak_kind = measured_peaks()
    nbytes = case_bytes(name, q)
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"case": name, "params": q, "tune": tune, "input_sets": args.sets,
                      "launches": args.steps,
                      "us_per_launch": round(ms * 1e3, 2), "bytes": nbytes, "gbs": round(gbs, 1),
                      "frac_of_measured": round(gbs / peak, 4), "peak_source": peak_kind}),
          flush=True)


# ------------------------------------------------------------ CPU oracle

def oracle_sample_step(rows_qk: int, rows_mx: int, state, pool=None, nthreads: int = 1):
    """One bounded sample of the step through the CPU oracle; returns the
    algorithmic bytes it covered.  With a thread pool, the rows of every
    call are split into `nthreads` contiguous chunks that run at once (the
    oracle's C entry points release the GIL, and rows are independent)."""
    import oracle
    Qb, gq, Kb, gk, Xb = state
    calls = [(lambda a, b: oracle.qknorm_rms(Qb[a:b], gq, EPS, QK_N), rows_qk),
             (lambda a, b: oracle.qknorm_rms(Kb[a:b], gk, EPS, QK_N), rows_qk),
             (lambda a, b: oracle.rmsnorm_mxcast(Xb[a:b], None, EPS, MX_B, 0), rows_mx),
             (lambda a, b: oracle.mxnorm_cast(Xb[a:b], None, EPS, MX_B, 0, 1), rows_mx),
             (lambda a, b: oracle.mxnorm_cast(Xb[a:b], None, EPS, MX_B, 0, 2), rows_mx)]
    for fn, rows in calls:
        if pool is None:
            fn(0, rows)
        else:
            cuts = [rows * k // nthreads for k in range(nthreads + 1)]
            list(pool.map(lambda k: fn(cuts[k], cuts[k + 1]), range(nthreads)))
    return 2 * qk_bytes(rows_qk, QK_H) + 3 * mx_bytes(rows_mx, MX_D, MX_B)


def oracle_inputs(rows_qk, rows_mx):
    import workloads
    Q, gq = workloads.qk_inputs(rows_qk, QK_H, seed=3000, outlier_frac=0.01)
    K, gk = workloads.qk_inputs(rows_qk, QK_H, seed=3001, outlier_frac=0.01)
    X, _ = workloads.mx_inputs(rows_mx, MX_D, seed=4000 + MX_T)
    return (workloads.bf16_bits(Q), gq.numpy(), workloads.bf16_bits(K), gk.numpy(),
            workloads.bf16_bits(X))


def host_threads() -> int:
    """The cores this process may run on (its affinity mask)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def time_oracle(seconds: float, nthreads: int):
    """The oracle on repeated row samples of the step for about `seconds`:
    16 rows of Q and of K and 128 rows of X per thread and pass."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    rows_qk, rows_mx = 16 * nthreads, 128 * nthreads
    state = oracle_inputs(rows_qk, rows_mx)
    pool = ThreadPoolExecutor(nthreads) if nthreads > 1 else None
    try:
        oracle_sample_step(rows_qk, rows_mx, state, pool, nthreads)   # warm-up
        done, passes, t0 = 0, 0, time.perf_counter()
        while True:
            done += oracle_sample_step(rows_qk, rows_mx, state, pool, nthreads)
            passes += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
    finally:
        if pool is not None:
            pool.shutdown()
    return done / dt / 1e9, passes, dt, rows_qk, rows_mx


def cpu_baseline(seconds: float):
    """The oracle as it stands, on the host cores: over tokens on every core
    of the affinity mask (the reported value), and single-threaded beside
    it, each for about half of `seconds`."""
    n = host_threads()
    v1, p1, d1, q1, m1 = time_oracle(seconds / 2, 1)
    vn, pn, dn, qn, mn = time_oracle(seconds / 2, n)
    return {"value": round(vn, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": (f"{pn} passes of {qn} rows of Q and of K (H=5120, N=4) and {mn} rows of "
                       f"X (D=4096) through qknorm_rms, rmsnorm_mxcast, mxnorm p=1, p=2, each "
                       f"call's rows split over {n} threads (over tokens); {dn:.1f} s"),
            "single_thread": {"value": round(v1, 4), "cores": 1,
                              "sample": f"{p1} passes of {q1} / {m1} rows; {d1:.1f} s"},
            "cpu": cpu_model()}


def cpu_model():
    """The host CPU's model name (lscpu), else what /proc/cpuinfo names."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


def run_reference(args):
    from concurrent.futures import ThreadPoolExecutor
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    n = host_threads()
    rows_qk, rows_mx = 4 * n, 32 * n
    state = oracle_inputs(rows_qk, rows_mx)
    with ThreadPoolExecutor(n) as pool:
        for _ in range(args.warmup):
            oracle_sample_step(rows_qk, rows_mx, state, pool, n)
        t0 = time.perf_counter()
        done = 0
        for _ in range(args.steps):
            done += oracle_sample_step(rows_qk, rows_mx, state, pool, n)
        dt = time.perf_counter() - t0
    value = round(done / dt / 1e9, 4)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n, "kind": "oracle",
                         "sample": (f"per step: {rows_qk} rows of Q and of K (H=5120, N=4), "
                                    f"{rows_mx} rows of X (D=4096) through qknorm_rms and the "
                                    f"three MX functions, rows split over {n} threads"),
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["nts", "reference"], default="nts")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", default=None,
                    help="time one kernel alone, e.g. mxnorm_cast:T=16384,D=1024,B=16,fmt=e2m1")
    ap.add_argument("--tune", default="",
                    help="--case: launch-shape overrides, e.g. vpt=4,rows=2,stages=3")
    ap.add_argument("--sets", type=int, default=1,
                    help="--case: input sets rotated between launches")
    args = ap.parse_args(argv)
    if args.case is not None:
        args.warmup = max(3, args.warmup)
        run_case(args)
        return
    if args.impl == "nts":
        args.warmup = max(3, args.warmup)     # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
