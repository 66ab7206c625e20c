#!/usr/bin/env python
"""Benchmark of the fused JSD forward+backward at the Qwen2.5 vocabulary.

Workload (one step): generalized JSD (beta = 0.5) forward and backward to both
inputs, gradients in bf16, on the causal-shift rows 0..N-2 of [N = 4 x 2048,
V = 151936] bf16 student and teacher logits (seeded synthetic logits with the
shape of the pages' Qwen2.5 runs; see softmax_divergence_lm_gb300/synth.py),
through the C-ABI call ``vpd_jsd_fwdbwd``.

Prints ONE JSON line (rank 0): tokens/s over all ranks, the roofline of the
dominant kernel (algorithmic bytes: read s and t once, write dS and dT once,
8 V bytes per token), the same metric end to end with host buffers, the CPU
oracle timed on a bounded sample, SM clocks sampled during the timed region,
and the library's kernel-launch count.

Multi-GPU (torchrun, one process per GPU): every rank runs the full workload
on its own GPU (rows are independent, so the op shards by token rows with no
data exchange); a barrier brackets the timed region and the time is the max
over ranks. ``--impl reference`` times the CPU oracle instead (rank 0 only).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "JSD fwd+bwd tokens/s at V=151936 bf16; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
BATCH, SEQ, VOCAB, BETA = 4, 2048, 151936, 0.5
ROWS = BATCH * SEQ - 1  # causal-shift rows 0..N-2 of the [N, V] buffer
BYTES_PER_TOKEN = 8 * VOCAB  # read s, t (bf16) once + write dS, dT (bf16) once
WORKLOAD = (f"qwen_vocab: JSD beta={BETA} fwd+bwd (both grads, bf16) on rows 0..N-2 of "
            f"[N={BATCH}x{SEQ}, V={VOCAB}] bf16 logits; vocab ids 151646..151935 = -inf")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--e2e-steps", type=int, default=8)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="target wall time of the CPU-oracle sample")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--sweep", action="store_true",
                   help="instead of the headline line, print one JSONL record per workload x op x phase")
    p.add_argument("--sweep-steps", type=int, default=10)
    p.add_argument("--profile-rows", type=int, default=0,
                   help="profiling mode: only the fused step on this many rows of the same vocabulary, "
                        "--warmup + --steps launches, one short line (for ncu captures of a small case)")
    p.add_argument("--profile-forward", action="store_true",
                   help="with --profile-rows: the forward-only call (no gradients) instead of fwd+bwd")
    p.add_argument("--profile-linear", type=int, default=0,
                   help="profiling mode: the fused-linear forward and backward on this many rows of the Qwen heads")
    p.add_argument("--cpu-sweep", action="store_true",
                   help="time the CPU oracle on every workload (the first four in full, 512 rows of the fifth) "
                        "with one thread and with all host threads; one JSONL record each")
    return p.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (barrier and max over ranks only; no data exchange)
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """The slowest rank's time: the job is done when every rank is."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def row_shard(n: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous rows [r0, r1) of an n-row batch owned by `rank` when a fixed
    batch is split over `world` GPUs. Rows are independent, so no data moves
    between ranks."""
    base, extra = divmod(n, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:  # noqa: BLE001
            sel = ["-i", str(device_index)]
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", *sel], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:10]))
            except ValueError:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r[0] <= self.t1 + 1] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3][1:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# the sources of the measured step: the single-read kernels, the streaming
# kernels that take the idle SMs' rows, and the call that splits the rows
FUSED_SOURCES = ("vpd_fused.cuh", "vpd_fused_bf16.cu", "vpd_fused_f16.cu", "vpd_fused.cu", "vpd_device.cuh",
                 "vpd_packed.cuh", "vpd_stream.cu", "vpd_api.cu", "vpd_internal.h")


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace runs collapsed, so that
    the hash follows the code and not its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def fused_source_hash() -> str:
    """Hash of the code of the sources the single-read kernels are built from."""
    h = hashlib.sha256()
    for name in FUSED_SOURCES:
        with open(os.path.join(ROOT, "softmax_divergence_lm_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this exact kernel source; None otherwise."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha") != kernel_hash:
        return None
    return rec.get("bytes_per_launch_full_workload")


def cpu_oracle_rate(s_rows, t_rows, seconds_target: float, threads: int):
    """Time the CPU oracle (fwd+bwd, beta = 0.5) on a bounded sample of rows."""
    from oracle import oracle as O
    import numpy as np

    O.build()
    n_all = s_rows.shape[0]
    probe = min(n_all, max(threads, 16))
    s64 = s_rows[:probe].float().cpu().double().numpy()
    t64 = t_rows[:probe].float().cpu().double().numpy()
    t0 = time.perf_counter()
    O.jsd(s64, t64, BETA, threads=threads)
    per_row = (time.perf_counter() - t0) / probe
    n = int(min(n_all, max(probe, seconds_target / max(per_row, 1e-9))))
    idx = torch.linspace(0, n_all - 1, n).round().long().to(s_rows.device)
    s64 = s_rows[idx].float().cpu().double().numpy()
    t64 = t_rows[idx].float().cpu().double().numpy()
    t0 = time.perf_counter()
    O.jsd(s64, t64, BETA, threads=threads)
    dt = time.perf_counter() - t0
    del np
    return n / dt, n, dt


def cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo; Arm hosts give the
    implementer and part numbers when no name is printed)."""
    try:
        text = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model Name", "Hardware"):
        m = re.search(rf"^{key}\s*:\s*(.+)$", text, flags=re.M)
        if m:
            return m.group(1).strip()
    impl = re.search(r"^CPU implementer\s*:\s*(\S+)", text, flags=re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", text, flags=re.M)
    if impl and part:
        # Arm Ltd. (implementer 0x41) core part numbers
        names = {"0xd0c": "Neoverse N1", "0xd40": "Neoverse V1", "0xd49": "Neoverse N2", "0xd4f": "Neoverse V2",
                 "0xd84": "Neoverse V3", "0xd8e": "Neoverse N3"}
        name = names.get(part.group(1).lower()) if impl.group(1).lower() == "0x41" else None
        return f"{name} (Arm part {part.group(1)})" if name else \
            f"Arm CPU implementer {impl.group(1)} part {part.group(1)}"
    return "unknown"


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    from softmax_divergence_lm_gb300 import binding as B
    from softmax_divergence_lm_gb300 import build as cuda_build
    from softmax_divergence_lm_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        cuda_build.build()
    barrier(world)
    B.load()
    # rank r holds the r-th contiguous share of a batch of `world` such
    # workloads: its own rows, drawn with the recipe's seed offset by r (rank 0
    # is the single-GPU workload)
    s3, t3 = synth.qwen_vocab(device=dev, seed=synth.SEEDS["qwen_vocab"] + rank)
    s = s3.view(BATCH * SEQ, VOCAB)[:-1]
    t = t3.view(BATCH * SEQ, VOCAB)[:-1]
    g = torch.full((ROWS,), 1.0 / ROWS, device=dev)
    loss = torch.empty(ROWS, device=dev)
    saved = torch.empty(ROWS, B.SAVED_PAIR, device=dev)
    ds = torch.empty(ROWS, VOCAB, dtype=torch.bfloat16, device=dev)
    dt = torch.empty(ROWS, VOCAB, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        B.vpd_jsd_fwdbwd(s, t, BETA, None, g, loss, saved, ds, dt, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    launches_per_step = None
    c0 = B.vpd_launch_count()
    step()
    torch.cuda.synchronize(dev)
    launches_per_step = B.vpd_launch_count() - c0

    clocks = ClockSampler(local)
    time.sleep(0.3)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    c0 = B.vpd_launch_count()
    start.record(stream)
    for i in range(args.steps):
        events[i][0].record(stream)
        step()
        events[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    launches = B.vpd_launch_count() - c0
    clocks.mark_end()
    barrier(world)
    clock_info = clocks.finish()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world)
    per_launch_ms = statistics.mean(a.elapsed_time(b) for a, b in events)
    ms_per_step = elapsed_ms / args.steps
    tokens_per_step = ROWS * world
    value = tokens_per_step / (ms_per_step / 1e3)

    peak, peak_kind = measured_peak()
    alg_bytes = BYTES_PER_TOKEN * ROWS
    achieved = alg_bytes / (per_launch_ms / 1e3) / 1e9
    kernel_hash = fused_source_hash()
    fused_rows, side_rows, planned = B.vpd_jsd_plan(s, t, None, ds, dt)
    single_read = fused_rows > 0 and planned == launches_per_step
    if single_read and side_rows:
        what = (f"k_jsd_fused on {fused_rows} rows with the streaming passes (k_pair_stats, k_jsd_div, k_pair_bwd) "
                f"on {side_rows} rows on the SMs its clusters leave idle, concurrently on a side stream; bytes and "
                f"time of the whole call ({launches_per_step} launches)")
    elif single_read:
        what = "k_jsd_fused (one launch per step)"
    else:
        what = f"{launches_per_step} streaming launches per step"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(kernel_hash) if single_read else None,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                "kernel": what, "fused_rows": fused_rows, "idle_sm_rows": side_rows,
                "algorithmic_bytes_per_launch": alg_bytes, "launch_ms": round(per_launch_ms, 4),
                "frac_of_8TBps_nameplate": round(achieved / 8000.0, 4)}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, B, s, t, g, dev, stream, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = host_threads()
        rate, n, secs = cpu_oracle_rate(s, t, args.cpu_seconds, threads)
        rate1, n1, secs1 = cpu_oracle_rate(s, t, max(2.0, args.cpu_seconds / 3), 1)
        cpu = {"value": round(rate, 2), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} of the {ROWS} workload rows (evenly spaced), fp64 oracle fwd+bwd, {secs:.1f} s wall",
               "single_thread": {"value": round(rate1, 2), "cores": 1,
                                 "sample": f"{n1} rows (evenly spaced), {secs1:.1f} s wall"},
               "cpu_model": cpu_model()}

    if rank == 0:
        out = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": WORKLOAD, "tokens_per_step_per_gpu": ROWS, "vocab": VOCAB, "beta": BETA,
                          "grads": "dS and dT, bf16", "l2": "inputs (4.98 GB per step) larger than the 129 MB L2",
                          "parallelism": (f"rows sharded contiguously: rank r holds rows [r x {ROWS}, (r + 1) x {ROWS})"
                                          f" of a {world} x {ROWS}-row batch, no collective")},
               "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clock_info,
               "gpu_launches": launches, "impl": "ours"}
        print(json.dumps(out), flush=True)


def run_e2e(args, B, s, t, g, dev, stream, world, chunks=8):
    """The same step through the C-ABI call with host buffers: every step copies
    the inputs from pinned host memory to the device and the loss and both
    gradients back. The rows are cut into chunks on three streams (copy in,
    compute, copy out) so both copy directions overlap each other and the
    kernel."""
    n, v = s.shape
    s_h = torch.empty(n, v, dtype=s.dtype, pin_memory=True)
    t_h = torch.empty(n, v, dtype=t.dtype, pin_memory=True)
    s_h.copy_(s)
    t_h.copy_(t)
    s_d = torch.empty_like(s)
    t_d = torch.empty_like(t)
    loss = torch.empty(n, device=dev)
    saved = torch.empty(n, 6, device=dev)
    ds = torch.empty(n, v, dtype=torch.bfloat16, device=dev)
    dt = torch.empty(n, v, dtype=torch.bfloat16, device=dev)
    loss_h = torch.empty(n, pin_memory=True)
    ds_h = torch.empty(n, v, dtype=torch.bfloat16, pin_memory=True)
    dt_h = torch.empty(n, v, dtype=torch.bfloat16, pin_memory=True)
    spans = [row_shard(n, chunks, c) for c in range(chunks)]
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    last_compute = [None] * chunks  # previous step's events per chunk (write-after-read order)
    last_out = [None] * chunks

    def step():
        for c, (a, b) in enumerate(spans):
            if last_compute[c] is not None:
                s_in.wait_event(last_compute[c])  # the kernel has finished reading s_d, t_d
            with torch.cuda.stream(s_in):
                s_d[a:b].copy_(s_h[a:b], non_blocking=True)
                t_d[a:b].copy_(t_h[a:b], non_blocking=True)
            arrived = torch.cuda.Event()
            arrived.record(s_in)
            s_run.wait_event(arrived)
            if last_out[c] is not None:
                s_run.wait_event(last_out[c])  # the host has the previous results
            B.vpd_jsd_fwdbwd(s_d[a:b], t_d[a:b], BETA, None, g[a:b], loss[a:b], saved[a:b], ds[a:b], dt[a:b],
                             s_run)
            computed = torch.cuda.Event()
            computed.record(s_run)
            s_out.wait_event(computed)
            with torch.cuda.stream(s_out):
                loss_h[a:b].copy_(loss[a:b], non_blocking=True)
                ds_h[a:b].copy_(ds[a:b], non_blocking=True)
                dt_h[a:b].copy_(dt[a:b], non_blocking=True)
            copied = torch.cuda.Event()
            copied.record(s_out)
            last_compute[c], last_out[c] = computed, copied
        stream.wait_stream(s_out)

    step()
    torch.cuda.synchronize(dev)
    # three windows of e2e_steps steps each; the median window is reported (the
    # host link is shared with the machine's other work, so one short window
    # can catch a transient slowdown) and every window is listed
    windows = []
    for _ in range(3):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for st in (s_in, s_run, s_out):
            st.wait_stream(stream)
        for _ in range(args.e2e_steps):
            step()
        end.record(stream)
        torch.cuda.synchronize(dev)
        windows.append(max_over_ranks(start.elapsed_time(end), world) / args.e2e_steps)
    ms = sorted(windows)[1]
    h2d = 2 * n * v * s.element_size()
    d2h = n * 4 + 2 * n * v * 2
    # the link alone: plain pinned copies of 1 GiB, each direction by itself
    # and both at once, so the e2e number can be read against them
    peaks = copy_peaks(dev, s_h.view(-1)[: 1 << 29], ds_h.view(-1)[: 1 << 29])
    # the link's bound for a step: each direction at its own rate, and both
    # together at the rate they reach when they run at once
    bound_ms = max(h2d / peaks["h2d_GBps"], d2h / peaks["d2h_GBps"], (h2d + d2h) / peaks["both_GBps"]) / 1e6
    return {"value": round(n * world / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "windows_ms_per_step": [round(w, 3) for w in windows],
            "copy_peaks": peaks, "copy_bound_ms_per_step": round(bound_ms, 3),
            "frac_of_copy_bound": round(bound_ms / ms, 4),
            "path": (f"pinned host -> device copies, vpd_jsd_fwdbwd, device -> pinned host copies of loss, dS, dT; "
                     f"{chunks} row chunks pipelined over 3 streams")}


def copy_peaks(dev, host_src, host_dst, reps=5):
    """GB/s of plain cudaMemcpyAsync between pinned host and device memory:
    host->device alone, device->host alone, and both directions at once
    (best of `reps`)."""
    d_in = torch.empty_like(host_src, device=dev)
    d_out = torch.empty_like(host_dst, device=dev)
    nbytes = host_src.numel() * host_src.element_size()
    a, b = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
        return best

    def h2d():
        with torch.cuda.stream(a):
            d_in.copy_(host_src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(b):
            host_dst.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_h2d, t_d2h, t_both = timed(h2d), timed(d2h), timed(both)
    return {"h2d_GBps": round(nbytes / t_h2d / 1e9, 1), "d2h_GBps": round(nbytes / t_d2h / 1e9, 1),
            "both_GBps": round(2 * nbytes / t_both / 1e9, 1), "bytes_each": nbytes}


# ---------------------------------------------------------------------------
def run_reference(args, world, rank):
    """The CPU oracle, as it stands, on a bounded sample of the same workload."""
    if rank != 0:
        return
    from oracle import oracle as O
    from softmax_divergence_lm_gb300 import synth

    O.build()
    threads = host_threads()
    rows = 256
    s3, t3 = synth.qwen_vocab(device="cpu", batch=1, seq=rows + 1)
    s64 = s3.view(rows + 1, VOCAB)[:-1].float().double().numpy()
    t64 = t3.view(rows + 1, VOCAB)[:-1].float().double().numpy()
    for _ in range(max(1, min(args.warmup, 2))):
        O.jsd(s64, t64, BETA, threads=threads)
    steps = max(1, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(steps):
        O.jsd(s64, t64, BETA, threads=threads)
    secs = time.perf_counter() - t0
    value = rows * steps / secs
    sample = f"{rows} rows of the same recipe per step (CPU-generated), fp64 oracle fwd+bwd, {steps} steps"
    out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": steps,
           "warmup": max(1, min(args.warmup, 2)), "ms_per_step": round(secs / steps * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "tokens_per_step_per_gpu": rows, "vocab": VOCAB, "beta": BETA},
           "impl": "reference",
           "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": threads, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# Sweep: every workload x op x phase (tokens/s, GB/s of minimum bytes, and
# the fraction of the measured peak). Minimum bytes: each input row read once
# and each gradient row written once.
# ---------------------------------------------------------------------------
def _trials(fn, trials, warmup, stream):
    """Per-call times (ms) of `trials` calls after `warmup` untimed ones, each
    bracketed by CUDA events on the launching stream."""
    for _ in range(max(3, warmup)):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(trials)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def source_hash() -> str:
    """Hash of the code of every CUDA source and the C header (comments and
    whitespace removed): names the library build a record was measured on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "softmax_divergence_lm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)) + ["../../include/vpd.h"]:
        path = os.path.normpath(os.path.join(csrc, name))
        if path.endswith((".cu", ".cuh", ".h")):
            with open(path, encoding="utf-8") as f:
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


# ncu summaries under profiles/ of the kernels a sweep record runs
NCU_SUMMARIES = {
    ("qwen_vocab", "jsd", "fwd+bwd"): "profiles/fused_jsd_qwen_vocab.md",
    ("qwen_vocab", "jsd", "fwd"): "profiles/fused_fwd_jsd_qwen_vocab.md",
    ("linear_heads", "jsd_linear", "fwd"): "profiles/linear_jsd_qwen_heads.md",
    ("linear_heads", "jsd_linear", "bwd"): "profiles/linear_jsd_qwen_heads.md",
}


def run_sweep(args):
    from softmax_divergence_lm_gb300 import binding as B
    from softmax_divergence_lm_gb300 import build as cuda_build
    from softmax_divergence_lm_gb300 import synth

    cuda_build.build()
    B.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    peak, kind = measured_peak()
    trials = max(10, args.sweep_steps)
    src = source_hash()

    def emit(workload, op, phase, dtype, beta, n, v, min_bytes, times, extra=None, flops=None):
        ms = statistics.median(times)
        gbs = min_bytes / (ms / 1e3) / 1e9
        key = next((k for k in NCU_SUMMARIES if workload.startswith(k[0]) and op == k[1] and phase.startswith(k[2])),
                   None)
        rec = {"workload": workload, "op": op, "phase": phase, "dtype": dtype, "beta": beta, "N": n, "V": v,
               "min_bytes": int(min_bytes), "ms": round(ms, 4), "ms_min": round(min(times), 4), "trials": len(times),
               "tokens_per_s": round(n / (ms / 1e3), 1), "GBps": round(gbs, 1),
               "frac_of_measured_peak": round(gbs / peak, 4), "peak_GBps": peak, "peak_source": kind,
               "frac_of_8TBps": round(gbs / 8000.0, 4), "source_sha": src,
               "ncu_summary": NCU_SUMMARIES.get(key)}
        if flops is not None:
            tf = flops / (ms / 1e3) / 1e12
            rec.update({"TFLOPs": round(tf, 1), "frac_of_bf16_sustained": round(tf / measured_tflops(), 4)})
        if extra:
            rec.update(extra)
        print(json.dumps(rec), flush=True)

    def pair_suite(name, s, t, betas, gdtype, segments=None, do_kl=True, fused_only=False, detached=False):
        n, v = s.shape[0] if s.dim() == 2 else s.shape[0] * s.shape[1], s.shape[-1]
        es, eg = s.element_size(), torch.empty((), dtype=gdtype).element_size()
        loss = torch.empty(n, device=dev)
        saved = torch.empty(n, 6, device=dev)
        ds = torch.empty(n, v, dtype=gdtype, device=dev)
        dt = torch.empty(n, v, dtype=gdtype, device=dev)
        g = torch.full((n,), 1.0 / n, device=dev)
        rd, wr = 2 * n * v * es, 2 * n * v * eg
        dt_name = str(s.dtype).replace("torch.", "")

        def plan(want_grads, want_t=True):
            fr, side, k = B.vpd_jsd_plan(s, t, segments, ds if want_grads else None,
                                         dt if want_grads and want_t else None)
            label = "single-read" if fr else ("two-pass" if not want_grads else "streaming")
            return {"path": label + (f" + {side} rows on idle SMs" if side else ""), "launches": k}

        for beta in betas:
            if not fused_only:
                ms = _trials(lambda: B.vpd_jsd_fwd(s, t, beta, segments, loss, saved), trials, 3, stream)
                # at beta = 0 / 1 the forward is the online KL kernel (one launch)
                fwd_path = {"path": "online KL kernel", "launches": 1} if beta in (0.0, 1.0) else plan(False)
                emit(name, "jsd", "fwd", dt_name, beta, n, v, rd, ms, fwd_path)
                ms = _trials(lambda: B.vpd_jsd_bwd(s, t, beta, segments, g, saved, ds, dt), trials, 3, stream)
                emit(name, "jsd", "bwd", dt_name, beta, n, v, rd + wr, ms)
            ms = _trials(lambda: B.vpd_jsd_fwdbwd(s, t, beta, segments, g, loss, saved, ds, dt), trials, 3, stream)
            emit(name, "jsd", "fwd+bwd", dt_name, beta, n, v, rd + wr, ms, plan(True))
            if detached:
                ms = _trials(lambda: B.vpd_jsd_fwdbwd(s, t, beta, segments, g, loss, saved, ds, None), trials, 3,
                             stream)
                emit(name, "jsd", "fwd+bwd detached teacher", dt_name, beta, n, v, rd + wr // 2, ms,
                     plan(True, want_t=False))
        if do_kl:
            for rev in (False, True):
                opn = "kl_reverse" if rev else "kl_forward"
                ms = _trials(lambda: B.vpd_kl_fwd(s, t, rev, segments, loss, saved), trials, 3, stream)
                emit(name, opn, "fwd (one read)", dt_name, None, n, v, rd, ms)
                ms = _trials(lambda: B.vpd_kl_bwd(s, t, rev, segments, g, saved, ds, dt), trials, 3, stream)
                emit(name, opn, "bwd", dt_name, None, n, v, rd + wr, ms)
        del ds, dt

    def single_suite(name, x, gdtype, ids=None, teacher=None):
        n, v = x.shape
        ex, eg = x.element_size(), torch.empty((), dtype=gdtype).element_size()
        dx = torch.empty(n, v, dtype=gdtype, device=dev)
        out = torch.empty(n, device=dev)
        saved = torch.empty(n, 3, device=dev)
        g = torch.full((n,), 1.0 / n, device=dev)
        dt_name = str(x.dtype).replace("torch.", "")
        ms = _trials(lambda: B.vpd_entropy_fwd(x, None, out, saved), trials, 3, stream)
        emit(name, "entropy", "fwd (single pass)", dt_name, None, n, v, n * v * ex, ms)
        ms = _trials(lambda: B.vpd_entropy_bwd(x, None, g, saved, dx), trials, 3, stream)
        emit(name, "entropy", "bwd", dt_name, None, n, v, n * v * (ex + eg), ms)
        if ids is not None:
            k = ids.shape[1]
            lp = torch.empty(n, k, device=dev)
            ls = torch.empty(n, 2, device=dev)
            err = torch.empty(1, dtype=torch.int32, device=dev)
            gk = torch.full((n, k), 1.0 / n, device=dev)
            ms = _trials(lambda: B.vpd_logprobs_fwd(x, None, ids, k, -100, lp, ls, err), trials, 3, stream)
            emit(name, f"logprobs_top{k}", "fwd", dt_name, None, n, v, n * v * ex, ms)
            ms = _trials(lambda: B.vpd_logprobs_bwd(x, None, ids, k, -100, gk, ls, dx), trials, 3, stream)
            emit(name, f"logprobs_top{k}", "bwd", dt_name, None, n, v, n * v * (ex + eg), ms)
            labels = ids[:, 0].contiguous()
            ms = _trials(lambda: B.vpd_cross_entropy_fwd(x, None, labels, -100, 1.0, out, ls, err), trials, 3, stream)
            emit(name, "cross_entropy", "fwd", dt_name, None, n, v, n * v * ex, ms)
            ms = _trials(lambda: B.vpd_cross_entropy_bwd(x, None, labels, -100, 1.0, g, ls, dx), trials, 3, stream)
            emit(name, "cross_entropy", "bwd", dt_name, None, n, v, n * v * (ex + eg), ms)
            if teacher is not None:
                tl = torch.log_softmax(teacher.float(), dim=1).gather(1, ids).contiguous()
                ms = _trials(lambda: B.vpd_topk_kl_fwd(x, None, ids, k, -100, tl, 1.0, out, ls, err), trials, 3,
                             stream)
                emit(name, f"topk{k}_forward_kl", "fwd", dt_name, None, n, v, n * v * ex, ms)
                ms = _trials(lambda: B.vpd_topk_kl_bwd(x, None, ids, k, -100, tl, 1.0, g, ls, dx), trials, 3, stream)
                emit(name, f"topk{k}_forward_kl", "bwd", dt_name, None, n, v, n * v * (ex + eg), ms)
                ms = _trials(lambda: B.vpd_topk_kl_fwd(x, None, ids, k, -100, tl, 2.0, out, ls, err), trials, 3,
                             stream)
                emit(name, f"topk{k}_forward_kl", "fwd, temperature 2", dt_name, None, n, v, n * v * ex, ms)
        del dx

    # page-shaped local shard, bf16
    s, t, ids = synth.page_shard(device=dev)
    pair_suite("page_shard 8192x16032", s, t, (0.1, 0.5, 0.9), torch.bfloat16)
    single_suite("page_shard 8192x16032", s, torch.bfloat16, ids, teacher=t)
    del s, t, ids
    torch.cuda.empty_cache()
    # Qwen2.5 vocabulary, rows 0..N-2 and the [4, 2047, V] causal view
    s3, t3 = synth.qwen_vocab(device=dev)
    n = BATCH * SEQ
    s, t = s3.view(n, VOCAB)[:-1], t3.view(n, VOCAB)[:-1]
    pair_suite("qwen_vocab rows 0..N-2", s, t, (0.5,), torch.bfloat16, do_kl=True, detached=True)
    pair_suite("qwen_vocab causal [4,2047,V]", s3[:, :-1], t3[:, :-1], (0.5,), torch.bfloat16, do_kl=False,
               fused_only=True)
    teacher_stream_suite(B, emit, s, t, dev, stream, trials)
    vocab_parallel_suite(B, emit, s, t, dev, stream, trials)
    del s, t, s3, t3
    torch.cuda.empty_cache()
    linear_suite(B, emit, synth, dev, stream, trials)
    torch.cuda.empty_cache()
    # numerical edge cases, fp32, 8 segments
    s, t, info = synth.edge_cases(device=dev)
    pair_suite("edge_cases 4096x128256 fp32 8 segments", s, t, (0.0, 0.25, 0.5, 0.75, 1.0), torch.float32,
               segments=info["segments"], do_kl=False)
    del s, t
    torch.cuda.empty_cache()
    # large throughput sweep, bf16 and fp16
    for dt_ in (torch.bfloat16, torch.float16):
        s, t = synth.large_sweep(device=dev, dtype=dt_)
        pair_suite("large_sweep 32768x262144", s, t, (0.5,), dt_, do_kl=False)
        n, v = s.shape
        loss = torch.empty(n, device=dev)
        saved = torch.empty(n, 6, device=dev)
        ds = torch.empty(n, v, dtype=dt_, device=dev)
        dtg = torch.empty(n, v, dtype=dt_, device=dev)
        g = torch.full((n,), 1.0 / n, device=dev)
        nm = str(dt_).replace("torch.", "")
        ms = _trials(lambda: B.vpd_kl_fwd(s, t, False, None, loss, saved), trials, 3, stream)
        emit("large_sweep 32768x262144", "kl_forward", "fwd (single pass)", nm, None, n, v, 2 * n * v * 2, ms)
        ms = _trials(lambda: B.vpd_kl_bwd(s, t, False, None, g, saved, ds, dtg), trials, 3, stream)
        emit("large_sweep 32768x262144", "kl_forward", "bwd", nm, None, n, v, 4 * n * v * 2, ms)
        del ds, dtg
        single_suite("large_sweep 32768x262144", s, dt_)
        del s, t
        torch.cuda.empty_cache()


def measured_tflops() -> float:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        return 1700.0


def teacher_stream_suite(B, emit, s, t, dev, stream, trials, chunk=1024):
    """JSD fwd+bwd with the teacher logits in a pinned host cache, student
    gradient only (the teacher is a cache): the teacher rows cross the
    host link once per step. Minimum HBM bytes: s read, t read once it has
    landed, dS written (6 V per token)."""
    n, v = s.shape
    t_host = t.cpu().pin_memory()
    staging = torch.empty(4 * chunk * v * 2, dtype=torch.uint8, device=dev)
    copy = torch.cuda.Stream(dev)
    loss = torch.empty(n, device=dev)
    saved = torch.empty(n, 6, device=dev)
    ds = torch.empty(n, v, dtype=torch.bfloat16, device=dev)
    g = torch.full((n,), 1.0 / n, device=dev)
    ms = _trials(lambda: B.vpd_jsd_fwdbwd_teacher_stream(s, t_host, 0.5, g, loss, saved, ds, None, staging, chunk,
                                                         stream, copy), trials, 3, stream)
    emit("qwen_vocab rows 0..N-2", "jsd", "fwd+bwd, teacher from a pinned host cache", "bfloat16", 0.5, n, v,
         3 * n * v * 2, ms, {"host_bytes_per_step": n * v * 2, "chunk_rows": chunk,
                             "host_GBps": round(n * v * 2 / (statistics.median(ms) / 1e3) / 1e9, 1)})


def vocab_parallel_suite(B, emit, s, t, dev, stream, trials):
    """The per-shard kernels of the vocabulary-parallel forward and backward
    for one of two shards (TP2) of the Qwen vocabulary; the all-reduces of the
    [N, 2] buffers between the steps are not timed (no second GPU here)."""
    n, v = s.shape
    h = v // 2
    sl, tl = s[:, :h], t[:, :h]
    loss = torch.empty(n, device=dev)
    saved = torch.empty(n, 6, device=dev)
    x = torch.empty(n, 2, device=dev)
    ds = torch.empty(n, h, dtype=torch.bfloat16, device=dev)
    dt = torch.empty(n, h, dtype=torch.bfloat16, device=dev)
    g = torch.full((n,), 1.0 / n, device=dev)

    def fwd():
        B.vpd_jsd_shard_stats(sl, tl, saved, x)
        B.vpd_jsd_shard_rescale(n, saved, x)
        B.vpd_jsd_shard_divergence(sl, tl, 0.5, loss, saved, x)
        B.vpd_jsd_shard_finish(n, 0.5, saved, x, loss)

    ms = _trials(fwd, trials, 3, stream)
    emit("qwen_vocab rows 0..N-2, TP2 shard", "jsd_vocab_parallel", "fwd (shard kernels)", "bfloat16", 0.5, n, h,
         2 * n * h * 2, ms)
    ms = _trials(lambda: B.vpd_jsd_bwd(sl, tl, 0.5, None, g, saved, ds, dt), trials, 3, stream)
    emit("qwen_vocab rows 0..N-2, TP2 shard", "jsd_vocab_parallel", "bwd (local)", "bfloat16", 0.5, n, h,
         4 * n * h * 2, ms)


def linear_suite(B, emit, synth, dev, stream, trials, n=8192):
    """Fused-linear JSD at the pages' heads (student Qwen2.5-0.5B hidden 896,
    teacher Qwen2.5-1.5B hidden 1536, vocabulary 151936): forward (two passes of
    logits tiles) and backward (logits tiles again, then dh and dW of the
    student); tensor-core FLOPs against the measured sustained bf16 peak."""
    h_s, w_s, h_t, w_t = synth.linear_heads(device=dev, n=n)
    heads = B.make_heads(h_s, w_s, h_t, w_t)
    fb, bb = B.vpd_jsd_linear_workspace(heads, True, False)
    ws = torch.empty(max(fb, bb), dtype=torch.uint8, device=dev)
    v, hs, ht = w_s.shape[0], h_s.shape[1], h_t.shape[1]
    loss = torch.empty(n, device=dev)
    saved = torch.empty(n, 6, device=dev)
    dh = torch.empty(n, hs, device=dev)
    dw = torch.empty(v, hs, device=dev)
    g = torch.full((n,), 1.0 / n, device=dev)
    logits_flops = 2 * n * v * (hs + ht)
    inputs = 2 * (n * hs + v * hs + n * ht + v * ht)
    ms = _trials(lambda: B.vpd_jsd_linear_fwd(heads, 0.5, loss, saved, ws), trials, 2, stream)
    emit("linear_heads 8192 x (896|1536) -> 151936", "jsd_linear", "fwd (two passes of logits tiles)", "bfloat16",
         0.5, n, v, inputs, ms, {"bound": "tensor"}, flops=2 * logits_flops)
    ms = _trials(lambda: B.vpd_jsd_linear_bwd(heads, 0.5, g, loss, saved, dh, dw, None, None, ws), trials, 2,
                 stream)
    emit("linear_heads 8192 x (896|1536) -> 151936", "jsd_linear", "bwd (student dh, dW)", "bfloat16", 0.5, n, v,
         inputs + 4 * (n * hs + v * hs), ms, {"bound": "tensor"},
         flops=logits_flops + 2 * 2 * (2 * n * v * hs))


def run_profile(args):
    """The headline step on a smaller row count, for profiler captures: the same
    kernel and launch shape per row, a few GB on the device."""
    from softmax_divergence_lm_gb300 import binding as B
    from softmax_divergence_lm_gb300 import build as cuda_build
    from softmax_divergence_lm_gb300 import synth

    dev = torch.device("cuda", 0)
    cuda_build.build()
    B.load()
    n = args.profile_rows
    s3, t3 = synth.qwen_vocab(device=dev, batch=1, seq=n)
    s, t = s3.view(n, VOCAB), t3.view(n, VOCAB)
    g = torch.full((n,), 1.0 / n, device=dev)
    loss = torch.empty(n, device=dev)
    saved = torch.empty(n, B.SAVED_PAIR, device=dev)
    if args.profile_forward:
        for _ in range(args.warmup + args.steps):
            B.vpd_jsd_fwd(s, t, BETA, None, loss, saved)
    else:
        ds = torch.empty(n, VOCAB, dtype=torch.bfloat16, device=dev)
        dt = torch.empty(n, VOCAB, dtype=torch.bfloat16, device=dev)
        for _ in range(args.warmup + args.steps):
            B.vpd_jsd_fwdbwd(s, t, BETA, None, g, loss, saved, ds, dt)
    torch.cuda.synchronize(dev)
    B.vpd_device_status()
    print(json.dumps({"profile_rows": n, "launches": args.warmup + args.steps, "vocab": VOCAB,
                      "step": "forward" if args.profile_forward else "fwd+bwd"}), flush=True)


def run_profile_linear(args):
    """The fused-linear forward and backward on a smaller row count of the Qwen
    heads, for profiler captures (the same kernels and tile shapes)."""
    from softmax_divergence_lm_gb300 import binding as B
    from softmax_divergence_lm_gb300 import build as cuda_build
    from softmax_divergence_lm_gb300 import synth

    dev = torch.device("cuda", 0)
    cuda_build.build()
    B.load()
    n = args.profile_linear
    h_s, w_s, h_t, w_t = synth.linear_heads(device=dev, n=n)
    heads = B.make_heads(h_s, w_s, h_t, w_t)
    fb, bb = B.vpd_jsd_linear_workspace(heads, True, False)
    ws = torch.empty(max(fb, bb), dtype=torch.uint8, device=dev)
    loss = torch.empty(n, device=dev)
    saved = torch.empty(n, 6, device=dev)
    dh = torch.empty(n, h_s.shape[1], device=dev)
    dw = torch.empty(w_s.shape[0], h_s.shape[1], device=dev)
    for _ in range(args.warmup + args.steps):
        B.vpd_jsd_linear_fwd(heads, 0.5, loss, saved, ws)
        B.vpd_jsd_linear_bwd(heads, 0.5, None, loss, saved, dh, dw, None, None, ws)
    torch.cuda.synchronize(dev)
    B.vpd_device_status()
    print(json.dumps({"profile_linear_rows": n, "calls": args.warmup + args.steps}), flush=True)


def run_cpu_sweep(args):
    """The CPU oracle, as it stands, on each workload: the tiny, page-shard,
    Qwen-vocabulary and edge-case workloads in full, and a seeded 512-row
    sample of the large sweep (its per-token rate, labelled an
    extrapolation); each with one thread and with every host thread."""
    from oracle import oracle as O
    from softmax_divergence_lm_gb300 import synth

    O.build()
    model = cpu_model()
    all_threads = host_threads()

    def emit(workload, op, n, v, fn, extrapolated=False):
        for threads in (1, all_threads):
            t0 = time.perf_counter()
            fn(threads)
            secs = time.perf_counter() - t0
            print(json.dumps({"workload": workload, "op": op, "N": n, "V": v, "threads": threads, "cpu_model": model,
                              "seconds": round(secs, 3), "tokens_per_s": round(n / secs, 2),
                              "kind": "oracle", "extrapolated": extrapolated}), flush=True)

    s, t = synth.tiny()
    s64, t64 = s.double().numpy(), t.double().numpy()
    emit("tiny 64x1024 fp32", "jsd fwd+bwd beta=0.5", 64, 1024, lambda k: O.jsd(s64, t64, 0.5, threads=k))
    s, t, _ = synth.page_shard()
    s64, t64 = s.float().double().numpy(), t.float().double().numpy()
    emit("page_shard 8192x16032", "jsd fwd+bwd beta=0.5", 8192, 16032, lambda k: O.jsd(s64, t64, 0.5, threads=k))
    del s64, t64
    s3, t3 = synth.qwen_vocab()
    n = BATCH * SEQ - 1
    s64 = s3.view(-1, VOCAB)[:-1].float().double().numpy()
    t64 = t3.view(-1, VOCAB)[:-1].float().double().numpy()
    del s3, t3
    emit("qwen_vocab rows 0..N-2", "jsd fwd+bwd beta=0.5", n, VOCAB, lambda k: O.jsd(s64, t64, 0.5, threads=k))
    del s64, t64
    s, t, info = synth.edge_cases()
    s64, t64 = s.double().numpy(), t.double().numpy()
    emit("edge_cases 4096x128256 fp32", "jsd fwd+bwd beta=0.5", 4096, 128256,
         lambda k: O.jsd(s64, t64, 0.5, threads=k))
    del s64, t64, s, t
    s, t = synth.large_sweep(n=512)
    s64, t64 = s.float().double().numpy(), t.float().double().numpy()
    emit("large_sweep 512-row sample of 32768x262144", "jsd fwd+bwd beta=0.5", 512, 262144,
         lambda k: O.jsd(s64, t64, 0.5, threads=k), extrapolated=True)


def main():
    args = parse_args()
    if args.profile_rows:
        run_profile(args)
        return
    if args.profile_linear:
        run_profile_linear(args)
        return
    if args.cpu_sweep:
        run_cpu_sweep(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup()
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
