"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long]

One step = one ``attn_fwd`` call over one batch of the workload (the whole
hot path: a single fused kernel).  The default workload is the long-sequence
causal configuration the throughput target is stated on: B=1, H=32, N=16384,
d=128, bf16, causal, Q,K,V ~ N(0,1) with 1% of the K rows scaled by 8.

Prints ONE JSON line (rank 0).  ``value`` is TFLOP/s with the inputs resident
in HBM (4*B*H*N^2*d FLOPs, halved for causal, counted per rank and summed over
ranks, divided by the slowest rank's time); ``e2e`` is the same metric through
the public API with pinned host buffers, the host->device copies of Q, K, V
and the device->host copies of O and LSE inside the timed region.

--impl reference times the fp64 CPU oracle (as it stands) on the host cores,
on bounded row samples of the same workload.  Under torchrun only rank 0 does
that; the other ranks exit without work.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_attention_51_gb300 import workloads as wl  # noqa: E402

METRIC = "attention fwd TFLOP/s (bf16, causal/non-causal) and % of GB300 dense BF16 peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# The sources that build the bf16 forward kernel this benchmark times: a
# committed DRAM-traffic figure is used only while they hash to what was
# profiled.
KERNEL_SOURCES = ["exact_attention_51_gb300/csrc/attn_fwd_kernel.cuh",
                  "exact_attention_51_gb300/csrc/ptx.cuh",
                  "exact_attention_51_gb300/csrc/launch.cuh",
                  "exact_attention_51_gb300/csrc/fwd_dispatch.h",
                  "exact_attention_51_gb300/csrc/attn_fwd_d*.cu",
                  "exact_attention_51_gb300/csrc/attn_api.cu"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for pat in KERNEL_SOURCES:
        for f in sorted(glob.glob(os.path.join(ROOT, pat))):
            h.update(os.path.basename(f).encode())
            h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str, causal: bool):
    """DRAM bytes per launch from a committed ncu capture, if the kernel
    sources still hash to what was profiled."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    key = f"{workload}-{'causal' if causal else 'full'}"
    e = d.get(key)
    if not e or e.get("kernel_source_sha") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples with host arrival times."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", gpu_id, "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [(t, s) for t, s in self.samples if t0 <= t <= t1 + 0.06]
        if not rows:  # timed region shorter than one sampling interval
            before = [(t, s) for t, s in self.samples if t <= t1 + 0.06]
            rows = before[-1:]
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, s in rows:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = max(smax, float(f[2]))
            except ValueError:
                continue
            for name, flag in zip(names, f[5:9]):
                if flag.lower() in ("active", "0x1", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": smax or None, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[device_index]
        return str(device_index)


# ---------------------------------------------------------------- CPU oracle

def row_flops(w: wl.Workload, causal: bool, rows) -> float:
    """Algorithmic FLOPs of the listed rows (4*d per visible key)."""
    if not causal:
        return 4.0 * w.d * w.N * len(rows)
    return float(sum(4.0 * w.d * ((r % w.N) + 1) for r in rows))


def time_oracle(w, causal, q, k, v, target_s: float, seed: int):
    """Oracle throughput (TFLOP/s) on seeded random row samples, grown until
    one sample takes about `target_s` seconds; returns (tflops, seconds, rows,
    threads)."""
    import numpy as np
    import oracle
    orc = oracle.Oracle()
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.H * w.N
    n = 256
    while True:
        rows = sorted(rng.choice(total_rows, size=min(n, total_rows), replace=False).tolist())
        t0 = time.perf_counter()
        orc.attn_bf16_rows(q, k, v, causal, w.scale, rows)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or len(rows) == total_rows:
            return row_flops(w, causal, rows) / dt / 1e12, dt, len(rows), orc.max_threads()
        n = int(len(rows) * min(8.0, max(1.5, target_s / max(dt, 1e-3))))


# ---------------------------------------------------------------- main arms

def reduce_max_over_ranks(values, device):
    """Element-wise max of `values` over all ranks (identity when not
    distributed).  The only collective in the benchmark; the data path has
    none."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_tflops(flops_per_rank: float, world: int, slowest_ms: float) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return world * flops_per_rank / (slowest_ms * 1e-3) / 1e12


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, w, causal):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    q, k, v = wl.workload_inputs(w)
    import numpy as np
    import oracle
    orc = oracle.Oracle()
    rng = np.random.default_rng(12345)
    total_rows = w.B * w.H * w.N
    # size each step to ~2 s of oracle work so K + W steps stay within minutes
    n = 256
    while True:
        rows = sorted(rng.choice(total_rows, size=min(n, total_rows), replace=False).tolist())
        t0 = time.perf_counter()
        orc.attn_bf16_rows(q, k, v, causal, w.scale, rows)
        dt = time.perf_counter() - t0
        if dt >= 1.0 or len(rows) == total_rows:
            break
        n = int(len(rows) * min(8.0, max(1.5, 2.0 / max(dt, 1e-3))))
    n = len(rows)
    times, flops = [], []
    for step in range(args.warmup + args.steps):
        rows = sorted(rng.choice(total_rows, size=n, replace=False).tolist())
        t0 = time.perf_counter()
        orc.attn_bf16_rows(q, k, v, causal, w.scale, rows)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            flops.append(row_flops(w, causal, rows))
    value = sum(flops) / sum(times) / 1e12
    sample = (f"{n} seeded random rows of {w.describe(causal)} per step "
              f"(full workload: {total_rows} rows)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.describe(causal), "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": causal, "sample_rows_per_step": n},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": orc.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w, causal):
    import torch
    import torch.distributed as dist

    import exact_attention_51_gb300 as ea
    from exact_attention_51_gb300 import build as eabuild

    ws, rank, local = dist_setup()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    eabuild.build()
    ea.load_library()

    q_h, k_h, v_h = wl.workload_inputs(w)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    flops = w.flops(causal)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws > 1:
            dist.barrier()

    # ---- device-resident timing
    splits = args.splits
    if splits == 0:
        splits = ea.attn_fwd_splitkv_num_splits(
            w.B, w.H, w.N, w.d, causal, torch.cuda.get_device_properties(dev).multi_processor_count)
    ws_bytes = ea.attn_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.d, splits) if splits > 1 else 0
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def fwd(qq, kk, vv, oo, ll, st=None):
        if splits > 1:
            ea.attn_fwd_splitkv(qq, kk, vv, causal=causal, num_splits=splits, out=oo, lse=ll,
                                workspace=workspace, stream=st)
        else:
            ea.attn_fwd(qq, kk, vv, causal=causal, out=oo, lse=ll, stream=st)

    for _ in range(args.warmup):
        fwd(q, k, v, o, lse)
    torch.cuda.synchronize(dev)
    st, detail = ea.attn_fwd_device_status()
    if st != ea.ATTN_OK:
        raise RuntimeError(f"device wait timed out during warm-up (code {detail:#x})")

    sampler = ClockSampler(gpu_id_for(local))
    time.sleep(0.3)  # let nvidia-smi start printing
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.monotonic()
    ev0.record(stream)
    for _ in range(args.steps):
        fwd(q, k, v, o, lse)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.monotonic()
    barrier()
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)
    ms = ev0.elapsed_time(ev1) / args.steps
    st, detail = ea.attn_fwd_device_status()
    if st != ea.ATTN_OK:
        raise RuntimeError(f"device wait timed out in the timed region (code {detail:#x})")

    # ---- end to end: pinned host buffers, copies inside the timed region.
    # Two device buffer sets; step i copies its inputs in on an H2D stream,
    # computes on the compute stream and copies O and LSE out on a D2H stream,
    # so the copies of one step overlap the kernel of the neighbouring steps
    # (the copy engines and the SMs are separate hardware).
    qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
    op = [torch.empty(q_h.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lp = [torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory() for _ in range(2)]
    bufs = [dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                 o=torch.empty_like(q), l=torch.empty_like(lse)) for _ in range(2)]
    del o, lse, q, k, v
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    for e in ev_free:
        e.record(s_d2h)

    def e2e_step(i):
        b = bufs[i % 2]
        s_h2d.wait_event(ev_free[i % 2])
        with torch.cuda.stream(s_h2d):
            b["q"].copy_(qp, non_blocking=True)
            b["k"].copy_(kp, non_blocking=True)
            b["v"].copy_(vp, non_blocking=True)
            ev_in[i % 2].record(s_h2d)
        stream.wait_event(ev_in[i % 2])
        fwd(b["q"], b["k"], b["v"], b["o"], b["l"], stream)
        ev_done[i % 2].record(stream)
        s_d2h.wait_event(ev_done[i % 2])
        with torch.cuda.stream(s_d2h):
            op[i % 2].copy_(b["o"], non_blocking=True)
            lp[i % 2].copy_(b["l"], non_blocking=True)
            ev_free[i % 2].record(s_d2h)

    for i in range(max(1, min(args.warmup, 3))):
        e2e_step(i)
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_d2h)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    st, detail = ea.attn_fwd_device_status()
    if st != ea.ATTN_OK:
        raise RuntimeError(f"device wait timed out in the end-to-end loop (code {detail:#x})")
    h2d = 3 * q_h.numel() * 2
    d2h = q_h.numel() * 2 + w.B * w.H * w.N * 4

    # ---- max over ranks
    ms, e2e_ms = reduce_max_over_ranks([ms, e2e_ms], dev)

    if rank == 0:
        peaks, peak_src = load_peaks()
        achieved = flops / (ms * 1e-3) / 1e12
        traffic = load_traffic(args.workload, causal)
        line = {
            "metric": METRIC,
            "value": whole_job_tflops(flops, ws, ms),
            "unit": "TFLOP/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.describe(causal), "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": causal, "scale": w.scale,
                       "l2": "inputs larger than L2 (3 x %d MiB bf16), no flush" % (
                           q_h.numel() * 2 >> 20),
                       "parallelism": f"replicas x{ws} (independent batches, no collective)",
                       "kv_splits": splits},
            "pct_of_bf16_peak": 100.0 * achieved / peaks["bf16_tflops"],
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                         "traffic": traffic, "peak_source": f"{peak_src} bf16 burst",
                         "kernel": f"attn_fwd_kernel<{w.d},{str(causal).lower()}>"},
            "clocks": clocks,
            "e2e": {"value": whole_job_tflops(flops, ws, e2e_ms), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps": e2e_steps,
                    "how": "pinned host buffers; H2D, kernel and D2H on three streams, "
                           "double-buffered across steps"},
            "gpu_launches": args.steps * (2 if splits > 1 else 1),
        }
        if ws == 1 and not args.no_cpu_baseline:
            tf, secs, nrows, cores = time_oracle(w, causal, q_h, k_h, v_h, args.cpu_seconds, 99)
            line["cpu_baseline"] = {
                "value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                "sample": f"{nrows} seeded random rows of {w.describe(causal)} "
                          f"({secs:.1f} s of fp64 oracle work)"}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--causal", choices=["default", "0", "1"], default="default")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--splits", type=int, default=1,
                    help="1: attn_fwd; >1: attn_fwd_splitkv with that many key splits; "
                         "0: attn_fwd_splitkv with its default split count")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = wl.WORKLOADS[args.workload]
    causal = w.causal[-1] if args.causal == "default" else args.causal == "1"
    if args.impl == "reference":
        return run_reference(args, w, causal)
    return run_ours(args, w, causal)


if __name__ == "__main__":
    sys.exit(main())
