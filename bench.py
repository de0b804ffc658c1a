"""Benchmark of the fused attention forward (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole path (one attn_fwd launch) over one batch of the
workload; the default workload is the causal B=2 H=32 N=8192 d=128 forward, the
configuration the throughput target is stated on.  Inputs are synthetic (seeded
generator), resident in HBM before the timed region, and larger than L2
(Q, K, V, O and LSE come to 537 MB per step), so no L2 flush is needed.

Metric: algorithmic TFLOP/s = 4*B*H*Nq*Nk*d (halved for causal; valid keys only
with key padding) per step / device time per step, summed over ranks.
Under torchrun each rank runs its own copy of the workload (weak scaling, no
collective on the data path); the barrier and the max-over-ranks time remain.

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample
of the same workload (rows computed one by one), on the same metric.
"""
from __future__ import annotations

import argparse
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
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16, d=128) and % of GB300 BF16 tensor peak"
DEFAULT_WORKLOAD = "causal_b2h32n8192d128"
FALLBACK_PEAK_TFLOPS = 1900.0
KERNEL_SOURCES = ["attn_fwd_kernel.cuh", "ptx.cuh", "attn_api.cu"]


def algorithmic_flops(B, H, Nq, Nk, d, causal, lens=None) -> float:
    """4*B*H*Nq*Nk*d, halved for causal; with key padding only valid keys count."""
    if lens is not None:
        nk = float(sum(min(max(int(L), 0), Nk) for L in lens))
        f = 4.0 * H * Nq * nk * d
    else:
        f = 4.0 * B * H * Nq * Nk * d
    return f / 2.0 if causal else f


def row_flops(i, Nq, Nk, d, causal, L) -> float:
    """Algorithmic flops of query row i: 4 * d * (visible keys)."""
    lim = L if not causal else min(L, i + Nk - Nq + 1)
    return 4.0 * d * max(lim, 0)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "online_softmax_flashattention_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured burst (MEASURED_PEAKS.json bf16_tflops)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_PEAK_TFLOPS, "fallback"


def load_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return float(e["dram_bytes_per_launch"])


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.perf_counter())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(t=t, sm=float(parts[1]), sm_max=float(parts[2]),
                                 reasons=dict(active=parts[4], hw_slowdown=parts[5], hw_thermal_slowdown=parts[6],
                                              sw_thermal_slowdown=parts[7], sw_power_cap=parts[8])))
            except ValueError:
                continue
        inside = [r for r in rows if self.t_start is not None and self.t_start <= r["t"] <= (self.t_stop or 1e30)]
        used = inside if len(inside) >= 2 else rows
        if not used:
            return None
        reasons = sorted({k for r in used for k, v in r["reasons"].items() if k != "active" and v == "Active"})
        return dict(sm_mhz=statistics.median(r["sm"] for r in used), sm_max_mhz=max(r["sm_max"] for r in used),
                    reasons=reasons, samples=len(used), window="timed region" if used is inside else "whole run")


# ------------------------------------------------------------------ CPU oracle (baseline and reference arm)

def _oracle_worker_init(name):
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    _oracle_inputs(name)  # input generation is not part of the measured oracle time


def _oracle_rows_job(args):
    name, picks = args
    import gen
    import oracle
    x = _oracle_inputs(name)
    t0 = time.perf_counter()
    oracle.attention_rows(x["Q"], x["K"], x["V"], x["scale"], x["causal"], x["lens"], picks)
    return time.perf_counter() - t0


_INPUT_CACHE = {}


def _oracle_inputs(name):
    if name not in _INPUT_CACHE:
        import gen
        _INPUT_CACHE[name] = gen.make_inputs(name)
    return _INPUT_CACHE[name]


class OraclePool:
    """The fp64 oracle on every host core: a spawn pool with one single-threaded worker per core."""

    def __init__(self, name: str, cores: int):
        import multiprocessing as mp
        self.name = name
        self.cores = cores
        self.pool = mp.get_context("spawn").Pool(cores, initializer=_oracle_worker_init, initargs=(name,))
        self.pool.map(_oracle_rows_job, [(name, [])] * cores, chunksize=1)

    def step(self, picks_per_worker):
        t0 = time.perf_counter()
        self.pool.map(_oracle_rows_job, [(self.name, p) for p in picks_per_worker], chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def sample_picks(w, n_rows, rng):
    import numpy as np  # noqa: F401
    picks = []
    for _ in range(n_rows):
        picks.append((int(rng.integers(w["B"])), int(rng.integers(w["H"])), int(rng.integers(w["Nq"]))))
    return picks


def picks_flops(w, picks, lens):
    Nk = w["Nk"]
    total = 0.0
    for b, h, i in picks:
        L = Nk if lens is None else min(max(int(lens[b]), 0), Nk)
        total += row_flops(i, w["Nq"], Nk, w["d"], w["causal"], L)
    return total


def run_oracle_sample(name, cores, rows_per_worker, steps, seed=1234, budget_s=None):
    """Time `steps` steps, each of cores x rows_per_worker oracle rows; returns (TFLOP/s, seconds, rows)."""
    import numpy as np
    import gen
    w = gen.WORKLOADS[name]
    lens = gen.make_lens(w)
    rng = np.random.default_rng(seed)
    pool = OraclePool(name, cores)
    try:
        flops = secs = 0.0
        rows = 0
        done = 0
        while done < steps:
            per = [sample_picks(w, rows_per_worker, rng) for _ in range(cores)]
            secs += pool.step(per)
            flops += sum(picks_flops(w, p, lens) for p in per)
            rows += cores * rows_per_worker
            done += 1
            if budget_s is not None and secs >= budget_s:
                break
    finally:
        pool.close()
    return flops / secs / 1e12, secs, rows, done


# ------------------------------------------------------------------ main

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=800)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def config_of(w, lens, world):
    return {"workload": w["name"], "B": w["B"], "H": w["H"], "Nq": w["Nq"], "Nk": w["Nk"], "d": w["d"],
            "causal": w["causal"], "key_padding": None if lens is None else [int(x) for x in lens],
            "layout": "[B,H,N,d] bf16, O bf16, LSE fp32",
            "l2": "no flush: inputs and outputs larger than L2 (537 MB per step vs 129 MB L2)"
            if w["name"] == DEFAULT_WORKLOAD else "no flush",
            "parallelism": f"replicas x{world} (each rank its own problem)"}


def reference_arm(args, w, lens, world, rank):
    if rank != 0:
        return
    cores = host_cores()
    rows_per_worker = 2
    t0 = time.perf_counter()
    # warm-up steps (untimed)
    if args.warmup > 0:
        run_oracle_sample(w["name"], cores, rows_per_worker, max(1, min(args.warmup, 3)), seed=99)
    value, secs, rows, done = run_oracle_sample(w["name"], cores, rows_per_worker, args.steps, seed=1234,
                                                budget_s=180.0)
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": world,
           "steps": done, "warmup": args.warmup, "ms_per_step": secs / max(done, 1) * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": config_of(w, lens, world),
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                            "sample": f"{rows} query rows drawn uniformly over (b, h, i), {rows_per_worker} per "
                                      f"worker per step, each computed alone by oracle.attention_rows in float64"},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "wall_s": time.perf_counter() - t0}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    world, rank, local = dist_env()
    import gen
    w = gen.WORKLOADS[args.workload]
    lens = gen.make_lens(w)
    if args.impl == "reference":
        reference_arm(args, w, lens, world, rank)
        return

    import numpy as np
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    from online_softmax_flashattention_attention_gb300 import build as pkgbuild

    pkgbuild.build_library()
    pkg.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    # CPU baseline pool first (spawned before any GPU work), rank 0 at N = 1 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        value, secs, rows, done = run_oracle_sample(w["name"], cores, 4, 10 ** 6, seed=4321, budget_s=15.0)
        cpu = {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{rows} query rows of {w['name']} drawn uniformly over (b, h, i), computed one by one "
                         f"by oracle.attention_rows in float64 on {cores} single-threaded worker processes "
                         f"({secs:.1f} s)"}

    x = gen.make_inputs(w)
    B, H, Nq, Nk, d = x["B"], x["H"], x["Nq"], x["Nk"], x["d"]
    scale, causal = x["scale"], x["causal"]

    def dev_tensor(codes):
        return torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(dev)

    Q, K, V = dev_tensor(x["Q"]), dev_tensor(x["K"]), dev_tensor(x["V"])
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    lt = None if lens is None else torch.as_tensor(lens, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flops = algorithmic_flops(B, H, Nq, Nk, d, causal, lens)

    def step():
        pkg.attn_fwd(Q, K, V, O, LSE, scale=scale, causal=causal, key_padding_lens=lt, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    pkg.status_sync(stream)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler.mark("t_start")
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark("t_stop")
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    pkg.status_sync(stream)
    ms_total = ev0.elapsed_time(ev1)
    if pg:
        t = torch.tensor([ms_total], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_step = ms_total / args.steps
    value = world * flops / (ms_step * 1e-3) / 1e12
    per_launch_tflops = flops / (ms_step * 1e-3) / 1e12

    # ---- end to end through the host-buffer C entry point (pinned host memory)
    e2e = None
    if args.e2e_steps > 0:
        def pinned(codes):
            return torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).pin_memory()

        Qh, Kh, Vh = pinned(x["Q"]), pinned(x["K"]), pinned(x["V"])
        Oh = torch.empty_like(Qh).pin_memory()
        Lh = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
        lh = None if lens is None else torch.as_tensor(lens, dtype=torch.int32)
        for _ in range(2):
            pkg.attn_fwd_host(Qh, Kh, Vh, Oh, Lh, scale=scale, causal=causal, key_padding_lens=lh, stream=stream)
        if pg:
            pg.barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            pkg.attn_fwd_host(Qh, Kh, Vh, Oh, Lh, scale=scale, causal=causal, key_padding_lens=lh, stream=stream)
        e2e_s = (time.perf_counter() - t0) / args.e2e_steps
        if pg:
            t = torch.tensor([e2e_s], device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            e2e_s = float(t.item())
        h2d = Qh.numel() * 2 + Kh.numel() * 2 + Vh.numel() * 2 + (0 if lh is None else lh.numel() * 4)
        d2h = Oh.numel() * 2 + Lh.numel() * 4
        e2e = {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
               "api": "attn_fwd_host (C ABI, pinned host buffers, copies inside the timed region)"}

    peak, peak_src = load_peaks()
    traffic = load_traffic(w["name"])
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": config_of(w, lens, world),
           "roofline": {"bound": "tensor", "achieved": per_launch_tflops, "peak": peak, "unit": "TFLOP/s",
                        "frac": per_launch_tflops / peak, "traffic": traffic,
                        "kernel": f"attn_fwd_kernel<{d}>", "peak_source": peak_src,
                        "flops_per_launch": flops},
           "e2e": e2e,
           "gpu_launches": args.steps,
           "clocks": clocks,
           "cpu_baseline": cpu}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
