"""Benchmark of the fused attention forward (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                    [--path fused|splitkv]

A step is one pass of the whole path (one attn_fwd launch) over one batch of the
workload; the default workload is the causal B=2 H=32 N=8192 d=128 forward, the
configuration the throughput target is stated on.  Inputs are synthetic (seeded
generator), resident in HBM before the timed region, and larger than L2
(Q, K, V, O and LSE come to 537 MB per step), so no L2 flush is needed.

Metric: algorithmic TFLOP/s = 4*B*H*Nq*Nk*d (halved for causal; valid keys only
with key padding) per step / device time per step, summed over ranks.
Under torchrun each rank runs its own copy of the workload (weak scaling, no
collective on the data path); the barrier and the max-over-ranks time remain.

--path splitkv times the split-KV route instead (attn_fwd_states over the automatic
split count, then attn_merge_states: two launches per step), the route for shapes
with few query tiles such as causal_b1h32q128k32768d128.

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample
of the same workload (rows computed one by one), on the same metric.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
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
FALLBACK_PEAK_GBS = 6800.0
KERNEL_SOURCES = ["attn_fwd_kernel.cuh", "attn_fwd_pair_kernel.cuh", "ptx.cuh", "attn_api.cu", "attn_merge_kernel.cuh"]


def algorithmic_flops(B, H, Nq, Nk, d, causal, lens=None) -> float:
    """4*B*H*Nq*Nk*d, halved for causal; with key padding only valid keys count.  For a
    causal problem with Nq != Nk (bottom-right aligned) the visible pairs are counted
    exactly: row i sees min(L, i + Nk - Nq + 1) keys."""
    if causal and Nq != Nk:
        Ls = [Nk] * B if lens is None else [min(max(int(L), 0), Nk) for L in lens]
        pairs = 0
        for L in Ls:
            lim = min(L, Nk - Nq + 1)          # row 0's limit; it grows by one per row up to L
            for i in range(Nq):
                pairs += max(min(L, lim + i), 0)
        return 4.0 * H * pairs * d
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
    """Identifies the kernel code a profile was taken on: the sources with comments and
    blank lines removed, so editing a comment does not void a recorded profile."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "online_softmax_flashattention_attention_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured burst (MEASURED_PEAKS.json bf16_tflops)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_PEAK_TFLOPS, "fallback"


def load_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured copy (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_PEAK_GBS, "fallback"


def algorithmic_bytes(B, H, Nq, Nk, d, lens=None, splits=0) -> float:
    """Bytes the kernel must move at least: Q, and K and V of the valid keys, read once;
    O (bf16) and LSE (fp32) written once -- or, for the partial-state kernel (splits > 0),
    the states o~ (fp32 d-vector), m and l of every (split, row) written instead."""
    nk = B * Nk if lens is None else sum(min(max(int(L), 0), Nk) for L in lens)
    read = 2.0 * H * d * (B * Nq + 2 * nk)
    write = (2.0 * d + 4) * B * H * Nq if splits == 0 else (4.0 * d + 8) * splits * B * H * Nq
    return read + write


def fused_kernel_name(B, H, Nq, d, sms, causal=True):
    """The kernel the library runs for a forward with O and LSE out: at d = 64, two query
    tiles per CTA once the pairs of tiles are at least as many as the SMs (causal) or more
    than half of them (no causal mask) (attn_api.cu, use_pair_kernel), else one tile per
    CTA."""
    pairs = B * H * ((-(-Nq // 128) + 1) // 2)
    if d == 64 and (pairs >= sms if causal else 2 * pairs > sms):
        return "attn_fwd_pair_kernel (d = 64, two query tiles per CTA)"
    return f"attn_fwd_kernel<{d}>"


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


# ------------------------------------------------------------------ NUMA placement of pinned buffers

def _cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        a, _, b = part.partition("-")
        cpus.update(range(int(a), int(b or a) + 1))
    return cpus


def gpu_numa(dev_index):
    """(node the GPU's PCI function reports, CPUs of that node) from sysfs, or (None, None)."""
    import torch
    try:
        p = torch.cuda.get_device_properties(dev_index)
        bdf = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bdf}/numa_node") as f:
            node = int(f.read().strip())
        if node < 0:
            return None, None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            return node, _cpulist(f.read())
    except (OSError, ValueError, AttributeError):
        return None, None


def pages_nodes(addr, nbytes):
    """NUMA nodes (and page counts) of the mapping holding [addr, addr + nbytes), read from
    /proc/self/numa_maps and /proc/self/maps; None if not found."""
    try:
        spans = {}
        with open("/proc/self/maps") as f:
            for ln in f:
                lo, hi = (int(x, 16) for x in ln.split()[0].split("-"))
                spans[lo] = hi
        with open("/proc/self/numa_maps") as f:
            for ln in f:
                parts = ln.split()
                lo = int(parts[0], 16)
                hi = spans.get(lo)
                if hi is None or not (lo <= addr < hi):
                    continue
                nodes = {}
                for tok in parts[1:]:
                    if tok.startswith("N") and "=" in tok:
                        k, v = tok[1:].split("=")
                        nodes[int(k)] = int(v)
                return nodes
    except (OSError, ValueError):
        return None
    return None


class near_gpu:
    """Run the body with this thread bound to the CPUs of the GPU's NUMA node (those the
    process may use), so that host memory pinned meanwhile is placed on that node."""

    def __init__(self, cpus):
        self.cpus = cpus
        self.saved = None

    def __enter__(self):
        try:
            allowed = os.sched_getaffinity(0)
            use = (self.cpus or set()) & allowed
            if use and use != allowed:
                self.saved = allowed
                os.sched_setaffinity(0, use)
        except (OSError, AttributeError):
            self.saved = None
        return self

    def __exit__(self, *exc):
        if self.saved:
            os.sched_setaffinity(0, self.saved)
        return False


def h2d_rate(host, devt, stream, reps=3):
    """GB/s of one pinned host -> device copy of `host` into `devt` (best of reps)."""
    import torch
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            devt.copy_(host, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    return host.numel() * host.element_size() / (best * 1e-3) / 1e9


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
    ap.add_argument("--no-variants", action="store_true", help="skip timing the lazy-rescale option")
    ap.add_argument("--path", choices=["fused", "splitkv"], default="fused")
    ap.add_argument("--layout", choices=["bhsd", "bshd", "varlen"], default="bhsd")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workloads of the sweep after the headline one")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def roofline_entry(intensity, ridge, tflops, peak, peak_src, kbytes, ms_kernel, hbm_peak, hbm_src, traffic, flops,
                   kernel):
    """The dominant kernel against the roof that bounds it: the tensor core when its
    arithmetic intensity (algorithmic flops / algorithmic bytes) is above the ridge of
    the measured peaks, HBM bandwidth below it."""
    common = {"traffic": traffic, "kernel": kernel, "kernel_ms": ms_kernel, "flops_per_launch": flops,
              "bytes_per_launch": kbytes, "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge}
    if intensity >= ridge:
        return {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                "peak_source": peak_src, **common}
    gbs = kbytes / (ms_kernel * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
            "peak_source": hbm_src, "tflops": tflops, **common}


def l2_note(w):
    mb = (2 * w["B"] * w["H"] * (2 * w["Nq"] + 2 * w["Nk"]) * w["d"] + 4 * w["B"] * w["H"] * w["Nq"]) / 1e6
    if mb > 129:
        return f"no flush: inputs and outputs larger than L2 ({mb:.0f} MB per step vs 129 MB L2)"
    return f"no flush: working set {mb:.1f} MB fits in the 129 MB L2 (repeated steps hit L2)"


def config_of(w, lens, world, path="fused", splits=1, layout="bhsd"):
    return {"workload": w["name"], "path": path if path == "fused" else f"splitkv (S={splits} + merge)",
            "tensor_layout": {"bhsd": "[B,H,N,d] contiguous", "bshd": "[B,N,H,d] via attn_fwd_strided"}[layout], "B": w["B"], "H": w["H"], "Nq": w["Nq"], "Nk": w["Nk"], "d": w["d"],
            "causal": w["causal"], "key_padding": None if lens is None else [int(x) for x in lens],
            "layout": "[B,H,N,d] bf16, O bf16, LSE fp32",
            "l2": l2_note(w),
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


def max_over_ranks(x: float, pg, device) -> float:
    """The largest value of x over the ranks of the process group (x itself without one):
    the job's time is its slowest rank's."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_rank: float, seconds: float) -> float:
    """Whole-job TFLOP/s: every rank ran its own copy of the workload (weak scaling), and the
    job took as long as its slowest rank."""
    return world * flops_per_rank / seconds / 1e12


def timed_region(step, steps, stream, dev, pg, local, kernel_events=False):
    """Time exactly `steps` calls of step() on `stream`, bracketed by a barrier and a
    device synchronisation on both sides, with nvidia-smi clocks sampled meanwhile.
    Returns (ms per step (max over ranks), ms of the dominant kernel per step, clocks).
    With kernel_events, step(evs) records evs[0] / evs[1] around its dominant kernel."""
    import torch
    kev = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
           if kernel_events else None)
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
        for i in range(steps):
            step(kev[i] if kev else None)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark("t_stop")
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), pg, dev)
    ms_step = ms_total / steps
    ms_kernel = ms_step if not kev else sum(a.elapsed_time(b) for a, b in kev) / steps
    return ms_step, ms_kernel, clocks


def e2e_region(e2e_step, steps, dev, pg):
    """Wall time per call of e2e_step() (which copies in, computes, copies out and
    synchronises), max over ranks."""
    import torch
    for _ in range(2):
        e2e_step()
    if pg:
        pg.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        e2e_step()
    return max_over_ranks((time.perf_counter() - t0) / steps, pg, dev)


def copy_e2e_step(stream, ins, step, outs):
    """One end-to-end step through device buffers: pinned host -> device copies, the
    step, device -> pinned host copies, then a synchronisation of the stream."""
    import torch

    def run():
        with torch.cuda.stream(stream):
            for host, devt in ins:
                devt.copy_(host, non_blocking=True)
            step()
            for host, devt in outs:
                host.copy_(devt, non_blocking=True)
        stream.synchronize()
    return run


# The workloads besides the headline one whose throughput the default run reports in its
# `configs` object, each timed on its own inputs after the headline workload.
SWEEP = ["b1h2n256d64", "causal_b4h16n2048d128", "padded_planted_b2h8n4096d128", "causal_b1h32n32768d128",
         "causal_b1h32n32768d64"]


def config_sweep(names, lib, pkg, stream, dev, pg, local, world, target_s=0.25):
    """Time one attn_fwd per step on each named workload (inputs resident, CUDA events on
    the launching stream, clocks sampled during each timed region); about target_s of
    timed work per workload."""
    import numpy as np
    import torch
    import gen
    peak, _ = load_peaks()
    hbm_peak, _ = load_hbm_peak()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {}
    for name in names:
        x = gen.make_inputs(name)
        B, H, Nq, Nk, d = x["B"], x["H"], x["Nq"], x["Nk"], x["d"]
        lens = x["lens"]
        dt = lambda c: torch.from_numpy(c.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
        Q, K, V = dt(x["Q"]), dt(x["K"]), dt(x["V"])
        O = torch.empty_like(Q)
        LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
        lt = None if lens is None else torch.as_tensor(lens, dtype=torch.int32, device=dev)
        sh = ctypes.c_void_p(stream.cuda_stream)
        a = (Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H, Nq, Nk, d, x["scale"],
             int(x["causal"]), None if lt is None else lt.data_ptr(), sh)

        def step(evs=None):
            rc = lib.attn_fwd(*a)
            if rc != 0:
                raise pkg.AttnError(rc, lib.attn_last_error().decode())
        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
        pkg.status_sync(stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(5):
                step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        est_ms = max(e0.elapsed_time(e1) / 5, 1e-3)
        steps = int(min(5000, max(20, target_s * 1e3 / est_ms)))
        ms, _, clocks = timed_region(step, steps, stream, dev, pg, local)
        pkg.status_sync(stream)
        flops = algorithmic_flops(B, H, Nq, Nk, d, x["causal"], lens)
        kbytes = algorithmic_bytes(B, H, Nq, Nk, d, lens)
        tflops = world * flops / (ms * 1e-3) / 1e12
        entry = {"ms_per_step": ms, "tflops": tflops, "frac": flops / (ms * 1e-3) / 1e12 / peak,
                 "achieved_gbs": kbytes / (ms * 1e-3) / 1e9, "hbm_frac": kbytes / (ms * 1e-3) / 1e9 / hbm_peak,
                 "steps": steps, "kernel": fused_kernel_name(B, H, Nq, d, sms, x["causal"]),
                 "flops_per_step": flops, "bytes_per_step": kbytes, "clocks": clocks,
                 "shape": {"B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d, "causal": x["causal"],
                           "key_padding": None if lens is None else [int(v) for v in lens]}}
        if lens is not None:
            entry["nominal_tflops"] = tflops * algorithmic_flops(B, H, Nq, Nk, d, x["causal"]) / flops
        out[name] = entry
        del Q, K, V, O, LSE, lt
        torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    world, rank, local = dist_env()
    import gen
    if args.layout == "varlen":
        return main_varlen(args, world, rank, local)
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
    lib = pkg.load_library()
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

    # the blocked CPU library on a sample of whole heads (host only, before any GPU work)
    cpu_blocked = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from online_softmax_flashattention_attention_gb300 import build as pkgb
        pkgb.build_cpu_library()
        per_head = algorithmic_flops(B, 1, Nq, Nk, d, causal, lens)
        hs = max(1, min(H, int(round(400e9 / max(per_head, 1.0)))))
        sub = [np.ascontiguousarray(x[t][:, :hs]) for t in ("Q", "K", "V")]
        pkg.attn_fwd_cpu(*[a[:, :1, :min(Nq, 256)] for a in sub], scale=scale)   # load + warm the library
        t0 = time.perf_counter()
        pkg.attn_fwd_cpu(*sub, scale=scale, causal=causal, key_padding_lens=lens)
        secs = time.perf_counter() - t0
        cpu_blocked = {"value": per_head * hs / secs / 1e12, "unit": "TFLOP/s", "cores": host_cores(),
                       "kind": "blocked C library (libattn_cpu.so, fp32, one thread per core)",
                       "sample": f"all rows of heads 0..{hs - 1} of every batch of {w['name']} ({secs:.2f} s)"}

    def dev_tensor(codes):
        return torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(dev)

    def pinned(codes):
        return torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).pin_memory()

    Q, K, V = dev_tensor(x["Q"]), dev_tensor(x["K"]), dev_tensor(x["V"])
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    lt = None if lens is None else torch.as_tensor(lens, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    lens_ptr = None if lt is None else lt.data_ptr()
    flops = algorithmic_flops(B, H, Nq, Nk, d, causal, lens)

    def check(rc):
        if rc != 0:
            raise pkg.AttnError(rc, lib.attn_last_error().decode())

    splits = 1
    kernel_events = False
    e2e_api = None
    if args.path == "splitkv":
        splits = pkg.splitkv_splits(B, H, Nq, Nk)
        launches_per_step = 2
        kernel_events = True
        o_st = torch.empty((splits, B, H, Nq, d), dtype=torch.float32, device=dev)
        m_st = torch.empty((splits, B, H, Nq), dtype=torch.float32, device=dev)
        l_st = torch.empty((splits, B, H, Nq), dtype=torch.float32, device=dev)
        st_args = (Q.data_ptr(), K.data_ptr(), V.data_ptr(), o_st.data_ptr(), m_st.data_ptr(), l_st.data_ptr(), B,
                   H, Nq, Nk, d, scale, int(causal), lens_ptr, splits, sh)
        mg_args = (o_st.data_ptr(), m_st.data_ptr(), l_st.data_ptr(), splits, B * H * Nq, d, O.data_ptr(),
                   LSE.data_ptr(), sh)

        def step(evs=None):
            if evs:
                evs[0].record(stream)
            check(lib.attn_fwd_states(*st_args))
            if evs:
                evs[1].record(stream)
            check(lib.attn_merge_states(*mg_args))
        e2e_api = "attn_fwd_states + attn_merge_states (C ABI) with pinned host copies inside the timed region"
    elif args.layout == "bshd":
        # the same values stored [B, N, H, d]; the tensors handed over are [B, H, N, d] views
        launches_per_step = 1
        Q, K, V = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (Q, K, V))
        O = torch.empty((B, Nq, H, d), dtype=torch.bfloat16, device=dev).transpose(1, 2)
        strides = [(ctypes.c_int64 * 3)(*t.stride()[:3]) for t in (Q, K, V, O)]
        sd_args = (Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H, Nq, Nk, d, scale,
                   int(causal), lens_ptr, *strides, sh)

        def step(evs=None):
            check(lib.attn_fwd_strided(*sd_args))
        e2e_api = "attn_fwd_strided (C ABI, [B, N, H, d] tensors) with pinned host copies inside the timed region"
    else:
        launches_per_step = 1
        fwd_args = (Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), B, H, Nq, Nk, d, scale,
                    int(causal), lens_ptr, sh)

        def step(evs=None):
            check(lib.attn_fwd(*fwd_args))

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    pkg.status_sync(stream)
    ms_step, ms_kernel, clocks = timed_region(step, args.steps, stream, dev, pg, local, kernel_events)
    pkg.status_sync(stream)
    value = job_throughput(world, flops, ms_step * 1e-3)
    per_launch_tflops = flops / (ms_kernel * 1e-3) / 1e12

    # the lazy-rescale option on the same inputs (not the headline: the pages' rule is)
    variants = None
    if args.path == "fused" and args.layout == "bhsd" and not args.no_variants:
        opts = pkg.AttnOptions(ctypes.sizeof(pkg.AttnOptions), 5.5, pkg.EXP2_HARDWARE)

        def lazy_step(evs=None):
            check(lib.attn_fwd_ex(*fwd_args[:-1], ctypes.byref(opts), sh))
        with torch.cuda.stream(stream):
            for _ in range(3):
                lazy_step()
        n_lazy = max(3, args.steps // 4)
        ms_lazy, _, _ = timed_region(lazy_step, n_lazy, stream, dev, pg, local)
        pkg.status_sync(stream)
        variants = {"lazy_rescale_threshold_5.5": {
            "value": world * flops / (ms_lazy * 1e-3) / 1e12, "unit": "TFLOP/s", "steps": n_lazy,
            "frac_of_peak": flops / (ms_lazy * 1e-3) / 1e12 / load_peaks()[0],
            "note": "attn_fwd_ex with rescale_threshold 5.5: the running max moves only when a block max passes it "
                    "by more than 5.5 (natural log); an option, not the pages' rule"}}
    # ---- end to end: pinned host buffers, copies in and out inside the timed region
    e2e = None
    if args.e2e_steps > 0:
        numa = None
        if e2e_api is None:  # the host-buffer C entry point does the copies itself
            # Where pinned buffers land and what that does to the host-to-device rate: one
            # copy of Q pinned under the process's default placement, then the buffers the
            # e2e steps use, pinned with this thread bound to the GPU's NUMA node.
            node, node_cpus = gpu_numa(local)
            Qd = pinned(x["Q"])
            numa = {"gpu_numa_node": node, "process_cpus": len(os.sched_getaffinity(0)),
                    "gpu_node_cpus_usable": len((node_cpus or set()) & os.sched_getaffinity(0)),
                    "default_pinned_pages_by_node": pages_nodes(Qd.data_ptr(), Qd.numel() * 2),
                    "default_h2d_gbs": h2d_rate(Qd, Q, stream)}
            with near_gpu(node_cpus):
                Qh, Kh, Vh = pinned(x["Q"]), pinned(x["K"]), pinned(x["V"])
                Oh = torch.empty_like(Qh).pin_memory()
                Lh = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
            numa.update({"e2e_pinned_pages_by_node": pages_nodes(Qh.data_ptr(), Qh.numel() * 2),
                         "e2e_h2d_gbs": h2d_rate(Qh, Q, stream),
                         "note": "e2e buffers pinned with the allocating thread bound to the GPU's NUMA node "
                                 "(when the process may use its CPUs); rates are one Q-sized pinned copy"})
            del Qd
            lh = None if lens is None else torch.as_tensor(lens, dtype=torch.int32)

            def e2e_step():
                pkg.attn_fwd_host(Qh, Kh, Vh, Oh, Lh, scale=scale, causal=causal, key_padding_lens=lh, stream=stream)
            e2e_api = "attn_fwd_host (C ABI, pinned host buffers, copies inside the timed region)"
            h2d = (Qh.numel() + Kh.numel() + Vh.numel()) * 2 + (0 if lh is None else lh.numel() * 4)
        else:
            # host buffers with the device tensors' strides: every copy is one plain memcpy
            hosts = [torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, pin_memory=True) for t in (Q, K, V)]
            for hst, t in zip(hosts, (Q, K, V)):
                hst.copy_(t.cpu())
            Oh = torch.empty_strided(O.shape, O.stride(), dtype=O.dtype, pin_memory=True)
            Lh = torch.empty(LSE.shape, dtype=LSE.dtype).pin_memory()
            e2e_step = copy_e2e_step(stream, list(zip(hosts, (Q, K, V))), step, [(Oh, O), (Lh, LSE)])
            h2d = sum(h.numel() for h in hosts) * 2
        e2e_s = e2e_region(e2e_step, args.e2e_steps, dev, pg)
        e2e = {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": Oh.numel() * 2 + Lh.numel() * 4, "ms_per_step": e2e_s * 1e3, "api": e2e_api,
               "numa": numa}

    # the other workloads of the sweep, each on its own inputs, after the headline one
    configs = None
    if (args.path == "fused" and args.layout == "bhsd" and w["name"] == DEFAULT_WORKLOAD and not args.no_configs):
        configs = config_sweep([n for n in SWEEP if n != w["name"]], lib, pkg, stream, dev, pg, local, world)

    peak, peak_src = load_peaks()
    hbm_peak, hbm_src = load_hbm_peak()
    kbytes = algorithmic_bytes(B, H, Nq, Nk, d, lens, 0 if args.path == "fused" else splits)
    intensity = flops / kbytes
    ridge = peak * 1e12 / (hbm_peak * 1e9)
    key = w["name"] + ("" if args.path == "fused" else ":splitkv") + ("" if args.layout == "bhsd" else ":" + args.layout)
    traffic = load_traffic(key)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    kname = (fused_kernel_name(B, H, Nq, d, sms, causal) if args.path == "fused"
             else f"attn_fwd_kernel<{d}> (states)")
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": config_of(w, lens, world, args.path, splits, args.layout),
           "roofline": roofline_entry(intensity, ridge, per_launch_tflops, peak, peak_src, kbytes, ms_kernel,
                                      hbm_peak, hbm_src, traffic, flops, kname),
           "e2e": e2e,
           "gpu_launches": args.steps * launches_per_step,
           "clocks": clocks,
           "cpu_baseline": cpu,
           "cpu_blocked": cpu_blocked,
           "variants": variants,
           "configs": configs}
    if lens is not None:  # key padding: `value` counts the valid keys; the nominal count beside it
        nominal = algorithmic_flops(B, H, Nq, Nk, d, causal)
        out["nominal"] = {"value": value * nominal / flops if flops > 0 else None, "unit": "TFLOP/s",
                          "flops_per_step": nominal, "flops_per_step_valid_keys": flops,
                          "note": "4 B H Nq Nk d (halved when causal): every key counted as if unpadded; "
                                  "the line's value counts only the keys the padding leaves visible"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def main_varlen(args, world, rank, local):
    """--layout varlen: a packed workload of sequences of different lengths through
    attn_fwd_varlen.  Flops count every sequence's causal triangle as n^2 / 2."""
    import gen
    import numpy as np
    import torch
    import online_softmax_flashattention_attention_gb300 as pkg
    from online_softmax_flashattention_attention_gb300 import build as pkgbuild

    name = args.workload if args.workload in gen.VARLEN_WORKLOADS else "varlen_causal_b16h16d128"
    x = gen.make_varlen(name)
    B, H, d, total = x["B"], x["H"], x["d"], x["total"]
    lengths = [int(n) for n in x["lengths"]]
    causal, scale = x["causal"], x["scale"]
    pairs = sum(n * n / 2.0 if causal else float(n * n) for n in lengths)
    flops = 4.0 * H * d * pairs
    config = {"workload": name, "layout": "packed [total, H, d] bf16, LSE [H, total] fp32", "B": B, "H": H, "d": d,
              "causal": causal, "lengths": lengths, "total_rows": total,
              "l2": f"no flush: inputs and outputs larger than L2 ({(4 * total * H * d * 2 + 4 * H * total) / 1e6:.0f}"
                    " MB per step vs 129 MB L2)",
              "parallelism": f"replicas x{world} (each rank its own problem)"}
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the oracle arm runs on the dense workloads; "
                              "packed sequences are timed against the dense route of the same library only"}))
        return
    pkgbuild.build_library()
    lib = pkg.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    to_dev = lambda c: torch.from_numpy(c.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    Q, K, V = to_dev(x["Q"]), to_dev(x["K"]), to_dev(x["V"])
    O = torch.empty_like(Q)
    LSE = torch.empty((H, total), dtype=torch.float32, device=dev)
    cu = torch.as_tensor(x["cu"], dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    args_v = (Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(), cu.data_ptr(), cu.data_ptr(),
              B, H, max(lengths), total, total, d, scale, int(causal), sh)

    def step(evs=None):
        rc = lib.attn_fwd_varlen(*args_v)
        if rc != 0:
            raise pkg.AttnError(rc, lib.attn_last_error().decode())

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    pkg.status_sync(stream)
    ms_step, ms_kernel, clocks = timed_region(step, args.steps, stream, dev, pg, local)
    pkg.status_sync(stream)
    tflops = flops / (ms_step * 1e-3) / 1e12
    e2e = None
    if args.e2e_steps > 0:
        hosts = [torch.from_numpy(c.view(np.int16)).view(torch.bfloat16).pin_memory() for c in (x["Q"], x["K"], x["V"])]
        Oh = torch.empty(O.shape, dtype=O.dtype).pin_memory()
        Lh = torch.empty(LSE.shape, dtype=LSE.dtype).pin_memory()
        e2e_s = e2e_region(copy_e2e_step(stream, list(zip(hosts, (Q, K, V))), step, [(Oh, O), (Lh, LSE)]),
                           args.e2e_steps, dev, pg)
        e2e = {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(h.numel() for h in hosts) * 2,
               "d2h_bytes_per_step": Oh.numel() * 2 + Lh.numel() * 4, "ms_per_step": e2e_s * 1e3,
               "api": "attn_fwd_varlen (C ABI) with pinned host copies inside the timed region"}
    peak, peak_src = load_peaks()
    hbm_peak, hbm_src = load_hbm_peak()
    kbytes = 2.0 * H * d * 4 * total + 4.0 * H * total
    out = {"metric": METRIC, "value": world * tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
           "roofline": roofline_entry(flops / kbytes, peak * 1e12 / (hbm_peak * 1e9), tflops, peak, peak_src, kbytes,
                                      ms_kernel, hbm_peak, hbm_src, load_traffic(name), flops,
                                      fused_kernel_name(B, H, max(lengths), d, torch.cuda.get_device_properties(dev)
                                                        .multi_processor_count, causal) + " (packed sequences)"),
           "e2e": e2e, "gpu_launches": args.steps, "clocks": clocks, "cpu_baseline": None}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
