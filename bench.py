"""Benchmark of the diagonal linear-recurrence scan (forward + backward).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 4] [--sets 3]
                    [--impl reference]

One step = one forward scan and one backward scan over one batch of the
workload: by default the largest named workload (near-unit bf16, B=16 T=4096
D=4096, bf16 storage, fp32 state; 268 M elements per tensor, 512 MiB, larger
than L2).  Inputs are resident in HBM before the timed region, and three
independent buffer sets rotate (each kernel reads the set that was written or
read two steps earlier).

The JSON line carries the step throughput (`value`), each direction timed
alone over back-to-back launches (`fwd`, `bwd`, `roofline` for the slower
one), the same figures for every other named workload (`per_config`), the
end-to-end figure through the host-buffer C ABI call (`e2e`), the next rows
on their own workloads (`extensions`) and the oracle on the host cores
(`cpu_baseline`).

Rank 0 prints one JSON line.  Under torchrun every rank runs the same
workload on its own GPU (independent replicas: the scan's lanes shard with
no exchange), and the value is the whole job's elements/s over the slowest
rank's time.

`--impl reference` times the CPU oracle (the reference arm) on the host
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "scan fwd+bwd elements/s and achieved HBM GB/s (% of GB300 roofline), 1 GPU"
L2_BYTES = 126 * 1024 * 1024


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def algorithmic_bytes(w) -> tuple[int, int]:
    """Forward reads a, b and writes out (+ the fp32 final state); backward
    reads a, out, grad_out and writes grad_a, grad_b."""
    E, s = w.elements, w.storage_bytes
    return 3 * E * s + 4 * w.B * w.D, 5 * E * s


# --------------------------------------------------------------- clocks ----
class ClockSampler:
    """Samples nvidia-smi during the timed region (SM clock, reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------- multi-rank job ----
def max_over_ranks(values, dist, device) -> list[float]:
    """Every rank's values replaced by the slowest rank's (element-wise max):
    the job's step ends when its slowest rank's does."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world: int, units_per_rank: int, ms: float) -> float:
    """Whole-job units per second: every rank processes its own units (weak
    scaling, independent replicas) in the slowest rank's time."""
    return world * units_per_rank / (ms * 1e-3)


# ------------------------------------------------------------ reference ----
def run_reference(args, w) -> dict:
    """The CPU oracle on the host cores: the reference arm of this benchmark."""
    import numpy as np

    import oracle
    from linear_recurrence_scan_lrscan_gb300.workloads import make_inputs, to_numpy_storage

    o = oracle.default()
    # A bounded sample: whole batch rows of the workload, every step of T,
    # a slice of the lanes sized for about a second of single-core work per step.
    lanes = max(1, min(w.D, int(args.ref_elements // max(1, w.T))))
    inp = make_inputs(w.cid, B=1, D=lanes)
    a, b, g = (to_numpy_storage(inp[k]) for k in ("a", "b", "grad_out"))
    E = a.size
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        out, _ = o.fwd(a, b, w.dtype)
        o.bwd(a, out, g, w.dtype)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    per_step = sum(times) / len(times)
    value = E / per_step
    sample = f"B=1 T={w.T} D={lanes} of {w.describe()} (fwd+bwd, single thread)"
    return {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "elements/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": config_of(w, None, None),
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _oracle_slice_worker(args):
    """One host process: the oracle's forward + backward on its own lanes of
    the sample, `reps` times; returns (elements, seconds)."""
    cid, lanes, lo, hi, reps = args
    sys.path.insert(0, ROOT)
    import oracle
    from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS, make_inputs, to_numpy_storage
    w = WORKLOADS[cid]
    inp = make_inputs(cid, B=1, D=lanes)
    a, b, g = (to_numpy_storage(inp[k])[:, :, lo:hi].copy() for k in ("a", "b", "grad_out"))
    o = oracle.default()
    t0 = time.perf_counter()
    for _ in range(reps):
        out, _ = o.fwd(a, b, w.dtype)
        o.bwd(a, out, g, w.dtype)
    return a.size * reps, time.perf_counter() - t0


def cpu_baseline(w, seconds: float = 12.0) -> dict:
    """The oracle as it stands on a bounded sample: single-threaded, and on
    every host core (the sample's lanes split into disjoint slices, one
    spawn-started process per core; lanes are independent)."""
    import multiprocessing as mp

    import oracle
    from linear_recurrence_scan_lrscan_gb300.workloads import make_inputs, to_numpy_storage

    o = oracle.default()
    lanes = max(1, min(w.D, 2_000_000 // max(1, w.T)))
    inp = make_inputs(w.cid, B=1, D=lanes)
    a, b, g = (to_numpy_storage(inp[k]) for k in ("a", "b", "grad_out"))
    E = a.size
    t_end = time.perf_counter() + seconds
    n, t_tot = 0, 0.0
    while n < 3 or time.perf_counter() < t_end:
        t0 = time.perf_counter()
        out, _ = o.fwd(a, b, w.dtype)
        o.bwd(a, out, g, w.dtype)
        t_tot += time.perf_counter() - t0
        n += 1
    single = E * n / t_tot
    cores = max(1, min(os.cpu_count() or 1, lanes))
    reps = max(1, n)
    cuts = [lanes * i // cores for i in range(cores + 1)]
    jobs = [(w.cid, lanes, cuts[i], cuts[i + 1], reps) for i in range(cores) if cuts[i + 1] > cuts[i]]
    from concurrent.futures import ProcessPoolExecutor
    # spawn-started workers (a fork after CUDA initialisation is unsafe); a
    # worker that dies raises here instead of hanging the pool
    with ProcessPoolExecutor(max_workers=len(jobs), mp_context=mp.get_context("spawn")) as pool:
        t0 = time.perf_counter()
        res = list(pool.map(_oracle_slice_worker, jobs))
        wall = time.perf_counter() - t0
    done = sum(r[0] for r in res)
    slowest = max(r[1] for r in res)
    multi = done / slowest
    return {"value": multi, "unit": "elements/s", "cores": len(jobs), "kind": "oracle",
            "sample": f"B=1 T={w.T} D={lanes} of {w.describe()}, fwd+bwd; {len(jobs)} spawn-started processes "
                      f"on disjoint lane slices, {reps} repetitions each (slowest process's compute time; "
                      f"{wall:.1f} s wall with start-up)",
            "single_thread": {"value": single, "cores": 1, "repetitions": n}}


def config_of(w, pf, pb, nsets: int = 3) -> dict:
    from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS
    c = {"workload": w.describe(), "B": w.B, "T": w.T, "D": w.D, "storage": w.dtype, "state": "f32",
         "elements_per_step": w.elements}
    big = w.elements * w.storage_bytes > L2_BYTES
    c["l2"] = (f"inputs larger than L2 ({w.elements * w.storage_bytes / 2**20:.0f} MiB per tensor) and "
               if big else "") + (f"{nsets} rotating buffer sets; each kernel reads the set written or read "
                                  f"{nsets - 1} steps earlier" if nsets > 1 else "one buffer set")
    if w.chunk:
        c["chunk"] = w.chunk
    if pf is not None:
        c["fwd_kernel"] = pf["name"]
        c["bwd_kernel"] = pb["name"]
    c["why_this_workload"] = ("the metric names no workload: the largest of the five named workloads "
                              "that fits one GPU (by elements per step)"
                              if w.elements == max(x.elements for x in WORKLOADS.values()) else
                              "chosen with --config")
    return c


# ------------------------------------------------------------------ ours ----
def device_sets(w, host: dict, dev, nsets: int, opts: dict) -> list[dict]:
    """`nsets` independent device copies of the workload's inputs with their
    output buffers; each set's `out` holds that set's forward result."""
    import torch

    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    sets = []
    for _ in range(nsets):
        a, b, g = host["a"].to(dev), host["b"].to(dev), host["grad_out"].to(dev)
        sets.append({"a": a, "b": b, "g": g, "out": torch.empty_like(a), "ga": torch.empty_like(a),
                     "gb": torch.empty_like(a),
                     "last": torch.empty(w.B, w.D, device=dev, dtype=torch.float32)})
    for s in sets:
        L.lrscan_fwd(s["a"], s["b"], s["out"], s["last"], **opts)
    torch.cuda.synchronize()
    return sets


def fwd_call(sets, opts):
    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    n = len(sets)

    def fn(i):
        s = sets[i % n]
        L.lrscan_fwd(s["a"], s["b"], s["out"], s["last"], **opts)
    return fn


def bwd_call(sets, opts):
    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    n = len(sets)

    def fn(i):
        s = sets[i % n]
        L.lrscan_bwd(s["a"], s["out"], s["g"], s["ga"], s["gb"], **opts)
    return fn


def kernel_timing(w, sets, opts, iters: int, stream, peak: float) -> dict:
    """Forward alone and backward alone, each over `iters` back-to-back
    launches rotating the buffer sets (CUDA events on the launching stream):
    mean device time per launch, algorithmic GB/s and its fraction of the
    measured copy peak, with the kernel the dispatcher ran."""
    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    fs = time_launch_samples(fwd_call(sets, opts), iters, stream)
    bs = time_launch_samples(bwd_call(sets, opts), iters, stream)
    fms, bms = sorted(fs)[1], sorted(bs)[1]  # medians of three samples
    if L.lrscan_sync_check() != 0:
        raise RuntimeError(f"device error while timing {w.describe()}")
    pf = L.lrscan_plan(w.B, w.T, w.D, w.dtype, "fwd", **opts)
    pb = L.lrscan_plan(w.B, w.T, w.D, w.dtype, "bwd", **opts)
    bf, bb = algorithmic_bytes(w)
    res = {"workload": w.describe(), "launches_per_direction": 3 * iters, "buffer_sets": len(sets),
           "timing": f"median of 3 samples of {iters} back-to-back launches"}
    for key, ms, smp, by, p in (("fwd", fms, fs, bf, pf), ("bwd", bms, bs, bb, pb)):
        gbs = by / (ms * 1e-3) / 1e9
        res[key] = {"us": ms * 1e3, "samples_us": [round(x * 1e3, 2) for x in smp], "GB/s": gbs,
                    "frac": gbs / peak, "algorithmic_bytes": by,
                    "elements/s": w.elements / (ms * 1e-3), "kernel": p["name"], "path": p["path"],
                    "kernels": p["kernels"], "traffic": load_traffic(w, key, p["name"])}
    res["elements/s"] = 2 * w.elements / ((fms + bms) * 1e-3)
    return res


def run_per_config(args, dev, stream, peak, headline: dict) -> dict:
    """Every named workload (1-5) at full size on its automatic plan, timed
    like the headline (back-to-back launches per direction, rotating buffer
    sets).  The headline workload's entry is the one measured above."""
    import torch

    from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS, make_inputs
    out = {}
    for cid, w in WORKLOADS.items():
        if cid == args.config:
            out[str(cid)] = headline
            continue
        host = make_inputs(cid)
        # tiny workloads are launch-latency bound: more launches per sample
        iters = max(20, min(args.steps, 200)) if w.elements > (1 << 20) else 200
        sets = device_sets(w, host, dev, min(3, args.sets), {})
        del host
        out[str(cid)] = kernel_timing(w, sets, {}, iters, stream, peak)
        del sets
        torch.cuda.empty_cache()
    return out


def run_ours(args, w, rank: int, world: int, dist) -> dict | None:
    import torch

    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    from linear_recurrence_scan_lrscan_gb300.workloads import make_inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    inp = make_inputs(w.cid)
    a_h, b_h, g_h = inp["a"], inp["b"], inp["grad_out"]
    opts = {}
    if args.path:
        opts["path"] = args.path
    if args.variant:
        opts["tile_variant"] = args.variant
    if w.chunk and args.path == "chunk":
        opts["chunk_len"] = w.chunk
    pf = L.lrscan_plan(w.B, w.T, w.D, w.dtype, "fwd", **opts)
    pb = L.lrscan_plan(w.B, w.T, w.D, w.dtype, "bwd", **opts)

    sets = device_sets(w, inp, dev, args.sets, opts)
    nsets = len(sets)
    fwd, bwd = fwd_call(sets, opts), bwd_call(sets, opts)

    def step(i):
        # the backward reads the set the previous step's forward wrote
        fwd(i)
        bwd(i + nsets - 1)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert L.lrscan_sync_check() == 0

    peaks = load_peaks()
    clocks = ClockSampler(dev.index if not os.environ.get("CUDA_VISIBLE_DEVICES") else
                          int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[dev.index]))
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # Device-timed region: K steps of forward + backward, nothing else on the stream.
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    rc = L.lrscan_sync_check()
    if rc != 0:
        raise RuntimeError(f"device error during the timed region: {rc}")
    total_ms = t_start.elapsed_time(t_end)
    # Per-kernel durations, right after the step loop and still under the clock
    # sampler: each direction alone over back-to-back launches.
    iters = max(20, min(args.steps, 200))
    kt = kernel_timing(w, sets, opts, iters, stream, peaks["hbm_gbs"])
    clk = clocks.stop() if rank == 0 else None
    total_ms, fwd_ms, bwd_ms = max_over_ranks([total_ms, kt["fwd"]["us"] * 1e-3, kt["bwd"]["us"] * 1e-3], dist,
                                              dev)
    ms_per_step = total_ms / args.steps

    # end to end through the host-buffer entry point: pinned host inputs ->
    # device -> fwd+bwd -> pinned host outputs, copies pipelined with the
    # kernels over batch-row chunks inside the library (lrscan_fwd_bwd_host)
    e2e = None
    if not args.no_e2e:
        pa, pbuf, pg = a_h.pin_memory(), b_h.pin_memory(), g_h.pin_memory()
        ho = torch.empty_like(pa).pin_memory()
        hga, hgb = torch.empty_like(pa).pin_memory(), torch.empty_like(pa).pin_memory()
        hl = torch.empty(w.B, w.D, dtype=torch.float32).pin_memory()
        e2e_steps = max(3, min(args.steps, args.e2e_steps))

        def e2e_step():
            L.lrscan_fwd_bwd_host(pa, pbuf, pg, out=ho, last=hl, grad_a=hga, grad_b=hgb, **opts)

        def timed(fn):
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            if dist is not None:
                dist.barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(e2e_steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / e2e_steps

        # the call returns when the host outputs are written, so events on the
        # idle current stream bracket the whole call
        e2e_ms = timed(e2e_step)
        s0 = sets[0]

        def serial_step():  # the same step without overlap: copy in, kernels, copy out on one stream
            s0["a"].copy_(pa, non_blocking=True)
            s0["b"].copy_(pbuf, non_blocking=True)
            s0["g"].copy_(pg, non_blocking=True)
            L.lrscan_fwd(s0["a"], s0["b"], s0["out"], s0["last"], **opts)
            L.lrscan_bwd(s0["a"], s0["out"], s0["g"], s0["ga"], s0["gb"], **opts)
            ho.copy_(s0["out"], non_blocking=True)
            hl.copy_(s0["last"], non_blocking=True)
            hga.copy_(s0["ga"], non_blocking=True)
            hgb.copy_(s0["gb"], non_blocking=True)
        serial_ms = timed(serial_step)
        e2e_ms, serial_ms = max_over_ranks([e2e_ms, serial_ms], dist, dev)
        s = w.storage_bytes
        e2e = {"value": job_throughput(world, w.elements, e2e_ms), "unit": "elements/s",
               "h2d_bytes_per_step": 3 * w.elements * s,
               "d2h_bytes_per_step": 3 * w.elements * s + 4 * w.B * w.D,
               "ms_per_step": e2e_ms,
               "path": "lrscan_fwd_bwd_host (C ABI, pinned host buffers): batch-row chunks, copies in / kernels / "
                       "copies out on three streams",
               "unpipelined_ms_per_step": serial_ms}
        del pa, pbuf, pg, ho, hga, hgb, hl
        assert L.lrscan_sync_check() == 0
    del inp, a_h, b_h, g_h

    if rank != 0:
        return None
    bf, bb = algorithmic_bytes(w)
    gbs_f = bf / (fwd_ms * 1e-3) / 1e9
    gbs_b = bb / (bwd_ms * 1e-3) / 1e9
    dominant = ("bwd", bb, bwd_ms, gbs_b, pb) if bwd_ms >= fwd_ms else ("fwd", bf, fwd_ms, gbs_f, pf)
    line = {
        "metric": METRIC,
        "value": job_throughput(world, w.elements, ms_per_step),
        "unit": "elements/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": config_of(w, pf, pb, nsets),
        "roofline": {"bound": "hbm", "kernel": f"{dominant[0]}:{dominant[4]['name']}",
                     "achieved": dominant[3], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": dominant[3] / peaks["hbm_gbs"], "peak_source": peaks["source"],
                     "algorithmic_bytes_per_launch": dominant[1], "launch_us": dominant[2] * 1e3,
                     "launches_timed": 3 * iters, "timing": kt["timing"],
                     "traffic": kt[dominant[0]]["traffic"]},
        "fwd": kt["fwd"],
        "bwd": kt["bwd"],
        "step_GB/s": (bf + bb) / (ms_per_step * 1e-3) / 1e9,
        "kernel_timing": f"each direction alone over {iters} back-to-back launches rotating {nsets} buffer "
                         "sets, CUDA events on the launching stream, right after the step loop (clocks "
                         "sampled over both)",
        "gpu_launches": args.steps * (pf["kernels"] + pb["kernels"]),
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_per_config:
        line["per_config"] = run_per_config(args, dev, stream, peaks["hbm_gbs"], kt)
    if not args.no_extensions:
        line["extensions"] = run_extensions(args, dev, peaks["hbm_gbs"])
    del sets
    torch.cuda.empty_cache()
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return line


# ------------------------------------------------------------ extensions ----
def time_launch_samples(fn, iters: int, stream, samples: int = 3) -> list[float]:
    """Mean device time (ms) of one call of fn(i) over `iters` back-to-back
    calls, `samples` times (after 3 untimed calls); CUDA events on the
    launching stream around each sample."""
    import torch
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    out = []
    for _ in range(samples):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(iters):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / iters)
    return out


def time_launches(fn, iters: int, stream) -> float:
    """Median over three samples of the mean device time of one call of fn(i)
    over `iters` back-to-back calls (a host stall that starves the device in
    one sample does not set the figure)."""
    return float(sorted(time_launch_samples(fn, iters, stream))[1])


def run_extensions(args, dev, peak) -> dict:
    """The next rows on their own workloads.  Here: the state-carrying scan
    on the gated workload (2): initial state h0, a segment start every 512
    tokens on average, grad_last in and grad_h0 out.  Each direction is timed
    over back-to-back launches rotating three buffer sets; GB/s counts the
    bytes the operation must move."""
    import numpy as np
    import torch

    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS, make_inputs
    stream = torch.cuda.current_stream()
    iters = max(20, min(args.steps, 200))
    w = WORKLOADS[2]
    opts = {}
    sets = device_sets(w, make_inputs(2), dev, 3, opts)
    B, T, D, E, s = w.B, w.T, w.D, w.elements, w.storage_bytes
    r = np.random.default_rng(7)
    pos = np.zeros((B, T), dtype=np.int32)
    starts = r.random((B, T)) < 1.0 / 512
    for t in range(1, T):
        pos[:, t] = np.where(starts[:, t], 0, pos[:, t - 1] + 1)
    seg = torch.from_numpy(pos).to(dev)
    h0 = torch.randn(B, D, device=dev)
    gl = torch.randn(B, D, device=dev)
    gh0 = torch.empty(B, D, device=dev)
    n = len(sets)

    def fwd(i):
        f = sets[i % n]
        L.lrscan_fwd_state(f["a"], f["b"], h0=h0, segment_pos=seg, out=f["out"], last=f["last"], **opts)

    def bwd(i):
        f = sets[i % n]
        L.lrscan_bwd_state(f["a"], f["out"], f["g"], h0=h0, segment_pos=seg, grad_last=gl, grad_a=f["ga"],
                           grad_b=f["gb"], grad_h0=gh0, **opts)
    fms = time_launches(fwd, iters, stream)
    bms = time_launches(bwd, iters, stream)
    if L.lrscan_sync_check() != 0:
        raise RuntimeError("device error while timing the state-carrying scan")
    fb = 3 * E * s + 4 * B * T + 2 * 4 * B * D
    bb = 5 * E * s + 4 * B * T + 3 * 4 * B * D
    del sets
    torch.cuda.empty_cache()
    return {"complex": run_complex(iters, dev, peak), "complex_long_t": run_complex_long_t(dev, peak),
            "complex_long_t_bf16": run_complex_long_t(dev, peak, "bf16"),
            "generated_decay": run_gated(iters, dev, peak),
            "generated_decay_fp32": run_gated(iters, dev, peak, "f32"),
            "long_t": run_long_t(dev, peak), "state": {
        "workload": w.describe(),
        "what": "carried state: h0 in, segment resets (int32 positions, ~1 start per 512 tokens), "
                "grad_last in, grad_h0 out",
        "launches_per_direction": 3 * iters, "timing": "median of 3 samples",
        "fwd": {"ms": fms, "GB/s": fb / (fms * 1e-3) / 1e9, "frac": fb / (fms * 1e-3) / 1e9 / peak,
                "algorithmic_bytes": fb},
        "bwd": {"ms": bms, "GB/s": bb / (bms * 1e-3) / 1e9, "frac": bb / (bms * 1e-3) / 1e9 / peak,
                "algorithmic_bytes": bb},
        "elements/s": 2 * E / ((fms + bms) * 1e-3)}}


def run_complex(iters: int, dev, peak) -> dict:
    """The complex scan on its workload (re/im planes, the gated workload's
    shape and decay magnitudes with random phases), three rotating buffer
    sets; forward moves 6 elements per (t, d) (+ the fp32 final state),
    backward 10."""
    import numpy as np
    import torch

    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    from linear_recurrence_scan_lrscan_gb300.workloads import COMPLEX_WORKLOAD as cw
    from linear_recurrence_scan_lrscan_gb300.workloads import make_complex_inputs
    stream = torch.cuda.current_stream()
    host = make_complex_inputs()
    sets = []
    for _ in range(3):
        st = {k: host[k].to(dev) for k in ("ar", "ai", "br", "bi", "go_r", "go_i")}
        st["out"] = [torch.empty_like(st["ar"]) for _ in range(2)]
        st["last"] = [torch.empty(cw.B, cw.D, device=dev) for _ in range(2)]
        st["grads"] = [torch.empty_like(st["ar"]) for _ in range(4)]
        sets.append(st)
    del host

    def fwd(i):
        st = sets[i % 3]
        L.lrscan_cfwd(st["ar"], st["ai"], st["br"], st["bi"], out_r=st["out"][0], out_i=st["out"][1],
                      last_r=st["last"][0], last_i=st["last"][1])

    def bwd(i):
        st = sets[i % 3]
        L.lrscan_cbwd(st["ar"], st["ai"], st["out"][0], st["out"][1], st["go_r"], st["go_i"], grads=st["grads"])
    fms = time_launches(fwd, iters, stream)
    bms = time_launches(bwd, iters, stream)
    if L.lrscan_sync_check() != 0:
        raise RuntimeError("device error while timing the complex scan")
    E, s = cw.elements, cw.storage_bytes
    B, T, D = cw.B, cw.T, cw.D
    fb, bb = 6 * E * s + 8 * B * D, 10 * E * s
    pf = L.lrscan_plan_complex(B, T, D, cw.dtype, "fwd")
    pb = L.lrscan_plan_complex(B, T, D, cw.dtype, "bwd")
    res = {"workload": cw.describe() + " complex (re/im planes)", "launches_per_direction": 3 * iters, "timing": "median of 3 samples",
           "fwd": {"ms": fms, "GB/s": fb / (fms * 1e-3) / 1e9, "frac": fb / (fms * 1e-3) / 1e9 / peak,
                   "algorithmic_bytes": fb, "kernel": pf["name"]},
           "bwd": {"ms": bms, "GB/s": bb / (bms * 1e-3) / 1e9, "frac": bb / (bms * 1e-3) / 1e9 / peak,
                   "algorithmic_bytes": bb, "kernel": pb["name"]},
           "elements/s": 2 * E / ((fms + bms) * 1e-3)}

    # the same workload with carried state: complex h0 in, a segment start
    # every 512 tokens on average, complex grad_last in, grad_h0 out
    r = np.random.default_rng(8)
    pos = np.zeros((B, T), dtype=np.int32)
    starts = r.random((B, T)) < 1.0 / 512
    for t in range(1, T):
        pos[:, t] = np.where(starts[:, t], 0, pos[:, t - 1] + 1)
    seg = torch.from_numpy(pos).to(dev)
    h0 = (torch.randn(B, D, device=dev), torch.randn(B, D, device=dev))
    gl = (torch.randn(B, D, device=dev), torch.randn(B, D, device=dev))
    gh0 = [torch.empty(B, D, device=dev) for _ in range(2)]

    def sfwd(i):
        st = sets[i % 3]
        L.lrscan_cfwd_state(st["ar"], st["ai"], st["br"], st["bi"], h0=h0, segment_pos=seg, out_r=st["out"][0],
                            out_i=st["out"][1], last_r=st["last"][0], last_i=st["last"][1])

    def sbwd(i):
        st = sets[i % 3]
        L.lrscan_cbwd_state(st["ar"], st["ai"], st["out"][0], st["out"][1], st["go_r"], st["go_i"], h0=h0,
                            segment_pos=seg, grad_last=gl, grads=st["grads"], grad_h0=gh0)
    sfms = time_launches(sfwd, iters, stream)
    sbms = time_launches(sbwd, iters, stream)
    if L.lrscan_sync_check() != 0:
        raise RuntimeError("device error while timing the state-carrying complex scan")
    sfb = fb + 4 * B * T + 8 * B * D
    sbb = bb + 4 * B * T + 3 * 8 * B * D
    psf = L.lrscan_plan_complex(B, T, D, cw.dtype, "fwd", state=True)
    psb = L.lrscan_plan_complex(B, T, D, cw.dtype, "bwd", state=True)
    res["state"] = {
        "what": "carried state: complex h0 in, segment resets (int32 positions, ~1 start per 512 tokens), "
                "complex grad_last in, grad_h0 out",
        "fwd": {"ms": sfms, "GB/s": sfb / (sfms * 1e-3) / 1e9, "frac": sfb / (sfms * 1e-3) / 1e9 / peak,
                "algorithmic_bytes": sfb, "kernel": psf["name"]},
        "bwd": {"ms": sbms, "GB/s": sbb / (sbms * 1e-3) / 1e9, "frac": sbb / (sbms * 1e-3) / 1e9 / peak,
                "algorithmic_bytes": sbb, "kernel": psb["name"]},
        "elements/s": 2 * E / ((sfms + sbms) * 1e-3)}
    del sets
    torch.cuda.empty_cache()
    return res


def run_complex_long_t(dev, peak, dtype="f32") -> dict:
    """The complex scan with few lanes and a long sequence: B=1 T=2^20 D=64
    re/im planes (fp32, or bf16 storage of the same draws), |a|~U(0.9,0.999)
    with phases ~U(-pi,pi), b and grad_out ~N(0,1), drawn on the device from a
    seeded generator.  The automatic plan (chunk streaming) beside the chunked
    path (complex chunk maps, grouped prefix), and the automatic plan with
    carried state and resets; algorithmic bytes are 6 (forward) and 10
    (backward) elements per (t, d)."""
    import math

    import torch

    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    B, T, D = 1, 1 << 20, 64
    gen = torch.Generator(device=dev).manual_seed(20298)
    rho = torch.empty(B, T, D, device=dev).uniform_(0.9, 0.999, generator=gen)
    th = torch.empty(B, T, D, device=dev).uniform_(-math.pi, math.pi, generator=gen)
    cv = (lambda x: x.bfloat16()) if dtype == "bf16" else (lambda x: x)
    ar, ai = cv(rho * torch.cos(th)), cv(rho * torch.sin(th))
    del rho, th
    br, bi, gr, gi = (cv(torch.empty(B, T, D, device=dev).normal_(generator=gen)) for _ in range(4))
    outs = L.lrscan_cfwd(ar, ai, br, bi)
    grads = L.lrscan_cbwd(ar, ai, outs[0], outs[1], gr, gi)
    stream = torch.cuda.current_stream()
    E = B * T * D
    es = 2 if dtype == "bf16" else 4
    fb, bb = 6 * E * es + 8 * B * D, 10 * E * es
    res = {"workload": f"B={B} T={T} D={D} {'bf16' if dtype == 'bf16' else 'fp32'} complex (few lanes, long sequence)"}
    for kw, name in ((dict(), "auto"), (dict(path="chunk"), "chunked")):
        fms = time_launches(lambda i: L.lrscan_cfwd(ar, ai, br, bi, out_r=outs[0], out_i=outs[1], last_r=outs[2],
                                                    last_i=outs[3], **kw), 10, stream)
        bms = time_launches(lambda i: L.lrscan_cbwd(ar, ai, outs[0], outs[1], gr, gi, grads=grads, **kw), 10, stream)
        if L.lrscan_sync_check() != 0:
            raise RuntimeError("device error while timing the long complex scan")
        part = {"fwd": {"ms": fms, "frac": fb / (fms * 1e-3) / 1e9 / peak,
                        "kernel": L.lrscan_plan_complex(B, T, D, dtype, "fwd", **kw)["name"]},
                "bwd": {"ms": bms, "frac": bb / (bms * 1e-3) / 1e9 / peak,
                        "kernel": L.lrscan_plan_complex(B, T, D, dtype, "bwd", **kw)["name"]},
                "elements/s": 2 * E / ((fms + bms) * 1e-3)}
        if name == "auto":
            res.update(part)
        else:
            res[name] = part
    # carried complex state: h0, a segment start every 4,096 steps, grad_last,
    # grad_h0 (the automatic plan)
    h0 = tuple(torch.empty(B, D, device=dev).normal_(generator=gen) for _ in range(2))
    gl = tuple(torch.empty(B, D, device=dev).normal_(generator=gen) for _ in range(2))
    gh0 = tuple(torch.empty(B, D, device=dev) for _ in range(2))
    seg = (torch.arange(T, device=dev, dtype=torch.int32) % 4096).view(1, T).repeat(B, 1).contiguous()
    fms = time_launches(lambda i: L.lrscan_cfwd_state(ar, ai, br, bi, h0=h0, segment_pos=seg, out_r=outs[0],
                                                      out_i=outs[1], last_r=outs[2], last_i=outs[3]), 10, stream)
    bms = time_launches(lambda i: L.lrscan_cbwd_state(ar, ai, outs[0], outs[1], gr, gi, h0=h0, segment_pos=seg,
                                                      grad_last=gl, grads=grads, grad_h0=gh0), 10, stream)
    if L.lrscan_sync_check() != 0:
        raise RuntimeError("device error while timing the long complex scan with carried state")
    sfb, sbb = fb + 4 * B * T + 8 * B * D, bb + 4 * B * T + 24 * B * D
    res["state"] = {"what": "complex h0, a segment start every 4,096 steps, grad_last, grad_h0",
                    "fwd": {"ms": fms, "frac": sfb / (fms * 1e-3) / 1e9 / peak,
                            "kernel": L.lrscan_plan_complex(B, T, D, dtype, "fwd", state=True)["name"]},
                    "bwd": {"ms": bms, "frac": sbb / (bms * 1e-3) / 1e9 / peak,
                            "kernel": L.lrscan_plan_complex(B, T, D, dtype, "bwd", state=True)["name"]},
                    "elements/s": 2 * E / ((fms + bms) * 1e-3)}
    del ar, ai, br, bi, gr, gi, outs, grads
    torch.cuda.empty_cache()
    return res


def run_gated(iters: int, dev, peak, dtype=None) -> dict:
    """The scan with decays generated in the kernel (exp(-exp(nu_log_d) exp(eta_t)))
    on the gated workload's shape (its bf16 storage, or `dtype`), three rotating
    buffer sets.  Forward moves b in and out out (2 elements per (t, d)) plus
    eta, nu_log and the fp32 final state; backward moves out, grad_out in and
    grad_b out (3 elements) plus eta, nu_log in and grad_eta, grad_nu_log out."""
    import torch

    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    from linear_recurrence_scan_lrscan_gb300.workloads import GATED_WORKLOAD as gw
    from linear_recurrence_scan_lrscan_gb300.workloads import make_gated_inputs
    stream = torch.cuda.current_stream()
    dtype = dtype or gw.dtype
    host = make_gated_inputs(dtype=dtype)
    sets = []
    for _ in range(3):
        st = {k: host[k].to(dev) for k in ("eta", "nu_log", "b", "grad_out")}
        st["out"], st["gb"] = torch.empty_like(st["b"]), torch.empty_like(st["b"])
        st["last"] = torch.empty(gw.B, gw.D, device=dev)
        L.lrscan_fwd_gated(st["eta"], st["nu_log"], st["b"], out=st["out"], last=st["last"])
        sets.append(st)
    del host

    def fwd(i):
        st = sets[i % 3]
        L.lrscan_fwd_gated(st["eta"], st["nu_log"], st["b"], out=st["out"], last=st["last"])

    def bwd(i):
        st = sets[i % 3]
        L.lrscan_bwd_gated(st["eta"], st["nu_log"], st["out"], st["grad_out"], grad_b=st["gb"])
    fms = time_launches(fwd, iters, stream)
    bms = time_launches(bwd, iters, stream)
    if L.lrscan_sync_check() != 0:
        raise RuntimeError("device error while timing the generated-decay scan")
    B, T, D, E = gw.B, gw.T, gw.D, gw.elements
    s = 4 if dtype == "f32" else 2
    fb = 2 * E * s + 4 * B * T + 4 * D + 4 * B * D
    bb = 3 * E * s + 2 * (4 * B * T + 4 * D)
    pf = L.lrscan_plan_gated(B, T, D, dtype, "fwd")
    pb = L.lrscan_plan_gated(B, T, D, dtype, "bwd")
    del sets
    torch.cuda.empty_cache()
    desc = gw.describe() if dtype == gw.dtype else f"B={B} T={T} D={D} {dtype}"
    return {"workload": desc + " with decays generated from eta [B,T] and nu_log [D]",
            "launches_per_direction": 3 * iters, "timing": "median of 3 samples",
            "fwd": {"ms": fms, "GB/s": fb / (fms * 1e-3) / 1e9, "frac": fb / (fms * 1e-3) / 1e9 / peak,
                    "algorithmic_bytes": fb, "kernel": pf["name"]},
            "bwd": {"ms": bms, "GB/s": bb / (bms * 1e-3) / 1e9, "frac": bb / (bms * 1e-3) / 1e9 / peak,
                    "algorithmic_bytes": bb, "kernel": pb["name"], "kernels": pb["kernels"]},
            "elements/s": 2 * E / ((fms + bms) * 1e-3)}


def run_long_t(dev, peak) -> dict:
    """Few lanes, very long sequence: B=1 T=2^22 D=64 fp32: the chunked path
    with chunk 64 (65,536 chunk maps per lane, 64 lanes) with the flat prefix
    (one warp per lane walks all maps) and with the grouped prefix, the
    chunked path at its own chunk lengths (grouped prefix over 512-step chunks
    forward, 128 backward), the single-pass chunk-streaming path, and the
    automatic plan (streaming), also with carried state and resets; then the
    automatic plan on bf16 storage of the same draws.  Inputs are drawn on the device from a seeded generator
    (a~U(0.9,0.9999), b,g~N(0,1))."""
    import torch

    from linear_recurrence_scan_lrscan_gb300 import lrscan as L
    B, T, D, C = 1, 1 << 22, 64, 64
    gen = torch.Generator(device=dev).manual_seed(20299)
    a = torch.empty(B, T, D, device=dev).uniform_(0.9, 0.9999, generator=gen)
    b = torch.empty(B, T, D, device=dev).normal_(generator=gen)
    g = torch.empty(B, T, D, device=dev).normal_(generator=gen)
    out, ga, gb = torch.empty_like(a), torch.empty_like(a), torch.empty_like(a)
    last = torch.empty(B, D, device=dev)
    stream = torch.cuda.current_stream()
    E = B * T * D
    res = {"workload": f"B={B} T={T} D={D} fp32 chunk {C} (few lanes, long sequence)"}
    for kw, name in ((dict(path="chunk", chunk_len=C, tile_variant=1), "flat_prefix"),
                     (dict(path="chunk", chunk_len=C, tile_variant=2), "grouped_prefix"),
                     (dict(path="chunk"), "chunked_own_length"),
                     (dict(path="stream"), "stream")):
        fms = time_launches(lambda i: L.lrscan_fwd(a, b, out, last, **kw), 10, stream)
        bms = time_launches(lambda i: L.lrscan_bwd(a, out, g, ga, gb, **kw), 10, stream)
        res[name] = {"fwd_ms": fms, "bwd_ms": bms,
                     "fwd_frac": 3 * E * 4 / (fms * 1e-3) / 1e9 / peak,
                     "bwd_frac": 5 * E * 4 / (bms * 1e-3) / 1e9 / peak,
                     "elements/s": 2 * E / ((fms + bms) * 1e-3)}
    fms = time_launches(lambda i: L.lrscan_fwd(a, b, out, last), 10, stream)
    bms = time_launches(lambda i: L.lrscan_bwd(a, out, g, ga, gb), 10, stream)
    res["auto_plan"] = {"fwd_ms": fms, "bwd_ms": bms,
                        "fwd_frac": 3 * E * 4 / (fms * 1e-3) / 1e9 / peak,
                        "bwd_frac": 5 * E * 4 / (bms * 1e-3) / 1e9 / peak,
                        "elements/s": 2 * E / ((fms + bms) * 1e-3)}
    if L.lrscan_sync_check() != 0:
        raise RuntimeError("device error while timing the long-sequence chunked path")
    res["auto"] = {d: L.lrscan_plan(B, T, D, "f32", d)["name"] for d in ("fwd", "bwd")}
    # carried state: h0, a segment start every 4,096 steps, grad_last, grad_h0
    # (the automatic plan); algorithmic bytes add the positions and the states
    h0 = torch.empty(B, D, device=dev).normal_(generator=gen)
    gl = torch.empty(B, D, device=dev).normal_(generator=gen)
    gh0 = torch.empty(B, D, device=dev)
    seg = (torch.arange(T, device=dev, dtype=torch.int32) % 4096).view(1, T).repeat(B, 1).contiguous()
    fms = time_launches(lambda i: L.lrscan_fwd_state(a, b, h0=h0, segment_pos=seg, out=out, last=last), 10, stream)
    bms = time_launches(lambda i: L.lrscan_bwd_state(a, out, g, h0=h0, segment_pos=seg, grad_last=gl, grad_a=ga,
                                                     grad_b=gb, grad_h0=gh0), 10, stream)
    if L.lrscan_sync_check() != 0:
        raise RuntimeError("device error while timing the long scan with carried state")
    fb, bb = 3 * E * 4 + 4 * B * T + 8 * B * D, 5 * E * 4 + 4 * B * T + 12 * B * D
    res["auto_plan_state"] = {"what": "h0, a segment start every 4,096 steps, grad_last, grad_h0",
                              "fwd_ms": fms, "bwd_ms": bms,
                              "fwd_frac": fb / (fms * 1e-3) / 1e9 / peak,
                              "bwd_frac": bb / (bms * 1e-3) / 1e9 / peak,
                              "elements/s": 2 * E / ((fms + bms) * 1e-3),
                              "kernels": {d: L.lrscan_plan(B, T, D, "f32", d, state=True)["name"]
                                          for d in ("fwd", "bwd")}}
    a, b, g = a.bfloat16(), b.bfloat16(), g.bfloat16()
    out, ga, gb = torch.empty_like(a), torch.empty_like(a), torch.empty_like(a)
    fms = time_launches(lambda i: L.lrscan_fwd(a, b, out, last), 10, stream)
    bms = time_launches(lambda i: L.lrscan_bwd(a, out, g, ga, gb), 10, stream)
    if L.lrscan_sync_check() != 0:
        raise RuntimeError("device error while timing the long bf16 scan")
    res["auto_plan_bf16"] = {"fwd_ms": fms, "bwd_ms": bms,
                             "fwd_frac": 3 * E * 2 / (fms * 1e-3) / 1e9 / peak,
                             "bwd_frac": 5 * E * 2 / (bms * 1e-3) / 1e9 / peak,
                             "elements/s": 2 * E / ((fms + bms) * 1e-3),
                             "kernels": {d: L.lrscan_plan(B, T, D, "bf16", d)["name"] for d in ("fwd", "bwd")}}
    del a, b, g, out, ga, gb
    torch.cuda.empty_cache()
    return res


# Sources of the time-tiled real-scan kernels the benchmark's step runs (their
# code, shapes, stage counts and launch): DRAM counters recorded under another
# hash of these files are stale.
TILED_KERNEL_SOURCES = ("scan_common.cuh", "state_args.h", "window_kernels.cuh", "wavefront_kernels.cuh",
                        "window_shapes.h", "window_launch.cuh", "kernels_window.cu")


def kernel_source_hash() -> str:
    """Hash of the tiled kernels' sources (TILED_KERNEL_SOURCES)."""
    import hashlib
    csrc = os.path.join(ROOT, "linear_recurrence_scan_lrscan_gb300", "csrc")
    h = hashlib.sha256()
    for f in TILED_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def load_traffic(w, direction: str, kernel: str):
    """DRAM bytes (read + write) per launch of this kernel on this workload from
    a committed ncu summary (profiles/traffic.json), or None when there is none
    or the kernel sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    if d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("entries", {}).get(f"{w.name}:{direction}:{kernel}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4,
                    help="workload id 1..5 (default 4, the largest: B=16 T=4096 D=4096 bf16)")
    ap.add_argument("--sets", type=int, default=3,
                    help="rotating device buffer sets (1 keeps the footprint small, e.g. for a profiler)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the timing of the other named workloads")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default=None, choices=[None, "auto", "seq", "window", "chunk", "plain"])
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extensions", action="store_true",
                    help="skip the timing of the state-carrying, complex, generated-decay and long-sequence scans")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-elements", type=float, default=2e6)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.sets < 1:
        ap.error("--sets must be >= 1")

    from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.config]
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, w)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    line = run_ours(args, w, rank, world, dist)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
