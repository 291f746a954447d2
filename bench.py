#!/usr/bin/env python
"""Benchmark of batched gapped y-drop seed extension on GB300.

One step = one fz_extend_batch call over the whole synthetic batch: inspector,
wide-band inspector, length binning, executor and CIGAR emission (every row of
the hot path).  Inputs are resident in HBM when a step starts; L2 is flushed
(a 256 MiB write) between timed steps, outside the timed region.

Default workload: the chromosome-scale batch, the largest configuration on one
GPU -- 1,000,000 seed anchors on a synthetic 50 Mbp target and a query derived
from it (15% substitutions, 3% indels, 10 kbp block inversions and moves),
extended on both sides in 6,000 bp windows (2,000,000 one-sided extensions),
HOXD70, gap open 400, extend 30, ydrop 9400.  --config 1|2|4|5 runs the others;
--wide runs a batch for the general-band path (512 extensions of 3 kbp windows
at a y-drop of 40,000, bands of about a thousand rows: workloads.make_wide), and
--dp edit|dtw the DPX article's other two dynamic programs.
Metric: GCUPS = live DP cells of the inspector sweeps per second of the whole
step; extensions/s is reported beside it.  The roofline line names the kernel
that took the most time in the timed steps (CUDA events on the library's stream
around its phases) and divides its own cells by its own time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fz|reference] [--config C | --wide | --dp P]

Multi-GPU (torchrun): the batch's seeds are split into contiguous shards, one
per rank (gapped_smith_waterman_gb300.multi.shard_bounds); every rank extends
its shard against its own copy of the sequences, with no collective on the
data path.  The total work is fixed (strong scaling); the step time is the max
over ranks and the cells are summed over them.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gapped_smith_waterman_gb300 import workloads as W  # noqa: E402

METRIC = "GCUPS and seed extensions/s (affine y-drop batch) at 1 GB300; % of DPX roofline"
# Roofline of the integer pipes: a Gotoh cell in DPX form is 2 add-max + 1 three-way max
# (64 lanes/clk/SM each on GB300) + 2 adds (128 lanes/clk/SM): 4/64 SM-clocks per lane and
# cell, i.e. 16 cells/clk/SM with one 32-bit cell per lane ("32").  The first-tier inspector
# keeps two cells in each 32-bit lane (16-bit halves) when the y-drop range allows it: the
# same instructions then advance two cells, 32 cells/clk/SM ("pair").  The traced pair sweep
# also decides each cell's four direction bits (4 packed subtractions per two cells, at
# 128 lanes/clk/SM): 6/64 SM-clocks per lane and two cells, 64/3 cells/clk/SM ("traced").
# SM count and maximum SM clock are read from the device at run time.
CELLS_PER_CLK_SM = {"32": 16.0, "pair": 32.0, "traced": 64.0 / 3.0}
MEASURED_RATE = {"32": "cell32_per_s", "pair": "cell16_per_s", "traced": "cell16_traced_per_s"}
CELL_BASIS = {"32": "2 DPX add-max + 1 DPX max3 at 64 lanes/clk, 2 adds at 128 lanes/clk, one 32-bit cell per lane",
              "pair": "2 DPX add-max + 1 DPX max3 at 64 lanes/clk, 2 adds at 128 lanes/clk per lane, two 16-bit "
                      "cells per lane (the first-tier pair sweep)",
              "traced": "2 DPX add-max + 1 DPX max3 at 64 lanes/clk, 2 adds + 4 direction tests at 128 lanes/clk "
                        "per lane, two 16-bit cells per lane (the traced pair sweep)"}

# Phases of one batch (fz_stats.phase_ms, index 6 = fz_stats.traced_ms) -> the kernel that
# runs in it: its name, source, cells (an fz_stats field, or a difference of two), its cell
# kind (pair kinds fall back to "32" when the pair sweep is off), and the committed
# DRAM-traffic summary of that kernel.
PHASES = {
    6: ("traced pair sweep (k_pair<true>: inspector that also stores direction codes and walks its best "
        "cell back; the extensions predicted long)", "extend_fast.cu", "traced_live_cells", "traced",
        "traced_traffic.json"),
    0: ("inspector (register-window sweep; first tier two 16-bit rows per register)", "extend_fast.cu",
        "plain_live_cells", "pair", "inspector_traffic.json"),
    1: ("inspector, wide band (k_wide<0>)", "extend_wide.cu", "live_cells", "32", None),
    3: ("executor (k_extend<K,1,*> / k_wide<1> replay with 4-bit direction codes)", "extend_fast.cu",
        "exec_live_cells", "32", "executor_traffic.json"),
    4: ("traceback walk and records (k_emit_*)", "pipeline.cu", None, "32", None),
}
LOCAL_KERNEL = ("local fill (k_local)", "local.cu", "live_cells", "32", "local_traffic.json")


def device_peaks(dev_index: int):
    """SM count (CUDA device properties) and maximum SM clock in GHz (nvidia-smi,
    else the driver's measured-peaks file, else GB300's nominal 2.07 GHz)."""
    import torch
    sms = torch.cuda.get_device_properties(dev_index).multi_processor_count
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(dev_index), "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20).stdout
        return sms, float(out.strip().splitlines()[0]) / 1e3, "nvidia-smi clocks.max.sm"
    except Exception:
        pass
    try:
        return sms, json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["sm_max_mhz"] / 1e3, \
            "MEASURED_PEAKS.json sm_max_mhz"
    except Exception:
        return sms, 2.07, "nominal GB300 maximum"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["fz", "reference"], default="fz")
    ap.add_argument("--config", type=int, default=3,
                    help="workload id (1-5); default: 3, 1M two-sided anchors on a 50 Mbp pair")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="bounded oracle sample for cpu_baseline")
    ap.add_argument("--ref-step-seconds", type=float, default=6.0,
                    help="reference arm: oracle time per step (sets its seeds per step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--seeds", type=int, default=0, help="use only the first N seeds (profiling captures)")
    ap.add_argument("--wide", action="store_true",
                    help="time the general-band path instead: 512 extensions of 3 kbp windows at y-drop 40,000")
    ap.add_argument("--dp", choices=["edit", "dtw"], default=None,
                    help="time the DPX article's other dynamic programs instead (512 edit distances of "
                         "1024 x 1024, or 256 DTWs of 800 x 800)")
    return ap.parse_args()


def rank_seeds(seeds, rank: int, ws: int):
    """The contiguous shard of the batch's seeds that rank `rank` of `ws`
    extends (all of them for one rank)."""
    from gapped_smith_waterman_gb300.multi import shard_bounds
    lo, hi = shard_bounds(len(seeds), rank, ws)
    return np.ascontiguousarray(seeds[lo:hi])


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    lrank = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, lrank


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clocks not sampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_model() -> str:
    """Host CPU model (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_sample(w, rng, seconds, threads):
    """A seeded sample of the workload's seeds sized to about `seconds` of oracle
    time on `threads` threads; returns (GCUPS, extensions/s, description)."""
    import oracle
    probe = np.sort(rng.choice(len(w.seeds), size=min(len(w.seeds), max(8, 4 * threads)), replace=False))
    t0 = time.perf_counter()
    oracle.extend_batch(w, seeds=w.seeds[probe], nthreads=threads)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(len(w.seeds), max(len(probe), len(probe) * seconds / dt)))
    idx = np.sort(rng.choice(len(w.seeds), size=n, replace=False))
    t0 = time.perf_counter()
    res, _, _ = oracle.extend_batch(w, seeds=w.seeds[idx], nthreads=threads)
    dt = time.perf_counter() - t0
    cells = int(res["live_cells"].sum())
    side = w.seeds["side"][idx]
    nx = int(np.count_nonzero(side & 1) + np.count_nonzero(side & 2))
    return cells / dt / 1e9, nx / dt, f"{n} of {len(w.seeds)} seeds (seeded), {cells} live cells, {dt:.1f} s"


def cpu_baseline(w, seconds: float):
    """The oracle, as it stands, on bounded seeded samples of the same workload:
    on all host cores (a pthread pool over independent extensions) and on one
    thread."""
    cores = os.cpu_count() or 1
    v, xs, desc = _oracle_sample(w, np.random.default_rng(123), seconds, cores)
    v1, xs1, desc1 = _oracle_sample(w, np.random.default_rng(124), max(2.0, seconds / 3), 1)
    return {"value": v, "unit": "GCUPS", "cores": cores, "kind": "oracle", "sample": desc,
            "extensions_per_s": xs, "cpu_model": cpu_model(),
            "single_thread": {"value": v1, "unit": "GCUPS", "cores": 1, "extensions_per_s": xs1,
                              "sample": desc1}}


def traffic_for_kernel(kernel, config):
    """DRAM bytes per step of the named kernel from its committed ncu summary, if
    it was taken on this workload and its source has not changed since the
    capture; else None."""
    import hashlib
    _, src_name, _, _, prof_name = kernel
    if not prof_name:
        return None
    try:
        prof = json.load(open(os.path.join(ROOT, "profiles", prof_name)))
        src = open(os.path.join(ROOT, "gapped_smith_waterman_gb300", "csrc", src_name), "rb").read()
        if prof.get("config") == config and prof.get("source_sha1") == hashlib.sha1(src).hexdigest():
            return prof.get("dram_bytes_per_launch_full_batch")
    except Exception:
        pass
    return None


def run_reference(args, ws, rank):
    """The reference arm: the oracle, as it stands, on the host cores.  Each step
    extends a fresh seeded sample of the workload's seeds, sized by a probe so
    that one step takes about --ref-step-seconds."""
    if rank != 0:
        return
    w = W.make_wide() if args.wide else W.make(args.config)
    import oracle
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(321)
    probe = np.sort(rng.choice(len(w.seeds), size=min(len(w.seeds), 2 * cores), replace=False))
    t0 = time.perf_counter()
    oracle.extend_batch(w, seeds=w.seeds[probe], nthreads=cores)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(len(w.seeds), max(cores, len(probe) * args.ref_step_seconds / dt)))
    times, cells = [], 0
    for step in range(args.warmup + args.steps):
        idx = np.sort(rng.choice(len(w.seeds), size=n, replace=False))
        t0 = time.perf_counter()
        res, _, _ = oracle.extend_batch(w, seeds=w.seeds[idx], nthreads=cores)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            cells += int(res["live_cells"].sum())
    tot = sum(times)
    v = cells / tot / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GCUPS", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": w.name, "note": w.note, "sample_per_step": f"{n} seeds"},
            "cpu_baseline": {"value": v, "unit": "GCUPS", "cores": cores, "kind": "oracle",
                             "sample": f"{n} random seeds per step of {len(w.seeds)}", "cpu_model": cpu_model()},
            "e2e": {"value": v, "unit": "GCUPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# Nominal integer-pipe peaks of the other two dynamic programs (cells/clk/SM,
# one 32-bit cell per lane): edit distance = DPX add-min (64 lanes/clk) + a
# min and an add (128 lanes/clk) = 2/64 SM-clocks per lane and cell; DTW =
# DPX 3-way min (64) + |x - y| as a subtraction and an absolute value + the
# add (128) = 2.5/64.
DP_CELLS_PER_CLK_SM = {"edit": 32.0, "dtw": 25.6}


def run_dp(args, ws, rank, lrank):
    """The DPX article's other dynamic programs: one step = one batch through
    fz_edit_distance_batch / fz_dtw_batch, inputs resident in HBM."""
    import torch
    from gapped_smith_waterman_gb300 import build as B
    from gapped_smith_waterman_gb300 import fz
    torch.cuda.set_device(lrank)
    dev = torch.device("cuda", lrank)
    B.build()
    w = W.make_edit_batch() if args.dp == "edit" else W.make_dtw_batch()
    if w.kind == "edit":
        da, db = (torch.from_numpy(W.pack2(x)).to(dev) for x in (w.a, w.b))
    else:
        da, db = (torch.from_numpy(np.ascontiguousarray(x, np.int32)).to(dev) for x in (w.a, w.b))
    dp = torch.from_numpy(np.ascontiguousarray(w.pairs).view(np.uint8)).to(dev)
    out = torch.empty(len(w.pairs), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fn = fz.fz_edit_distance_batch if w.kind == "edit" else fz.fz_dtw_batch
    call = lambda: fn(da.data_ptr(), len(w.a), db.data_ptr(), len(w.b), dp.data_ptr(), len(w.pairs),  # noqa: E731
                      out.data_ptr(), stream.cuda_stream)
    cells = int((w.pairs["a_len"].astype(np.int64) * w.pairs["b_len"].astype(np.int64)).sum())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(lrank)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0.0
    for _ in range(args.steps):
        flush.fill_(1)
        torch.cuda.synchronize()
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    clocks = sampler.stop()
    value = cells * args.steps / (tot * 1e-3) / 1e9
    sms, ghz, clock_src = device_peaks(lrank)
    peak = sms * ghz * DP_CELLS_PER_CLK_SM[w.kind]
    # e2e: host inputs copied in, results copied out, inside the timed region
    h_a = torch.from_numpy(W.pack2(w.a) if w.kind == "edit" else np.ascontiguousarray(w.a, np.int32)).pin_memory()
    h_b = torch.from_numpy(W.pack2(w.b) if w.kind == "edit" else np.ascontiguousarray(w.b, np.int32)).pin_memory()
    h_p = torch.from_numpy(np.ascontiguousarray(w.pairs).view(np.uint8)).pin_memory()
    h_o = torch.empty(len(w.pairs), dtype=torch.int32).pin_memory()
    ne, e2e_s = max(1, min(args.steps, 5)), 0.0
    for _ in range(ne):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        da.copy_(h_a, non_blocking=True)
        db.copy_(h_b, non_blocking=True)
        dp.copy_(h_p, non_blocking=True)
        call()
        h_o.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        e2e_s += time.perf_counter() - t0
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        f = oracle.edit_distance if w.kind == "edit" else oracle.dtw
        n = 0
        t0 = time.perf_counter()
        while n < len(w.pairs) and time.perf_counter() - t0 < max(1.0, args.cpu_seconds / 3):
            oracle.pairs_batch(f, w.a, w.b, w.pairs[n:n + 1])
            n += 1
        dt = time.perf_counter() - t0
        c = int((w.pairs["a_len"][:n].astype(np.int64) * w.pairs["b_len"][:n].astype(np.int64)).sum())
        cpu = {"value": c / dt / 1e9, "unit": "GCUPS", "cores": 1, "kind": "oracle",
               "sample": f"{n} of {len(w.pairs)} pairs, one thread, {dt:.1f} s", "cpu_model": cpu_model()}
    line = {"metric": f"GCUPS of the batched {'edit distance' if w.kind == 'edit' else 'dynamic time warping'} "
                      "at 1 GB300", "value": value, "unit": "GCUPS", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": w.name, "note": w.note, "cells_per_step": cells,
                       "l2": "flushed between steps (256 MiB write)"},
            "roofline": {"bound": "alu", "kernel": f"k_dp<{w.kind == 'dtw'}>", "achieved": value, "peak": peak,
                         "unit": "Gcell/s", "frac": value / peak,
                         "peak_basis": f"{sms} SM x {ghz:.3f} GHz ({clock_src}) x {DP_CELLS_PER_CLK_SM[w.kind]} "
                                       "cells/clk/SM", "traffic": None},
            "gpu_launches": args.steps, "clocks": clocks,
            "e2e": {"value": cells * ne / e2e_s / 1e9, "unit": "GCUPS",
                    "h2d_bytes_per_step": int(h_a.numel() * h_a.element_size() + h_b.numel() * h_b.element_size()
                                              + h_p.numel()),
                    "d2h_bytes_per_step": int(h_o.numel() * 4)},
            "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, lrank = dist_env()
    if args.dp:
        if rank == 0:
            run_dp(args, ws, rank, lrank)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    import torch
    import torch.distributed as dist
    from gapped_smith_waterman_gb300 import build as B
    from gapped_smith_waterman_gb300 import fz
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(lrank)
    dev = torch.device("cuda", lrank)
    if rank == 0:
        B.build()
    if ws > 1:
        dist.barrier()
    w = W.make_wide() if args.wide else W.make(args.config)
    t2, q2 = W.pack2(w.target), W.pack2(w.query)
    seeds = rank_seeds(w.seeds[:args.seeds] if args.seeds else w.seeds, rank, ws)
    ext = fz.Extender.for_workload(w, device=dev)
    fz.fz_set_profiling(ext.ctx, True)
    d_t, d_q, d_s = ext.upload(t2, q2, seeds)
    d_out = ext.alloc_out(len(seeds))
    side = seeds["side"].astype(np.int64)
    n_req = int(((side & 1) != 0).sum() + ((side & 2) != 0).sum())   # one-sided problems per step
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        ext.run(d_t, w.target.size, d_q, w.query.size, d_s, len(seeds), d_out)
        ext.stats()
    rates = None
    if rank == 0:
        # integer-pipe rates on a warm GPU, the better of two runs of each (a run
        # in a process's first moments once read 200x low)
        r1, r2 = fz.fz_bench_int_rates(), fz.fz_bench_int_rates()
        rates = {k: max(r1[k], r2[k]) for k in r1}
    sampler = ClockSampler(lrank)
    step_ms, cells, launches, exts = [], 0, 0, 0
    phase_tot = [0.0] * 7                      # device ms per phase over the timed steps (6: traced sweep)
    stat_tot = {"live_cells": 0, "exec_live_cells": 0, "traced_live_cells": 0, "plain_live_cells": 0}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    for _ in range(args.steps):
        flush.fill_(1)
        torch.cuda.synchronize()
        e0.record(stream)
        ext.run(d_t, w.target.size, d_q, w.query.size, d_s, len(seeds), d_out)
        e1.record(stream)
        st = ext.stats()                       # synchronises the stream
        step_ms.append(e0.elapsed_time(e1))
        for k in range(6):
            phase_tot[k] += st.phase_ms[k]
        phase_tot[6] += st.traced_ms
        stat_tot["live_cells"] += st.live_cells
        stat_tot["exec_live_cells"] += st.exec_live_cells
        stat_tot["traced_live_cells"] += st.traced_live_cells
        stat_tot["plain_live_cells"] += st.live_cells - st.traced_live_cells
        cells += st.live_cells
        launches += st.launches
        exts += st.extensions if w.mode == 0 else n_req
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if ws > 1:
        dist.barrier()
    tot_ms = sum(step_ms)
    if ws > 1:
        t = torch.tensor([tot_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        tot_ms = float(t.item())
        c = torch.tensor([float(cells), float(exts)], dtype=torch.float64, device=dev)
        dist.all_reduce(c, op=dist.ReduceOp.SUM)      # every rank's shard
        cells, exts = int(c[0].item()), int(c[1].item())
    value = cells / (tot_ms * 1e-3) / 1e9
    ext_per_s = exts / (tot_ms * 1e-3)

    e2e = None
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(a).pin_memory().numpy()  # noqa: E731
        h_t, h_q, h_s = pin(t2), pin(q2), pin(seeds.view(np.uint8)).view(W.SEED_DTYPE)
        h_out = pin(np.zeros(2 * len(seeds), fz.RESULT_DTYPE).view(np.uint8)).view(fz.RESULT_DTYPE)
        res_dev = np.frombuffer(d_out[:2 * len(seeds) * fz.RESULT_DTYPE.itemsize].cpu().numpy().tobytes(),
                                dtype=fz.RESULT_DTYPE)
        h_cig = pin(np.zeros(int(res_dev["cigar_len"].astype(np.int64).sum()) + 16, np.uint32))   # runs written
        ne, e2e_s, e2e_cells, d2h = max(1, min(args.steps, 5)), 0.0, 0, 0
        fz.fz_extend_batch_host(ext.ctx, h_t, w.target.size, h_q, w.query.size, h_s, h_out, h_cig, stream.cuda_stream)
        for _ in range(ne):
            flush.fill_(1)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            used = fz.fz_extend_batch_host(ext.ctx, h_t, w.target.size, h_q, w.query.size, h_s, h_out, h_cig,
                                           stream.cuda_stream)
            e2e_s += time.perf_counter() - t0
            e2e_cells += ext.stats().live_cells
            d2h = h_out.nbytes + 4 * used
        e2e_x = ne * n_req
        if ws > 1:
            t = torch.tensor([e2e_s], dtype=torch.float64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            c = torch.tensor([float(e2e_cells), float(e2e_x)], dtype=torch.float64, device=dev)
            dist.all_reduce(c, op=dist.ReduceOp.SUM)
            e2e_s, e2e_cells, e2e_x = float(t.item()), int(c[0].item()), int(c[1].item())
        e2e = {"value": e2e_cells / e2e_s / 1e9, "unit": "GCUPS",
               "extensions_per_s": e2e_x / e2e_s,
               "h2d_bytes_per_step": int(t2.nbytes + q2.nbytes + seeds.nbytes), "d2h_bytes_per_step": int(d2h)}

    if rank != 0:
        ext.close()
        if ws > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline(w, args.cpu_seconds)
    # the roofline names the kernel with the largest share of the timed steps
    if w.mode == W.MODE_LOCAL:
        kernel, kphase = LOCAL_KERNEL, 0
    else:
        kphase = max(PHASES, key=lambda k: phase_tot[k])
        if PHASES[kphase][2] is None:         # (the walk has no cell count: report the sweeps)
            kphase = 0
        kernel = PHASES[kphase]
    kname, _, kcells_field, kind, _ = kernel
    pair = fz.fz_pair_sweep_used(w.sub, w.gap_open, w.gap_extend, w.ydrop, w.mode)
    if kind == "pair" and not pair:
        kind = "32"
    sms, ghz, clock_src = device_peaks(lrank)
    peak = sms * ghz * CELLS_PER_CLK_SM[kind]
    k_ms = phase_tot[kphase]
    achieved = stat_tot[kcells_field] / (k_ms * 1e-3) / 1e9 if k_ms > 0 else None
    measured_peak = rates[MEASURED_RATE[kind]] / 1e9 if rates else None
    line = {
        "metric": METRIC, "value": value, "unit": "GCUPS", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_ms / args.steps, "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": w.name, "note": w.note, "extensions": int(exts / args.steps),
                   "scoring": "HOXD70, gap open 400, extend 30", "ydrop": w.ydrop, "max_len": w.max_len,
                   "l2": "flushed between steps (256 MiB write)",
                   "parallelism": f"contiguous seed shards x{ws}" if ws > 1 else "one GPU"},
        "extensions_per_s": ext_per_s,
        "live_cells_per_step": int(cells / args.steps),
        "roofline": {"bound": "alu", "kernel": kname,
                     "achieved": achieved, "peak": peak, "unit": "Gcell/s",
                     "frac": (achieved / peak) if achieved else None,
                     "cells": f"{kcells_field} of the timed steps / the kernel's phase time (CUDA events)",
                     "kernel_share_of_step": k_ms / tot_ms if tot_ms > 0 else None,
                     "peak_basis": (f"{sms} SM x {ghz:.3f} GHz ({clock_src}) x {CELLS_PER_CLK_SM[kind]:.2f} "
                                    f"cells/clk/SM ({CELL_BASIS[kind]})"),
                     "peak_measured_int_pipes": measured_peak,
                     "frac_of_measured": (achieved / measured_peak) if (achieved and measured_peak) else None,
                     "measured_basis": f"fz_bench_int_rates {MEASURED_RATE[kind]} (the costed cell loop)",
                     "int_rates_gops": {k: v / 1e9 for k, v in (rates or {}).items()},
                     "traffic": traffic_for_kernel(kernel, "wide" if args.wide else args.config),
                     "traffic_unit": "DRAM bytes per step of this kernel (ncu, scaled to the full batch)",
                     "kernel_ms_per_step": k_ms / args.steps},
        "phase_ms_per_step": [round(x / args.steps, 4) for x in phase_tot],
        "phases": ("plain inspector, wide inspector, bins+scans, executors, traceback+records, whole batch, "
                   "traced sweep (with the work order)"),
        "batch_stats": {"eager": int(st.eager), "bins": [int(b) for b in st.bin], "traced": int(st.traced),
                        "traced_live_cells": int(st.traced_live_cells), "live_cells": int(st.live_cells),
                        "wide": int(st.wide), "retried_512": int(st.retried),
                        "executor_window_cells": int(st.exec_cells), "executor_live_cells": int(st.exec_live_cells),
                        "trace_bytes": int(st.trace_bytes),
                        "cigar_slot_runs": int(st.cigar_runs)},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    ext.close()
    if ws > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
