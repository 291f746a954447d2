#!/usr/bin/env python
"""Benchmark of batched gapped y-drop seed extension on GB300.

One step = one fz_extend_batch call over the whole synthetic batch: inspector,
wide-band inspector, length binning, executor and CIGAR emission (every row of
the hot path).  Inputs are resident in HBM when a step starts; L2 is flushed
(a 256 MiB write) between timed steps, outside the timed region.

Default workload: 100,000 right extensions in 6,000 bp windows with skewed
homology lengths (97% of homologies 8-128 bp), HOXD70, gap open 400, extend 30,
ydrop 9400.  Metric: GCUPS = live DP cells of the inspector sweeps per second
of the whole step; extensions/s is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fz|reference]

Multi-GPU (torchrun): every rank extends its own copy of the batch (weak
scaling), no collective on the data path; the step time is the max over ranks.
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
# (64 lanes/clk/SM each on GB300) + 2 adds (128 lanes/clk/SM): 4/64 SM-clocks per lane
# and cell, i.e. 16 cells/clk/SM with 32-bit lanes; x 152 SMs x 2.07 GHz max SM clock.
# The first-tier inspector keeps two cells in each 32-bit lane (16-bit halves) when the
# y-drop range allows it: the same instructions then advance two cells, 32 cells/clk/SM.
SMS, SM_MAX_GHZ, CELLS_PER_CLK_SM = 152, 2.07, 16.0
PEAK_GCUPS = SMS * SM_MAX_GHZ * CELLS_PER_CLK_SM


# Dominant kernel per mode: (name, source file, committed DRAM-traffic summary).
DOMINANT = {
    "extend": ("inspector (register-window sweep; first tier two 16-bit rows per register)", "extend_fast.cu",
               "inspector_traffic.json"),
    "local": ("local fill (k_local)", "local.cu", "local_traffic.json"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["fz", "reference"], default="fz")
    ap.add_argument("--config", type=int, default=2, help="workload id (1-5); default: the 100k x 6 kbp batch")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="bounded oracle sample for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--seeds", type=int, default=0, help="use only the first N seeds (profiling captures)")
    return ap.parse_args()


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


def cpu_baseline(w, seconds: float):
    """The oracle, as it stands, on a bounded seeded sample of the same workload,
    all host cores (a pthread pool over independent extensions)."""
    import oracle
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(123)
    probe = np.sort(rng.choice(len(w.seeds), size=min(len(w.seeds), 64), replace=False))
    t0 = time.perf_counter()
    res, _, _ = oracle.extend_batch(w, seeds=w.seeds[probe], nthreads=cores)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(len(w.seeds), max(64, len(probe) * seconds / dt)))
    idx = np.sort(rng.choice(len(w.seeds), size=n, replace=False))
    t0 = time.perf_counter()
    res, _, _ = oracle.extend_batch(w, seeds=w.seeds[idx], nthreads=cores)
    dt = time.perf_counter() - t0
    cells = int(res["live_cells"].sum())
    return {"value": cells / dt / 1e9, "unit": "GCUPS", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {len(w.seeds)} seeds (seeded), {cells} live cells, {dt:.1f} s",
            "extensions_per_s": int(np.count_nonzero(w.seeds[idx]["side"] & 1) +
                                    np.count_nonzero(w.seeds[idx]["side"] & 2)) / dt}


def traffic_for_current_kernel(mode, config):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, if it was taken on this workload and its source has not changed
    since the capture; else None."""
    import hashlib
    _, src_name, prof_name = DOMINANT[mode]
    try:
        prof = json.load(open(os.path.join(ROOT, "profiles", prof_name)))
        src = open(os.path.join(ROOT, "gapped_smith_waterman_gb300", "csrc", src_name), "rb").read()
        if prof.get("config") == config and prof.get("source_sha1") == hashlib.sha1(src).hexdigest():
            return prof.get("dram_bytes_per_launch_full_batch")
    except Exception:
        pass
    return None


def run_reference(args, ws, rank):
    if rank != 0:
        return
    w = W.make(args.config)
    import oracle
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(321)
    n = min(len(w.seeds), 200)
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
                             "sample": f"{n} random seeds per step of {len(w.seeds)}"},
            "e2e": {"value": v, "unit": "GCUPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, lrank = dist_env()
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
    w = W.make(args.config)
    t2, q2 = W.pack2(w.target), W.pack2(w.query)
    seeds = np.ascontiguousarray(w.seeds[:args.seeds] if args.seeds else w.seeds)
    ext = fz.Extender.for_workload(w, device=dev)
    fz.fz_set_profiling(ext.ctx, True)
    d_t, d_q, d_s = ext.upload(t2, q2, seeds)
    d_out = ext.alloc_out(len(seeds))
    side = seeds["side"].astype(np.int64)
    n_req = int(((side & 1) != 0).sum() + ((side & 2) != 0).sum())   # one-sided problems per step
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    rates = fz.fz_bench_int_rates() if rank == 0 else None

    for _ in range(args.warmup):
        ext.run(d_t, w.target.size, d_q, w.query.size, d_s, len(seeds), d_out)
        ext.stats()
    sampler = ClockSampler(lrank)
    step_ms, insp_ms, cells, launches, exts = [], [], 0, 0, 0
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
        insp_ms.append(st.phase_ms[0])
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
    value = ws * cells / (tot_ms * 1e-3) / 1e9
    ext_per_s = ws * exts / (tot_ms * 1e-3)
    insp_gcups = cells / (sum(insp_ms) * 1e-3) / 1e9 if sum(insp_ms) > 0 else None

    e2e = None
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(a).pin_memory().numpy()  # noqa: E731
        h_t, h_q, h_s = pin(t2), pin(q2), pin(seeds.view(np.uint8)).view(W.SEED_DTYPE)
        h_out = np.zeros(2 * len(seeds), fz.RESULT_DTYPE)
        st0 = ext.stats()
        h_cig = pin(np.zeros(int(st0.cigar_runs) + 16, np.uint32))
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
        e2e = {"value": ws * e2e_cells / e2e_s / 1e9, "unit": "GCUPS",
               "extensions_per_s": ws * ne * n_req / e2e_s,
               "h2d_bytes_per_step": int(t2.nbytes + q2.nbytes + seeds.nbytes), "d2h_bytes_per_step": int(d2h)}

    if rank != 0:
        ext.close()
        if ws > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline(w, args.cpu_seconds)
    mode = "local" if w.mode == W.MODE_LOCAL else "extend"
    cells_per_lane = 2 if fz.fz_pair_sweep_used(w.sub, w.gap_open, w.gap_extend, w.ydrop, w.mode) else 1
    peak = PEAK_GCUPS * cells_per_lane
    measured_peak = None
    if rates:
        r = rates
        measured_peak = cells_per_lane / (2.0 / r["viaddmax"] + 1.0 / r["vimax3"] + 2.0 / r["iadd"]) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GCUPS", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": w.name, "note": w.note, "extensions": int(exts / args.steps),
                   "scoring": "HOXD70, gap open 400, extend 30", "ydrop": w.ydrop, "max_len": w.max_len,
                   "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas x{ws}"},
        "extensions_per_s": ext_per_s,
        "live_cells_per_step": int(cells / args.steps),
        "roofline": {"bound": "alu", "kernel": DOMINANT[mode][0],
                     "achieved": insp_gcups, "peak": peak, "unit": "Gcell/s",
                     "frac": (insp_gcups / peak) if insp_gcups else None,
                     "peak_basis": (f"152 SM x 2.07 GHz x {16 * cells_per_lane} cells/clk/SM (2 DPX add-max + 1 DPX "
                                    "max3 at 64 lanes/clk, 2 adds at 128 lanes/clk per lane-cell; "
                                    + ("two 16-bit cells per 32-bit lane: the first-tier pair sweep)" if cells_per_lane == 2
                                       else "one 32-bit cell per lane)")),
                     "peak_measured_int_pipes": measured_peak,
                     "int_rates_gops": {k: v / 1e9 for k, v in (rates or {}).items()},
                     "traffic": traffic_for_current_kernel(mode, args.config),
                     "kernel_ms_per_step": sum(insp_ms) / args.steps},
        "phase_ms_last_step": [round(x, 4) for x in st.phase_ms],
        "phases": "inspector, wide inspector, bins+scans, executors, traceback+records, whole batch",
        "batch_stats": {"eager": int(st.eager), "bins": [int(b) for b in st.bin], "wide": int(st.wide), "retried_512": int(st.retried),
                        "executor_window_cells": int(st.exec_cells), "trace_bytes": int(st.trace_bytes),
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
