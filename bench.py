#!/usr/bin/env python3
"""Benchmark of the uniform-grid build on GB300; prints one JSON line.

A step is one whole build (count, scan, scatter, gather: grid_build, one
cooperative launch of the bucketed build kernel) of the headline scene: 1,000,000 particles uniform in
[-5, 5)^3 on a 128^3 grid, 32-byte records, inputs resident in HBM.  L2 is
flushed (a 2 x L2-size buffer is written) between steps, outside the timed
events.  Per step the build is bracketed by CUDA events on the stream it is
launched on.

Further passes in the same run:
  * phase pass   — each per-phase entry point alone, L2 flushed before it:
                   per-kernel microseconds and the gather kernel's roofline;
  * end to end   — host buffers: pinned host origen -> device, build,
                   destino and inicios -> pinned host, all inside the events:
                   steps in turn on three streams, each with its own device
                   and host result arrays, over one timed region (`e2e`), and
                   each step alone between its own events (`e2e_serial`);
  * neighbours   — the neighbour query on SPH-like scenes (20 and 50
                   particles per cell on 64^3 cells), in linear and Morton
                   cell order, on the reordered records and through ordenado:
                   the reorder's gain and the Z-curve's;
  * workloads    — every workload (tiny, scan-dominated, headline,
                   contention, stress with its ten ping-pong builds), whole
                   builds with L2 flushed before each: microseconds,
                   algorithmic GB/s and the fraction of the HBM peak;
  * cpu baseline — the CPU oracle (single thread) on the same scene.

``--impl reference`` times the CPU oracle alone (the reference arm).
Under torchrun every rank builds its own replica of the scene ("replicas
only": the build does not shard); the reported time is the maximum over
ranks and the value counts every rank's particles.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grid-build Mparticles/s (count+scan+scatter+gather) at 1M/128³; HBM GB/s"
UNIT = "Mparticles/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers

def algorithmic_bytes(n: int, cells: int) -> dict:
    """Minimal bytes each phase must move (every array touched the fewest times
    the method allows; counter atomics stay in L2 and are not counted)."""
    return {
        "clear": 4 * cells,
        "count": 16 * n + 4 * n,          # pos+vida read, celdaDe write
        "scan": 4 * cells + 4 * (cells + 1),
        "clear_cursor": 4 * cells,
        "scatter": 12 * n,                # celdaDe, inicios[c], ordenado
        "gather": 68 * n,                 # ordenado, 32-B read, 32-B write
    }


def hbm_peak() -> tuple[float, str]:
    try:
        with open(PEAKS_FILE) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_traffic(sources: list[str]) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel (sha256 over its source files, in
    order, as named in the summary's first column joined by '+')."""
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "uniform_grid_particle_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    key, digest = "+".join(sources), h.hexdigest()
    for line in lines:
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == key:
            return float(parts[2]) if parts[1] == digest else None
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        self.out.flush()
        self.out.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.out.read())) if len(r) >= 9]
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = sorted({name for r in rows for name, v in zip(self.REASONS, r[5:9]) if "Active" in v and "Not" not in v})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    if int(os.environ.get("WORLD_SIZE", "1")) <= 1:
        return None
    import torch.distributed as dist

    backend = "nccl" if _cuda_ok() else "gloo"
    dist.init_process_group(backend)
    return dist


def _cuda_ok() -> bool:
    import torch

    return torch.cuda.is_available()


def max_over_ranks(value: float, dist) -> float:
    """Largest `value` over all ranks (the job is as slow as its slowest rank)."""
    if dist is None:
        return value
    import torch

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, n_per_rank: int, ms_per_step: float) -> float:
    """Whole-job Mparticles/s: every rank builds n_per_rank particles per step and
    the step lasts as long as the slowest rank's (ms_per_step is that maximum)."""
    return world * n_per_rank / (ms_per_step / 1e3) / 1e6


def barrier(dist) -> None:
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle

def oracle_timing(scene, rows, budget_s: float, min_runs: int = 3) -> dict:
    import oracle

    o = oracle.load()
    times = []
    start = time.perf_counter()
    while len(times) < min_runs or time.perf_counter() - start < budget_s:
        t0 = time.perf_counter()
        o.build(rows, scene.dims, scene.origin, scene.cell_size)
        times.append(time.perf_counter() - t0)
    per_build = statistics.median(times)
    return {"value": scene.n / per_build / 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"{len(times)} whole builds of the {scene.name} scene (N={scene.n}, "
                       f"{scene.dims[0]}^3 cells), single-threaded C oracle, median "
                       f"{per_build * 1e3:.1f} ms/build; host has {os.cpu_count()} cores")}


def run_reference(args) -> None:
    """The reference arm: the CPU oracle timed on this host's cores.

    Each step is one oracle build with the full grid.  When K + W whole builds
    would overrun the time budget, each step builds the first n_s particles of
    the scene instead (n_s chosen from a one-build calibration), and the
    sample says so."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from uniform_grid_particle_gb300 import scenes

    import oracle

    scene = scenes.SCENES[args.scene]
    rows = scene.particles()
    o = oracle.load()
    t0 = time.perf_counter()
    o.build(rows, scene.dims, scene.origin, scene.cell_size)
    t_full = time.perf_counter() - t0
    per_step = args.reference_budget / (args.steps + args.warmup)
    n_s = scene.n if t_full <= per_step else max(10_000, int(scene.n * per_step / t_full))
    sample = rows[:n_s]
    for _ in range(args.warmup):
        o.build(sample, scene.dims, scene.origin, scene.cell_size)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        o.build(sample, scene.dims, scene.origin, scene.cell_size)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = n_s / (ms / 1e3) / 1e6
    what = "whole builds" if n_s == scene.n else f"builds of the first {n_s:,} particles (full grid)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": workload_config(scene, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} {what} of the {scene.name} scene, single-threaded C oracle "
                                   f"({t_full * 1e3:.1f} ms per whole build); host has {os.cpu_count()} cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# fp32 lanes of the GPU (152 SMs x 128) and its maximum SM clock, for the
# neighbour query's arithmetic ceiling; operations in one distance test.
ALU_LANES = 152 * 128
ALU_CLOCK_GHZ = 2.07
PAIR_TEST_OPS = 7


def pair_tests(conteos, dims) -> int:
    """Distance tests of one neighbour query: for every particle, the
    particles of the (up to) 27 cells around its cell, itself included.
    conteos is in linear order (x fastest)."""
    import numpy as np

    gx, gy, gz = (int(d) for d in dims)
    c = conteos.astype(np.int64).reshape(gz, gy, gx)
    pad = np.pad(c, 1)
    around = np.zeros_like(c)
    for dz in range(3):
        for dy in range(3):
            for dx in range(3):
                around += pad[dz:dz + gz, dy:dy + gy, dx:dx + gx]
    return int((c * around).sum())


# The kernel one grid_build launches, non-stable and stable, and the sources
# its committed DRAM traffic is keyed by (None: no capture of that kernel).
BUILD_KERNEL = ("build_bucketed_kernel<false>", ["build_bucketed.cu", "fused_common.cuh"])
STABLE_KERNEL = ("build_bucketed_kernel<true>", None)


# The committed DRAM traffic was captured on this workload only.
TRAFFIC_SCENE = "headline"


def build_kernel(n: int, cells: int, stable: bool, sms: int) -> str:
    """The kernel grid_build launches for a scene of n particles on `cells`
    cells: the plan limits of the library's grid_build (cluster, one-CTA,
    sparse, bucketed), restated to label the timed launch."""
    mode = "true" if stable else "false"
    if n and not stable and n <= 32768 and cells <= 131072:
        return "build_cluster_kernel"
    if n and n <= 8192 and cells <= 8192:
        return f"build_small_kernel<{mode}>"
    if n and 4 * n <= cells and n <= 2 * sms * 1024:
        return f"build_sparse_kernel<{mode}>"
    return f"build_bucketed_kernel<{mode}>"


def roofline_entry(flags: int, total_alg: int, ms_per_step: float, peak: float, peak_kind: str,
                   scene_name: str = TRAFFIC_SCENE, kernel: str | None = None) -> dict:
    """The timed step is one launch of the build kernel: its algorithmic
    bytes are the whole build's, its duration the step's event time."""
    achieved = total_alg / (ms_per_step * 1e-3) / 1e9
    default_kernel, sources = BUILD_KERNEL if flags == 0 else STABLE_KERNEL
    kernel = kernel or default_kernel
    if scene_name != TRAFFIC_SCENE or kernel != default_kernel:
        sources = None
    return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
            "unit": "GB/s", "frac": achieved / peak, "algorithmic_bytes_per_launch": total_alg,
            "traffic": kernel_traffic(sources) if sources else None,
            "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS}


def workload_config(scene, args, kernel: str | None = None) -> dict:
    return {
        "workload": (f"{scene.name}: N={scene.n:,} particles, grid {scene.dims[0]}x{scene.dims[1]}x{scene.dims[2]}"
                     f" over [-5,5)^3, 32-byte Particula AoS, {scene.kind} positions"),
        "build": ("stable (ordenado ordered by particle index inside each cell)" if args.stable
                  else "atomic (order inside a cell unspecified)"),
        "l2": "flushed between steps (a 2x L2 buffer is written outside the timed events)",
        "launch": ("grid_build on a stream (C ABI): one launch of "
                   + (kernel or (STABLE_KERNEL[0] if args.stable else BUILD_KERNEL[0]))),
    }


# The five workloads, each timed as whole builds with L2 flushed before every
# build (the headline is the line's own value; it is timed again here so that
# every row comes from the same pass).
CONFIG_SCENES = ["tiny", "scan_dominated", "headline", "contention", "stress"]


def time_configs(ug, scenes, flags: int, steps: int, warmup: int, timed, settle, stream, peak: float,
                 sms: int) -> dict:
    """Per workload: mean and median microseconds per build, Mparticles/s,
    algorithmic GB/s and the fraction of the HBM peak.  The stress workload
    runs its ten ping-pong builds (each reads the previous build's destino)
    `max(1, steps // 10)` times from the original scene and reports build 1 and
    builds 2-10 apart."""
    import statistics

    import torch

    out = {}
    for name in CONFIG_SCENES:
        scene = scenes.SCENES[name]
        rows = scene.particles()
        n, cells = scene.n, scene.cells
        alg = sum(algorithmic_bytes(n, cells).values())
        p = ug.make_params(n, scene.dims, scene.origin, scene.cell_size)
        origen = torch.from_numpy(rows).cuda()
        del rows
        b = ug.GridBuffers.allocate(p, flags)

        def one(src, dst):
            ug.grid_build(src, dst.destino, dst.conteos, dst.celdaDe, dst.inicios, dst.ordenado, dst.ws, p,
                          flags, stream)

        def row(us: list[float]) -> dict:
            mean = statistics.mean(us)
            gbs = alg / (mean * 1e-6) / 1e9
            return {"us_mean": mean, "us_median": statistics.median(us), "mparticles_per_s": n / mean,
                    "achieved_gbs": gbs, "frac": gbs / peak, "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS}

        entry = {"n": n, "cells": cells, "algorithmic_bytes": alg, "kernel": build_kernel(n, cells, bool(flags), sms)}
        if scene.builds > 1:
            pong = ug.GridBuffers.allocate(p, flags)
            first, rest = [], []
            for k in range(warmup):
                settle(k)
                one(origen, b)
            for rep in range(max(1, steps // scene.builds)):
                src, bufs = origen, [b, pong]
                for k in range(scene.builds):
                    dst = bufs[k % 2]
                    ms = timed(lambda: one(src, dst), 1)[0]
                    (first if k == 0 else rest).append(1e3 * ms)
                    src = dst.destino
            for bufs_ in (b, pong):
                if ug.grid_status(bufs_.ws) != 0:
                    raise RuntimeError(f"device status set during the {name} builds")
            entry["build1"] = row(first)
            entry["builds_2_on"] = row(rest)
            entry["steps"] = {"build1": len(first), "builds_2_on": len(rest)}
            del pong
        else:
            for k in range(warmup):
                settle(k)
                one(origen, b)
            us = [1e3 * ms for ms in timed(lambda: one(origen, b), steps)]
            if ug.grid_status(b.ws) != 0:
                raise RuntimeError(f"device status set during the {name} builds")
            entry.update(row(us))
            entry["steps"] = steps
        out[name] = entry
        del b, origen
        torch.cuda.empty_cache()
    return out


def neighbour_query(ug, sph, warmup: int, steps: int, timed, settle, stream) -> dict:
    """grid_density on one SPH-like scene, in linear and Morton order, on the
    reordered records and through ordenado, L2 flushed before every step:
    microseconds, the reorder's gain, the Z-curve's, and the ALU roofline of
    the linear query on the reordered records."""
    import statistics

    import numpy as np
    import torch

    origen_s = torch.from_numpy(sph.particles()).cuda()
    rho = torch.empty(sph.n, dtype=torch.float32, device="cuda")
    h = sph.cell_size
    out = {
        "scene": f"{sph.name}: N={sph.n:,}, grid {sph.dims[0]}^3, h = cellSize = {h:.6f}",
        "mean_particles_per_cell": sph.n / sph.cells,
        "l2": "flushed between steps",
        "steps": steps,
    }
    tests = 0
    for order_name, order in (("linear", ug.GRID_ORDER_LINEAR), ("morton", ug.GRID_ORDER_MORTON)):
        ps = ug.make_params(sph.n, sph.dims, sph.origin, sph.cell_size, order=order)
        bs = ug.GridBuffers.allocate(ps)
        bs.build(origen_s, ps, stream=stream)

        def q_sorted():
            ug.grid_density(bs.destino, bs.inicios, rho, bs.ws, ps, h, stream=stream)

        def q_indirect():
            ug.grid_density(origen_s, bs.inicios, rho, bs.ws, ps, h, ordenado=bs.ordenado, stream=stream)

        for k in range(warmup):
            settle(k)
            q_sorted()
            q_indirect()
        sorted_ms = statistics.mean(timed(q_sorted, steps))
        indirect_ms = statistics.mean(timed(q_indirect, steps))
        if ug.grid_status(bs.ws) != 0:
            raise RuntimeError(f"device status {ug.grid_status(bs.ws)} after the neighbour query")
        out[f"us_{order_name}_sorted"] = 1e3 * sorted_ms
        out[f"us_{order_name}_indirect"] = 1e3 * indirect_ms
        if order == ug.GRID_ORDER_LINEAR:
            tests = pair_tests(bs.conteos.cpu().numpy().view(np.uint32), sph.dims)
        del bs
    out["reorder_gain"] = out["us_linear_indirect"] / out["us_linear_sorted"]
    out["morton_gain_sorted"] = out["us_linear_sorted"] / out["us_morton_sorted"]
    out["morton_gain_indirect"] = out["us_linear_indirect"] / out["us_morton_indirect"]
    best = min(out[f"us_{o}_sorted"] for o in ("linear", "morton"))
    out["mparticles_per_s_best"] = sph.n / best
    # The query does one distance test per (particle, candidate in its 27
    # cells): 7 fp32 operations (3 differences, 1 product, 2 fused
    # multiply-adds, 1 comparison).  Its ceiling is the fp32 lanes at the
    # maximum SM clock: 152 SMs x 128 lanes x 2.07 GHz / 7.
    tests_per_s = tests / (out["us_linear_sorted"] * 1e-6) / 1e9
    alu_peak = ALU_LANES * ALU_CLOCK_GHZ / PAIR_TEST_OPS
    out["roofline"] = {"bound": "alu", "kernel": "density_tile_kernel<0> (linear, reordered records)",
                       "achieved": tests_per_s, "peak": alu_peak, "unit": "Gpair-tests/s",
                       "frac": tests_per_s / alu_peak, "pair_tests_per_query": int(tests),
                       "peak_derivation": f"{ALU_LANES} fp32 lanes x {ALU_CLOCK_GHZ} GHz / "
                                          f"{PAIR_TEST_OPS} ops per test"}
    del origen_s, rho
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------- GPU arm

def run_gpu(args) -> None:
    import numpy as np
    import torch

    from uniform_grid_particle_gb300 import build as ugbuild
    from uniform_grid_particle_gb300 import scenes

    dist = dist_setup()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    ugbuild.build()
    from uniform_grid_particle_gb300 import ugrid as ug

    scene = scenes.SCENES[args.scene]
    rows = scene.particles()
    n, cells = scene.n, scene.cells
    flags = ug.GRID_STABLE if args.stable else 0
    p = ug.make_params(n, scene.dims, scene.origin, scene.cell_size)
    b = ug.GridBuffers.allocate(p, flags)
    origen = torch.from_numpy(rows).cuda()
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    step_kernel = build_kernel(n, cells, bool(flags), torch.cuda.get_device_properties(local).multi_processor_count)
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device="cuda")
    sleep = getattr(torch.cuda, "_sleep", None)

    def step():
        ug.grid_build(origen, b.destino, b.conteos, b.celdaDe, b.inicios, b.ordenado, b.ws, p, flags,
                      torch.cuda.current_stream())

    def settle(k, cold=True):
        """Untimed: flush L2 (unless warm), then hold the stream (~100 us of
        spinning on the GPU) so that the host has enqueued the whole step
        before the GPU reaches its start event."""
        if cold:
            flush.fill_(k & 0x7F)
        if sleep is not None:
            sleep(200_000)

    def timed(run, steps, cold=True):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier(dist)
        torch.cuda.synchronize()
        for k in range(steps):
            settle(k, cold)
            starts[k].record(stream)
            run()
            ends[k].record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        return [a.elapsed_time(e) for a, e in zip(starts, ends)]

    def check_status(where):
        if ug.grid_status(b.ws) != 0:
            raise RuntimeError(f"device status set during {where}")

    for k in range(args.warmup):
        settle(k)
        step()
    torch.cuda.synchronize()
    check_status("warm-up")

    # ---- the timed region: K whole builds ----
    with ClockSampler(local) as clocks:
        step_ms = timed(step, args.steps)
    check_status("the timed steps")
    total_ms = max_over_ranks(sum(step_ms), dist)
    ms_per_step = total_ms / args.steps
    value = job_rate(world, n, ms_per_step)
    kernels_per_step = 1   # one cooperative launch of the build kernel, stable or not

    # ---- the same build replayed from a CUDA graph ----
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step()
    for k in range(args.warmup):
        settle(k)
        graph.replay()
    graph_ms = timed(graph.replay, min(args.steps, args.graph_steps))
    check_status("the graph steps")

    # ---- warm L2, and an input already in cell order (context) ----
    warm_ms = timed(step, min(args.steps, args.graph_steps), cold=False)
    sorted_in = b.destino.clone()     # the last build's records: already in cell order
    b_sorted = ug.GridBuffers.allocate(p, flags)

    def step_sorted():
        ug.grid_build(sorted_in, b_sorted.destino, b_sorted.conteos, b_sorted.celdaDe, b_sorted.inicios,
                      b_sorted.ordenado, b_sorted.ws, p, flags, torch.cuda.current_stream())

    for k in range(args.warmup):
        settle(k)
        step_sorted()
    sorted_ms = timed(step_sorted, min(args.steps, args.graph_steps))
    if ug.grid_status(b_sorted.ws) != 0:
        raise RuntimeError("device status set during the sorted-input builds")
    del sorted_in, b_sorted
    context = {"warm_l2_us": 1e3 * statistics.mean(warm_ms),
               "sorted_input_us": 1e3 * statistics.mean(sorted_ms),
               "sorted_input": "the previous build's destino (particles already in cell order), L2 flushed"}

    # ---- repeated builds of one scene, origen and destino swapped (stress) ----
    if scene.builds > 1:
        pong = ug.GridBuffers.allocate(p, flags)
        src, bufs = origen.clone(), [b, pong]
        seq_ms = []
        for k in range(scene.builds):
            dst = bufs[k % 2]
            settle(k)
            a_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            ug.grid_build(src, dst.destino, dst.conteos, dst.celdaDe, dst.inicios, dst.ordenado, dst.ws, p, flags,
                          stream)
            e_ev.record(stream)
            torch.cuda.synchronize()
            seq_ms.append(a_ev.elapsed_time(e_ev))
            if ug.grid_status(dst.ws) != 0:
                raise RuntimeError("device status set during the ping-pong builds")
            src = dst.destino  # the next build reads this one's output, into the other buffers
        context["ping_pong"] = {"builds": scene.builds, "build1_us": 1e3 * seq_ms[0],
                                "builds_2_on_mean_us": 1e3 * statistics.mean(seq_ms[1:]),
                                "note": "build k+1 reads build k's destino; L2 flushed before each"}
        del pong, src

    # ---- phase pass: each phase alone, L2 flushed before each (cold) ----
    phase_names = ["clear", "count", "scan", "clear_cursor", "scatter", "gather"]
    calls = {
        "clear": lambda: ug.grid_clear(b.conteos, p, stream),
        "count": lambda: ug.grid_count(origen, b.conteos, b.celdaDe, p, stream),
        "scan": lambda: ug.grid_scan(b.conteos, b.inicios, b.ws, p, stream),
        "clear_cursor": lambda: ug.grid_clear(b.conteos, p, stream),
        "scatter": lambda: ug.grid_scatter(b.celdaDe, b.inicios, b.conteos, b.ordenado, b.ws, p, flags, stream),
        "gather": lambda: ug.grid_reorder(b.ordenado, origen, b.destino, b.ws, p, stream),
    }
    phase_ms = {k: [] for k in phase_names}
    for k in range(args.warmup + args.phase_steps):
        evs = []
        for name in phase_names:
            settle(k)
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            calls[name]()
            e.record(stream)
            evs.append((name, a, e))
        torch.cuda.synchronize()
        if k >= args.warmup:
            for name, a, e in evs:
                phase_ms[name].append(a.elapsed_time(e))
    check_status("the phase pass")
    phase_us = {k: 1e3 * statistics.mean(v) for k, v in phase_ms.items()}
    alg = algorithmic_bytes(n, cells)
    peak, peak_kind = hbm_peak()
    gather_gbs = alg["gather"] / (phase_us["gather"] * 1e-6) / 1e9

    # ---- the overflow diagnostics (f3) and the two-array gather (f4), cold ----
    diag = torch.zeros(2, dtype=torch.int32, device="cuda")
    hot = origen[:, :4].contiguous()    # pos, vida: the per-step state
    cold = origen[:, 4:].contiguous()   # vel, masa
    hot_out, cold_out = torch.empty_like(hot), torch.empty_like(cold)
    next_calls = {
        "diagnostics": lambda: ug.grid_diagnostics(b.conteos, diag, p, 64, stream),
        "reorder_many": lambda: ug.grid_reorder_many(b.ordenado, [(hot, hot_out), (cold, cold_out)], b.ws, p, stream),
    }
    next_ms = {k: [] for k in next_calls}
    for k in range(args.warmup + args.phase_steps):
        evs = []
        for name, call in next_calls.items():
            settle(k)
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            e.record(stream)
            evs.append((name, a, e))
        torch.cuda.synchronize()
        if k >= args.warmup:
            for name, a, e in evs:
                next_ms[name].append(a.elapsed_time(e))
    check_status("the diagnostics and the two-array gather")
    next_rows = {}
    for name, bytes_moved, what in (
            ("diagnostics", 4 * cells, "conteos read once (4 B per cell)"),
            ("reorder_many", 4 * n + 2 * 32 * n, "ordenado once, a 16-B hot and a 16-B cold record read and written")):
        us = 1e3 * statistics.mean(next_ms[name])
        achieved = bytes_moved / (us * 1e-6) / 1e9
        next_rows[name] = {"us": us, "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                                                  "unit": "GB/s", "frac": achieved / peak,
                                                  "algorithmic_bytes_per_launch": bytes_moved, "bytes": what}}
    next_rows["diagnostics"]["maxPorCelda_desbordes_at_64"] = [int(v) for v in diag.cpu().tolist()]
    del hot, cold, hot_out, cold_out

    # ---- end to end: host buffers, copies inside the events ----
    host_in = torch.from_numpy(rows).pin_memory()
    host_dest = torch.empty((n, 8), dtype=torch.float32).pin_memory()
    host_inicios = torch.empty(cells + 1, dtype=torch.int32).pin_memory()
    dev_in = torch.empty_like(origen)

    def e2e_step():
        # One C-ABI call: pinned host origen in, the build, destino and inicios out.
        ug.grid_build_host(host_in, host_dest, host_inicios, dev_in, b.destino, b.conteos, b.celdaDe, b.inicios,
                           b.ordenado, b.ws, p, flags, stream)

    for k in range(args.warmup):
        e2e_step()
    e2e_ms = timed(e2e_step, args.e2e_steps)
    check_status("the end-to-end pass")
    e2e_total = max_over_ranks(sum(e2e_ms), dist)
    e2e_value = job_rate(world, n, e2e_total / len(e2e_ms))
    e2e_serial = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(host_in.numel() * 4),
                  "d2h_bytes_per_step": int(host_dest.numel() * 4 + host_inicios.numel() * 4),
                  "ms_per_step": e2e_total / len(e2e_ms),
                  "note": "each step alone: L2 flushed and the stream held before it, one event pair per step"}
    if not np.array_equal(host_inicios.numpy()[[0, cells]], np.array([0, n], dtype=np.int32)):
        raise RuntimeError("end-to-end result is inconsistent")

    # ---- end to end, pipelined: --e2e-streams streams, each with its own
    # device and host result arrays, so that one step's copy in overlaps
    # another's copies out and the builds hide under the copies ----
    e2e_pipe = None
    if args.e2e_steps > 0:
        ways = max(2, args.e2e_streams)
        pipe_streams = [stream] + [torch.cuda.Stream() for _ in range(ways - 1)]
        pipe_bufs = [b] + [ug.GridBuffers.allocate(p, flags) for _ in range(ways - 1)]
        pipe_in = [dev_in] + [torch.empty_like(origen) for _ in range(ways - 1)]
        pipe_dest = [host_dest] + [torch.empty((n, 8), dtype=torch.float32).pin_memory() for _ in range(ways - 1)]
        pipe_inicios = [host_inicios] + [torch.empty(cells + 1, dtype=torch.int32).pin_memory()
                                         for _ in range(ways - 1)]

        def pipelined(count):
            for k in range(count):
                j = k % ways
                bj = pipe_bufs[j]
                ug.grid_build_host(host_in, pipe_dest[j], pipe_inicios[j], pipe_in[j], bj.destino, bj.conteos,
                                   bj.celdaDe, bj.inicios, bj.ordenado, bj.ws, p, flags, pipe_streams[j])

        pipelined(max(4, args.warmup))
        torch.cuda.synchronize()
        barrier(dist)
        settle(0)  # L2 flushed once, then the stream held while the host enqueues
        start = torch.cuda.Event(enable_timing=True)
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(ways)]
        start.record(pipe_streams[0])
        for j in range(1, ways):
            pipe_streams[j].wait_event(start)
        pipelined(args.e2e_steps)
        for j in range(ways):
            ends[j].record(pipe_streams[j])
        torch.cuda.synchronize()
        pipe_ms = max(start.elapsed_time(e) for e in ends)
        for bj in pipe_bufs:
            if ug.grid_status(bj.ws) != 0:
                raise RuntimeError("device status set during the pipelined end-to-end pass")
        for j in range(min(ways, args.e2e_steps)):
            if not np.array_equal(pipe_inicios[j].numpy()[[0, cells]], np.array([0, n], dtype=np.int32)):
                raise RuntimeError("pipelined end-to-end result is inconsistent")
        pipe_total = max_over_ranks(pipe_ms, dist)
        e2e_pipe = {"value": job_rate(world, n, pipe_total / args.e2e_steps), "unit": UNIT,
                    "ms_per_step": pipe_total / args.e2e_steps, "steps": args.e2e_steps, "streams": ways,
                    "h2d_bytes_per_step": int(host_in.numel() * 4),
                    "d2h_bytes_per_step": int(host_dest.numel() * 4 + host_inicios.numel() * 4),
                    "note": f"grid_build_host on {ways} streams in turn, one timed region over all steps; "
                            "L2 flushed once before it"}
        del pipe_bufs, pipe_in, pipe_dest, pipe_inicios

    # ---- neighbour query on SPH-like scenes: cell order x access path ----
    neighbour = neighbour_dense = None
    if args.density_steps > 0:
        neighbour = neighbour_query(ug, scenes.SCENES["sph"], args.warmup, args.density_steps, timed, settle, stream)
        neighbour_dense = neighbour_query(ug, scenes.SCENES["sph_dense"], args.warmup,
                                          max(3, args.density_steps // 4), timed, settle, stream)

    # ---- every workload, whole builds, L2 flushed before each ----
    configs = None
    if args.config_steps > 0:
        configs = time_configs(ug, scenes, flags, args.config_steps, args.warmup, timed, settle, stream, peak,
                               torch.cuda.get_device_properties(local).multi_processor_count)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    cpu = oracle_timing(scene, rows, args.cpu_budget) if world == 1 else None
    total_alg = sum(alg.values())
    gbs = lambda us: total_alg / (us * 1e-6) / 1e9  # noqa: E731
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": workload_config(scene, args, step_kernel),
        "roofline": roofline_entry(flags, total_alg, ms_per_step, peak, peak_kind, scene.name, step_kernel),
        "gather_roofline": {"kernel": "reorder_kernel (grid_reorder alone, L2 flushed before it)",
                            "achieved": gather_gbs, "peak": peak, "unit": "GB/s", "frac": gather_gbs / peak,
                            "algorithmic_bytes_per_launch": alg["gather"],
                            "traffic": kernel_traffic(["reorder.cu"]) if scene.name == TRAFFIC_SCENE else None},
        "build_hbm": {"algorithmic_bytes": total_alg, "us_per_build": ms_per_step * 1e3,
                      "us_min": 1e3 * min(step_ms), "us_median": 1e3 * statistics.median(step_ms),
                      "us_max": 1e3 * max(step_ms), "us_steps": [round(1e3 * t, 2) for t in step_ms[:200]],
                      "achieved_gbs": gbs(ms_per_step * 1e3),
                      "frac_of_nominal_8tbs": gbs(ms_per_step * 1e3) / NOMINAL_HBM_GBS,
                      "frac_of_measured": gbs(ms_per_step * 1e3) / peak},
        "graph": {"us_per_build": 1e3 * statistics.mean(graph_ms),
                  "us_median": 1e3 * statistics.median(graph_ms),
                  "value": n / (statistics.mean(graph_ms) / 1e3) / 1e6,
                  "frac_of_nominal_8tbs": gbs(1e3 * statistics.mean(graph_ms)) / NOMINAL_HBM_GBS},
        "context": context,
        "phases_us_cold": phase_us,
        "next_rows_cold": next_rows,
        "phases_gbs_cold": {k: alg[k] / (phase_us[k] * 1e-6) / 1e9 for k in phase_names},
        "cpu_baseline": cpu,
        # End to end through grid_build_host: scenes in turn on several streams
        # (the way a caller with a stream of scenes uses it), and each step alone.
        "e2e": e2e_pipe if e2e_pipe is not None else e2e_serial,
        "e2e_serial": e2e_serial,
        "neighbour_query": neighbour,
        "neighbour_query_dense": neighbour_dense,
        "configs": configs,
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--scene", default="headline")
    ap.add_argument("--stable", action="store_true", help="time the stable (reproducible) build")
    ap.add_argument("--graph-steps", type=int, default=2000)
    ap.add_argument("--density-steps", type=int, default=20,
                    help="steps of the neighbour-query leg (0 skips it)")
    ap.add_argument("--config-steps", type=int, default=30,
                    help="timed builds of each of the five workloads (0 skips that leg)")
    ap.add_argument("--phase-steps", type=int, default=500)
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="streams the end-to-end steps take in turn (at least 2)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time")
    ap.add_argument("--reference-budget", type=float, default=150.0,
                    help="seconds the --impl reference steps may take in all")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
