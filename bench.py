#!/usr/bin/env python
"""Throughput of the WaveFilter per-layer, per-step KV-filtering path.

One step = one pass of the whole path (Haar low-pass, coarse scoring + Top-K,
recursive filtering, sparse gather + eq. (3) attention) over one layer of the
workload, through the C ABI.  Metric: cached prompt tokens filtered+attended
per second per layer-step (batch * layers * N_p per step), plus the achieved
HBM bandwidth of the dominant kernel against the measured peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the float64 CPU oracle as the reference arm

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the units of the path are independent; there is no data-path collective)
and rank 0 prints one JSON line with the whole-job throughput.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from wavelet_guided_sparse_gb300 import workloads as wl  # noqa: E402

METRIC = "cached prompt tokens filtered+attended/sec per layer-step; HBM GB/s vs peak"
DEFAULT_CONFIG = "llada8b_layer"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) of one dwt_lowpass launch on the default workload,
# from an ncu capture of the kernel source with this SHA-256 prefix; null
# once the kernel has changed since the counters were taken.
# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture
# of the 4096-token layer (profiles/), valid while the kernel sources (without
# comments and blank space) hash to source_sha.
DWT_TRAFFIC = {"sources": ("wf_dwt.cu",), "source_sha": "65d64d392b075f89",
               "bytes_per_launch": 33577984}  # 33.58 MB read + 0 B written (A_L stays in L2)
PATH_TRAFFIC = {"sources": ("wf_path.cu", "wf_common.cuh", "wf_mma.cuh", "wf_umma.cuh"),
                "source_sha": "4e8b7fafc8ea55e4",
                "bytes_per_launch": 38690048}  # 38.69 MB read + 3.3 KB written
# One cold launch: the reads are the K/V bytes exactly; most of the 71.6 MB
# of cache writes are still in L2 when the kernel ends (written back later).
CACHE_TRAFFIC = {"sources": ("wf_cache.cu", "wf_common.cuh"), "source_sha": "d9a8f99a6f16b2e0",
                 "bytes_per_launch": 81929216}  # 67.65 MB read + 14.28 MB written


def _rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _workload_desc(cfg: wl.WorkloadConfig) -> str:
    ks = cfg.k_per_level()
    return (f"{cfg.name}: batch={cfg.batch}, layers=1 of {cfg.layers}, H={cfg.heads}, "
            f"d={cfg.head_dim}, N_p={cfg.n_prompt}, G={cfg.n_gen}, {cfg.dtype}, "
            f"Haar L={cfg.levels}, k_L={ks[-1]}, budget B={cfg.budget}")


def _config_obj(cfg, extra=None):
    ks = cfg.k_per_level()
    obj = {"workload": _workload_desc(cfg), "batch": cfg.batch, "layers_per_step": 1,
           "heads": cfg.heads, "head_dim": cfg.head_dim, "n_prompt": cfg.n_prompt,
           "n_gen": cfg.n_gen, "levels": cfg.levels, "k_per_level": ks,
           "budget": cfg.budget, "parallelism": "replicas"}
    if extra:
        obj.update(extra)
    return obj


def tokens_per_step(cfg) -> int:
    return cfg.batch * 1 * cfg.n_prompt


def path_bytes(cfg) -> dict:
    """Algorithmic HBM bytes of one step (one layer), by stage."""
    e = 2 if cfg.dtype == "bf16" else 4
    U, d, n, g, L = cfg.units_per_layer, cfg.head_dim, cfg.n_prompt, cfg.n_gen, cfg.levels
    ks = cfg.k_per_level()
    P, B = n >> L, ks[0]
    rows = ks[L] << L
    return {
        "dwt": U * (n * d * e + P * d * 4),
        "score": U * (P * d * 4 + g * d * e + ks[L] * 4),
        "filter": U * (rows * d * e + g * d * e + ks[L] * 4 + B * 4),
        "attn": U * (2 * B * d * e + 2 * g * d * e + g * d * e + B * 4 + g * d * 4),
    }


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def allreduce_max(value: float, world: int, device) -> float:
    """The largest of every rank's value (the slowest rank's time); one rank: itself."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, tokens: int, steps: int, t_ms: float) -> float:
    """Whole-job throughput: every replica processes `tokens` per step."""
    return world * tokens * steps / (t_ms / 1e3)


def cache_init_bytes(cfg) -> int:
    """Algorithmic HBM bytes of one wf_cache_init: K and V of every position
    read once and written once, plus the fp32 A_L of the prompt keys."""
    e = 2 if cfg.dtype == "bf16" else 4
    rows = cfg.n_prompt + cfg.n_gen
    return (4 * cfg.units_per_layer * rows * cfg.head_dim * e +
            cfg.units_per_layer * (cfg.n_prompt >> cfg.levels) * cfg.head_dim * 4)


def step_bytes(cfg, fused: bool) -> int:
    """Algorithmic HBM bytes of one wf_step; the fused step never writes or
    reads A_L in global memory."""
    total = sum(path_bytes(cfg).values())
    if fused:
        total -= 2 * cfg.units_per_layer * (cfg.n_prompt >> cfg.levels) * cfg.head_dim * 4
    return total


def _strip_comments(text: str) -> str:
    """C++ source without comments and blank space (comment edits leave the
    kernel, and so its measured traffic, unchanged)."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return "".join("".join(out).split())


def _source_sha(names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "wavelet_guided_sparse_gb300", "csrc", n)) as f:
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic(table):
    """ncu DRAM bytes per launch, if the kernel sources are the profiled ones."""
    try:
        sha = _source_sha(table["sources"])
    except OSError:
        return None
    return table["bytes_per_launch"] if table["source_sha"] == sha else None


class ClockSampler:
    """nvidia-smi clock/throttle samples while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", device_index],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # Samples under load: power above the midpoint of the observed range.
        lo, hi = min(power), max(power)
        loaded = [s for s, p in zip(sm, power) if p >= (lo + hi) / 2] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": hi}


# ------------------------------------------------------------------ CPU oracle

def _oracle_unit(args):
    q, kp, vp, kg, vg, levels, ks = args
    import oracle.wavefilter_oracle as wo
    wo.wavefilter_step(q, kp, vp, kg, vg, levels, ks)
    return 1


def _oracle_pool(workers):
    import concurrent.futures
    import multiprocessing
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    ctx = multiprocessing.get_context("spawn")
    return concurrent.futures.ProcessPoolExecutor(max_workers=workers, mp_context=ctx)


def _unit_jobs(arrs, cfg, units):
    ks = cfg.k_per_level()
    jobs = []
    for u in units:
        b, h = divmod(u, cfg.heads)
        jobs.append((arrs["Q"][b, h], arrs["Kp"][b, h], arrs["Vp"][b, h], arrs["Kg"][b, h],
                     arrs["Vg"][b, h], cfg.levels, ks))
    return jobs


def cpu_oracle_rate(arrs, cfg, budget_s: float, workers: int):
    """Oracle tokens/s on a bounded sample: whole units, all host cores."""
    U = cfg.units_per_layer
    with _oracle_pool(workers) as pool:
        list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, [0] * workers)))  # start workers
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            n = min(U, max(workers, 1))
            units = [(done + i) % U for i in range(n)]
            list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, units)))
            done += n
        elapsed = time.perf_counter() - t0
    tokens = done / U * tokens_per_step(cfg)
    return tokens / elapsed, done, elapsed


# ------------------------------------------------------------------ arms

def run_reference(args, cfg):
    rank, world, _ = _rank_env()
    if rank != 0:
        return 0
    arrs = wl.generate_layer(cfg, 0, workers=min(16, os.cpu_count() or 1))
    workers = os.cpu_count() or 1
    U = cfg.units_per_layer
    # Size each step's sample so the whole run takes about two minutes.
    with _oracle_pool(workers) as pool:
        list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, [0] * workers)))
        t0 = time.perf_counter()
        list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, list(range(min(U, workers))))))
        per_round = time.perf_counter() - t0
        rounds = max(1, min(math.ceil(U / workers),
                            int(120.0 / max(per_round * (args.steps + args.warmup), 1e-9))))
        sample_units = min(U, rounds * workers)
        for i in range(args.warmup):
            list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, list(range(sample_units)))))
        t0 = time.perf_counter()
        for i in range(args.steps):
            units = [(i * sample_units + j) % U for j in range(sample_units)]
            list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, units)))
        elapsed = time.perf_counter() - t0
    frac = sample_units / U
    value = args.steps * frac * tokens_per_step(cfg) / elapsed
    sample = (f"{sample_units} of {U} (sequence, head) units per step, float64 numpy oracle, "
              f"{workers} single-threaded worker processes")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed / args.steps * 1e3 / frac, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator with planted needle spans)",
            "config": _config_obj(cfg),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": workers,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, cfg):
    import torch
    import torch.distributed as dist

    from wavelet_guided_sparse_gb300 import binding as bd

    rank, world, local = _rank_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bd.lib()
    ks = cfg.k_per_level()
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    arrs = wl.generate_layer(cfg, 0, workers=min(16, os.cpu_count() or 1))
    base = {k: torch.from_numpy(v).to(device=dev, dtype=dt) for k, v in arrs.items()}
    per_copy = sum(t.numel() * t.element_size() for t in base.values())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    touched = path_bytes(cfg)
    touched_bytes = sum(touched.values())
    n_copies = max(2, math.ceil(4 * l2 / max(touched_bytes, 1)))
    copies = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(n_copies - 1)]
    dims = bd.make_dims(base["Q"], base["Kp"], cfg.levels)
    ws = bd.alloc_workspace(dims, ks, dev)
    launches = bd.step_launch_count(dims, ks)
    out = torch.empty(base["Q"].shape, dtype=torch.float32, device=dev)
    lse = torch.empty(base["Q"].shape[:3], dtype=torch.float32, device=dev)
    idx = torch.empty((cfg.batch, cfg.heads, ks[0]), dtype=torch.int32, device=dev)

    def step(c, stream=None):
        bd.step(c["Q"], c["Kp"], c["Vp"], c["Kg"], c["Vg"], cfg.levels, ks, ws, out=out,
                lse=lse, idx_out=idx, stream=stream)

    for c in copies:  # eager pass (sets kernel attributes before capture)
        step(c)
    torch.cuda.synchronize()
    # One graph per input copy (one step each) and one graph that runs a step
    # on every copy in turn: the timed loop replays the latter, so that graph
    # launch latency is paid once per n_copies steps, as it would be for a
    # model's layers captured together.
    graphs = []
    cap_stream = torch.cuda.Stream(device=dev)
    for c in copies:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream):
            step(c)
        graphs.append(g)
    cycle = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cycle, stream=cap_stream):
        for c in copies:
            step(c)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = vis.split(",")[local] if vis else str(local)
    sampler = ClockSampler(smi_index) if rank == 0 else None
    time.sleep(0.3)

    # ---- warm-up + timed region (CUDA graph of wf_step per input copy)
    for i in range(args.warmup):
        graphs[i % n_copies].replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps // n_copies):
        cycle.replay()
    for i in range(args.steps % n_copies):
        graphs[i].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_ms = allreduce_max(ev0.elapsed_time(ev1), world, dev)
    ms_per_step = t_ms / args.steps
    value = job_value(world, tokens_per_step(cfg), args.steps, t_ms)

    # ---- steps 2-5 with A_L cached from an earlier step (unchanged prompt keys)
    als = [bd.dwt_lowpass(c["Kp"], cfg.levels) for c in copies]
    torch.cuda.synchronize()

    def step_cached(c, al):
        bd.step_cached_al(c["Q"], c["Kp"], c["Vp"], c["Kg"], c["Vg"], al, cfg.levels, ks, ws,
                          out=out, lse=lse, idx_out=idx)

    for c, al in zip(copies, als):
        step_cached(c, al)
    torch.cuda.synchronize()
    cyc_cached = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cyc_cached, stream=cap_stream):
        for c, al in zip(copies, als):
            step_cached(c, al)
    for _ in range(max(1, args.warmup // n_copies)):
        cyc_cached.replay()
    torch.cuda.synchronize()
    r_reps = max(1, args.steps // n_copies)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(r_reps):
        cyc_cached.replay()
    c1.record(stream)
    torch.cuda.synchronize()
    cached_ms = c0.elapsed_time(c1) / (r_reps * n_copies)
    del cyc_cached, als

    # ---- per-stage kernel durations (same launches, events on the launch stream)
    stage_ms = {"dwt": [], "score": [], "filter": [], "attn": []}
    al = torch.empty((cfg.batch, cfg.heads, cfg.n_prompt >> cfg.levels, cfg.head_dim),
                     dtype=torch.float32, device=dev)
    idx_l = torch.empty((cfg.batch, cfg.heads, ks[-1]), dtype=torch.int32, device=dev)
    lib = bd.lib()
    sp = bd._stream(stream)
    karr = bd._k_array(ks)
    n_stage_steps = max(args.steps, 20)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_stage_steps)]
    for i in range(n_stage_steps):
        c = copies[i % n_copies]
        e = evs[i]
        e[0].record(stream)
        lib.wf_dwt_lowpass(bd.ctypes.byref(dims), bd._ptr(c["Kp"]), bd._ptr(al), None, sp)
        e[1].record(stream)
        lib.wf_score_topk(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(al), ks[-1],
                          bd._ptr(idx_l), None, bd._ptr(ws), ws.numel(), sp)
        e[2].record(stream)
        lib.wf_recursive_filter(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(c["Kp"]),
                                bd._ptr(idx_l), karr, bd._ptr(idx), bd._ptr(ws), ws.numel(), sp)
        e[3].record(stream)
        lib.wf_sparse_gather_attn(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(c["Kp"]),
                                  bd._ptr(c["Vp"]), bd._ptr(c["Kg"]), bd._ptr(c["Vg"]),
                                  bd._ptr(idx), ks[0], bd._ptr(out), bd._ptr(lse), bd._ptr(ws),
                                  ws.numel(), sp)
        e[4].record(stream)
    torch.cuda.synchronize()
    for e in evs[3:]:  # the first launches include one-time effects
        for j, name in enumerate(("dwt", "score", "filter", "attn")):
            stage_ms[name].append(e[j].elapsed_time(e[j + 1]))
    stage_us = {k: 1e3 * statistics.mean(v) for k, v in stage_ms.items()}
    # The standalone DWT entry point: average duration over back-to-back launches (rotating
    # input copies, as in the timed region) between one event pair.
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_dwt = max(args.steps, 20)
    d0.record(stream)
    for i in range(n_dwt):
        lib.wf_dwt_lowpass(bd.ctypes.byref(dims), bd._ptr(copies[i % n_copies]["Kp"]), bd._ptr(al),
                           None, sp)
    d1.record(stream)
    torch.cuda.synchronize()
    dwt_us = 1e3 * d0.elapsed_time(d1) / n_dwt

    # ---- first-step cache write (eq. (2)) with A_L, from token-major K/V:
    # two input/output sets alternate (each launch touches more than L2), and
    # the launches are replayed from one CUDA graph so that host call
    # overhead stays out of the kernel time.
    cache_sets = []
    for c in copies[:2]:
        tk = torch.cat([c["Kp"], c["Kg"]], dim=2).transpose(1, 2).contiguous()
        tv = torch.cat([c["Vp"], c["Vg"]], dim=2).transpose(1, 2).contiguous()
        cache_sets.append((tk, tv, bd.cache_init(tk, tv, cfg.n_prompt, cfg.levels)))
    torch.cuda.synchronize()
    n_cache = 20
    cache_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cache_graph, stream=cap_stream):
        for i in range(n_cache):
            tk, tv, o = cache_sets[i % 2]
            bd.cache_init(tk, tv, cfg.n_prompt, cfg.levels, out=o)
    for _ in range(3):
        cache_graph.replay()
    torch.cuda.synchronize()
    cache_reps = max(1, min(50, args.steps // n_cache))
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    for _ in range(cache_reps):
        cache_graph.replay()
    k1.record(stream)
    torch.cuda.synchronize()
    cache_us = 1e3 * k0.elapsed_time(k1) / (cache_reps * n_cache)
    del cache_graph, cache_sets

    # ---- the step with a longer basis (eight-tap Daubechies filter): the
    # general path (pyramid launches, level-by-level filter CTA per unit,
    # gather + attention), from a CUDA graph over the rotating input copies.
    db4 = bd.daubechies_lowpass(4)
    basis_ws = torch.zeros(bd.basis_workspace_bytes(dims, db4, ks), dtype=torch.uint8,
                           device=dev)

    def step_basis(c):
        bd.step_basis(c["Q"], c["Kp"], c["Vp"], c["Kg"], c["Vg"], cfg.levels, ks, db4,
                      ws=basis_ws, out=out, lse=lse, idx_out=idx)

    for c in copies:
        step_basis(c)
    torch.cuda.synchronize()
    basis_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(basis_graph, stream=cap_stream):
        for c in copies:
            step_basis(c)
    for _ in range(2):
        basis_graph.replay()
    torch.cuda.synchronize()
    basis_reps = max(1, min(20, args.steps // n_copies))
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(basis_reps):
        basis_graph.replay()
    b1.record(stream)
    torch.cuda.synchronize()
    basis_ms = b0.elapsed_time(b1) / (basis_reps * n_copies)
    del basis_graph, basis_ws

    # ---- end to end through the host-buffer entry point (pinned host memory)
    host = {k: v.cpu().pin_memory() for k, v in base.items()}
    host["O"] = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    stage = {k: torch.empty_like(v) for k, v in base.items()}
    stage["O"] = torch.empty_like(out)
    h2d = sum(host[k].numel() * host[k].element_size() for k in ("Q", "Kp", "Vp", "Kg", "Vg"))
    d2h = host["O"].numel() * host["O"].element_size()
    e2e_steps = max(10, min(args.steps, 200))
    for _ in range(3):
        bd.step_host(dims, host, ks, stage, ws, stream=stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        bd.step_host(dims, host, ks, stage, ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allreduce_max(e0.elapsed_time(e1), world, dev)
    e2e_value = job_value(world, tokens_per_step(cfg), e2e_steps, e2e_ms)
    # ---- end to end with a device-resident cache (the serving loop): per step
    # the host sends Q and the generation block's new K/V rows (token-major),
    # eq. (4) writes them into the cache, steps 2-5 run from the A_L that
    # wf_cache_init wrote, and O comes back.  One resident cache per input copy,
    # as each layer of a model keeps its own.
    res_caches = []
    for c in copies:
        tk = torch.cat([c["Kp"], c["Kg"]], dim=2).transpose(1, 2).contiguous()
        tv = torch.cat([c["Vp"], c["Vg"]], dim=2).transpose(1, 2).contiguous()
        res_caches.append(bd.cache_init(tk, tv, cfg.n_prompt, cfg.levels))
        del tk, tv
    # Q and the new rows sit back to back on both sides (one H2D copy per step).
    new_k = base["Kg"].transpose(1, 2).contiguous()
    new_v = base["Vg"].transpose(1, 2).contiguous()
    n_gen_el = base["Q"].numel()
    h_pack = torch.empty(3 * n_gen_el, dtype=base["Q"].dtype).pin_memory()
    d_pack = torch.empty(3 * n_gen_el, dtype=base["Q"].dtype, device=dev)
    dhost, dstage = {}, {}
    for i, (name, src) in enumerate((("Q", base["Q"]), ("K", new_k), ("V", new_v))):
        dhost[name] = h_pack[i * n_gen_el:(i + 1) * n_gen_el].view(src.shape)
        dhost[name].copy_(src.cpu())
        dstage[name] = d_pack[i * n_gen_el:(i + 1) * n_gen_el].view(src.shape)
    dhost["O"] = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    dstage["O"] = torch.empty_like(out)
    res_h2d = sum(dhost[k].numel() * dhost[k].element_size() for k in ("Q", "K", "V"))
    res_d2h = dhost["O"].numel() * dhost["O"].element_size()
    for i in range(3):
        bd.decode_step_host(dims, dhost, ks, dstage, res_caches[i % n_copies], ws, stream=stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for i in range(e2e_steps):
        bd.decode_step_host(dims, dhost, ks, dstage, res_caches[i % n_copies], ws, stream=stream)
    r1.record(stream)
    torch.cuda.synchronize()
    res_ms = allreduce_max(r0.elapsed_time(r1), world, dev)
    res_value = job_value(world, tokens_per_step(cfg), e2e_steps, res_ms)
    del res_caches
    clocks = sampler.stop() if sampler else None
    status = bd.read_device_status(ws)

    if rank != 0:
        dist.barrier()
        return 0
    peak, peak_kind = _peaks()
    peak_source = (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                   else "fallback 6.8 TB/s")
    dwt_bytes = touched["dwt"]
    cache_bytes = cache_init_bytes(cfg)
    dwt_achieved = dwt_bytes / (dwt_us * 1e-6) / 1e9
    fused = launches == 1
    total_bytes = step_bytes(cfg, fused)
    dwt_roofline = {"kernel": "dwt_stream_kernel (wf_dwt_lowpass, fp32 A_L)", "bound": "hbm",
                    "achieved": dwt_achieved, "peak": peak, "unit": "GB/s",
                    "frac": dwt_achieved / peak, "peak_source": peak_source,
                    "traffic": _traffic(DWT_TRAFFIC), "algorithmic_bytes_per_launch": dwt_bytes,
                    "launch_us": dwt_us,
                    "timing": f"{n_dwt} back-to-back launches, rotating input copies"}
    if fused:
        # One kernel per step: its average duration is the timed region / K.
        step_ach = total_bytes / (ms_per_step * 1e-3) / 1e9
        roofline = {"kernel": "path_kernel (whole step: Haar low-pass, scoring, filter, gather,"
                              " attention)", "bound": "hbm", "achieved": step_ach, "peak": peak,
                    "unit": "GB/s", "frac": step_ach / peak, "peak_source": peak_source,
                    "traffic": _traffic(PATH_TRAFFIC), "algorithmic_bytes_per_launch": total_bytes,
                    "launch_us": ms_per_step * 1e3,
                    "timing": "CUDA events over the timed region / K (one launch per step)"}
    else:
        # Two launches per step: the roofline line is the longer of the two
        # kernels; the path kernel alone is what wf_step_cached_al times.
        rest_bytes = touched["score"] + touched["filter"] + touched["attn"]
        if cached_ms * 1e3 > dwt_us:
            rest_ach = rest_bytes / (cached_ms * 1e-3) / 1e9
            roofline = {"kernel": "path_kernel (steps 2-5; the longer of the step's two launches)",
                        "bound": "hbm", "achieved": rest_ach, "peak": peak, "unit": "GB/s",
                        "frac": rest_ach / peak, "peak_source": peak_source, "traffic": None,
                        "algorithmic_bytes_per_launch": rest_bytes,
                        "launch_us": cached_ms * 1e3,
                        "timing": "graph replays of wf_step_cached_al (the same kernel without "
                                  "the DWT launch) / steps"}
        else:
            roofline = dwt_roofline
    cpu_rate, cpu_units, cpu_s = (None, 0, 0.0)
    workers = os.cpu_count() or 1
    if world == 1 and not args.no_cpu_baseline:
        cpu_rate, cpu_units, cpu_s = cpu_oracle_rate(arrs, cfg, args.cpu_seconds, workers)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic (seeded generator with planted needle spans)",
        "config": _config_obj(cfg, {
            "l2": f"rotating {n_copies} device input copies ({n_copies * per_copy / 2**20:.0f} MiB,"
                  f" {n_copies} x {touched_bytes / 2**20:.1f} MiB touched per step > "
                  f"{l2 / 2**20:.0f} MiB L2)",
            "timing": f"CUDA events around K steps: replays of one CUDA graph holding one wf_step"
                      f" per input copy ({n_copies} steps per replay), remainder from per-copy graphs"}),
        "roofline": roofline,
        "path_roofline": {"bytes_per_step": total_bytes,
                          "achieved": total_bytes / (ms_per_step * 1e-3) / 1e9,
                          "peak": peak, "unit": "GB/s",
                          "frac": total_bytes / (ms_per_step * 1e-3) / 1e9 / peak},
        "dwt_roofline": dwt_roofline,
        "cached_al_step": {
            "what": "wf_step_cached_al: steps 2-5 with A_L from an earlier wf_dwt_lowpass "
                    "(prompt keys unchanged between denoising steps)",
            "value": tokens_per_step(cfg) / (cached_ms * 1e-3), "unit": "tokens/s",
            "ms_per_step": cached_ms,
            "algorithmic_bytes_per_step": touched["score"] + touched["filter"] + touched["attn"],
            "achieved_gbs": (touched["score"] + touched["filter"] + touched["attn"]) /
                            (cached_ms * 1e-3) / 1e9},
        "cache_init_roofline": {
            "kernel": "cache_write_kernel (wf_cache_init: eq. (2) cache write of K/V from "
                      "token-major projections + fp32 A_L of the prompt keys)",
            "bound": "hbm", "achieved": cache_bytes / (cache_us * 1e-6) / 1e9, "peak": peak,
            "unit": "GB/s", "frac": cache_bytes / (cache_us * 1e-6) / 1e9 / peak,
            "peak_source": peak_source, "traffic": _traffic(CACHE_TRAFFIC),
            "algorithmic_bytes_per_launch": cache_bytes, "launch_us": cache_us,
            "timing": "CUDA graph of 20 launches over two alternating input/output sets, "
                      "events around its replays"},
        "basis_step": {
            "what": "wf_step_basis with the eight-tap Daubechies low-pass (periodic pyramid, "
                    "level-by-level filter, gather + attention): the general path for a "
                    "longer basis",
            "value": tokens_per_step(cfg) / (basis_ms * 1e-3), "unit": "tokens/s",
            "ms_per_step": basis_ms,
            "launches_per_step": cfg.levels + 2},
        "stages_us": stage_us,
        "cpu_baseline": None if cpu_rate is None else {
            "value": cpu_rate, "unit": "tokens/s", "cores": workers, "kind": "oracle",
            "sample": f"{cpu_units} (sequence, head) units of this workload in {cpu_s:.1f} s, "
                      f"float64 numpy oracle, {workers} single-threaded worker processes"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "entry_point": "wf_step_host (pinned host Q/Kp/Vp/Kg/Vg in, O out)"},
        "e2e_resident_cache": {
            "value": res_value, "unit": "tokens/s", "h2d_bytes_per_step": res_h2d,
            "d2h_bytes_per_step": res_d2h, "steps": e2e_steps,
            "ms_per_step": res_ms / e2e_steps,
            "entry_point": "wf_decode_step_host (pinned host Q and new token-major K/V rows in, "
                           "back to back: one H2D copy; eq. (4) update + steps 2-5 on a "
                           "device-resident cache written by wf_cache_init; O out)"},
        "gpu_launches": launches * args.steps,  # path_kernel (+ dwt_stream_kernel unless fused)
        "clocks": clocks,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(wl.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = wl.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
