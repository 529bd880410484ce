#!/usr/bin/env python
"""Throughput of the WaveFilter per-layer, per-step KV-filtering path.

One step = one pass of the whole path (Haar low-pass, coarse scoring + Top-K,
recursive filtering, sparse gather + eq. (3) attention) over every layer of
the workload, through the C ABI; the default workload is the full denoising
step (32 layers of 32 heads over a 65536-token prompt).  Metric: cached prompt tokens filtered+attended
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
DEFAULT_CONFIG = "full_step"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per launch of each kernel on a workload:
# dram__bytes_read.sum + dram__bytes_write.sum of one launch from a one-pass
# ncu capture of `bench.py` on that workload (profiles/), valid while the
# kernel's sources (without comments and blank space) hash to source_sha.
TRAFFIC = {
    # 536.9 MB read + 16.1 MB written (full step); 268.5 + 12.5 MB (long prompt)
    "dwt": {"sources": ("wf_dwt.cu", "wf_common.cuh", "wf_mma.cuh", "wf_internal.h"),
            "source_sha": "e40d91781866bcc9",
            "bytes": {"full_step": 553035520, "long_prompt": 280975872}},
    # 122.3 MB read + 0.1 MB written (full step); 68.1 MB read (long prompt)
    "path": {"sources": ("wf_path.cu", "wf_common.cuh", "wf_mma.cuh", "wf_umma.cuh",
                         "wf_internal.h"),
             "source_sha": "7f6aa126a9aa4548",
             "bytes": {"full_step": 122388224, "long_prompt": 68129536}},
    # 1076.7 MB read + 1042.5 MB written (one full-step layer)
    "cache": {"sources": ("wf_cache.cu", "wf_common.cuh", "wf_internal.h"),
              "source_sha": "167dcdf5ab135297", "bytes": {"full_step": 2119244544}},
}


def _rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _workload_desc(cfg: wl.WorkloadConfig) -> str:
    ks = cfg.k_per_level()
    return (f"{cfg.name}: batch={cfg.batch}, layers={cfg.layers}, H={cfg.heads}, "
            f"d={cfg.head_dim}, N_p={cfg.n_prompt}, G={cfg.n_gen}, {cfg.dtype}, "
            f"Haar L={cfg.levels}, k_L={ks[-1]}, budget B={cfg.budget}")


def _config_obj(cfg, extra=None):
    ks = cfg.k_per_level()
    obj = {"workload": _workload_desc(cfg), "batch": cfg.batch, "layers_per_step": cfg.layers,
           "heads": cfg.heads, "head_dim": cfg.head_dim, "n_prompt": cfg.n_prompt,
           "n_gen": cfg.n_gen, "levels": cfg.levels, "k_per_level": ks,
           "budget": cfg.budget, "parallelism": "replicas"}
    if extra:
        obj.update(extra)
    return obj


def tokens_per_step(cfg) -> int:
    """Cached prompt tokens filtered+attended per step: batch * layers * N_p."""
    return cfg.batch * cfg.layers * cfg.n_prompt


def tokens_per_unit(cfg) -> float:
    """Share of one (sequence, layer, head) unit in tokens_per_step."""
    return cfg.n_prompt / cfg.heads


def path_bytes(cfg) -> dict:
    """Algorithmic HBM bytes of one layer of the step, by stage (the staged
    entry points; each stage reads its own inputs)."""
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


def layer_bytes(cfg) -> int:
    """Algorithmic HBM bytes of one layer of the step, term by term as the
    measurement plan defines them: the K_p stream, the A_L write and read, the
    span rows of the coarse survivors, the gathered K/V rows, K_g/V_g, Q, O
    and the selected indices."""
    e = 2 if cfg.dtype == "bf16" else 4
    U, d, n, g, L = cfg.units_per_layer, cfg.head_dim, cfg.n_prompt, cfg.n_gen, cfg.levels
    ks = cfg.k_per_level()
    P, B = n >> L, ks[0]
    return U * (n * d * e + 2 * P * d * 4 + (ks[L] << L) * d * e + 2 * B * d * e +
                2 * g * d * e + g * d * e + g * d * 4 + 4 * B)


def stream_bytes(cfg) -> int:
    """The share of layer_bytes that the K_p stream moves: K_p read once and
    the A_L write."""
    e = 2 if cfg.dtype == "bf16" else 4
    return cfg.units_per_layer * (cfg.n_prompt * cfg.head_dim * e +
                                  (cfg.n_prompt >> cfg.levels) * cfg.head_dim * 4)


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


def _traffic(kind, cfg):
    """ncu DRAM bytes per launch of a kernel on this workload, if captured for
    the current kernel sources; else None."""
    table = TRAFFIC[kind]
    try:
        sha = _source_sha(table["sources"])
    except OSError:
        return None
    return table["bytes"].get(cfg.name) if table["source_sha"] == sha else None


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
    n_b, n_h = arrs["Q"].shape[:2]
    jobs = []
    for u in units:
        b, h = divmod(u % (n_b * n_h), n_h)
        jobs.append((arrs["Q"][b, h], arrs["Kp"][b, h], arrs["Vp"][b, h], arrs["Kg"][b, h],
                     arrs["Vg"][b, h], cfg.levels, ks))
    return jobs


def _oracle_sample(cfg, workers):
    """Seeded units of layer 0 for the CPU legs (numpy generator): every unit of
    the layer when that is cheap, else as many as there are workers."""
    heads = list(range(cfg.heads)) if cfg.units_per_layer * cfg.n_prompt <= (1 << 22) else \
        list(range(min(cfg.heads, max(workers, 1))))
    return wl.generate_layer(cfg, 0, seqs=[0], heads=heads, workers=min(16, max(workers, 1)))


def cpu_oracle_rate(arrs, cfg, budget_s: float, workers: int):
    """Oracle tokens/s on a bounded sample: whole (sequence, layer, head) units
    of the workload, all host cores."""
    n_units = arrs["Q"].shape[0] * arrs["Q"].shape[1]
    with _oracle_pool(workers) as pool:
        list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, [0] * workers)))  # start workers
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            n = max(workers, 1)
            units = [(done + i) % n_units for i in range(n)]
            list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, units)))
            done += n
        elapsed = time.perf_counter() - t0
    return done * tokens_per_unit(cfg) / elapsed, done, elapsed


# ------------------------------------------------------------------ arms

def run_reference(args, cfg):
    rank, world, _ = _rank_env()
    if rank != 0:
        return 0
    workers = os.cpu_count() or 1
    arrs = _oracle_sample(cfg, workers)
    n_units = arrs["Q"].shape[0] * arrs["Q"].shape[1]
    units_per_step = cfg.units_per_layer * cfg.layers
    # Size each step's sample so that the whole run takes about two minutes.
    with _oracle_pool(workers) as pool:
        list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, [0] * workers)))
        t0 = time.perf_counter()
        list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, list(range(workers)))))
        per_round = time.perf_counter() - t0
        rounds = max(1, min(math.ceil(units_per_step / workers),
                            int(120.0 / max(per_round * (args.steps + args.warmup), 1e-9))))
        sample_units = min(units_per_step, rounds * workers)
        for i in range(args.warmup):
            list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, list(range(sample_units)))))
        t0 = time.perf_counter()
        for i in range(args.steps):
            units = [(i * sample_units + j) % n_units for j in range(sample_units)]
            list(pool.map(_oracle_unit, _unit_jobs(arrs, cfg, units)))
        elapsed = time.perf_counter() - t0
    frac = sample_units / units_per_step
    value = args.steps * frac * tokens_per_step(cfg) / elapsed
    sample = (f"{sample_units} of the {units_per_step} (sequence, layer, head) units of a step, "
              f"drawn from {n_units} seeded units of layer 0; float64 numpy oracle, "
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


def _event():
    import torch
    return torch.cuda.Event(enable_timing=True)


def _capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def _input_sets(cfg, dev, l2_bytes):
    """Device-resident inputs the timed steps cycle through.  A multi-layer
    workload holds every layer (independent seeds; one step = one call per
    layer).  A one-layer workload holds enough copies of its layer that the
    bytes one step touches times the copies exceed 4x L2, so that no step
    finds its inputs in L2."""
    import torch
    if cfg.layers > 1:
        return [wl.generate_layer_torch(cfg, layer, dev) for layer in range(cfg.layers)], 1
    base = wl.generate_layer_torch(cfg, 0, dev)
    n = max(2, math.ceil(4 * l2_bytes / max(layer_bytes(cfg), 1)))
    return [base] + [{k: v.clone() for k, v in base.items()} for _ in range(n - 1)], n


def _time_cycles(cycle, graphs, steps, steps_per_cycle, stream):
    """CUDA-event time of `steps` steps: replays of the cycle graph (one call
    per input set) plus, for a remainder, per-set graphs."""
    e0, e1 = _event(), _event()
    e0.record(stream)
    for _ in range(steps // steps_per_cycle):
        cycle.replay()
    for i in range(steps % steps_per_cycle):
        graphs[i].replay()
    e1.record(stream)
    import torch
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


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
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sets, n_copies = _input_sets(cfg, dev, l2)
    steps_per_cycle = 1 if cfg.layers > 1 else n_copies
    base = sets[0]
    per_set = sum(t.numel() * t.element_size() for t in base.values())
    dims = bd.make_dims(base["Q"], base["Kp"], cfg.levels)
    ws = bd.alloc_workspace(dims, ks, dev)
    plan = bd.step_plan(dims, ks)
    launches = plan["launches"]
    out = torch.empty(base["Q"].shape, dtype=torch.float32, device=dev)
    lse = torch.empty(base["Q"].shape[:3], dtype=torch.float32, device=dev)
    idx = torch.empty((cfg.batch, cfg.heads, ks[0]), dtype=torch.int32, device=dev)

    def step(c):
        bd.step(c["Q"], c["Kp"], c["Vp"], c["Kg"], c["Vg"], cfg.levels, ks, ws, out=out,
                lse=lse, idx_out=idx)

    for c in sets:  # eager pass (sets kernel attributes before capture)
        step(c)
    torch.cuda.synchronize()
    # One graph per input set and one graph with a call on every set in turn:
    # the timed loop replays the latter (for a multi-layer workload it is one
    # whole step, the layers in order, as a model's layers would be captured).
    cap_stream = torch.cuda.Stream(device=dev)
    graphs = [_capture(lambda c=c: step(c), cap_stream) for c in sets] \
        if steps_per_cycle > 1 else []
    cycle = _capture(lambda: [step(c) for c in sets], cap_stream)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = vis.split(",")[local] if vis else str(local)
    sampler = ClockSampler(smi_index) if rank == 0 else None
    time.sleep(0.3)

    # ---- warm-up + timed region
    for i in range(args.warmup):
        (graphs[i % n_copies] if graphs else cycle).replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_ms = allreduce_max(_time_cycles(cycle, graphs, args.steps, steps_per_cycle, stream),
                         world, dev)
    if world > 1:
        dist.barrier()
    ms_per_step = t_ms / args.steps
    value = job_value(world, tokens_per_step(cfg), args.steps, t_ms)
    layer_us = ms_per_step * 1e3 / cfg.layers

    # ---- the first launch of a two-launch step, alone (the standalone DWT
    # entry point over the same keys): a CUDA graph of back-to-back launches
    # over the sets (host call overhead stays out of short launches).
    lib = bd.lib()
    sp = bd._stream(stream)
    al = torch.empty((cfg.batch, cfg.heads, cfg.n_prompt >> cfg.levels, cfg.head_dim),
                     dtype=torch.float32, device=dev)
    n_dwt = max(20, len(sets))

    def dwt_cycle():
        for i in range(n_dwt):
            lib.wf_dwt_lowpass(bd.ctypes.byref(dims), bd._ptr(sets[i % len(sets)]["Kp"]),
                               bd._ptr(al), None, bd._stream())

    dwt_graph = _capture(dwt_cycle, cap_stream)
    dwt_graph.replay()
    torch.cuda.synchronize()
    d_reps = 3
    dwt_us = 1e3 * _time_cycles(dwt_graph, [], d_reps, 1, stream) / (d_reps * n_dwt)
    del dwt_graph

    # ---- steps 2-5 with A_L cached from an earlier step (unchanged prompt keys)
    als = [bd.dwt_lowpass(c["Kp"], cfg.levels) for c in sets]
    torch.cuda.synchronize()

    def step_cached(c, a):
        bd.step_cached_al(c["Q"], c["Kp"], c["Vp"], c["Kg"], c["Vg"], a, cfg.levels, ks, ws,
                          out=out, lse=lse, idx_out=idx)

    # ---- the two launches of a two-launch step, each timed where it runs:
    # when wf_step's stream launch is exactly wf_dwt_lowpass and its second
    # launch exactly that of wf_step_cached_al, a CUDA graph of those calls per
    # input set (the step's launches, in its order) carries CUDA events
    # recorded as graph nodes around every launch.
    split_us = None
    if launches == 2 and plan.get("stream_is_dwt_lowpass"):
        try:
            sev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
                   for _ in sets]
        except TypeError:  # a torch without graph-node events
            sev = None
        if sev is not None:
            def split_cycle():
                for i, c in enumerate(sets):
                    sev[i][0].record()
                    lib.wf_dwt_lowpass(bd.ctypes.byref(dims), bd._ptr(c["Kp"]), bd._ptr(al), None,
                                       bd._stream())
                    sev[i][1].record()
                    step_cached(c, al)
                    sev[i][2].record()

            split_cycle()
            torch.cuda.synchronize()
            split_graph = _capture(split_cycle, cap_stream)
            d_us, p_us = [], []
            for rep in range(3):
                split_graph.replay()
                torch.cuda.synchronize()
                if rep:  # the first replay includes one-time effects
                    d_us += [1e3 * e[0].elapsed_time(e[1]) for e in sev]
                    p_us += [1e3 * e[1].elapsed_time(e[2]) for e in sev]
            split_us = {"dwt": statistics.mean(d_us), "path": statistics.mean(p_us)}
            del split_graph

    for c, a in zip(sets, als):
        step_cached(c, a)
    torch.cuda.synchronize()
    cyc_cached = _capture(lambda: [step_cached(c, a) for c, a in zip(sets, als)], cap_stream)
    for _ in range(max(1, args.warmup // steps_per_cycle)):
        cyc_cached.replay()
    torch.cuda.synchronize()
    r_reps = max(1, args.steps // steps_per_cycle)
    cached_ms = _time_cycles(cyc_cached, [], r_reps * steps_per_cycle, steps_per_cycle,
                             stream) / (r_reps * steps_per_cycle)
    cached_layer_us = cached_ms * 1e3 / cfg.layers
    del cyc_cached

    # ---- per-stage kernel durations (the staged entry points in order, per
    # input set): a CUDA graph with events recorded as graph nodes around
    # every launch where this torch has them, else host-launched with events
    # on the stream (those durations then include any gap while the host
    # enqueues the next call).
    stage_ms = {"dwt": [], "score": [], "filter": [], "attn": []}
    idx_l = torch.empty((cfg.batch, cfg.heads, ks[-1]), dtype=torch.int32, device=dev)
    karr = bd._k_array(ks)
    n_stage = min(len(sets), 32)
    try:
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
               for _ in range(n_stage)]
        stage_graphed = True
    except TypeError:  # a torch without graph-node events
        evs = [[_event() for _ in range(5)] for _ in range(n_stage)]
        stage_graphed = False

    def stage_cycle():
        for i in range(n_stage):
            c, e, cs = sets[i], evs[i], bd._stream()
            e[0].record()
            lib.wf_dwt_lowpass(bd.ctypes.byref(dims), bd._ptr(c["Kp"]), bd._ptr(al), None, cs)
            e[1].record()
            lib.wf_score_topk(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(al), ks[-1],
                              bd._ptr(idx_l), None, bd._ptr(ws), ws.numel(), cs)
            e[2].record()
            lib.wf_recursive_filter(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(c["Kp"]),
                                    bd._ptr(idx_l), karr, bd._ptr(idx), bd._ptr(ws), ws.numel(),
                                    cs)
            e[3].record()
            lib.wf_sparse_gather_attn(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(c["Kp"]),
                                      bd._ptr(c["Vp"]), bd._ptr(c["Kg"]), bd._ptr(c["Vg"]),
                                      bd._ptr(idx), ks[0], bd._ptr(out), bd._ptr(lse),
                                      bd._ptr(ws), ws.numel(), cs)
            e[4].record()

    def stage_collect(first):
        for e in evs[first:]:
            for j, name in enumerate(("dwt", "score", "filter", "attn")):
                stage_ms[name].append(e[j].elapsed_time(e[j + 1]))

    if stage_graphed:
        stage_graph = _capture(stage_cycle, cap_stream)
        for rep in range(3):
            stage_graph.replay()
            torch.cuda.synchronize()
            if rep:  # the first replay includes one-time effects
                stage_collect(0)
        del stage_graph
    else:
        stage_cycle()
        torch.cuda.synchronize()
        stage_collect(min(3, n_stage - 1))
    stage_us = {k: 1e3 * statistics.mean(v) for k, v in stage_ms.items()}

    # ---- the gather + eq. (3) attention launch on its own: the index lists
    # of (up to) eight input sets, formed once by the staged entry points,
    # then a CUDA graph of back-to-back wf_sparse_gather_attn launches that
    # cycles through the sets (each set's K/V rows are read again only after
    # the other sets', so no launch finds its rows in L2).
    gsets = sets[:8]
    g_idx = []
    for c in gsets:
        gi = torch.empty((cfg.batch, cfg.heads, ks[0]), dtype=torch.int32, device=dev)
        lib.wf_dwt_lowpass(bd.ctypes.byref(dims), bd._ptr(c["Kp"]), bd._ptr(al), None, sp)
        lib.wf_score_topk(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(al), ks[-1],
                          bd._ptr(idx_l), None, bd._ptr(ws), ws.numel(), sp)
        lib.wf_recursive_filter(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(c["Kp"]),
                                bd._ptr(idx_l), karr, bd._ptr(gi), bd._ptr(ws), ws.numel(), sp)
        g_idx.append(gi)
    torch.cuda.synchronize()

    def gather_cycle():
        for c, gi in zip(gsets, g_idx):
            lib.wf_sparse_gather_attn(bd.ctypes.byref(dims), bd._ptr(c["Q"]), bd._ptr(c["Kp"]),
                                      bd._ptr(c["Vp"]), bd._ptr(c["Kg"]), bd._ptr(c["Vg"]),
                                      bd._ptr(gi), ks[0], bd._ptr(out), bd._ptr(lse),
                                      bd._ptr(ws), ws.numel(), bd._stream())

    gather_graph = _capture(gather_cycle, cap_stream)
    for _ in range(3):
        gather_graph.replay()
    torch.cuda.synchronize()
    g_reps = max(2, min(20, 160 // len(gsets)))
    gather_us = 1e3 * _time_cycles(gather_graph, [], g_reps, 1, stream) / (g_reps * len(gsets))
    del gather_graph, g_idx

    # ---- first-step cache write (eq. (2)) with A_L, from token-major K/V:
    # two input/output sets alternate (each launch touches more than L2),
    # replayed from one CUDA graph so host call overhead stays out.
    cache_sets = []
    for c in sets[:2]:
        tk = torch.cat([c["Kp"], c["Kg"]], dim=2).transpose(1, 2).contiguous()
        tv = torch.cat([c["Vp"], c["Vg"]], dim=2).transpose(1, 2).contiguous()
        cache_sets.append((tk, tv, bd.cache_init(tk, tv, cfg.n_prompt, cfg.levels)))
    torch.cuda.synchronize()
    n_cache = 20
    cache_graph = _capture(lambda: [bd.cache_init(cache_sets[i % 2][0], cache_sets[i % 2][1],
                                                  cfg.n_prompt, cfg.levels,
                                                  out=cache_sets[i % 2][2])
                                    for i in range(n_cache)], cap_stream)
    for _ in range(3):
        cache_graph.replay()
    torch.cuda.synchronize()
    cache_reps = max(1, min(50, args.steps // n_cache))
    cache_us = 1e3 * _time_cycles(cache_graph, [], cache_reps, 1, stream) / (cache_reps * n_cache)
    del cache_graph, cache_sets
    torch.cuda.empty_cache()

    # ---- the step with a longer basis (eight-tap Daubechies filter), from a
    # CUDA graph over (up to four) input sets: with the default schedule
    # (every level between L and 0 keeps all children) the composed level-L
    # filter's logits and the path kernel; otherwise the general path
    # (pyramid launches, level-by-level filter CTA per unit, gather +
    # attention).
    db4 = bd.daubechies_lowpass(4)
    keep_all = all(ks[j] == 2 * ks[j + 1] for j in range(1, cfg.levels))
    basis_launches = 2 if keep_all and cfg.dtype == "bf16" else cfg.levels + 2
    basis_ws = torch.zeros(bd.basis_workspace_bytes(dims, db4, ks), dtype=torch.uint8,
                           device=dev)
    bsets = sets[:4]

    def step_basis(c):
        bd.step_basis(c["Q"], c["Kp"], c["Vp"], c["Kg"], c["Vg"], cfg.levels, ks, db4,
                      ws=basis_ws, out=out, lse=lse, idx_out=idx)

    for c in bsets:
        step_basis(c)
    torch.cuda.synchronize()
    basis_graph = _capture(lambda: [step_basis(c) for c in bsets], cap_stream)
    basis_graph.replay()
    torch.cuda.synchronize()
    basis_reps = max(1, min(10, args.steps // len(bsets)))
    basis_ms = _time_cycles(basis_graph, [], basis_reps, 1, stream) / (basis_reps * len(bsets))
    del basis_graph, basis_ws
    torch.cuda.empty_cache()

    # ---- end to end through the host-buffer entry point: every layer-step
    # sends its Q/K_p/V_p/K_g/V_g from pinned host memory and reads O back.
    # The host side holds (up to) two layers' inputs, used alternately.
    host_sets = []
    for c in sets[:2]:
        h = {k: v.cpu().pin_memory() for k, v in c.items()}
        h["O"] = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        host_sets.append(h)
    stage = {k: torch.empty_like(v) for k, v in base.items()}
    stage["O"] = torch.empty_like(out)
    h2d_layer = sum(host_sets[0][k].numel() * host_sets[0][k].element_size()
                    for k in ("Q", "Kp", "Vp", "Kg", "Vg"))
    d2h_layer = host_sets[0]["O"].numel() * host_sets[0]["O"].element_size()
    e2e_steps = max(3, min(args.steps, 200 // cfg.layers))

    def e2e_step():
        for layer in range(cfg.layers):
            bd.step_host(dims, host_sets[layer % len(host_sets)], ks, stage, ws, stream=stream)

    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = _event(), _event()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allreduce_max(e0.elapsed_time(e1), world, dev)
    e2e_value = job_value(world, tokens_per_step(cfg), e2e_steps, e2e_ms)
    del host_sets, stage

    # ---- end to end with device-resident caches (the serving loop): per
    # layer-step the host sends Q and the generation block's new K/V rows
    # (token-major, back to back: one copy), eq. (4) writes them into that
    # layer's cache, steps 2-5 run from its cached A_L, and O comes back.
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
    caches = [{"Kp": c["Kp"], "Vp": c["Vp"], "Kg": c["Kg"], "Vg": c["Vg"], "AL": a}
              for c, a in zip(sets, als)]
    res_h2d = sum(dhost[k].numel() * dhost[k].element_size() for k in ("Q", "K", "V"))
    res_d2h = dhost["O"].numel() * dhost["O"].element_size()
    res_steps = max(10, min(args.steps, 400 // cfg.layers))

    def res_step(i):
        for layer in range(cfg.layers):
            cache = caches[(i * cfg.layers + layer) % len(caches)]
            bd.decode_step_host(dims, dhost, ks, dstage, cache, ws, stream=stream)

    for i in range(2):
        res_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    r0, r1 = _event(), _event()
    r0.record(stream)
    for i in range(res_steps):
        res_step(i)
    r1.record(stream)
    torch.cuda.synchronize()
    res_ms = allreduce_max(r0.elapsed_time(r1), world, dev)
    res_value = job_value(world, tokens_per_step(cfg), res_steps, res_ms)
    del caches, als
    clocks = sampler.stop() if sampler else None
    status = bd.read_device_status(ws)

    if rank != 0:
        dist.barrier()
        return 0
    peak, peak_kind = _peaks()
    peak_source = (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                   else "fallback 6.8 TB/s")
    lbytes = layer_bytes(cfg)
    sbytes = stream_bytes(cfg)
    dwt_roofline = {"kernel": "dwt_stream_kernel (wf_dwt_lowpass: K_p stream, fp32 A_L)",
                    "bound": "hbm", "achieved": sbytes / (dwt_us * 1e-6) / 1e9, "peak": peak,
                    "unit": "GB/s", "frac": sbytes / (dwt_us * 1e-6) / 1e9 / peak,
                    "peak_source": peak_source, "traffic": _traffic("dwt", cfg),
                    "algorithmic_bytes_per_launch": sbytes, "launch_us": dwt_us,
                    "timing": f"CUDA graph of {n_dwt} back-to-back launches over the input "
                              "sets, events around its replays"}
    gbytes = path_bytes(cfg)["attn"]
    gather_roofline = {"kernel": "path_kernel, gather + attention phase only (wf_sparse_gather_attn: "
                                 "selected K/V rows, K_g/V_g, Q in; O, lse out)",
                       "bound": "hbm", "achieved": gbytes / (gather_us * 1e-6) / 1e9,
                       "peak": peak, "unit": "GB/s",
                       "frac": gbytes / (gather_us * 1e-6) / 1e9 / peak,
                       "peak_source": peak_source, "traffic": None,
                       "algorithmic_bytes_per_launch": gbytes, "launch_us": gather_us,
                       "timing": f"CUDA graph of back-to-back launches over {len(gsets)} input "
                                 "sets' index lists, events around its replays"}
    dg_bytes, dg_us = sbytes + gbytes, dwt_us + gather_us
    dwt_gather = {"what": "the K_p stream (wf_dwt_lowpass) and the gather + attention "
                          "(wf_sparse_gather_attn) of one layer, each launch timed on its own",
                  "bytes": dg_bytes, "us": dg_us, "achieved": dg_bytes / (dg_us * 1e-6) / 1e9,
                  "peak": peak, "unit": "GB/s", "frac": dg_bytes / (dg_us * 1e-6) / 1e9 / peak}
    if launches == 1:
        # One kernel per layer-step: its average duration is the timed region
        # divided by the layer-steps in it.
        roofline = {"kernel": "path_kernel (the whole layer-step: Haar low-pass, scoring, "
                              "filter, gather, attention)", "bound": "hbm",
                    "achieved": lbytes / (layer_us * 1e-6) / 1e9, "peak": peak, "unit": "GB/s",
                    "frac": lbytes / (layer_us * 1e-6) / 1e9 / peak, "peak_source": peak_source,
                    "traffic": _traffic("path", cfg), "algorithmic_bytes_per_launch": lbytes,
                    "launch_us": layer_us,
                    "timing": "CUDA events over the timed region / layer-steps (one launch each)"}
    else:
        # Two launches per layer-step; the dominant one is the path kernel
        # (steps 2-5): its bytes are the layer's minus the stream's; its
        # duration from the events around each of its launches in a graph of
        # the step's two launches, else the layer-step's minus the separately
        # timed stream launch.
        if split_us is not None:
            pk_us, dwt_step_us = split_us["path"], split_us["dwt"]
            timing = ("CUDA events recorded as graph nodes around every launch of a CUDA graph "
                      "of the step's two launches per input set (wf_dwt_lowpass, then "
                      "wf_step_cached_al on its A_L: the launches wf_step issues)")
            dwt_roofline["in_step_launch_us"] = dwt_step_us
        else:
            pk_us, dwt_step_us = layer_us - dwt_us, dwt_us
            timing = "layer-step time from the timed region minus the separately timed stream launch"
        pk_bytes = lbytes - sbytes
        big = pk_us >= dwt_step_us
        roofline = {"kernel": "path_kernel (steps 2-5 of the layer-step)", "bound": "hbm",
                    "achieved": pk_bytes / (pk_us * 1e-6) / 1e9, "peak": peak, "unit": "GB/s",
                    "frac": pk_bytes / (pk_us * 1e-6) / 1e9 / peak, "peak_source": peak_source,
                    "traffic": _traffic("path", cfg), "algorithmic_bytes_per_launch": pk_bytes,
                    "launch_us": pk_us, "timing": timing} if big else dwt_roofline
    cpu_rate, cpu_units, cpu_s = (None, 0, 0.0)
    workers = os.cpu_count() or 1
    if world == 1 and not args.no_cpu_baseline:
        arrs = _oracle_sample(cfg, workers)
        cpu_rate, cpu_units, cpu_s = cpu_oracle_rate(arrs, cfg, args.cpu_seconds, workers)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic (seeded generator with planted needle spans, "
                                    "drawn on the device)",
        "config": _config_obj(cfg, {
            "l2": (f"{len(sets)} distinct device-resident layers, "
                   f"{len(sets) * per_set / 2**30:.1f} GiB, each step reads every one"
                   if cfg.layers > 1 else
                   f"rotating {n_copies} device input copies ({n_copies * per_set / 2**20:.0f} "
                   f"MiB, {n_copies} x {layer_bytes(cfg) / 2**20:.1f} MiB touched per step > "
                   f"{l2 / 2**20:.0f} MiB L2)"),
            "timing": "CUDA events around K steps: replays of one CUDA graph holding one wf_step "
                      "per input set in order"}),
        "roofline": roofline,
        "path_roofline": {"what": "whole step, algorithmic bytes of every term",
                          "bytes_per_step": lbytes * cfg.layers,
                          "achieved": lbytes / (layer_us * 1e-6) / 1e9, "peak": peak,
                          "unit": "GB/s", "frac": lbytes / (layer_us * 1e-6) / 1e9 / peak},
        "dwt_roofline": dwt_roofline,
        "gather_roofline": gather_roofline,
        "dwt_gather": dwt_gather,
        "plan": plan,
        "layer_step_us": layer_us,
        "cached_al_step": {
            "what": "wf_step_cached_al: steps 2-5 with A_L from an earlier wf_dwt_lowpass "
                    "(prompt keys unchanged between denoising steps)",
            "value": tokens_per_step(cfg) / (cached_ms * 1e-3), "unit": "tokens/s",
            "ms_per_step": cached_ms, "layer_step_us": cached_layer_us,
            "algorithmic_bytes_per_layer": lbytes - sbytes,
            "achieved_gbs": (lbytes - sbytes) / (cached_layer_us * 1e-6) / 1e9},
        "cache_init_roofline": {
            "kernel": "cache_write_kernel (wf_cache_init: eq. (2) cache write of K/V from "
                      "token-major projections + fp32 A_L of the prompt keys), one layer",
            "bound": "hbm", "achieved": cache_init_bytes(cfg) / (cache_us * 1e-6) / 1e9,
            "peak": peak, "unit": "GB/s",
            "frac": cache_init_bytes(cfg) / (cache_us * 1e-6) / 1e9 / peak,
            "peak_source": peak_source, "traffic": _traffic("cache", cfg),
            "algorithmic_bytes_per_launch": cache_init_bytes(cfg), "launch_us": cache_us,
            "timing": "CUDA graph of 20 launches over two alternating input/output sets, "
                      "events around its replays"},
        "basis_step": {
            "what": "wf_step_basis with the eight-tap Daubechies low-pass, one layer: "
                    + ("level-L logits of the composed periodic filter, then the path kernel"
                       if basis_launches == 2 else
                       "periodic pyramid, level-by-level filter, gather + attention"),
            "value": tokens_per_step(cfg) / cfg.layers / (basis_ms * 1e-3), "unit": "tokens/s",
            "layer_step_ms": basis_ms, "launches_per_layer_step": basis_launches},
        "stages_us": stage_us,
        "stages_timing": ("CUDA graph of the four staged entry points per input set, events "
                          "recorded as graph nodes around every launch" if stage_graphed else
                          "host-launched, events on the stream around every launch"),
        "cpu_baseline": None if cpu_rate is None else {
            "value": cpu_rate, "unit": "tokens/s", "cores": workers, "kind": "oracle",
            "sample": f"{cpu_units} (sequence, layer, head) units of this workload in "
                      f"{cpu_s:.1f} s, float64 numpy oracle, {workers} single-threaded "
                      f"worker processes"},
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d_layer * cfg.layers,
                "d2h_bytes_per_step": d2h_layer * cfg.layers, "steps": e2e_steps,
                "entry_point": "wf_step_host per layer (pinned host Q/Kp/Vp/Kg/Vg in, O out)"},
        "e2e_resident_cache": {
            "value": res_value, "unit": "tokens/s", "h2d_bytes_per_step": res_h2d * cfg.layers,
            "d2h_bytes_per_step": res_d2h * cfg.layers, "steps": res_steps,
            "ms_per_step": res_ms / res_steps,
            "entry_point": "wf_decode_step_host per layer (pinned host Q and new token-major "
                           "K/V rows in, one H2D copy; eq. (4) update + steps 2-5 on the "
                           "layer's device-resident cache and A_L; O out)"},
        "gpu_launches": launches * cfg.layers * args.steps,
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
