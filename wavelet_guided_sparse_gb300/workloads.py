"""Seeded synthetic inputs for the WaveFilter KV-filtering path.

This module only draws random numbers and lays them out; it contains none of
the filtering arithmetic (no DWT, no scoring, no selection, no attention).
Both the float64 oracle (through the tests) and the CUDA path consume the
arrays it returns, so the two sides always see identical inputs.

Workload shapes follow the synthetic stand-in for the long-context needle
retrieval setting used by "WaveFilter: Enhancing the Long-Context Capability
of Diffusion LLMs via Wavelet-Guided KV Cache Filtering" (§1, Fig. 1: RULER
``niah_single_1`` with LLaDA-8B-Instruct).  The real suite and model weights
are not used; instead keys carry planted "needle" spans that are aligned with
the query direction.

Key recipe, per (sequence, layer, head) unit, over the N = N_p + G token
positions of the cache (prompt positions first, then the generation block):

    K[n, c] = s_c * (0.6 * z[n, c] + 0.8 * r[n, c])
        z ~ N(0, 1)
        r = per-channel Gaussian random walk over n, standardised over n to
            zero mean and unit variance
        s_c ~ log-uniform [0.5, 2], shared by all heads of a (sequence, layer)
    K[n, :] += 3 * u   for n inside a planted span (prompt positions only)
    Q[i, :]  = N(0, 1) + 3 * u           (G generation-block queries)
    V        ~ N(0, 1)

u is one seeded unit vector per (sequence, layer, head).  Planted spans are
non-overlapping: the prompt is cut into ``n_spans`` equal segments and one
span starts at a uniform seeded offset inside each segment (so spans are not
aligned to the wavelet blocks).  Values are drawn in float64 and rounded to
the workload dtype (bf16 round-to-nearest-even, or fp32) before anything
consumes them.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Sequence

import numpy as np

__all__ = [
    "WorkloadConfig",
    "CONFIGS",
    "default_k_per_level",
    "generate_unit",
    "generate_layer",
    "generate_layer_torch",
    "round_to_bf16",
]


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    """One synthetic workload: shapes, wavelet depth, budget and span layout."""

    name: str
    batch: int
    layers: int
    heads: int
    head_dim: int
    n_prompt: int
    n_gen: int
    dtype: str  # "f32" or "bf16"
    levels: int
    budget: int
    n_spans: int
    span_len: int
    seed: int
    k_coarse: Optional[int] = None  # explicit coarse Top-K; None = default rule

    @property
    def units_per_layer(self) -> int:
        return self.batch * self.heads

    def k_per_level(self) -> list:
        """Per-level survivors k_0..k_L (k_0 = final budget)."""
        return default_k_per_level(self.n_prompt, self.levels, self.budget, self.k_coarse)

    def with_budget(self, budget: int, name: Optional[str] = None) -> "WorkloadConfig":
        return dataclasses.replace(self, budget=budget, name=name or self.name, k_coarse=None)


def default_k_per_level(n_prompt: int, levels: int, budget: int,
                        k_coarse: Optional[int] = None) -> list:
    """Survivor count per level, index j = 0 (tokens) .. L (coarsest).

    k_L = ceil(2B / 2^L) (or ``k_coarse``) capped at the N_p / 2^L coarse
    positions; k_j = min(2^(L-j) k_L, N_p / 2^j) for 1 <= j < L, which keeps
    every child of every survivor; k_0 = B.  This is a reading of the pages
    (they give no per-level rule); it reproduces the coarse k stated for the
    1024-token (k_3 = 16, B = 64) and 4096-token (k_4 = 64, B = 512) workloads.
    """
    if levels < 1:
        raise ValueError("levels must be >= 1")
    if n_prompt % (1 << levels):
        raise ValueError("n_prompt must be a multiple of 2^levels")
    top = n_prompt >> levels
    k_l = k_coarse if k_coarse is not None else -(-2 * budget // (1 << levels))
    k_l = max(1, min(k_l, top))
    ks = [0] * (levels + 1)
    ks[levels] = k_l
    for j in range(levels - 1, 0, -1):
        ks[j] = min(k_l << (levels - j), n_prompt >> j)
    ks[0] = budget
    return ks


def _cfg(name, **kw) -> WorkloadConfig:
    return WorkloadConfig(name=name, **kw)


# The five workloads: Tiny, an LLaDA-8B-shaped layer, a long prompt, a full
# 32-layer denoising step and a batched long-context budget sweep.
CONFIGS: Dict[str, WorkloadConfig] = {
    "tiny": _cfg("tiny", batch=1, layers=1, heads=2, head_dim=64, n_prompt=1024,
                 n_gen=32, dtype="f32", levels=3, budget=64, n_spans=4, span_len=8,
                 seed=0x5EED + 0, k_coarse=16),
    "llada8b_layer": _cfg("llada8b_layer", batch=1, layers=1, heads=32, head_dim=128,
                          n_prompt=4096, n_gen=32, dtype="bf16", levels=4, budget=512,
                          n_spans=8, span_len=16, seed=0x5EED + 1, k_coarse=64),
    "long_prompt": _cfg("long_prompt", batch=1, layers=1, heads=32, head_dim=128,
                        n_prompt=32768, n_gen=32, dtype="bf16", levels=5, budget=2048,
                        n_spans=16, span_len=16, seed=0x5EED + 2),
    "full_step": _cfg("full_step", batch=1, layers=32, heads=32, head_dim=128,
                      n_prompt=65536, n_gen=32, dtype="bf16", levels=6, budget=4096,
                      n_spans=32, span_len=16, seed=0x5EED + 3),
}
for _frac, _tag in ((0.01, "1pct"), (0.025, "2p5pct"), (0.05, "5pct"), (0.10, "10pct")):
    CONFIGS[f"batched_long_{_tag}"] = _cfg(
        f"batched_long_{_tag}", batch=2, layers=1, heads=32, head_dim=128,
        n_prompt=131072, n_gen=64, dtype="bf16", levels=7,
        budget=int(math.floor(_frac * 131072)), n_spans=64, span_len=16,
        seed=0x5EED + 4)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bf16 (ties to even); returns float32.

    Inputs here are finite, so the plain bit-level round-to-nearest-even on
    the float32 pattern is exact.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).reshape(f.shape)


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def _rng(cfg: WorkloadConfig, *key: int) -> np.random.Generator:
    return np.random.default_rng([cfg.seed, *key])


def _channel_scale(cfg: WorkloadConfig, seq: int, layer: int) -> np.ndarray:
    rng = _rng(cfg, seq, layer, 1_000_001)
    return np.exp(rng.uniform(math.log(0.5), math.log(2.0), size=cfg.head_dim))


def span_starts(cfg: WorkloadConfig, seq: int, layer: int) -> np.ndarray:
    """Start positions of the planted spans of one (sequence, layer)."""
    rng = _rng(cfg, seq, layer, 1_000_002)
    seg = cfg.n_prompt // cfg.n_spans
    if seg < cfg.span_len:
        raise ValueError("spans do not fit in the prompt")
    offs = rng.integers(0, seg - cfg.span_len + 1, size=cfg.n_spans)
    return np.arange(cfg.n_spans, dtype=np.int64) * seg + offs


def generate_unit(cfg: WorkloadConfig, seq: int, layer: int, head: int) -> Dict[str, np.ndarray]:
    """Inputs of one (sequence, layer, head) unit, rounded to ``cfg.dtype``.

    Returns float32 arrays Q [G,d], Kp [N_p,d], Vp [N_p,d], Kg [G,d], Vg [G,d].
    """
    d, n_p, g = cfg.head_dim, cfg.n_prompt, cfg.n_gen
    n = n_p + g
    scale = _channel_scale(cfg, seq, layer)
    starts = span_starts(cfg, seq, layer)
    rng = _rng(cfg, seq, layer, head)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    z = rng.standard_normal((n, d))
    walk = np.cumsum(rng.standard_normal((n, d)), axis=0)
    walk -= walk.mean(axis=0, keepdims=True)
    walk /= walk.std(axis=0, keepdims=True)
    keys = scale[None, :] * (0.6 * z + 0.8 * walk)
    for s in starts:
        keys[s:s + cfg.span_len] += 3.0 * u
    q = rng.standard_normal((g, d)) + 3.0 * u[None, :]
    v = rng.standard_normal((n, d))
    return {
        "Q": _round(q, cfg.dtype),
        "Kp": _round(keys[:n_p], cfg.dtype),
        "Vp": _round(v[:n_p], cfg.dtype),
        "Kg": _round(keys[n_p:], cfg.dtype),
        "Vg": _round(v[n_p:], cfg.dtype),
    }


def _unit_job(args):
    cfg, s, layer, h = args
    return generate_unit(cfg, s, layer, h)


def generate_layer(cfg: WorkloadConfig, layer: int = 0,
                   seqs: Optional[Sequence[int]] = None,
                   heads: Optional[Sequence[int]] = None,
                   workers: int = 0) -> Dict[str, np.ndarray]:
    """Stack units of one layer into [b, H, rows, d] float32 arrays.

    ``seqs`` / ``heads`` select a subset (default: all); a unit's values do
    not depend on which other units are generated with it.  ``workers`` > 1
    draws units in a spawn-started process pool (safe after CUDA is
    initialised in the parent).
    """
    seqs = list(range(cfg.batch)) if seqs is None else list(seqs)
    heads = list(range(cfg.heads)) if heads is None else list(heads)
    out: Dict[str, np.ndarray] = {}
    shapes = {"Q": cfg.n_gen, "Kp": cfg.n_prompt, "Vp": cfg.n_prompt,
              "Kg": cfg.n_gen, "Vg": cfg.n_gen}
    for name, rows in shapes.items():
        out[name] = np.empty((len(seqs), len(heads), rows, cfg.head_dim), dtype=np.float32)
    jobs = [(cfg, s, layer, h) for s in seqs for h in heads]
    if workers and workers > 1 and len(jobs) > 1:
        import concurrent.futures
        import multiprocessing
        ctx = multiprocessing.get_context("spawn")
        with concurrent.futures.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as pool:
            units = pool.map(_unit_job, jobs)
            for i, unit in enumerate(units):
                bi, hi = divmod(i, len(heads))
                for name in shapes:
                    out[name][bi, hi] = unit[name]
        return out
    for i, job in enumerate(jobs):
        unit = _unit_job(job)
        bi, hi = divmod(i, len(heads))
        for name in shapes:
            out[name][bi, hi] = unit[name]
    return out


def generate_layer_torch(cfg: WorkloadConfig, layer: int = 0, device="cuda",
                         seqs: Optional[Sequence[int]] = None):
    """The recipe of :func:`generate_unit` for every head of one layer, drawn
    with torch's generator on ``device`` (a 32-layer workload of 65536-token
    prompts takes seconds this way instead of tens of minutes on the host).

    Same distributions, planted-span layout rules and rounding as the numpy
    generator, but a different random stream: the values differ from
    :func:`generate_layer`'s, so parity tests use that one and this serves
    throughput measurements.  Returns tensors of the workload dtype (bf16 by
    round-to-nearest-even, or fp32): Q, Kp, Vp, Kg, Vg as [b, H, rows, d].
    """
    import torch

    seqs = list(range(cfg.batch)) if seqs is None else list(seqs)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    d, n_p, g, H = cfg.head_dim, cfg.n_prompt, cfg.n_gen, cfg.heads
    n = n_p + g
    out = {k: torch.empty((len(seqs), H, rows, d), dtype=dt, device=device)
           for k, rows in (("Q", g), ("Kp", n_p), ("Vp", n_p), ("Kg", g), ("Vg", g))}
    for bi, s in enumerate(seqs):
        # Host-side draws of the small per-(sequence, layer) parameters, from
        # the numpy generator (identical to generate_unit's).
        scale = torch.from_numpy(_channel_scale(cfg, s, layer)).to(device, torch.float32)
        starts = span_starts(cfg, s, layer)
        gen = torch.Generator(device=device)
        gen.manual_seed(int(np.random.SeedSequence([cfg.seed, s, layer, 7]).generate_state(1)[0]))
        for h in range(H):
            u = torch.randn(d, generator=gen, device=device, dtype=torch.float32)
            u /= u.norm()
            walk = torch.randn((n, d), generator=gen, device=device, dtype=torch.float32)
            walk = walk.cumsum(0)
            walk -= walk.mean(0, keepdim=True)
            walk /= walk.std(0, unbiased=False, keepdim=True)
            keys = torch.randn((n, d), generator=gen, device=device, dtype=torch.float32)
            keys.mul_(0.6).add_(walk, alpha=0.8).mul_(scale[None, :])
            del walk
            for st in starts:
                keys[int(st):int(st) + cfg.span_len] += 3.0 * u
            q = torch.randn((g, d), generator=gen, device=device, dtype=torch.float32) + 3.0 * u
            v = torch.randn((n, d), generator=gen, device=device, dtype=torch.float32)
            out["Q"][bi, h] = q.to(dt)
            out["Kp"][bi, h] = keys[:n_p].to(dt)
            out["Kg"][bi, h] = keys[n_p:].to(dt)
            out["Vp"][bi, h] = v[:n_p].to(dt)
            out["Vg"][bi, h] = v[n_p:].to(dt)
    return out
