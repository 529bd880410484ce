"""Shared helpers of the GPU parity tests (not collected as tests)."""

from __future__ import annotations

import os

import numpy as np
import torch

import oracle.wavefilter_oracle as wo
from wavelet_guided_sparse_gb300 import binding as bd
from wavelet_guided_sparse_gb300 import workloads as wl

# Tolerances of the parity contract.
GAP_TOL = 1e-4      # index sets must agree where the oracle's boundary gap exceeds this
AL_RTOL = 1e-3      # DWT coefficients, relative
OUT_ATOL = 2e-2     # attention output, max-abs (bf16 inputs, fp32 accumulation)

WORKERS = min(16, os.cpu_count() or 1)


def _unit_with_gaps(args):
    """Worker: one seeded unit and the oracle's boundary gap at every selecting
    level of its recursive filter (inf where a level keeps every candidate)."""
    name, seq, layer, head = args
    cfg = wl.CONFIGS[name]
    u = wl.generate_unit(cfg, seq, layer, head)
    res = wo.recursive_filter(u["Q"], u["Kp"], cfg.levels, cfg.k_per_level())
    return u, min(lv["gap"] for lv in res["levels"].values())


def layer_with_gaps(name: str, layer: int = 0, workers: int = WORKERS):
    """All units of one layer ([b, H, rows, d] float32 arrays, as
    ``wl.generate_layer``) plus, per (b, h), the smallest oracle boundary gap
    over its selecting levels.  Runs in a spawn-started process pool (safe
    after CUDA is initialised in the parent)."""
    import concurrent.futures
    import multiprocessing
    cfg = wl.CONFIGS[name]
    jobs = [(name, b, layer, h) for b in range(cfg.batch) for h in range(cfg.heads)]
    shapes = {"Q": cfg.n_gen, "Kp": cfg.n_prompt, "Vp": cfg.n_prompt, "Kg": cfg.n_gen,
              "Vg": cfg.n_gen}
    arrs = {k: np.empty((cfg.batch, cfg.heads, r, cfg.head_dim), np.float32)
            for k, r in shapes.items()}
    gaps = {}
    ctx = multiprocessing.get_context("spawn")
    with concurrent.futures.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as pool:
        for (_, b, _, h), (u, gap) in zip(jobs, pool.map(_unit_with_gaps, jobs)):
            for k in shapes:
                arrs[k][b, h] = u[k]
            gaps[(b, h)] = gap
    return arrs, gaps


def pick_units(gaps: dict, n_decisive: int = 2, n_near: int = 2):
    """Units to compare in full: the first `n_decisive` whose every selecting
    level is decisive (gap > GAP_TOL; compared element by element) plus the
    first `n_near` with a near tie (validated), plus the layer's last unit."""
    units = sorted(gaps)
    dec = [u for u in units if gaps[u] > GAP_TOL][:n_decisive]
    near = [u for u in units if gaps[u] <= GAP_TOL][:n_near]
    return sorted(set(dec + near + [units[-1]]))


def torch_dtype(cfg_dtype: str):
    return torch.bfloat16 if cfg_dtype == "bf16" else torch.float32


def to_device(arrs: dict, cfg_dtype: str, device="cuda") -> dict:
    dt = torch_dtype(cfg_dtype)
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(device=device, dtype=dt)
            for k, v in arrs.items()}


def unit_inputs(arrs: dict, b: int, h: int) -> dict:
    return {k: v[b, h] for k, v in arrs.items()}


def oracle_unit(arrs: dict, b: int, h: int, levels: int, ks) -> dict:
    u = unit_inputs(arrs, b, h)
    return wo.wavefilter_step(u["Q"], u["Kp"], u["Vp"], u["Kg"], u["Vg"], levels, ks)


def selection_is_decisive(res: dict, tol: float = GAP_TOL) -> bool:
    """True if every level that discards candidates has an oracle gap > tol."""
    return all(lv["gap"] > tol for lv in res["levels"].values())


def check_index_set(idx: np.ndarray, n_prompt: int, budget: int) -> None:
    assert idx.shape == (budget,)
    assert (np.diff(idx) > 0).all(), "indices must be strictly ascending"
    assert idx[0] >= 0 and idx[-1] < n_prompt


def _band(scores, cand, k, tol):
    """Candidates that any correct selection of k must keep (score more than
    `tol` relative above the oracle's k-th largest) and those it may keep or
    drop (within `tol` of the k-th / (k+1)-th largest).  Scores that a
    correct fp32 computation could reorder lie inside that band."""
    order = np.lexsort((cand, -scores))
    s_k, s_k1 = scores[order[k - 1]], scores[order[k]]
    must = cand[scores > s_k * (1.0 + tol)]
    free = cand[(scores <= s_k * (1.0 + tol)) & (scores >= s_k1 * (1.0 - tol))]
    return must, free


def selection_is_valid(q, kp, levels, ks, gpu_idx, tol=GAP_TOL, budget=20000, lowpass=None):
    """True if the final token set `gpu_idx` is what the recursive filter
    (Fig. 2(c)-(d) of the WaveFilter page, as the oracle reads it) can return
    when scores are known only to `tol` relative: at every selecting level
    the survivors contain every candidate scoring more than `tol` above the
    oracle's k-th score and no candidate more than `tol` below the (k+1)-th,
    and the candidates of the next level are the children of those survivors.

    The GPU reports only the final set, so the survivors of the upper levels
    are reconstructed: they contain the ancestors of the final tokens, and the
    near-tie band's remaining slots are enumerated (depth first; `budget`
    bounds the number of candidate sets scored).  Scores are the oracle's
    float64 attention masses over each hypothesised candidate set.  `lowpass`:
    None for the Haar pyramid, else the low-pass of a longer basis."""
    pyr = (wo.haar_pyramid(kp, levels) if lowpass is None
           else wo.wavelet_pyramid(kp, levels, lowpass))
    gpu = np.asarray(gpu_idx, dtype=np.int64)
    gpu_set = set(gpu.tolist())
    if len(gpu_set) != len(gpu) or len(gpu) != ks[0]:
        return False
    count = [0]

    def rec(j, cand):
        count[0] += 1
        if count[0] > budget:
            raise AssertionError("near-tie enumeration exceeds its budget")
        k = int(ks[j])
        if k >= len(cand):
            must, free = cand, cand[:0]
        else:
            s = wo.attention_mass(q, pyr[j][cand])
            must, free = _band(s, cand, k, tol)
        must_s, free_s = set(must.tolist()), set(free.tolist())
        if j == 0:
            return must_s <= gpu_set <= (must_s | free_s)
        anc = set((gpu >> j).tolist())
        if not anc <= (must_s | free_s):
            return False
        need = must_s | (anc & free_s)
        rest = k - len(need)
        if rest < 0:
            return False
        pool = sorted(free_s - need)
        import itertools
        for combo in itertools.combinations(pool, rest):
            surv = np.array(sorted(need | set(combo)), dtype=np.int64)
            nxt = np.sort(np.concatenate([2 * surv, 2 * surv + 1]))
            if rec(j - 1, nxt):
                return True
        return False

    return rec(levels, np.arange(pyr[levels].shape[0], dtype=np.int64))


def compare_step_unit(arrs, b, h, levels, ks, gpu_idx, gpu_out, gpu_lse=None, res=None,
                      lowpass=None):
    """Parity of one unit of a full step.  Returns "exact" (every selecting
    level decisive: the index set equals the oracle's) or "valid" (a near-tie
    at some level: the GPU's set passes :func:`selection_is_valid`, and the
    attention output is compared with the oracle's eq. (3) on that set)."""
    res = res if res is not None else oracle_unit(arrs, b, h, levels, ks)
    n_prompt = arrs["Kp"].shape[2]
    check_index_set(gpu_idx, n_prompt, ks[0])
    if selection_is_decisive(res):
        np.testing.assert_array_equal(gpu_idx, res["idx"], err_msg=f"unit ({b},{h})")
        ref_out, ref_lse = res["out"], res["lse"]
        kind = "exact"
    else:
        u = unit_inputs(arrs, b, h)
        assert selection_is_valid(u["Q"], u["Kp"], levels, ks, gpu_idx, lowpass=lowpass), \
            f"unit ({b},{h}): selection is not a valid near-tie outcome"
        ref_out, ref_lse = wo.sparse_attention(u["Q"], u["Kp"], u["Vp"], u["Kg"], u["Vg"],
                                               gpu_idx)
        kind = "valid"
    err = np.abs(gpu_out - ref_out).max()
    assert err <= OUT_ATOL, f"unit ({b},{h}) max-abs {err}"
    if gpu_lse is not None:
        np.testing.assert_allclose(gpu_lse, ref_lse, rtol=0, atol=OUT_ATOL)
    return kind


def run_step(dev: dict, levels: int, ks, with_idx=True, al=None):
    """wf_step, or (al given: A_L from an earlier wf_dwt_lowpass) wf_step_cached_al."""
    q = dev["Q"]
    dims = bd.make_dims(q, dev["Kp"], levels)
    ws = bd.alloc_workspace(dims, ks, q.device)
    b, h, g, d = q.shape
    out = torch.empty((b, h, g, d), dtype=torch.float32, device=q.device)
    lse = torch.empty((b, h, g), dtype=torch.float32, device=q.device)
    idx = torch.empty((b, h, ks[0]), dtype=torch.int32, device=q.device) if with_idx else None
    if al is None:
        bd.step(dev["Q"], dev["Kp"], dev["Vp"], dev["Kg"], dev["Vg"], levels, ks, ws,
                out=out, lse=lse, idx_out=idx)
    else:
        bd.step_cached_al(dev["Q"], dev["Kp"], dev["Vp"], dev["Kg"], dev["Vg"], al, levels, ks,
                          ws, out=out, lse=lse, idx_out=idx)
    status = bd.read_device_status(ws)
    return out, lse, idx, status
