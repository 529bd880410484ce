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


def compare_step_unit(arrs, b, h, levels, ks, gpu_idx, gpu_out, gpu_lse=None, res=None):
    """Parity of one unit of a full step.  Returns "exact" or "conditional"."""
    res = res if res is not None else oracle_unit(arrs, b, h, levels, ks)
    n_prompt = arrs["Kp"].shape[2]
    check_index_set(gpu_idx, n_prompt, ks[0])
    if selection_is_decisive(res):
        np.testing.assert_array_equal(gpu_idx, res["idx"], err_msg=f"unit ({b},{h})")
        ref_out, ref_lse = res["out"], res["lse"]
        kind = "exact"
    else:
        # Near-tie boundary: the oracle's own eq. (3) on the GPU's index set.
        u = unit_inputs(arrs, b, h)
        ref_out, ref_lse = wo.sparse_attention(u["Q"], u["Kp"], u["Vp"], u["Kg"], u["Vg"],
                                               gpu_idx)
        kind = "conditional"
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
