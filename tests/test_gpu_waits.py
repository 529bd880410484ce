"""Bounded device waits, driven to their limit.

Every wait of the kernels on an mbarrier (bulk-copy stages, tensor-core
commits) gives up after a bounded number of polls, raises
WF_DEV_WAIT_TIMEOUT in the workspace status word and lets the kernel finish,
so a lost copy never hangs the GPU.  wf_debug_inject_wait_timeout makes one
such wait run out on purpose — the first copy of the streaming ring is never
issued, nothing else is in flight when the wait gives up — and these tests
check that the flag is raised, that the launch itself succeeds, and that the
context stays usable: the next clean call returns the same bits as before.
"""

import numpy as np
import pytest
import torch

from gpu_common import run_step, to_device
from wavelet_guided_sparse_gb300 import binding as bd
from wavelet_guided_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _shape(kind):
    if kind == "single_launch":     # step 1 fused into the path kernel
        cfg = wl.CONFIGS["tiny"]
        return wl.generate_layer(cfg), cfg.levels, cfg.k_per_level(), cfg.dtype
    cfg = wl.CONFIGS["long_prompt"]  # separate streaming DWT launch first
    arrs = wl.generate_layer(cfg, heads=[0, 1])
    return arrs, cfg.levels, cfg.k_per_level(), cfg.dtype


@pytest.mark.parametrize("kind", ["single_launch", "two_launches"])
def test_injected_wait_timeout_is_reported_and_recovers(kind):
    arrs, levels, ks, dtype = _shape(kind)
    dev = to_device(arrs, dtype)
    dims = bd.make_dims(dev["Q"], dev["Kp"], levels)
    assert bd.step_launch_count(dims, ks) == (1 if kind == "single_launch" else 2)
    ref_out, ref_lse, ref_idx, status = run_step(dev, levels, ks)
    assert status == 0
    bd.inject_wait_timeout(1000)
    _, _, _, status = run_step(dev, levels, ks)  # synchronises: the launch completed
    assert status & bd.DEV_WAIT_TIMEOUT, status
    bd.inject_wait_timeout(0)
    out, lse, idx, status = run_step(dev, levels, ks)
    assert status == 0
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse) and torch.equal(idx, ref_idx)


def test_injection_is_one_shot():
    arrs, levels, ks, dtype = _shape("single_launch")
    dev = to_device(arrs, dtype)
    bd.inject_wait_timeout(1000)
    _, _, _, first = run_step(dev, levels, ks)
    _, _, _, second = run_step(dev, levels, ks)
    assert first & bd.DEV_WAIT_TIMEOUT and second == 0
