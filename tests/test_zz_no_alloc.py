"""The allocation-free entry point, wf_step_static_scratch.

Some callers cannot allocate device memory: plugin or enqueue interfaces of
inference engines that forbid allocation inside the call, and latency-critical
loops that cannot afford cudaMalloc's implicit device synchronisation.  For
them the library keeps its scratch in a fixed device array.  This test calls
that entry point twice in a row through the C ABI and checks each result
against the ordinary workspace entry point, wf_step, on the same inputs.

The file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""

import numpy as np
import pytest
import torch

from wavelet_guided_sparse_gb300 import binding as bd
from wavelet_guided_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

def _inputs(name, layer=0):
    cfg = wl.CONFIGS[name]
    arrs = wl.generate_layer(cfg, layer)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    return cfg, {k: torch.from_numpy(v).to(device="cuda", dtype=dt) for k, v in arrs.items()}


@pytest.mark.parametrize("name", ["tiny", "llada8b_layer"])
def test_static_scratch_matches_workspace_entry_point(name):
    # Both entry points run the same deterministic kernels on the same inputs,
    # so their outputs are bit-equal; the fixed array keeps the previous
    # call's contents, which the second call must not pick up.
    cfg, dev = _inputs(name)
    ks = cfg.k_per_level()
    dims = bd.make_dims(dev["Q"], dev["Kp"], cfg.levels)
    ws = bd.alloc_workspace(dims, ks, dev["Q"].device)
    ref_idx = torch.empty((cfg.batch, cfg.heads, ks[0]), dtype=torch.int32, device="cuda")
    ref_lse = torch.empty(dev["Q"].shape[:3], dtype=torch.float32, device="cuda")
    ref = bd.step(dev["Q"], dev["Kp"], dev["Vp"], dev["Kg"], dev["Vg"], cfg.levels, ks, ws,
                  lse=ref_lse, idx_out=ref_idx)
    assert bd.read_device_status(ws) == 0
    outs = []
    for call in range(2):
        outs.append((torch.empty_like(ref), torch.empty_like(ref_lse), torch.empty_like(ref_idx)))
    torch.cuda.synchronize()
    free_before = None
    for call, (out, lse, idx) in enumerate(outs):
        if call == 1:  # no device memory is taken by the call itself
            free_before = torch.cuda.mem_get_info()[0]
        bd.step_static_scratch(dev["Q"], dev["Kp"], dev["Vp"], dev["Kg"], dev["Vg"],
                               cfg.levels, ks, out=out, lse=lse, idx_out=idx)
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before
        assert torch.equal(out, ref), call
        assert torch.equal(lse, ref_lse), call
        assert torch.equal(idx, ref_idx), call


def test_static_scratch_rejects_sizes_beyond_its_limit():
    # Eight sequences of 32 heads over a 131072-token prompt at L = 5 need
    # far more scratch than the fixed array holds: rejected on the host
    # before anything runs.
    dims = bd.Dims(8, 32, 131072, 64, 128, 5, 0)
    ks = bd.default_k_per_level(131072, 5, 4096)
    assert bd.workspace_bytes(dims, ks) > (48 << 20)
    small = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = bd.lib().wf_step_static_scratch(bd.ctypes.byref(dims), bd._ptr(small), bd._ptr(small),
                                         bd._ptr(small), bd._ptr(small), bd._ptr(small),
                                         bd._k_array(ks), bd._ptr(small), None, None, None)
    assert st == 4  # WF_ERR_WORKSPACE
