"""GPU parity of the path for longer orthonormal bases (WaveFilter §3.1 leaves
the basis psi open): the periodic pyramid of wf_dwt_lowpass_basis and the
whole step of wf_step_basis against the float64 oracle, through the C ABI.

The library's filter taps come from its own generator (wf_daubechies_lowpass,
C++); the oracle builds its own (numpy).  Bars: pyramid levels within 1e-3
relative with a floor of 1e-5 of the level's rms (the filters' signed taps
cancel, so near-zero coefficients carry the fp32 rounding of their
neighbours); selections and outputs as for the Haar step.
"""

import numpy as np
import pytest
import torch

import oracle.wavefilter_oracle as wo
from gpu_common import compare_step_unit, to_device
from wavelet_guided_sparse_gb300 import binding as bd
from wavelet_guided_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

LEVEL_FLOOR = 1e-5


def _rand(seed, b, h, n, g, d, dtype):
    rng = np.random.default_rng(seed)
    arrs = {"Q": rng.standard_normal((b, h, g, d)) * 1.5,
            "Kp": rng.standard_normal((b, h, n, d)) * 1.5,
            "Vp": rng.standard_normal((b, h, n, d)),
            "Kg": rng.standard_normal((b, h, g, d)) * 1.5,
            "Vg": rng.standard_normal((b, h, g, d))}
    rnd = wl.round_to_bf16 if dtype == "bf16" else (lambda x: x.astype(np.float32))
    return {k: rnd(v) for k, v in arrs.items()}


@pytest.mark.parametrize("moments,n,levels,d,dtype", [
    (2, 256, 3, 64, "bf16"), (4, 512, 4, 128, "f32"), (3, 128, 5, 128, "bf16"),
    (1, 256, 4, 64, "f32"), (8, 64, 3, 64, "bf16"),
])
def test_basis_pyramid_matches_oracle(moments, n, levels, d, dtype):
    arrs = _rand(n + moments, 2, 2, n, 4, d, dtype)
    dev = to_device(arrs, dtype)
    got = [a.cpu().numpy() for a in bd.dwt_lowpass_basis(dev["Kp"], levels,
                                                         bd.daubechies_lowpass(moments))]
    g = wo.daubechies_lowpass(moments)
    for b in range(2):
        for h in range(2):
            pyr = wo.wavelet_pyramid(arrs["Kp"][b, h], levels, g)
            for j in range(1, levels + 1):
                ref = pyr[j]
                tol = 1e-3 * np.abs(ref) + LEVEL_FLOOR * np.sqrt((ref ** 2).mean())
                assert (np.abs(got[j - 1][b, h] - ref) <= tol).all(), (b, h, j)


def _check_step(arrs, dtype, levels, ks, moments):
    dev = to_device(arrs, dtype)
    b, h, g, d = arrs["Q"].shape
    idx = torch.empty((b, h, ks[0]), dtype=torch.int32, device="cuda")
    lse = torch.empty((b, h, g), dtype=torch.float32, device="cuda")
    out = bd.step_basis(dev["Q"], dev["Kp"], dev["Vp"], dev["Kg"], dev["Vg"], levels, ks,
                        bd.daubechies_lowpass(moments), lse=lse, idx_out=idx)
    torch.cuda.synchronize()
    out, lse, idx = out.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()
    low = wo.daubechies_lowpass(moments)
    kinds = []
    for bi in range(b):
        for hi in range(h):
            u = {k: v[bi, hi] for k, v in arrs.items()}
            res = wo.wavefilter_step(u["Q"], u["Kp"], u["Vp"], u["Kg"], u["Vg"], levels, ks,
                                     lowpass=low)
            kinds.append(compare_step_unit(arrs, bi, hi, levels, ks, idx[bi, hi], out[bi, hi],
                                           lse[bi, hi], res=res, lowpass=low))
    return kinds


@pytest.mark.parametrize("moments,n,levels,g,d,h,budget,dtype", [
    (2, 512, 3, 20, 64, 3, 96, "bf16"),
    (4, 1024, 4, 32, 128, 2, 128, "f32"),
    (3, 2048, 4, 64, 128, 2, 200, "bf16"),
    (1, 1024, 3, 7, 64, 2, 64, "bf16"),
    (8, 64, 3, 5, 64, 2, 16, "bf16"),  # 106-tap composed filter over 64 tokens: windows wrap
])
def test_step_basis_shapes(moments, n, levels, g, d, h, budget, dtype):
    arrs = _rand(n + g + moments, 1, h, n, g, d, dtype)
    _check_step(arrs, dtype, levels, bd.default_k_per_level(n, levels, budget), moments)


def test_step_basis_nontrivial_levels():
    # Every level discards candidates (k_j < 2 k_{j+1}).
    arrs = _rand(31, 1, 3, 512, 9, 64, "bf16")
    _check_step(arrs, "bf16", 4, [40, 30, 20, 12, 8], 2)


def test_step_basis_workload_db4():
    # The 4096-token layer with the eight-tap Daubechies basis, every unit.
    cfg = wl.CONFIGS["llada8b_layer"]
    arrs = wl.generate_layer(cfg, 0)
    kinds = _check_step(arrs, cfg.dtype, cfg.levels, cfg.k_per_level(), 4)
    assert kinds.count("exact") >= len(kinds) // 2
