"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before anything reaches the GPU.  No call
here launches a kernel, so the suite runs without a GPU."""

import ctypes
import os
import re

import pytest

from wavelet_guided_sparse_gb300 import binding as bd
from wavelet_guided_sparse_gb300 import workloads as wl

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "wavefilter.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(bd.LIB_PATH):
        from wavelet_guided_sparse_gb300 import build
        build.build()
    return bd.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(wf_\w+)\s*\(", text, re.M)))


def test_header_declares_the_path(lib):
    names = _declared()
    for want in ("wf_dwt_lowpass", "wf_score_topk", "wf_recursive_filter",
                 "wf_sparse_gather_attn", "wf_step", "wf_workspace_bytes"):
        assert want in names
    assert set(names) == set(bd.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(8):
        assert lib.wf_status_string(code)
    assert lib.wf_status_string(0) == b"ok"
    assert lib.wf_status_string(99) == b"unknown status"


@pytest.mark.parametrize("name", sorted(wl.CONFIGS))
def test_default_k_matches_generator(lib, name):
    cfg = wl.CONFIGS[name]
    if cfg.k_coarse is not None:
        pytest.skip("explicit coarse k")
    assert bd.default_k_per_level(cfg.n_prompt, cfg.levels, cfg.budget) == cfg.k_per_level()


def test_default_k_rejects_bad_input(lib):
    out = (ctypes.c_int32 * 4)()
    assert lib.wf_default_k_per_level(1004, 3, 64, out) == 2  # 1004 % 8 != 0
    assert lib.wf_default_k_per_level(1024, 3, 0, out) == 2
    assert lib.wf_default_k_per_level(1024, 0, 64, out) == 2
    assert lib.wf_default_k_per_level(1024, 3, 64, None) == 1


def _dims(**kw):
    base = dict(batch=1, heads=32, n_prompt=4096, n_gen=32, head_dim=128, levels=4, dtype=0)
    base.update(kw)
    return bd.Dims(**base)


def _ws(dims, k):
    n = ctypes.c_size_t(0)
    st = bd.lib().wf_workspace_bytes(ctypes.byref(dims), bd._k_array(k), ctypes.byref(n))
    return st, n.value


def test_workspace_bytes_validation(lib):
    k = [512, 512, 256, 128, 64]
    st, n = _ws(_dims(), k)
    assert st == 0 and n >= 32 * 256 * 32 * 4   # coarse logits [U, P, G] fp32
    assert _ws(_dims(head_dim=96), k)[0] == 3
    assert _ws(_dims(dtype=7), k)[0] == 3
    assert _ws(_dims(n_gen=65), k)[0] == 3
    assert _ws(_dims(n_prompt=4008), k)[0] == 2
    assert _ws(_dims(levels=0), k)[0] == 2
    assert _ws(_dims(), [512, 512, 256, 128, 300])[0] == 2   # k_L > N_p / 2^L
    assert _ws(_dims(), [512, 512, 256, 100, 64])[0] == 2    # k_2 > 2 k_3
    assert _ws(_dims(), [1025, 512, 256, 128, 64])[0] == 2   # B > 2 k_1
    assert _ws(_dims(), [0, 512, 256, 128, 64])[0] == 2
    assert lib.wf_workspace_bytes(None, bd._k_array(k), ctypes.byref(ctypes.c_size_t())) == 1


def test_entry_points_reject_before_launch(lib):
    # Every failure below is decided on the host; no kernel is enqueued.
    dims = _dims()
    k = bd._k_array([512, 512, 256, 128, 64])
    p16 = ctypes.c_void_p(1 << 20)  # aligned dummy (never dereferenced on these paths)
    p17 = ctypes.c_void_p((1 << 20) + 4)
    st = lib.wf_step(ctypes.byref(dims), p16, p16, p16, p16, p16, k, p16, None, None,
                     p16, 16, None)
    assert st == 4  # workspace too small
    st = lib.wf_step(ctypes.byref(dims), p17, p16, p16, p16, p16, k, p16, None, None,
                     p16, 1 << 40, None)
    assert st == 7  # misaligned Q
    st = lib.wf_step(ctypes.byref(dims), None, p16, p16, p16, p16, k, p16, None, None,
                     p16, 1 << 40, None)
    assert st == 1
    st = lib.wf_step(ctypes.byref(_dims(n_prompt=4100)), p16, p16, p16, p16, p16, k, p16,
                     None, None, p16, 1 << 40, None)
    assert st == 2
    assert lib.wf_dwt_lowpass(ctypes.byref(dims), None, p16, None, None) == 1
    assert lib.wf_dwt_lowpass(ctypes.byref(dims), p17, p16, None, None) == 7
    assert lib.wf_score_topk(ctypes.byref(dims), p16, p16, 0, p16, None, p16, 1 << 20, None) == 2
    assert lib.wf_score_topk(ctypes.byref(dims), p16, p16, 257, p16, None, p16, 1 << 20, None) == 2
    assert lib.wf_score_topk(ctypes.byref(dims), p16, p16, 64, p16, None, p16, 8, None) == 4
    assert lib.wf_recursive_filter(ctypes.byref(dims), p16, p16, p16,
                                   bd._k_array([2000, 512, 256, 128, 64]), p16, p16, 1 << 40,
                                   None) == 2
    assert lib.wf_sparse_gather_attn(ctypes.byref(dims), p16, p16, p16, p16, p16, p16, -1, p16,
                                     None, p16, 1 << 20, None) == 2
    assert lib.wf_sparse_gather_attn(ctypes.byref(dims), p16, p16, p16, p16, p16, None, 5, p16,
                                     None, p16, 1 << 20, None) == 1
    assert lib.wf_clear_device_status(None, 256, None) == 1
    assert lib.wf_clear_device_status(p16, 8, None) == 4
    # Cached A_L: the extra pointer is validated like the others.
    assert lib.wf_step_cached_al(ctypes.byref(dims), p16, p16, p16, p16, p16, None, k, p16, None,
                                 None, p16, 1 << 40, None) == 1
    assert lib.wf_step_cached_al(ctypes.byref(dims), p16, p16, p16, p16, p16, p17, k, p16, None,
                                 None, p16, 1 << 40, None) == 7
    assert lib.wf_step_cached_al(ctypes.byref(dims), p16, p16, p16, p16, p16, p16, k, p16, None,
                                 None, p16, 16, None) == 4


def test_product_path_has_no_oracle_dependency():
    # The package must never import the oracle (test infrastructure only).
    pkg = os.path.dirname(bd.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


@pytest.mark.parametrize("name", sorted(wl.CONFIGS))
def test_every_workload_is_planned(lib, name):
    # Every configuration fits the kernels' shared-memory plans (no launch).
    cfg = wl.CONFIGS[name]
    dims = bd.Dims(cfg.batch, cfg.heads, cfg.n_prompt, cfg.n_gen, cfg.head_dim, cfg.levels,
                   0 if cfg.dtype == "bf16" else 1)
    st, n = _ws(dims, cfg.k_per_level())
    assert st == 0, name
    assert n >= cfg.units_per_layer * (cfg.n_prompt >> cfg.levels) * ((cfg.n_gen + 3) // 4 * 4) * 4
    # The fused single-launch step is planned where each CTA's coarse slice is
    # small (the 4096-token layer and the tiny case); the long prompts keep a
    # separate streaming DWT launch.
    assert bd.step_launch_count(dims, cfg.k_per_level()) == (
        1 if name in ("tiny", "llada8b_layer") else 2), name


def test_step_launch_count_validates(lib):
    dims = bd.Dims(1, 2, 1024, 32, 64, 3, 1)
    k = (ctypes.c_int32 * 4)(64, 64, 32, 16)
    out = ctypes.c_int32(-1)
    assert lib.wf_step_launch_count(ctypes.byref(dims), k, None) == 1  # WF_ERR_NULL
    assert lib.wf_step_launch_count(ctypes.byref(dims), None, ctypes.byref(out)) == 1
    bad = bd.Dims(1, 2, 1004, 32, 64, 3, 1)  # N_p not a multiple of 2^L: WF_ERR_SHAPE
    assert lib.wf_step_launch_count(ctypes.byref(bad), k, ctypes.byref(out)) == 2
    assert out.value == -1
    assert lib.wf_step_launch_count(ctypes.byref(dims), k, ctypes.byref(out)) == 0
    assert out.value in (1, 2)


def test_cache_writes_reject_before_launch(lib):
    # wf_cache_init / wf_cache_update validate like the step entry points;
    # every case below fails on the host, so nothing is enqueued.
    dims = _dims()
    p16 = ctypes.c_void_p(1 << 20)
    p17 = ctypes.c_void_p((1 << 20) + 4)
    init = lib.wf_cache_init
    assert init(None, p16, p16, p16, p16, p16, p16, p16, None) == 1
    assert init(ctypes.byref(dims), None, p16, p16, p16, p16, p16, None, None) == 1
    assert init(ctypes.byref(dims), p16, p16, p16, p16, p16, None, None, None) == 1
    assert init(ctypes.byref(dims), p17, p16, p16, p16, p16, p16, None, None) == 7
    assert init(ctypes.byref(dims), p16, p16, p16, p16, p16, p16, p17, None) == 7  # AL
    assert init(ctypes.byref(_dims(n_prompt=4100)), p16, p16, p16, p16, p16, p16, p16,
                None) == 2
    assert init(ctypes.byref(_dims(head_dim=96)), p16, p16, p16, p16, p16, p16, p16, None) == 3
    assert init(ctypes.byref(_dims(dtype=3)), p16, p16, p16, p16, p16, p16, p16, None) == 3
    upd = lib.wf_cache_update
    assert upd(ctypes.byref(dims), p16, p16, None, p16, None) == 1
    assert upd(ctypes.byref(dims), p16, p17, p16, p16, None) == 7
    assert upd(ctypes.byref(_dims(n_gen=0)), p16, p16, p16, p16, None) == 2
    assert upd(ctypes.byref(_dims(n_gen=65)), p16, p16, p16, p16, None) == 3


def test_decode_step_host_rejects_before_copies(lib):
    # Every argument of the host-buffer decode step is validated before its
    # first copy is enqueued.
    dims = _dims()
    k = bd._k_array([512, 512, 256, 128, 64])
    p16 = ctypes.c_void_p(1 << 20)
    p17 = ctypes.c_void_p((1 << 20) + 4)
    f = lib.wf_decode_step_host

    def call(dims=dims, k=k, h=p16, dq=p16, al=p16, ws=p16, wsb=1 << 40):
        return f(ctypes.byref(dims), h, h, h, k, h, dq, p16, p16, p16, p16, p16, p16, al, p16,
                 ws, wsb, None)

    assert call(h=None) == 1
    assert call(al=None) == 1
    assert call(ws=None) == 1
    assert call(dq=p17) == 7
    assert call(al=p17) == 7
    assert call(wsb=16) == 4
    assert call(k=bd._k_array([512, 512, 256, 128, 300])) == 2
    assert call(dims=_dims(n_prompt=4100)) == 2
    assert call(dims=_dims(head_dim=96)) == 3


def test_daubechies_lowpass_host_helper(lib):
    # The library's own filter generator (root finding in C++) against the
    # oracle's numpy spectral factorisation: independent code, same filters.
    import numpy as np

    import oracle.wavefilter_oracle as wo
    for n in range(1, 9):
        np.testing.assert_allclose(bd.daubechies_lowpass(n), wo.daubechies_lowpass(n), rtol=0,
                                   atol=1e-12)
    out = (ctypes.c_double * 32)()
    assert lib.wf_daubechies_lowpass(0, out) == 3
    assert lib.wf_daubechies_lowpass(9, out) == 3
    assert lib.wf_daubechies_lowpass(2, None) == 1


def test_basis_entry_points_reject_before_launch(lib):
    dims = _dims()
    k = bd._k_array([512, 512, 256, 128, 64])
    p16 = ctypes.c_void_p(1 << 20)
    p17 = ctypes.c_void_p((1 << 20) + 4)
    taps = (ctypes.c_double * 8)(*bd.daubechies_lowpass(4))
    n = ctypes.c_size_t(0)
    # Every level between L and 0 keeps all children: the level-L logits and
    # the path kernel's scratch; a level that discards: A_1..A_L in fp32.
    assert lib.wf_basis_workspace_bytes(ctypes.byref(dims), 8, k, ctypes.byref(n)) == 0
    assert 32 * 256 * 32 * 4 < n.value < 32 * 4096 * 128 * 4 // 2
    k_sel = bd._k_array([400, 500, 256, 128, 64])
    n_sel = ctypes.c_size_t(0)
    assert lib.wf_basis_workspace_bytes(ctypes.byref(dims), 8, k_sel, ctypes.byref(n_sel)) == 0
    assert n_sel.value > 32 * 4096 * 128 * 4 // 2
    assert lib.wf_basis_workspace_bytes(ctypes.byref(dims), 7, k, ctypes.byref(n)) == 3
    assert lib.wf_basis_workspace_bytes(ctypes.byref(dims), 18, k, ctypes.byref(n)) == 3
    assert lib.wf_dwt_lowpass_basis(ctypes.byref(dims), None, 8, p16, p16, None) == 1
    assert lib.wf_dwt_lowpass_basis(ctypes.byref(dims), taps, 0, p16, p16, None) == 3
    assert lib.wf_dwt_lowpass_basis(ctypes.byref(dims), taps, 8, p17, p16, None) == 7

    def step(dims=dims, taps=taps, nt=8, q=p16, ws=p16, wsb=1 << 40, k=k):
        return lib.wf_step_basis(ctypes.byref(dims), taps, nt, q, p16, p16, p16, p16, k, p16,
                                 None, None, ws, wsb, None)

    assert step(taps=None) == 1
    assert step(nt=3) == 3
    assert step(q=None) == 1
    assert step(q=p17) == 7
    assert step(wsb=n.value - 1) == 4
    assert step(k=k_sel, wsb=n_sel.value - 1) == 4
    assert step(k=bd._k_array([512, 512, 256, 128, 300])) == 2
    assert step(dims=_dims(n_prompt=4100)) == 2


@pytest.mark.parametrize("name,launches,stream_is_dwt,al_stages", [
    ("llada8b_layer", 1, 0, 0),       # one launch: the stream fused into the path kernel
    ("long_prompt", 2, 1, 4),         # wf_dwt_lowpass + the cached-A_L launch, 4 stages
    ("full_step", 2, 1, 4),
    ("batched_long_10pct", 2, 0, 0),  # 512 positions per CTA: the stream forms the logits
])
def test_step_plan_routes(name, launches, stream_is_dwt, al_stages):
    # wf_step's launch plan on a 152-SM device for the workloads' shapes (host
    # only): which of the three routes each takes.
    cfg = wl.CONFIGS[name]
    dims = bd.Dims(cfg.batch, cfg.heads, cfg.n_prompt, cfg.n_gen, cfg.head_dim, cfg.levels,
                   bd.WF_BF16)
    plan = bd.step_plan(dims, cfg.k_per_level())
    assert plan["launches"] == launches
    assert plan["stream_is_dwt_lowpass"] == stream_is_dwt
    assert plan["al_stages"] == al_stages
    n = ctypes.c_int32(0)
    assert bd.lib().wf_step_launch_count(ctypes.byref(dims), bd._k_array(cfg.k_per_level()),
                                         ctypes.byref(n)) == 0
    assert n.value == launches
