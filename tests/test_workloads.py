"""Host-side checks of the seeded input generator (no filtering arithmetic)."""

import numpy as np
import pytest
import torch

from wavelet_guided_sparse_gb300 import workloads as wl


def test_configs_present_and_shaped():
    names = {"tiny", "llada8b_layer", "long_prompt", "full_step", "batched_long_1pct",
             "batched_long_2p5pct", "batched_long_5pct", "batched_long_10pct"}
    assert names <= set(wl.CONFIGS)
    for cfg in wl.CONFIGS.values():
        assert cfg.n_prompt % (1 << cfg.levels) == 0
        ks = cfg.k_per_level()
        assert len(ks) == cfg.levels + 1 and ks[0] == cfg.budget
        assert ks[cfg.levels] <= cfg.n_prompt >> cfg.levels
        for j in range(cfg.levels):
            assert 1 <= ks[j] <= 2 * ks[j + 1]


def test_default_k_rule_reproduces_stated_coarse_k():
    assert wl.CONFIGS["tiny"].k_per_level() == [64, 64, 32, 16]
    assert wl.CONFIGS["llada8b_layer"].k_per_level() == [512, 512, 256, 128, 64]
    assert wl.default_k_per_level(4096, 4, 512) == [512, 512, 256, 128, 64]
    assert wl.CONFIGS["long_prompt"].k_per_level()[-1] == 128
    assert wl.CONFIGS["full_step"].k_per_level()[-1] == 128
    assert [wl.CONFIGS[f"batched_long_{t}"].k_per_level()[-1]
            for t in ("1pct", "2p5pct", "5pct", "10pct")] == [21, 52, 103, 205]
    assert [wl.CONFIGS[f"batched_long_{t}"].budget
            for t in ("1pct", "2p5pct", "5pct", "10pct")] == [1310, 3276, 6553, 13107]


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(10000) * np.exp(
        np.random.default_rng(1).uniform(-20, 20, 10000))
    x = np.concatenate([x, [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8)]])
    want = torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(wl.round_to_bf16(x), want)


def test_generation_is_deterministic_and_subset_consistent():
    cfg = wl.CONFIGS["tiny"]
    a = wl.generate_layer(cfg)
    b = wl.generate_layer(cfg)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    one = wl.generate_layer(cfg, heads=[1])
    for k in a:
        np.testing.assert_array_equal(one[k][0, 0], a[k][0, 1])
    assert a["Kp"].shape == (1, 2, 1024, 64) and a["Q"].shape == (1, 2, 32, 64)


def test_bf16_workload_values_are_exact_bf16():
    cfg = wl.CONFIGS["llada8b_layer"]
    u = wl.generate_unit(cfg, 0, 0, 3)
    for name, arr in u.items():
        np.testing.assert_array_equal(wl.round_to_bf16(arr), arr, err_msg=name)


@pytest.mark.parametrize("name", ["tiny", "llada8b_layer", "full_step", "batched_long_1pct"])
def test_spans_do_not_overlap_and_fit(name):
    cfg = wl.CONFIGS[name]
    st = wl.span_starts(cfg, 0, 0)
    assert len(st) == cfg.n_spans
    assert (np.diff(st) >= cfg.span_len).all()
    assert st[0] >= 0 and st[-1] + cfg.span_len <= cfg.n_prompt


def test_planted_direction_present():
    # Queries and planted keys share the unit direction u (times 3).
    cfg = wl.CONFIGS["tiny"]
    u = wl.generate_unit(cfg, 0, 0, 0)
    st = wl.span_starts(cfg, 0, 0)
    qdir = u["Q"].mean(axis=0)
    qdir /= np.linalg.norm(qdir)
    planted = np.concatenate([np.arange(s, s + cfg.span_len) for s in st])
    proj = u["Kp"] @ qdir
    others = np.setdiff1d(np.arange(cfg.n_prompt), planted)
    assert proj[planted].mean() > proj[others].mean() + 2.0
