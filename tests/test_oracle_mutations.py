"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
of ``test_oracle.py`` catch each one.  A pin set that lets a dropped term, a
wrong index, a transposed softmax or a reversed tie-break through is too weak.
"""

import math

import numpy as np
import pytest

import oracle.wavefilter_oracle as wo
import test_oracle as pins


def _analysis_unscaled(x):
    x = np.asarray(x, dtype=np.float64)
    return x[0::2] + x[1::2], x[0::2] - x[1::2]


def _analysis_misaligned(x):
    x = np.roll(np.asarray(x, dtype=np.float64), 1, axis=0)
    return (x[0::2] + x[1::2]) / math.sqrt(2), (x[0::2] - x[1::2]) / math.sqrt(2)


def _mass_wrong_axis(q, keys):
    z = np.asarray(q, np.float64) @ np.asarray(keys, np.float64).T / math.sqrt(q.shape[-1])
    p = np.exp(z - z.max(axis=0, keepdims=True))
    return (p / p.sum(axis=0, keepdims=True)).sum(axis=0)


def _mass_no_scale(q, keys):
    z = np.asarray(q, np.float64) @ np.asarray(keys, np.float64).T
    p = np.exp(z - z.max(axis=1, keepdims=True))
    return (p / p.sum(axis=1, keepdims=True)).sum(axis=0)


def _mass_max_over_queries(q, keys):
    z = np.asarray(q, np.float64) @ np.asarray(keys, np.float64).T / math.sqrt(q.shape[-1])
    p = np.exp(z - z.max(axis=1, keepdims=True))
    return (p / p.sum(axis=1, keepdims=True)).max(axis=0)


def _topk_high_tiebreak(scores, positions, k):
    scores = np.asarray(scores, np.float64)
    positions = np.asarray(positions, np.int64)
    order = np.lexsort((-positions, -scores))
    if k >= len(positions):
        return np.sort(positions), math.inf
    return np.sort(positions[order[:k]]), 0.0


def _topk_smallest(scores, positions, k):
    scores = np.asarray(scores, np.float64)
    positions = np.asarray(positions, np.int64)
    order = np.lexsort((positions, scores))
    if k >= len(positions):
        return np.sort(positions), math.inf
    return np.sort(positions[order[:k]]), 0.0


def _attn_drop_generation_rows(q, kp, vp, kg, vg, idx):
    return _ORIG_ATTN(q, kp, vp, kg[:0], vg[:0], idx)


def _attn_no_scale(q, kp, vp, kg, vg, idx):
    return _ORIG_ATTN(np.asarray(q, np.float64) * math.sqrt(np.shape(q)[-1]), kp, vp, kg, vg, idx)


_ORIG_ATTN = wo.sparse_attention
_ORIG_INIT = wo.cache_init


def _init_gen_block_first(k_all, v_all, n_prompt, levels):
    # The generation block taken from the front of the sequence.
    n_gen = np.shape(k_all)[0] - n_prompt
    roll = lambda a: np.roll(np.asarray(a, np.float64), -n_gen, axis=0)
    return _ORIG_INIT(roll(k_all), roll(v_all), n_prompt, levels)


def _init_reshape_not_swap(k_all, v_all, n_prompt, levels):
    # [N, H, d] reinterpreted as [H, N, d] instead of swapping the axes.
    k = np.asarray(k_all, np.float64)
    v = np.asarray(v_all, np.float64)
    n, h, d = k.shape
    flip = lambda a: np.swapaxes(a.reshape(h, n, d), 0, 1)
    return _ORIG_INIT(flip(k), flip(v), n_prompt, levels)


def _init_lowpass_of_values(k_all, v_all, n_prompt, levels):
    c = _ORIG_INIT(k_all, v_all, n_prompt, levels)
    c["a_l"] = _ORIG_INIT(v_all, k_all, n_prompt, levels)["a_l"]
    return c


def _init_keys_values_swapped(k_all, v_all, n_prompt, levels):
    c = _ORIG_INIT(k_all, v_all, n_prompt, levels)
    c["Vp"], c["Vg"] = _ORIG_INIT(v_all, v_all, n_prompt, levels)["Kp"], c["Kg"]
    return c


def _init_lowpass_unscaled(k_all, v_all, n_prompt, levels):
    c = _ORIG_INIT(k_all, v_all, n_prompt, levels)
    c["a_l"] = c["a_l"] * 2.0 ** (levels / 2)
    return c


_ORIG_DB = wo.daubechies_lowpass
_ORIG_DWT = wo.dwt_analysis_step
_ORIG_RF = wo.recursive_filter


def _db_reversed(n):
    return _ORIG_DB(n)[::-1].copy()


def _db_unit_sum(n):
    g = _ORIG_DB(n)
    return g / g.sum()


def _dwt_zero_padded(x, g):
    x = np.asarray(x, np.float64)
    padded = np.concatenate([x, np.zeros((len(g),) + x.shape[1:])])
    a, d = _ORIG_DWT(padded, g)
    return a[: x.shape[0] // 2], d[: x.shape[0] // 2]


def _dwt_shifted(x, g):
    return _ORIG_DWT(np.roll(np.asarray(x, np.float64), -1, axis=0), g)


def _dwt_mirror_without_signs(x, g):
    x = np.asarray(x, np.float64)
    m = x.shape[0]
    base = 2 * np.arange(m // 2)
    a = sum(g[k] * x[(base + k) % m] for k in range(len(g)))
    d = sum(g[len(g) - 1 - k] * x[(base + k) % m] for k in range(len(g)))
    return a, d


def _rf_ignores_basis(q, kp, levels, k_per_level, lowpass=None):
    return _ORIG_RF(q, kp, levels, k_per_level)


def _update_heads_reshaped(k_gen, v_gen):
    k = np.asarray(k_gen, np.float64)
    g, h, d = k.shape
    return {"Kg": k.reshape(h, g, d), "Vg": np.asarray(v_gen, np.float64).reshape(h, g, d)}

def _scatter_off_by_one(kp, vp, kg, vg, k_new, v_new, positions):
    return _real_scatter(kp, vp, kg, vg, k_new, v_new, np.minimum(np.asarray(positions) + 1,
                                                                  kp.shape[1] + kg.shape[1] - 1))


def _scatter_all_to_generation(kp, vp, kg, vg, k_new, v_new, positions):
    kg2, vg2 = np.array(kg, np.float64), np.array(vg, np.float64)
    for m, n in enumerate(np.asarray(positions)):
        g = int(n) % kg2.shape[1]
        kg2[:, g], vg2[:, g] = np.asarray(k_new)[m], np.asarray(v_new)[m]
    return {"Kp": np.array(kp, np.float64), "Vp": np.array(vp, np.float64), "Kg": kg2, "Vg": vg2}


def _scatter_keys_values_swapped(kp, vp, kg, vg, k_new, v_new, positions):
    return _real_scatter(kp, vp, kg, vg, v_new, k_new, positions)


def _repair_unscaled(a_l, kp_new, positions, levels):
    out = _real_repair(a_l, kp_new, positions, levels)
    touched = {int(n) >> levels for n in positions if n < kp_new.shape[1]}
    for c in touched:
        out[:, c] *= 2.0 ** (levels / 2)
    return out


def _repair_wrong_span(a_l, kp_new, positions, levels):
    return _real_repair(a_l, kp_new, [int(n) + (1 << levels) for n in positions
                                      if int(n) + (1 << levels) < kp_new.shape[1]], levels)


def _repair_nothing(a_l, kp_new, positions, levels):
    return np.array(a_l, np.float64)


_real_scatter = wo.cache_scatter
_real_repair = wo.al_repair

PIN_TESTS = [
    lambda: pins.test_haar_worked_example(),
    lambda: pins.test_haar_parseval(3),
    lambda: pins.test_haar_delta_lands_in_its_block(5),
    lambda: pins.test_haar_lowpass_is_scaled_span_sum(3),
    lambda: pins.test_attention_mass_worked_example(),
    lambda: pins.test_attention_mass_matches_sdpa_probabilities(3, 17, 8),
    lambda: pins.test_attention_mass_sums_to_number_of_queries(),
    lambda: pins.test_top_k_matches_bruteforce_with_ties(),
    lambda: pins.test_top_k_all_equal_takes_lowest_positions(),
    lambda: pins.test_recursive_filter_keep_all_is_token_topk(),
    lambda: pins.test_recursive_filter_all_equal_keys_picks_lowest(),
    lambda: pins.test_sparse_attention_worked_example(),
    lambda: pins.test_full_budget_is_full_attention(),
    lambda: pins.test_sparse_attention_uses_only_selected_rows(),
    lambda: pins.test_lse_closed_forms(),
    lambda: pins.test_cache_init_places_every_row(16, 3, 2, 3, 2),
    lambda: pins.test_cache_init_lowpass_closed_form(2),
    lambda: pins.test_cache_init_round_trip_and_rejects(),
    lambda: pins.test_cache_update_places_every_row(),
    lambda: pins.test_cache_scatter_places_every_row(),
    lambda: pins.test_al_repair_equals_full_pyramid_and_keeps_untouched_rows(2),
    lambda: pins.test_al_repair_closed_form(),
    lambda: pins.test_daubechies_db1_is_haar(),
    lambda: pins.test_daubechies_db2_closed_form(),
    lambda: pins.test_daubechies_filter_conditions(4),
    lambda: pins.test_wavelet_perfect_reconstruction_and_parseval(2, 3),
    lambda: pins.test_wavelet_pyramid_equals_equivalent_filter(2, 3),
    lambda: pins.test_recursive_filter_basis_matches_dense_bruteforce(2, 64, 3, [5, 7, 6, 4], 3),
]

MUTANTS = [
    ("haar_analysis_step", _analysis_unscaled),
    ("haar_analysis_step", _analysis_misaligned),
    ("attention_mass", _mass_wrong_axis),
    ("attention_mass", _mass_no_scale),
    ("attention_mass", _mass_max_over_queries),
    ("top_k", _topk_high_tiebreak),
    ("top_k", _topk_smallest),
    ("sparse_attention", _attn_drop_generation_rows),
    ("sparse_attention", _attn_no_scale),
    ("cache_init", _init_gen_block_first),
    ("cache_init", _init_reshape_not_swap),
    ("cache_init", _init_lowpass_of_values),
    ("cache_init", _init_keys_values_swapped),
    ("cache_init", _init_lowpass_unscaled),
    ("cache_update", _update_heads_reshaped),
    ("cache_scatter", _scatter_off_by_one),
    ("cache_scatter", _scatter_all_to_generation),
    ("cache_scatter", _scatter_keys_values_swapped),
    ("al_repair", _repair_unscaled),
    ("al_repair", _repair_wrong_span),
    ("al_repair", _repair_nothing),
    ("daubechies_lowpass", _db_reversed),
    ("daubechies_lowpass", _db_unit_sum),
    ("dwt_analysis_step", _dwt_zero_padded),
    ("dwt_analysis_step", _dwt_shifted),
    ("dwt_analysis_step", _dwt_mirror_without_signs),
    ("recursive_filter", _rf_ignores_basis),
]


@pytest.mark.parametrize("target,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, target, mutant):
    monkeypatch.setattr(wo, target, mutant)
    caught = 0
    for pin in PIN_TESTS:
        try:
            pin()
        except (AssertionError, ValueError):
            caught += 1
    assert caught > 0, f"no pin catches the mutant {mutant.__name__}"
