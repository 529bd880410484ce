"""Pins of the near-tie selection validator used by the GPU parity tests.

The GPU's index set is compared element by element with the oracle's where
every selecting level of the recursive filter (Fig. 2(c)-(d) of the
WaveFilter page) has a boundary gap above 1e-4; elsewhere it must pass
``selection_is_valid``.  These CPU tests hold that validator to what it
claims: the oracle's own selection passes; a selection computed from
slightly perturbed keys (what a correct fp32 kernel produces) passes; an
exact tie resolved the other way passes; and plain mistakes — a confidently
selected token swapped for a confidently rejected one, a token that is not a
candidate, a duplicate, a missing token — are rejected.
"""

import numpy as np
import pytest

import oracle.wavefilter_oracle as wo
from gpu_common import GAP_TOL, selection_is_valid

CASES = [  # (seed, n_prompt, levels, k_per_level, G, d)
    (1, 256, 3, [20, 14, 10, 8], 5, 64),     # every level selects
    (2, 512, 4, [40, 30, 20, 12, 8], 16, 32),
    (3, 256, 3, [32, 32, 16, 8], 8, 64),     # keep-all levels above a token Top-B
    (4, 1024, 2, [100, 90, 60], 3, 32),
]


def _inputs(seed, n, g, d):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((g, d)) * 1.5, rng.standard_normal((n, d)) * 1.5


@pytest.mark.parametrize("seed,n,levels,ks,g,d", CASES)
def test_oracle_selection_is_valid(seed, n, levels, ks, g, d):
    q, kp = _inputs(seed, n, g, d)
    res = wo.recursive_filter(q, kp, levels, ks)
    assert selection_is_valid(q, kp, levels, ks, res["idx"])


@pytest.mark.parametrize("seed,n,levels,ks,g,d", CASES)
def test_perturbed_selection_is_valid(seed, n, levels, ks, g, d):
    # Keys perturbed by ~1e-7 relative change every score by far less than the
    # tolerance: whatever the oracle selects from them must be accepted.
    q, kp = _inputs(seed, n, g, d)
    rng = np.random.default_rng(seed + 100)
    for _ in range(3):
        kp2 = kp * (1.0 + 1e-7 * rng.standard_normal(kp.shape))
        idx = wo.recursive_filter(q, kp2, levels, ks)["idx"]
        assert selection_is_valid(q, kp, levels, ks, idx)


def _token_scores(q, kp, levels, ks):
    res = wo.recursive_filter(q, kp, levels, ks)
    lv = res["levels"][0]
    return res, lv["cand"], lv["scores"]


@pytest.mark.parametrize("seed,n,levels,ks,g,d", CASES)
def test_confident_swap_is_invalid(seed, n, levels, ks, g, d):
    q, kp = _inputs(seed, n, g, d)
    res, cand, s = _token_scores(q, kp, levels, ks)
    sel = set(res["idx"].tolist())
    best = int(cand[np.argmax(s)])          # selected with the largest margin
    out = [c for c in cand.tolist() if c not in sel]
    worst = int(min(out, key=lambda c: s[list(cand).index(c)]))
    bad = np.array(sorted((sel - {best}) | {worst}))
    assert not selection_is_valid(q, kp, levels, ks, bad)


@pytest.mark.parametrize("seed,n,levels,ks,g,d", CASES)
def test_malformed_sets_are_invalid(seed, n, levels, ks, g, d):
    q, kp = _inputs(seed, n, g, d)
    res, cand, _ = _token_scores(q, kp, levels, ks)
    idx = res["idx"].copy()
    not_cand = sorted(set(range(n)) - set(cand.tolist()))
    if not_cand:  # a token whose ancestors were all rejected
        bad = idx.copy()
        bad[0] = not_cand[0]
        assert not selection_is_valid(q, kp, levels, ks, np.sort(bad))
    dup = idx.copy()
    dup[1] = dup[0]
    assert not selection_is_valid(q, kp, levels, ks, dup)
    assert not selection_is_valid(q, kp, levels, ks, idx[:-1])


def test_exact_tie_resolved_either_way_is_valid():
    # Two sibling tokens with identical keys share every ancestor and tie at
    # level 0.  Find inputs where the budget boundary falls between them: the
    # oracle keeps the lower position; keeping the higher one instead is an
    # equally correct outcome and must pass, while the same swap on a pair
    # that does not tie must fail.
    levels, ks, g, d = 3, [21, 16, 8, 4], 4, 32
    for seed in range(200):
        q, kp = _inputs(seed, 128, g, d)
        res, cand, s = _token_scores(q, kp, levels, ks)
        order = np.lexsort((cand, -s))
        a, b = int(cand[order[ks[0] - 1]]), int(cand[order[ks[0]]])
        # make b's key equal a's where they are siblings
        if a // 2 != b // 2:
            continue
        kp2 = kp.copy()
        kp2[b] = kp2[a]
        res2, cand2, s2 = _token_scores(q, kp2, levels, ks)
        if res2["levels"][0]["gap"] != 0.0:
            continue
        sel = set(res2["idx"].tolist())
        lo, hi = min(a, b), max(a, b)
        if lo not in sel or hi in sel:
            continue
        other = np.array(sorted((sel - {lo}) | {hi}))
        assert selection_is_valid(q, kp2, levels, ks, other)
        assert res2["levels"][0]["gap"] <= GAP_TOL
        return
    pytest.skip("no sibling pair at the boundary in the scanned seeds")


def test_longer_basis_selection_is_validated_on_its_own_pyramid():
    # With a Daubechies basis the scores come from that basis's pyramid: the
    # oracle's selection passes when the validator is given the basis, and
    # the same set need not pass under the Haar pyramid's scores.
    q, kp = _inputs(9, 512, 8, 32)
    ks, levels = [40, 30, 20, 12, 8], 4
    low = wo.daubechies_lowpass(3)
    idx = wo.recursive_filter(q, kp, levels, ks, lowpass=low)["idx"]
    assert selection_is_valid(q, kp, levels, ks, idx, lowpass=low)
    haar_idx = wo.recursive_filter(q, kp, levels, ks)["idx"]
    if not np.array_equal(idx, haar_idx):
        assert not selection_is_valid(q, kp, levels, ks, idx)
