"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test ties one oracle function to a hand-worked example from the pages'
definitions, a closed form, an invariant of the orthonormal Haar transform,
a library special case (torch float64 scaled-dot-product attention) or brute
force on tiny inputs.  ``test_oracle_mutations.py`` plants plausible mistakes
in the oracle and checks that one of these pins catches each of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.wavefilter_oracle as wo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ev(expr):
    return float(eval(str(expr), {"__builtins__": {}}, {"sqrt": math.sqrt, "log": math.log}))


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _sdpa(q, k, v):
    """torch float64 scaled-dot-product attention (scale 1/sqrt(d), no mask)."""
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.as_tensor(q, dtype=torch.float64)[None, None],
        torch.as_tensor(k, dtype=torch.float64)[None, None],
        torch.as_tensor(v, dtype=torch.float64)[None, None])
    return out[0, 0].numpy()


def _mass_by_sdpa(q, keys):
    """Attention probabilities via SDPA with identity values, summed over queries."""
    n = keys.shape[0]
    return _sdpa(q, keys, np.eye(n)).sum(axis=0)


def _brute_topk(scores, positions, k):
    ranked = sorted(zip(scores.tolist(), positions.tolist()), key=lambda t: (-t[0], t[1]))
    return np.array(sorted(p for _, p in ranked[:k]), dtype=np.int64)


# --------------------------------------------------------------------- Haar DWT

def test_haar_worked_example():
    g = _load("haar_ramp8.json")
    x = np.array(g["x"], dtype=np.float64)[:, None]
    pyr = wo.haar_pyramid(x, 3)
    a3, details = wo.haar_dwt(x, 3)
    for j in (1, 2, 3):
        want_a = np.array([_ev(e) for e in g["A"][str(j)]])
        want_d = np.array([_ev(e) for e in g["D"][str(j)]])
        np.testing.assert_allclose(pyr[j][:, 0], want_a, rtol=0, atol=1e-13)
        np.testing.assert_allclose(details[j - 1][:, 0], want_d, rtol=0, atol=1e-13)
    np.testing.assert_allclose(a3[:, 0], [_ev("18/sqrt(2)")], rtol=0, atol=1e-13)


@pytest.mark.parametrize("levels", [1, 2, 3, 5, 7])
def test_haar_perfect_reconstruction(levels):
    rng = np.random.default_rng(levels)
    x = rng.standard_normal((1 << (levels + 2), 5))
    a, details = wo.haar_dwt(x, levels)
    np.testing.assert_allclose(wo.haar_idwt(a, details), x, rtol=0, atol=1e-12)


@pytest.mark.parametrize("levels", [1, 3, 6])
def test_haar_parseval(levels):
    rng = np.random.default_rng(100 + levels)
    x = rng.standard_normal((1 << (levels + 3), 7)) * rng.uniform(0.1, 10, size=7)
    a, details = wo.haar_dwt(x, levels)
    energy = (a ** 2).sum(axis=0) + sum((d ** 2).sum(axis=0) for d in details)
    np.testing.assert_allclose(energy, (x ** 2).sum(axis=0), rtol=1e-12)


def test_haar_matrix_orthonormal():
    # The full L-level transform of R^N is an orthogonal matrix: build it column by column.
    n, levels = 32, 4
    cols = []
    for i in range(n):
        e = np.zeros((n, 1))
        e[i] = 1.0
        a, details = wo.haar_dwt(e, levels)
        cols.append(np.concatenate([a[:, 0]] + [d[:, 0] for d in reversed(details)]))
    w = np.stack(cols, axis=1)
    np.testing.assert_allclose(w @ w.T, np.eye(n), atol=1e-13)


@pytest.mark.parametrize("levels", [1, 4, 7])
def test_haar_constant_signal(levels):
    c = np.array([3.25, -1.5])
    x = np.tile(c, (1 << (levels + 1), 1))
    a, details = wo.haar_dwt(x, levels)
    np.testing.assert_allclose(a, np.tile(c * 2 ** (levels / 2), (2, 1)), rtol=1e-14)
    for d in details:
        np.testing.assert_array_equal(d, 0.0)


@pytest.mark.parametrize("levels", [1, 3, 4, 7])
def test_haar_lowpass_is_scaled_span_sum(levels):
    rng = np.random.default_rng(7 * levels)
    n = 1 << (levels + 3)
    x = rng.standard_normal((n, 6))
    span_sum = x.reshape(n >> levels, 1 << levels, 6).sum(axis=1)
    np.testing.assert_allclose(wo.haar_pyramid(x, levels)[levels],
                               span_sum * 2.0 ** (-levels / 2), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("pos", [0, 1, 5, 8, 31])
def test_haar_delta_lands_in_its_block(pos):
    # Reading of eq. (5): coarse position p covers tokens [p 2^L, (p+1) 2^L).
    levels, n = 3, 32
    x = np.zeros((n, 1))
    x[pos] = 1.0
    a = wo.haar_pyramid(x, levels)[levels][:, 0]
    want = np.zeros(n >> levels)
    want[pos >> levels] = 2 ** (-levels / 2)
    np.testing.assert_allclose(a, want, atol=1e-15)


# ------------------------------------------------------------ scoring + Top-K

def test_attention_mass_worked_example():
    g = _load("attention_mass_2x2.json")
    q = np.array(g["Q"], dtype=np.float64)
    k = np.array([[_ev(e) for e in row] for row in g["K"]])
    s = wo.attention_mass(q, k)
    np.testing.assert_allclose(s, [_ev(e) for e in g["scores"]], rtol=1e-14)


@pytest.mark.parametrize("g,n,d", [(1, 5, 4), (3, 17, 8), (32, 64, 64)])
def test_attention_mass_matches_sdpa_probabilities(g, n, d):
    rng = np.random.default_rng(g * 1000 + n)
    q = rng.standard_normal((g, d)) * 2
    keys = rng.standard_normal((n, d)) * 2
    np.testing.assert_allclose(wo.attention_mass(q, keys), _mass_by_sdpa(q, keys),
                               rtol=1e-12, atol=1e-14)


def test_attention_mass_sums_to_number_of_queries():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((7, 16))
    keys = rng.standard_normal((40, 16)) * 3
    s = wo.attention_mass(q, keys)
    assert s.shape == (40,)
    assert abs(s.sum() - 7.0) < 1e-12
    assert (s >= 0).all()


def test_top_k_matches_bruteforce_with_ties():
    rng = np.random.default_rng(11)
    for trial in range(50):
        n = int(rng.integers(2, 40))
        scores = rng.integers(0, 6, size=n).astype(np.float64) / 7.0  # many ties
        positions = rng.permutation(1000)[:n]
        k = int(rng.integers(1, n + 1))
        got, _ = wo.top_k(scores, positions, k)
        np.testing.assert_array_equal(got, _brute_topk(scores, positions, k))


def test_top_k_all_equal_takes_lowest_positions():
    positions = np.array([9, 3, 7, 1, 12, 4])
    got, gap = wo.top_k(np.full(6, 0.25), positions, 3)
    np.testing.assert_array_equal(got, [1, 3, 4])
    assert gap == 0.0


def test_top_k_gap_definition():
    got, gap = wo.top_k(np.array([0.5, 0.4, 0.1, 0.3]), np.arange(4), 2)
    np.testing.assert_array_equal(got, [0, 1])
    assert math.isclose(gap, (0.4 - 0.3) / 0.4)
    _, gap_all = wo.top_k(np.array([0.5, 0.4]), np.arange(2), 2)
    assert gap_all == math.inf


# ----------------------------------------------------------- recursive filter

def _equivalent_filter(g, j):
    """Level-j equivalent low-pass: w_1 = g, w_j = (g upsampled by 2^(j-1)) * w_(j-1)."""
    w = np.array([1.0])
    for i in range(1, j + 1):
        up = np.zeros((len(g) - 1) * 2 ** (i - 1) + 1)
        up[:: 2 ** (i - 1)] = g
        w = np.convolve(up, w)
    return w


def _direct_level(x, g, j):
    """A_j[p] = sum_m w_j[m] x[(2^j p + m) mod N], summed directly."""
    n = x.shape[0]
    w = _equivalent_filter(g, j)
    out = np.zeros((n >> j,) + x.shape[1:])
    for p in range(n >> j):
        for m, wm in enumerate(w):
            out[p] += wm * x[((p << j) + m) % n]
    return out


def _dense_reference_levels(q, kp, levels, ks, lowpass=None):
    """Same selection written densely: every level's A_j from span sums (or,
    for another basis, its equivalent filter summed directly), a candidate
    mask from the parents, SDPA probabilities, brute-force Top-K."""
    n = kp.shape[0]
    out = {}
    parents = None
    for j in range(levels, -1, -1):
        if lowpass is None:
            a_j = kp.reshape(n >> j, 1 << j, -1).sum(axis=1) * 2.0 ** (-j / 2)
        else:
            a_j = _direct_level(kp, lowpass, j)
        pos = np.arange(n >> j)
        mask = np.ones(n >> j, bool) if parents is None else np.isin(pos >> 1, parents)
        cand = pos[mask]
        s = _mass_by_sdpa(q, a_j[cand])
        parents = _brute_topk(s, cand, ks[j])
        out[j] = parents
    return out


@pytest.mark.parametrize("n,levels,ks,g", [
    (64, 3, [5, 7, 6, 4], 3),
    (128, 3, [20, 18, 10, 6], 4),
    (256, 4, [30, 16, 9, 6, 4], 2),
    (256, 2, [50, 33, 20], 5),
    (128, 4, [16, 16, 8, 4, 2], 1),
])
def test_recursive_filter_matches_dense_bruteforce(n, levels, ks, g):
    rng = np.random.default_rng(n + levels * 17 + g)
    d = 8
    q = rng.standard_normal((g, d)) * 1.5
    kp = rng.standard_normal((n, d)) * 1.5
    got = wo.recursive_filter(q, kp, levels, ks)
    want = _dense_reference_levels(q, kp, levels, ks)
    for j in range(levels + 1):
        np.testing.assert_array_equal(got["levels"][j]["sel"], want[j], err_msg=f"level {j}")
    np.testing.assert_array_equal(got["idx"], want[0])


def test_recursive_filter_keep_all_is_token_topk():
    # Keeping every candidate down to level 1 makes level 0 a Top-B over all tokens.
    rng = np.random.default_rng(5)
    n, levels, b, d = 128, 3, 19, 16
    q = rng.standard_normal((4, d))
    kp = rng.standard_normal((n, d)) * 2
    ks = [b] + [n >> j for j in range(1, levels + 1)]
    got = wo.recursive_filter(q, kp, levels, ks)["idx"]
    want = _brute_topk(_mass_by_sdpa(q, kp), np.arange(n), b)
    np.testing.assert_array_equal(got, want)


def test_recursive_filter_all_equal_keys_picks_lowest():
    n, levels = 64, 3
    q = np.random.default_rng(0).standard_normal((3, 4))
    kp = np.ones((n, 4))
    got = wo.recursive_filter(q, kp, levels, [5, 6, 4, 2])
    np.testing.assert_array_equal(got["levels"][3]["sel"], [0, 1])
    np.testing.assert_array_equal(got["levels"][2]["sel"], [0, 1, 2, 3])
    np.testing.assert_array_equal(got["idx"], [0, 1, 2, 3, 4])


# ------------------------------------------------------------------ attention

def test_sparse_attention_worked_example():
    g = _load("attention_mass_2x2.json")
    q = np.array(g["Q"], dtype=np.float64)
    k = np.array([[_ev(e) for e in row] for row in g["K"]])
    v = np.array(g["V"], dtype=np.float64)
    out, lse = wo.sparse_attention(q, k, v, np.zeros((0, 2)), np.zeros((0, 2)), [0, 1])
    np.testing.assert_allclose(out, [[_ev(e) for e in r] for r in g["out"]], rtol=1e-14)
    np.testing.assert_allclose(lse, [_ev(e) for e in g["lse"]], rtol=1e-14)


def test_full_budget_is_full_attention():
    # B = N_p with every level kept: the sparse cache is the whole cache (eq. 3).
    rng = np.random.default_rng(9)
    n, g, d, levels = 64, 6, 16, 3
    q, kp, vp = (rng.standard_normal(s) for s in ((g, d), (n, d), (n, d)))
    kg, vg = rng.standard_normal((g, d)), rng.standard_normal((g, d))
    ks = [n] + [n >> j for j in range(1, levels + 1)]
    res = wo.wavefilter_step(q, kp, vp, kg, vg, levels, ks)
    np.testing.assert_array_equal(res["idx"], np.arange(n))
    want = _sdpa(q, np.concatenate([kp, kg]), np.concatenate([vp, vg]))
    np.testing.assert_allclose(res["out"], want, rtol=1e-12, atol=1e-13)


def test_sparse_attention_uses_only_selected_rows():
    rng = np.random.default_rng(12)
    n, g, d = 40, 3, 8
    q, kp, vp = (rng.standard_normal(s) for s in ((g, d), (n, d), (n, d)))
    kg, vg = rng.standard_normal((2, d)), rng.standard_normal((2, d))
    idx = np.array([2, 5, 6, 30])
    out, _ = wo.sparse_attention(q, kp, vp, kg, vg, idx)
    want = _sdpa(q, np.concatenate([kp[idx], kg]), np.concatenate([vp[idx], vg]))
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-13)


def test_lse_closed_forms():
    g, d = 3, 8
    q = np.random.default_rng(1).standard_normal((g, d))
    out, lse = wo.sparse_attention(q, np.zeros((10, d)), np.arange(10 * d, dtype=float).reshape(10, d),
                                   np.zeros((2, d)), np.ones((2, d)), [1, 4, 7])
    np.testing.assert_allclose(lse, np.full(g, math.log(5)), rtol=1e-14)
    want = (np.arange(10 * d).reshape(10, d)[[1, 4, 7]].sum(0) + 2.0) / 5.0
    np.testing.assert_allclose(out, np.tile(want, (g, 1)), rtol=1e-13)
    # One key: lse is its logit.
    k1 = np.random.default_rng(2).standard_normal((1, d))
    _, lse1 = wo.sparse_attention(q, k1, np.ones((1, d)), np.zeros((0, d)), np.zeros((0, d)), [0])
    np.testing.assert_allclose(lse1, (q @ k1.T)[:, 0] / math.sqrt(d), rtol=1e-13)


# ------------------------------------------------------------ sanity statistic

@pytest.mark.parametrize("name", ["tiny", "llada8b_layer"])
def test_planted_span_recall_sanity(name):
    """Not parity: the synthetic needles should mostly survive the filter
    (chance level is B / N_p = 1/16 here)."""
    from wavelet_guided_sparse_gb300 import workloads as wl
    cfg = wl.CONFIGS[name]
    st = wl.span_starts(cfg, 0, 0)
    planted = np.concatenate([np.arange(s, s + cfg.span_len) for s in st])
    recalls = []
    for h in range(2):
        u = wl.generate_unit(cfg, 0, 0, h)
        idx = wo.recursive_filter(u["Q"], u["Kp"], cfg.levels, cfg.k_per_level())["idx"]
        assert len(idx) == cfg.budget and (np.diff(idx) > 0).all()
        recalls.append(np.isin(planted, idx).mean())
    assert min(recalls) > 0.5, recalls


# ------------------------------------------------- cache write (eqs. (2), (4))

def _coded_kv(n, h, d):
    """K[n, h, c] = n + 1000 h + 10^6 c and V = -(K + 1/2): every entry names
    its own (position, head, channel), exactly in float64."""
    nn, hh, cc = np.meshgrid(np.arange(n), np.arange(h), np.arange(d), indexing="ij")
    k = (nn + 1000.0 * hh + 1e6 * cc).astype(np.float64)
    return k, -(k + 0.5)


@pytest.mark.parametrize("n_prompt,n_gen,heads,d,levels", [(16, 3, 2, 3, 2), (32, 5, 3, 4, 3),
                                                           (8, 1, 1, 2, 1)])
def test_cache_init_places_every_row(n_prompt, n_gen, heads, d, levels):
    # Eq. (2): cache row n of head h holds position n of head h, prompt and
    # generation block split at n_prompt, values beside their keys.
    k, v = _coded_kv(n_prompt + n_gen, heads, d)
    c = wo.cache_init(k, v, n_prompt, levels)
    assert c["Kp"].shape == (heads, n_prompt, d) and c["Kg"].shape == (heads, n_gen, d)
    for h in range(heads):
        for n in range(n_prompt + n_gen):
            for ch in range(d):
                want = n + 1000 * h + 1e6 * ch
                if n < n_prompt:
                    assert c["Kp"][h, n, ch] == want and c["Vp"][h, n, ch] == -(want + 0.5)
                else:
                    g = n - n_prompt
                    assert c["Kg"][h, g, ch] == want and c["Vg"][h, g, ch] == -(want + 0.5)


@pytest.mark.parametrize("levels", [1, 2, 3])
def test_cache_init_lowpass_closed_form(levels):
    # A_L of the coded keys in closed form: the span of coarse position p
    # holds positions p 2^L .. p 2^L + 2^L - 1, so
    #   sum = 2^L (1000 h + 10^6 c) + 2^(2L) p + 2^(L-1) (2^L - 1)
    # and A_L = 2^(-L/2) * sum (orthonormal Haar, scaled span sum).
    n_prompt, n_gen, heads, d = 32, 4, 2, 3
    k, v = _coded_kv(n_prompt + n_gen, heads, d)
    a = wo.cache_init(k, v, n_prompt, levels)["a_l"]
    span = 1 << levels
    assert a.shape == (heads, n_prompt >> levels, d)
    for h in range(heads):
        for p in range(n_prompt >> levels):
            for ch in range(d):
                s = span * (1000 * h + 1e6 * ch) + span * span * p + (span // 2) * (span - 1)
                assert a[h, p, ch] == pytest.approx(s * 2.0 ** (-levels / 2), rel=1e-14)


def test_cache_init_round_trip_and_rejects():
    rng = np.random.default_rng(11)
    k, v = rng.standard_normal((2, 40, 3, 5))
    c = wo.cache_init(k, v, 32, 2)
    back = np.concatenate([c["Kp"], c["Kg"]], axis=1)
    np.testing.assert_array_equal(np.swapaxes(back, 0, 1), k)
    with pytest.raises(ValueError):
        wo.cache_init(k, v[:, :2], 32, 2)
    with pytest.raises(ValueError):
        wo.cache_init(k, v, 0, 2)


def test_cache_update_places_every_row():
    # Eq. (4): generation row g of head h takes the new key of position g.
    k, v = _coded_kv(5, 3, 2)
    c = wo.cache_update(k, v)
    for h in range(3):
        for g in range(5):
            for ch in range(2):
                want = g + 1000 * h + 1e6 * ch
                assert c["Kg"][h, g, ch] == want and c["Vg"][h, g, ch] == -(want + 0.5)


def _scatter_case(n_prompt=16, n_gen=4, heads=2, d=3, seed=5):
    """A cache holding coded rows and M new coded rows (offset by 0.25 so they
    differ from every old entry) for a scattered position set that mixes
    prompt and generation positions."""
    k, v = _coded_kv(n_prompt + n_gen, heads, d)
    c = wo.cache_init(k, v, n_prompt, 1)
    rng = np.random.default_rng(seed)
    pos = rng.choice(n_prompt + n_gen, size=7, replace=False)
    nk = np.stack([k[n] + 0.25 for n in pos])
    nv = np.stack([v[n] - 0.25 for n in pos])
    return c, pos, nk, nv


def test_cache_scatter_places_every_row():
    # Eq. (4) over a scattered set: row n of head h holds the new coded row of
    # position n if n was written, else its old coded row.
    n_prompt, n_gen, heads, d = 16, 4, 2, 3
    c, pos, nk, nv = _scatter_case(n_prompt, n_gen, heads, d)
    out = wo.cache_scatter(c["Kp"], c["Vp"], c["Kg"], c["Vg"], nk, nv, pos)
    written = set(pos.tolist())
    for h in range(heads):
        for n in range(n_prompt + n_gen):
            for ch in range(d):
                base = n + 1000 * h + 1e6 * ch
                want_k = base + 0.25 if n in written else base
                want_v = -(base + 0.5) - 0.25 if n in written else -(base + 0.5)
                kk = out["Kp"][h, n, ch] if n < n_prompt else out["Kg"][h, n - n_prompt, ch]
                vv = out["Vp"][h, n, ch] if n < n_prompt else out["Vg"][h, n - n_prompt, ch]
                assert kk == want_k and vv == want_v, (h, n, ch)


def test_cache_scatter_rejects():
    c, pos, nk, nv = _scatter_case()
    with pytest.raises(ValueError):
        wo.cache_scatter(c["Kp"], c["Vp"], c["Kg"], c["Vg"], nk, nv, np.r_[pos[:-1], pos[0]])
    with pytest.raises(ValueError):
        wo.cache_scatter(c["Kp"], c["Vp"], c["Kg"], c["Vg"], nk, nv, np.r_[pos[:-1], 20])
    with pytest.raises(ValueError):
        wo.cache_scatter(c["Kp"], c["Vp"], c["Kg"], c["Vg"], nk[:, :1], nv[:, :1], pos)


@pytest.mark.parametrize("levels", [1, 2, 3])
def test_al_repair_equals_full_pyramid_and_keeps_untouched_rows(levels):
    # The repaired A_L equals the pyramid of the whole updated prompt cache,
    # and coarse positions whose span holds no rewritten row are the input's
    # rows bit for bit.
    n_prompt = 32
    rng = np.random.default_rng(levels)
    kp = rng.standard_normal((3, n_prompt, 4))
    a_l = np.stack([wo.haar_pyramid(kp[h], levels)[levels] for h in range(3)])
    pos = np.array([3, 17, 18, 33])  # 33: a generation position
    nk = rng.standard_normal((4, 3, 4))
    kp_new = kp.copy()
    for m, n in enumerate(pos):
        if n < n_prompt:
            kp_new[:, n] = nk[m]
    out = wo.al_repair(a_l, kp_new, pos, levels)
    full = np.stack([wo.haar_pyramid(kp_new[h], levels)[levels] for h in range(3)])
    np.testing.assert_allclose(out, full, rtol=1e-14, atol=1e-14)
    touched = {int(n) >> levels for n in pos if n < n_prompt}
    for c in range(n_prompt >> levels):
        if c not in touched:
            assert np.array_equal(out[:, c], a_l[:, c]), c
        else:
            assert not np.array_equal(out[:, c], a_l[:, c]), c


def test_al_repair_closed_form():
    # Coded keys, prompt position 5 rewritten to K + 0.25 at L = 2: the span
    # of coarse position 1 (tokens 4..7) sums to its old closed form plus 0.25,
    # scaled by 2^(-L/2); the other coarse positions keep theirs.
    n_prompt, heads, d, L = 16, 2, 3, 2
    k, v = _coded_kv(n_prompt + 2, heads, d)
    c = wo.cache_init(k, v, n_prompt, L)
    kp_new = c["Kp"].copy()
    kp_new[:, 5] += 0.25
    out = wo.al_repair(c["a_l"], kp_new, [5], L)
    span = 1 << L
    for h in range(heads):
        for p in range(n_prompt >> L):
            for ch in range(d):
                s = span * (1000 * h + 1e6 * ch) + span * span * p + (span // 2) * (span - 1)
                s += 0.25 if p == 1 else 0.0
                assert out[h, p, ch] == pytest.approx(s * 2.0 ** (-L / 2), rel=1e-14)


# ----------------------------------------------------- Daubechies bases (psi)

def test_daubechies_db1_is_haar():
    g = wo.daubechies_lowpass(1)
    np.testing.assert_allclose(g, [1 / math.sqrt(2)] * 2, rtol=1e-15)
    x = np.random.default_rng(3).standard_normal((32, 5))
    a, d = wo.dwt_analysis_step(x, g)
    ha, hd = wo.haar_analysis_step(x)
    np.testing.assert_allclose(a, ha, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(d, hd, rtol=1e-14, atol=1e-15)


def test_daubechies_db2_closed_form():
    # The four-tap Daubechies filter in closed form: (1+√3, 3+√3, 3−√3, 1−√3) / (4√2).
    s3 = math.sqrt(3.0)
    want = np.array([1 + s3, 3 + s3, 3 - s3, 1 - s3]) / (4 * math.sqrt(2.0))
    np.testing.assert_allclose(wo.daubechies_lowpass(2), want, rtol=1e-13)


@pytest.mark.parametrize("n", [2, 3, 4, 6])
def test_daubechies_filter_conditions(n):
    g = wo.daubechies_lowpass(n)
    f = len(g)
    assert f == 2 * n
    assert math.isclose(g.sum(), math.sqrt(2.0), rel_tol=1e-13)
    # Orthonormal to its own even shifts.
    for m in range(n):
        dot = float(np.dot(g[:f - 2 * m], g[2 * m:]))
        assert abs(dot - (1.0 if m == 0 else 0.0)) < 1e-12, m
    # N vanishing moments: the mirror high-pass kills polynomials of degree < N.
    k = np.arange(f, dtype=np.float64)
    for p in range(n):
        assert abs(np.sum((-1.0) ** k * k ** p * g)) < 1e-9 * max(1.0, (f - 1) ** p), p
    # Extremal phase: apart from the N zeros at -1, every zero inside the unit
    # circle (a root of multiplicity N comes back from np.roots split by about
    # eps^(1/N), hence the loose test for "at -1"; the others lie > 1 away).
    zeros = np.roots(g)
    inner = zeros[np.abs(zeros + 1) > 0.05]
    assert len(inner) == n - 1 and (np.abs(inner) < 1).all()


@pytest.mark.parametrize("n,levels", [(2, 3), (4, 2), (3, 4)])
def test_wavelet_perfect_reconstruction_and_parseval(n, levels):
    g = wo.daubechies_lowpass(n)
    x = np.random.default_rng(n * 10 + levels).standard_normal((64, 3))
    a, details = x, []
    for _ in range(levels):
        a, d = wo.dwt_analysis_step(a, g)
        details.append(d)
    energy = (a ** 2).sum() + sum((d ** 2).sum() for d in details)
    assert math.isclose(energy, (x ** 2).sum(), rel_tol=1e-12)
    for d in reversed(details):
        a = wo.dwt_synthesis_step(a, d, g)
    np.testing.assert_allclose(a, x, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n", [2, 3, 4])
def test_wavelet_polynomial_details_vanish(n):
    # Away from the periodic wrap, the details of a degree < N polynomial are 0.
    g = wo.daubechies_lowpass(n)
    t = np.arange(64, dtype=np.float64) / 64
    x = sum((j + 1) * t ** j for j in range(n))[:, None]
    _, d = wo.dwt_analysis_step(x, g)
    interior = d[: (64 - len(g)) // 2 + 1]
    assert np.abs(interior).max() < 1e-10


@pytest.mark.parametrize("n,levels", [(1, 3), (2, 3), (4, 2), (3, 3)])
def test_wavelet_pyramid_equals_equivalent_filter(n, levels):
    # Cascade identity: A_L[p] = sum_m w_L[m] x[(2^L p + m) mod N] with
    # w_1 = g and w_j = (g upsampled by 2^(j-1)) convolved with w_(j-1).
    g = wo.daubechies_lowpass(n)
    w = g.copy()
    for j in range(2, levels + 1):
        up = np.zeros((len(g) - 1) * 2 ** (j - 1) + 1)
        up[:: 2 ** (j - 1)] = g
        w = np.convolve(up, w)
    size = 128
    x = np.random.default_rng(n + levels).standard_normal((size, 4))
    want = np.zeros((size >> levels, 4))
    for p in range(size >> levels):
        for m, wm in enumerate(w):
            want[p] += wm * x[((p << levels) + m) % size]
    np.testing.assert_allclose(wo.wavelet_pyramid(x, levels, g)[levels], want, rtol=1e-12,
                               atol=1e-12)



@pytest.mark.parametrize("n_mom,n,levels,ks,g", [
    (2, 64, 3, [5, 7, 6, 4], 3),
    (4, 128, 3, [20, 18, 10, 6], 4),
    (3, 256, 4, [30, 16, 9, 6, 4], 2),
])
def test_recursive_filter_basis_matches_dense_bruteforce(n_mom, n, levels, ks, g):
    rng = np.random.default_rng(n + levels * 17 + g + 100 * n_mom)
    d = 8
    q = rng.standard_normal((g, d)) * 1.5
    kp = rng.standard_normal((n, d)) * 1.5
    low = wo.daubechies_lowpass(n_mom)
    got = wo.recursive_filter(q, kp, levels, ks, lowpass=low)
    want = _dense_reference_levels(q, kp, levels, ks, lowpass=low)
    for j in range(levels + 1):
        np.testing.assert_array_equal(got["levels"][j]["sel"], want[j], err_msg=f"level {j}")


@pytest.mark.parametrize("n_mom", [2, 4])
def test_recursive_filter_basis_keep_all_is_token_topk(n_mom):
    rng = np.random.default_rng(50 + n_mom)
    n, levels, b, d = 128, 3, 19, 16
    q = rng.standard_normal((4, d))
    kp = rng.standard_normal((n, d)) * 2
    ks = [b] + [n >> j for j in range(1, levels + 1)]
    got = wo.recursive_filter(q, kp, levels, ks, lowpass=wo.daubechies_lowpass(n_mom))["idx"]
    np.testing.assert_array_equal(got, _brute_topk(_mass_by_sdpa(q, kp), np.arange(n), b))


def test_recursive_filter_db1_equals_haar():
    rng = np.random.default_rng(21)
    q = rng.standard_normal((5, 8))
    kp = rng.standard_normal((256, 8))
    ks = [40, 30, 20, 12, 8]
    a = wo.recursive_filter(q, kp, 4, ks)
    b = wo.recursive_filter(q, kp, 4, ks, lowpass=wo.daubechies_lowpass(1))
    for j in range(5):
        np.testing.assert_array_equal(a["levels"][j]["sel"], b["levels"][j]["sel"])
