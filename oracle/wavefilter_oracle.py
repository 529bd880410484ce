"""Float64 CPU oracle of the WaveFilter per-layer, per-step KV filtering path.

TEST INFRASTRUCTURE ONLY.  This module is the checker the CUDA path is held
to.  Only the test suite, the package smoke check and the benchmark's CPU
baseline leg may import it; the product path never calls it and shares no
code with it.

Source: "WaveFilter: Enhancing the Long-Context Capability of Diffusion LLMs
via Wavelet-Guided KV Cache Filtering" (arXiv 2606.00724).  The pages give
eq. (3) (cached attention, §2.1), eq. (5) (one DWT level, §2.2), the DWT
pyramid {A_L, D_L..D_1} (§2.2), the DWT of the cached prompt keys with a
basis psi (§3.1), and a prose pipeline (§1, Fig. 2 (b)-(d), §3 overview):
extract low-frequency key features, score them against the queries with
attention, keep a Top-K of candidate regions, refine those regions
recursively across scales down to tokens, build a sparse KV cache from the
final tokens plus the generation positions and attend over it.  §3.2 and
Appendix A are not on the pages, so the following readings are taken (each
one plainest consistent with the rest):

  * psi is the orthonormal Haar pair g = [1/sqrt2, 1/sqrt2],
    h = [1/sqrt2, -1/sqrt2]; eq. (5) pairs 0-based samples (2n, 2n+1), so
    A_j[p] covers tokens [p 2^j, (p+1) 2^j).
  * Score of a candidate = attention mass: for each query of the generation
    block, softmax over the current candidate set of Q . A_j / sqrt(d), then
    summed over the queries.  Raw orthonormal coefficients are used.
  * Candidates at level j < L are the two children {2p, 2p+1} of every level
    j+1 survivor; k_j survivors are kept per level, k_0 = final budget B.
  * Top-K order: larger score first, equal scores -> lower position first.
  * The sparse cache is the selected prompt tokens (ascending) followed by
    all generation positions; eq. (3) attention over it, no mask.
  * Longer bases (psi is open): the extremal-phase Daubechies filters with N
    vanishing moments (N = 1 is Haar), each level extended periodically; the
    recursive filter then keeps the pyramid's index tree (children 2p, 2p+1)
    and scores A_j of that basis.
  * Cache writes: eq. (2) stores the keys/values of every position at t = 1
    (token-major input, head-major cache, prompt positions first), eq. (4)
    replaces the generation rows at t > 1.

Everything is float64 numpy, one unit (sequence, layer, head) at a time,
with no blocking or fusion beyond the definitions above.
"""

from __future__ import annotations

import math
from typing import Dict, List, Sequence

import numpy as np

SQRT2 = math.sqrt(2.0)

__all__ = [
    "haar_analysis_step",
    "haar_synthesis_step",
    "haar_dwt",
    "haar_idwt",
    "haar_pyramid",
    "attention_mass",
    "top_k",
    "recursive_filter",
    "sparse_attention",
    "wavefilter_step",
    "wavefilter_step_batched",
    "cache_init",
    "cache_update",
    "cache_scatter",
    "al_repair",
    "daubechies_lowpass",
    "dwt_analysis_step",
    "dwt_synthesis_step",
    "wavelet_pyramid",
]


def haar_analysis_step(x: np.ndarray):
    """One level of eq. (5) (WaveFilter §2.2) along axis 0 with Haar filters.

    A_1[n] = (x[2n] + x[2n+1]) / sqrt2 (low-pass g), D_1[n] = (x[2n] -
    x[2n+1]) / sqrt2 (high-pass h); the factor-2 downsampling of eq. (5) is
    the step of 2 in n.  Axis 0 must have even length.
    """
    x = np.asarray(x, dtype=np.float64)
    if x.shape[0] % 2:
        raise ValueError("length must be even")
    even, odd = x[0::2], x[1::2]
    return (even + odd) / SQRT2, (even - odd) / SQRT2


def haar_synthesis_step(a: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Inverse of :func:`haar_analysis_step` (orthonormal Haar synthesis)."""
    a = np.asarray(a, dtype=np.float64)
    d = np.asarray(d, dtype=np.float64)
    out = np.empty((2 * a.shape[0],) + a.shape[1:], dtype=np.float64)
    out[0::2] = (a + d) / SQRT2
    out[1::2] = (a - d) / SQRT2
    return out


def haar_dwt(x: np.ndarray, levels: int):
    """L-level pyramid of WaveFilter §2.2: returns (A_L, [D_1, ..., D_L]).

    The approximation A_j is fed back into eq. (5) for the next level.
    """
    a = np.asarray(x, dtype=np.float64)
    details = []
    for _ in range(levels):
        a, d = haar_analysis_step(a)
        details.append(d)
    return a, details


def haar_idwt(a_l: np.ndarray, details: Sequence[np.ndarray]) -> np.ndarray:
    """Rebuild the signal from (A_L, [D_1..D_L]) (used for self-tests)."""
    a = np.asarray(a_l, dtype=np.float64)
    for d in reversed(list(details)):
        a = haar_synthesis_step(a, d)
    return a


def haar_pyramid(x: np.ndarray, levels: int) -> List[np.ndarray]:
    """Approximations [A_0 = x, A_1, ..., A_L] (WaveFilter §2.2, §3.1).

    A_L of the prompt keys is the low-frequency component K_low of §3.1.
    """
    out = [np.asarray(x, dtype=np.float64)]
    for _ in range(levels):
        out.append(haar_analysis_step(out[-1])[0])
    return out


def attention_mass(q: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Importance of each candidate key (WaveFilter Fig. 2(c), §1).

    z[i, c] = Q[i] . keys[c] / sqrt(d) (the eq. (3) logits), a softmax over
    the candidates for every query i, and the per-candidate sum over the
    queries.  Returns s[c] (non-negative, summing to the number of queries).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    d = q.shape[-1]
    z = q @ keys.T / math.sqrt(d)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    return p.sum(axis=0)


def top_k(scores: np.ndarray, positions: np.ndarray, k: int):
    """Top-k candidate positions (WaveFilter Fig. 2(c)-(d) "Top-K").

    Order: larger score first; equal scores -> lower position first.
    Returns (selected positions sorted ascending, boundary gap), where the
    gap is (s_(k) - s_(k+1)) / s_(k) for the scores sorted in that order, or
    +inf when every candidate is kept.
    """
    scores = np.asarray(scores, dtype=np.float64)
    positions = np.asarray(positions, dtype=np.int64)
    if not 1 <= k:
        raise ValueError("k must be >= 1")
    order = np.lexsort((positions, -scores))  # last key is primary
    if k >= len(positions):
        return np.sort(positions), math.inf
    kth, nxt = scores[order[k - 1]], scores[order[k]]
    gap = (kth - nxt) / kth if kth > 0 else 0.0
    return np.sort(positions[order[:k]]), gap


def recursive_filter(q: np.ndarray, kp: np.ndarray, levels: int,
                     k_per_level: Sequence[int], lowpass=None) -> Dict:
    """Coarse Top-K plus multi-scale recursive filtering (WaveFilter §3.1-§3.2,
    Fig. 2(b)-(d)).

    Level L: candidates are all N_p / 2^L positions of A_L; keep k_L.
    Level j = L-1 .. 0: candidates are the children {2p, 2p+1} of the level
    j+1 survivors, scored against A_j; keep k_j.  Level 0 yields the final
    token set S (k_0 = B tokens, ascending).

    ``lowpass``: None for the Haar pyramid, else the low-pass filter of
    another orthonormal basis (``daubechies_lowpass``); the candidates still
    follow the pyramid's index tree, A_j comes from :func:`wavelet_pyramid`.

    Returns {"idx": S, "levels": {j: {"cand", "scores", "sel", "gap"}}}.
    """
    q = np.asarray(q, dtype=np.float64)
    pyr = haar_pyramid(kp, levels) if lowpass is None else wavelet_pyramid(kp, levels, lowpass)
    if len(k_per_level) != levels + 1:
        raise ValueError("k_per_level needs levels + 1 entries")
    per_level = {}
    cand = np.arange(pyr[levels].shape[0], dtype=np.int64)
    sel = None
    for j in range(levels, -1, -1):
        if j < levels:
            cand = np.sort(np.concatenate([2 * sel, 2 * sel + 1]))
        if k_per_level[j] > len(cand):
            raise ValueError(f"k_{j}={k_per_level[j]} exceeds {len(cand)} candidates")
        s = attention_mass(q, pyr[j][cand])
        sel, gap = top_k(s, cand, int(k_per_level[j]))
        per_level[j] = {"cand": cand, "scores": s, "sel": sel, "gap": gap}
    return {"idx": sel, "levels": per_level}


def sparse_attention(q, kp, vp, kg, vg, idx):
    """Eq. (3) of WaveFilter §2.1 over the sparse cache (Fig. 2(d)).

    Keys/values are the prompt rows at ``idx`` followed by every generation
    row; O = softmax(Q K^T / sqrt(d)) V with no mask.  Also returns the
    natural-log normaliser lse[i] = log sum_j exp(Q[i] . K_j / sqrt(d)).
    """
    q = np.asarray(q, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    k = np.concatenate([np.asarray(kp, np.float64)[idx], np.asarray(kg, np.float64)])
    v = np.concatenate([np.asarray(vp, np.float64)[idx], np.asarray(vg, np.float64)])
    z = q @ k.T / math.sqrt(q.shape[-1])
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    denom = e.sum(axis=1, keepdims=True)
    out = (e / denom) @ v
    lse = (m + np.log(denom))[:, 0]
    return out, lse


def wavefilter_step(q, kp, vp, kg, vg, levels: int, k_per_level: Sequence[int],
                    lowpass=None) -> Dict:
    """Whole path for one unit: DWT -> coarse Top-K -> recursive filtering ->
    sparse cache -> eq. (3) attention.  Returns the selection record plus
    "out" [G, d], "lse" [G] and "a_l" (the level-L approximation).
    ``lowpass`` as in :func:`recursive_filter` (None: Haar)."""
    sel = recursive_filter(q, kp, levels, k_per_level, lowpass)
    out, lse = sparse_attention(q, kp, vp, kg, vg, sel["idx"])
    sel["out"] = out
    sel["lse"] = lse
    sel["a_l"] = (haar_pyramid(kp, levels) if lowpass is None
                  else wavelet_pyramid(kp, levels, lowpass))[levels]
    return sel


def wavefilter_step_batched(inputs: Dict[str, np.ndarray], levels: int,
                            k_per_level: Sequence[int]) -> List[Dict]:
    """Apply :func:`wavefilter_step` to every unit of [b, H, rows, d] arrays
    (units are independent).  Returns a flat list in (b, h) order."""
    b, h = inputs["Q"].shape[:2]
    res = []
    for bi in range(b):
        for hi in range(h):
            res.append(wavefilter_step(inputs["Q"][bi, hi], inputs["Kp"][bi, hi],
                                       inputs["Vp"][bi, hi], inputs["Kg"][bi, hi],
                                       inputs["Vg"][bi, hi], levels, k_per_level))
    return res


def cache_init(k_all, v_all, n_prompt: int, levels: int) -> Dict:
    """KV-cache initialisation at the first denoising step t = 1 (WaveFilter
    §2.1 eq. (2)) plus the low-frequency component of the cached prompt keys
    (§3.1), which §1 extracts at that initial step.

    ``k_all``, ``v_all``: [N, H, d], one sequence in token-major order (the
    keys and values eq. (1) computes for every position I, heads side by
    side per token).  Positions [0, n_prompt) form the prompt I_p, the rest
    [n_prompt, N) the generation block I_g.  Eq. (2) stores them unchanged:
    the cache keeps each head's rows in position order.

    Returns {"Kp": [H, N_p, d], "Vp", "Kg": [H, N - N_p, d], "Vg",
    "a_l": [H, N_p / 2^L, d]} with a_l = A_L of Kp per head (haar_pyramid).
    """
    k = np.asarray(k_all, dtype=np.float64)
    v = np.asarray(v_all, dtype=np.float64)
    if k.ndim != 3 or k.shape != v.shape:
        raise ValueError("K and V must both be [N, H, d]")
    if not 0 < n_prompt <= k.shape[0]:
        raise ValueError("n_prompt out of range")
    # Per head h, cache row n is position n of that head: a swap of the
    # token and head axes.
    kp = np.swapaxes(k[:n_prompt], 0, 1)
    vp = np.swapaxes(v[:n_prompt], 0, 1)
    kg = np.swapaxes(k[n_prompt:], 0, 1)
    vg = np.swapaxes(v[n_prompt:], 0, 1)
    a_l = np.stack([haar_pyramid(kp[h], levels)[levels] for h in range(kp.shape[0])])
    return {"Kp": kp, "Vp": vp, "Kg": kg, "Vg": vg, "a_l": a_l}


def cache_update(k_gen, v_gen) -> Dict:
    """Cache update at a later step t > 1 (WaveFilter §2.1 eq. (4)): the keys
    and values just computed for the generation positions replace the cached
    ones, K~^t[I~] = K^t[I~], V~^t[I~] = V^t[I~].

    ``k_gen``, ``v_gen``: [G, H, d] token-major.  Returns {"Kg": [H, G, d],
    "Vg"}: the new generation-block cache, rows in position order per head.
    The prompt part of the cache is untouched, so an A_L computed from it
    stays valid.
    """
    k = np.asarray(k_gen, dtype=np.float64)
    v = np.asarray(v_gen, dtype=np.float64)
    if k.ndim != 3 or k.shape != v.shape:
        raise ValueError("K and V must both be [G, H, d]")
    return {"Kg": np.swapaxes(k, 0, 1), "Vg": np.swapaxes(v, 0, 1)}


def cache_scatter(kp, vp, kg, vg, k_new, v_new, positions) -> Dict:
    """Cache update over an arbitrary inferred set (WaveFilter §2.1 eq. (4):
    K~^t[I~] = K^t[I~], V~^t[I~] = V^t[I~]), where I~ may hold generation
    positions and prompt positions alike (caching schemes that refresh part of
    the prompt cache write those rows too).

    ``kp``, ``vp``: [H, N_p, d] and ``kg``, ``vg``: [H, G, d], the cache of one
    sequence (position n < N_p is prompt row n, position N_p + g is generation
    row g).  ``k_new``, ``v_new``: [M, H, d] token-major rows for the M
    distinct ``positions`` (0 <= position < N_p + G).  Returns new arrays
    {"Kp", "Vp", "Kg", "Vg"}; every row not in ``positions`` is unchanged.
    """
    kp, vp = np.array(kp, np.float64), np.array(vp, np.float64)
    kg, vg = np.array(kg, np.float64), np.array(vg, np.float64)
    k_new = np.asarray(k_new, np.float64)
    v_new = np.asarray(v_new, np.float64)
    pos = np.asarray(positions, np.int64)
    n_prompt, n_gen = kp.shape[1], kg.shape[1]
    if k_new.shape != v_new.shape or k_new.ndim != 3 or k_new.shape[0] != len(pos):
        raise ValueError("new rows must be [M, H, d] for M positions")
    if k_new.shape[1:] != (kp.shape[0], kp.shape[2]):
        raise ValueError("new rows disagree with the cache on heads / head_dim")
    if len(set(pos.tolist())) != len(pos):
        raise ValueError("positions must be distinct")
    if ((pos < 0) | (pos >= n_prompt + n_gen)).any():
        raise ValueError("position outside the cache")
    for m, n in enumerate(pos):
        if n < n_prompt:
            kp[:, n], vp[:, n] = k_new[m], v_new[m]
        else:
            kg[:, n - n_prompt], vg[:, n - n_prompt] = k_new[m], v_new[m]
    return {"Kp": kp, "Vp": vp, "Kg": kg, "Vg": vg}


def al_repair(a_l, kp_new, positions, levels: int) -> np.ndarray:
    """The level-L approximation (WaveFilter §2.2 pyramid, §3.1) of the
    prompt keys after a scatter, without recomputing all of it: a coarse
    position p covers tokens [p 2^L, (p+1) 2^L), so only the coarse positions
    whose span holds a rewritten prompt position change; each of them is the
    pyramid of its span's new keys, every other row of ``a_l`` is kept.

    ``a_l``: [H, N_p / 2^L, d] of the cache before the scatter; ``kp_new``:
    [H, N_p, d] after it; ``positions`` as for :func:`cache_scatter`
    (generation positions do not touch A_L).
    """
    out = np.array(a_l, np.float64)
    kp_new = np.asarray(kp_new, np.float64)
    n_prompt = kp_new.shape[1]
    touched = sorted({int(n) >> levels for n in np.asarray(positions) if n < n_prompt})
    for c in touched:
        for h in range(kp_new.shape[0]):
            span = kp_new[h, c << levels:(c + 1) << levels]
            out[h, c] = haar_pyramid(span, levels)[levels][0]
    return out


# ------------------------------------------------------------------------
# Longer orthonormal bases.  §3.1 leaves the basis psi open; the Haar pair is
# the shortest member of the Daubechies family, whose longer members trade
# span locality for smoother low-pass responses.  Readings: the filters are
# the extremal-phase Daubechies filters with N vanishing moments, and each
# level extends its input periodically, which keeps every level an
# orthonormal transform for any even length.


def daubechies_lowpass(n_moments: int) -> np.ndarray:
    """Low-pass filter g (length 2N) of the orthonormal Daubechies wavelet
    with N = ``n_moments`` vanishing moments, from its defining polynomial.

    The filter's frequency response satisfies
        |m0(w)|^2 = cos(w/2)^(2N) * P(sin(w/2)^2),
        P(y) = sum_{k=0}^{N-1} binom(N-1+k, k) y^k,
    so m0 has N zeros at z = -1 and, for every root y_k of P, one zero of
    z^2 - (2 - 4 y_k) z + 1 (the substitution y = (2 - z - 1/z) / 4); of each
    such reciprocal pair the zero inside the unit circle is taken (extremal
    phase, energy front-loaded).  g holds the coefficients of the polynomial
    with those zeros, highest power first, scaled so that sum(g) = sqrt2.
    N = 1 gives the Haar filter [1/sqrt2, 1/sqrt2].
    """
    n = int(n_moments)
    if n < 1:
        raise ValueError("need at least one vanishing moment")
    zeros = [-1.0] * n
    if n > 1:
        p_desc = [math.comb(n - 1 + k, k) for k in range(n - 1, -1, -1)]
        for y in np.roots(p_desc):
            b = 1.0 - 2.0 * y
            r = np.sqrt(b * b - 1.0 + 0j)
            z1, z2 = b + r, b - r
            zeros.append(z1 if abs(z1) < 1.0 else z2)
    g = np.real(np.poly(np.array(zeros, dtype=complex)))
    return g * (SQRT2 / g.sum())


def _highpass(g: np.ndarray) -> np.ndarray:
    """Quadrature-mirror partner h[k] = (-1)^k g[F-1-k] of a low-pass g."""
    g = np.asarray(g, dtype=np.float64)
    return np.array([(-1.0) ** k * g[len(g) - 1 - k] for k in range(len(g))])


def dwt_analysis_step(x: np.ndarray, g: np.ndarray):
    """One level of eq. (5) (WaveFilter §2.2) along axis 0 for a general
    orthonormal low-pass g, input extended periodically:
        A[n] = sum_k g[k] x[(2n + k) mod M],  D[n] = sum_k h[k] x[(2n + k) mod M]
    with h the quadrature mirror of g.  With the Haar g this is
    :func:`haar_analysis_step`.  Axis 0 must have even length M.
    """
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    h = _highpass(g)
    m = x.shape[0]
    if m % 2:
        raise ValueError("length must be even")
    base = 2 * np.arange(m // 2)
    a = np.zeros((m // 2,) + x.shape[1:])
    d = np.zeros_like(a)
    for k in range(len(g)):
        rows = x[(base + k) % m]
        a += g[k] * rows
        d += h[k] * rows
    return a, d


def dwt_synthesis_step(a: np.ndarray, d: np.ndarray, g: np.ndarray) -> np.ndarray:
    """Inverse of :func:`dwt_analysis_step`: the transpose of the orthonormal
    analysis map, x[(2n + k) mod M] += g[k] A[n] + h[k] D[n]."""
    a = np.asarray(a, dtype=np.float64)
    d = np.asarray(d, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    h = _highpass(g)
    m = 2 * a.shape[0]
    x = np.zeros((m,) + a.shape[1:])
    base = 2 * np.arange(m // 2)
    for k in range(len(g)):
        np.add.at(x, (base + k) % m, g[k] * a + h[k] * d)
    return x


def wavelet_pyramid(x: np.ndarray, levels: int, g: np.ndarray) -> List[np.ndarray]:
    """Approximations [A_0 = x, A_1, ..., A_L] of the pyramid of WaveFilter
    §2.2 for the low-pass g (each A_j fed back into eq. (5))."""
    out = [np.asarray(x, dtype=np.float64)]
    for _ in range(levels):
        out.append(dwt_analysis_step(out[-1], g)[0])
    return out
