"""The bench's algorithmic byte counts (the numerators of every roofline
fraction it prints), written out term by term for the 4096-token layer:
32 units, N_p = 4096, d = 128, bf16, G = 32, L = 4, k_L = 64, B = 512."""

import bench
from wavelet_guided_sparse_gb300 import workloads as wl

U, N, D, E, G, L, KL, B = 32, 4096, 128, 2, 32, 4, 64, 512
P = N >> L


def test_workload_is_the_one_written_out():
    cfg = wl.CONFIGS["llada8b_layer"]
    assert (cfg.units_per_layer, cfg.n_prompt, cfg.head_dim, cfg.n_gen, cfg.levels) == (U, N, D, G, L)
    assert cfg.k_per_level()[L] == KL and cfg.budget == B and cfg.dtype == "bf16"


def test_single_launch_step_bytes():
    kp_stream = U * N * D * E                 # every prompt key once
    span_rows = U * (KL << L) * D * E         # the coarse survivors' spans
    gathered = U * 2 * B * D * E              # selected keys and values
    small = U * (3 * G * D * E                # Q, read by scoring, filtering, attention
                 + 2 * G * D * E              # K_g, V_g
                 + G * D * 4                  # O written
                 + (KL + KL + B + B) * 4)     # survivor and token index lists
    assert bench.step_bytes(wl.CONFIGS["llada8b_layer"], fused=True) == (
        kp_stream + span_rows + gathered + small)
    # Two launches: A_L written by the stream and read back by the scoring.
    assert bench.step_bytes(wl.CONFIGS["llada8b_layer"], fused=False) == (
        kp_stream + span_rows + gathered + small + 2 * U * P * D * 4)


def test_cache_init_bytes():
    # K and V of every position read once and written once, plus fp32 A_L.
    assert bench.cache_init_bytes(wl.CONFIGS["llada8b_layer"]) == (
        4 * U * (N + G) * D * E + U * P * D * 4) == 139_460_608
