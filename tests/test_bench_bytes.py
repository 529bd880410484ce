"""The bench's algorithmic byte counts (the numerators of every roofline
fraction it prints), written out term by term: the 4096-token layer (32
units, N_p = 4096, d = 128, bf16, G = 32, L = 4, k_L = 64, B = 512) and the
32-layer full denoising step."""

import bench
from wavelet_guided_sparse_gb300 import workloads as wl

U, N, D, E, G, L, KL, B = 32, 4096, 128, 2, 32, 4, 64, 512
P = N >> L


def test_workload_is_the_one_written_out():
    cfg = wl.CONFIGS["llada8b_layer"]
    assert (cfg.units_per_layer, cfg.n_prompt, cfg.head_dim, cfg.n_gen, cfg.levels) == (U, N, D, G, L)
    assert cfg.k_per_level()[L] == KL and cfg.budget == B and cfg.dtype == "bf16"


def test_layer_bytes_term_by_term():
    kp_stream = U * N * D * E                 # every prompt key once
    al = 2 * U * P * D * 4                    # A_L written and read back (fp32)
    span_rows = U * (KL << L) * D * E         # the coarse survivors' spans
    gathered = U * 2 * B * D * E              # selected keys and values
    small = U * (2 * G * D * E                # K_g, V_g
                 + G * D * E                  # Q
                 + G * D * 4                  # O written
                 + 4 * B)                     # selected token indices
    cfg = wl.CONFIGS["llada8b_layer"]
    assert bench.layer_bytes(cfg) == kp_stream + al + span_rows + gathered + small
    assert round(bench.layer_bytes(cfg) / 1e6, 2) == 60.10
    assert bench.stream_bytes(cfg) == kp_stream + al // 2


def test_full_step_bytes():
    cfg = wl.CONFIGS["full_step"]
    assert cfg.layers == 32 and cfg.k_per_level()[cfg.levels] == 128
    assert bench.tokens_per_step(cfg) == 32 * 65536
    assert round(bench.layer_bytes(cfg) * cfg.layers / 1e9, 1) == 22.6


def test_cache_init_bytes():
    # K and V of every position read once and written once, plus fp32 A_L.
    assert bench.cache_init_bytes(wl.CONFIGS["llada8b_layer"]) == (
        4 * U * (N + G) * D * E + U * P * D * 4) == 139_460_608


def test_gather_bytes_term_by_term():
    # The stand-alone gather + attention launch: the selected key and value
    # rows, K_g/V_g, Q, O and the indices; with the K_p stream it is the
    # "DWT + gather" figure.
    gathered = U * 2 * B * D * E
    small = U * (2 * G * D * E + G * D * E + G * D * 4 + 4 * B)
    cfg = wl.CONFIGS["llada8b_layer"]
    assert bench.path_bytes(cfg)["attn"] == gathered + small
    full = wl.CONFIGS["full_step"]
    assert bench.path_bytes(full)["attn"] == 68_943_872
    assert bench.stream_bytes(full) + bench.path_bytes(full)["attn"] == 622_592_000
