"""GPU parity of the KV-cache writes around the filtering path, through the C
ABI: the first-step initialisation of WaveFilter §2.1 eq. (2) with A_L of the
prompt keys (§3.1), and the generation-row update of eq. (4).

Bars: every cache row bit-exact (the operation is a copy); A_L within 1e-3
relative of the float64 oracle and bit-identical to wf_dwt_lowpass of the
written prompt keys (the same summation order); the step that then reads the
cache (wf_step_cached_al with this A_L) meets the whole-step contract.
Inputs are rounded to the device type on the host, so the oracle sees the
values the GPU sees.
"""

import numpy as np
import pytest
import torch

import oracle.wavefilter_oracle as wo
from gpu_common import AL_RTOL, compare_step_unit, run_step, to_device, torch_dtype
from wavelet_guided_sparse_gb300 import binding as bd
from wavelet_guided_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _rounder(dtype):
    return wl.round_to_bf16 if dtype == "bf16" else (lambda x: x.astype(np.float32))


def _token_major(arrs):
    """[b, H, rows, d] prompt and generation arrays -> token-major K, V
    [b, N_p + G, H, d] (the projections' output layout)."""
    k = np.concatenate([arrs["Kp"], arrs["Kg"]], axis=2).transpose(0, 2, 1, 3)
    v = np.concatenate([arrs["Vp"], arrs["Vg"]], axis=2).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(k), np.ascontiguousarray(v)


def _al_close(got, ref):
    tol = AL_RTOL * np.abs(ref) + 1e-6 * np.sqrt((ref ** 2).mean())
    return (np.abs(got - ref) <= tol).all()


def _check_init(k, v, n_prompt, levels, dtype):
    """Runs wf_cache_init on host-rounded K, V and compares every output."""
    dt = torch_dtype(dtype)
    kd = torch.from_numpy(k).to("cuda", dt)
    vd = torch.from_numpy(v).to("cuda", dt)
    out = bd.cache_init(kd, vd, n_prompt, levels)
    al_dwt = bd.dwt_lowpass(out["Kp"], levels)
    torch.cuda.synchronize()
    assert torch.equal(out["AL"], al_dwt), "A_L differs from wf_dwt_lowpass"
    got = {n: out[n].cpu().double().numpy() for n in ("Kp", "Vp", "Kg", "Vg", "AL")}
    b, _, h, _ = k.shape
    for bi in range(b):
        ref = wo.cache_init(k[bi], v[bi], n_prompt, levels)
        for n in ("Kp", "Vp", "Kg", "Vg"):
            np.testing.assert_array_equal(got[n][bi], ref[n], err_msg=f"{n} sequence {bi}")
        for hi in range(h):
            assert _al_close(got["AL"][bi, hi], ref["a_l"][hi]), (bi, hi)
    return out


@pytest.mark.parametrize("b,h,n_prompt,g,d,levels,dtype", [
    (2, 3, 128, 7, 128, 4, "bf16"),    # ragged G, two sequences
    (1, 2, 256, 33, 64, 5, "f32"),     # d = 64 fp32, 32-row spans
    (2, 2, 64, 1, 64, 1, "bf16"),      # one generation row, pairs
    (1, 2, 3 * 128, 5, 64, 7, "bf16"), # 128-row spans (eight 16-row blocks)
    (1, 1, 4096, 64, 128, 12, "f32"),  # one span of 4096 rows, G at its maximum
])
def test_cache_init_shapes(b, h, n_prompt, g, d, levels, dtype):
    rng = np.random.default_rng(n_prompt * 7 + g)
    rnd = _rounder(dtype)
    k = rnd(rng.standard_normal((b, n_prompt + g, h, d)) * 1.5)
    v = rnd(rng.standard_normal((b, n_prompt + g, h, d)))
    _check_init(k, v, n_prompt, levels, dtype)


@pytest.mark.parametrize("name", ["tiny", "llada8b_layer"])
def test_cache_init_workload_then_step(name):
    # The full layer of the workload: initialise the cache from token-major
    # K/V, then run steps 2-5 on it with the A_L the initialisation wrote;
    # every unit is held to the whole-step contract against the oracle.
    cfg = wl.CONFIGS[name]
    ks = cfg.k_per_level()
    arrs = wl.generate_layer(cfg, 0)
    arrs = {n: _rounder(cfg.dtype)(a) for n, a in arrs.items()}
    k, v = _token_major(arrs)
    out = _check_init(k, v, cfg.n_prompt, cfg.levels, cfg.dtype)
    q = to_device({"Q": arrs["Q"]}, cfg.dtype)["Q"]
    dev = {"Q": q, "Kp": out["Kp"], "Vp": out["Vp"], "Kg": out["Kg"], "Vg": out["Vg"]}
    o, lse, idx, status = run_step(dev, cfg.levels, ks, al=out["AL"])
    assert status == 0
    o, lse, idx = o.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()
    kinds = [compare_step_unit(arrs, 0, hi, cfg.levels, ks, idx[0, hi], o[0, hi], lse[0, hi])
             for hi in range(cfg.heads)]
    assert kinds.count("exact") >= len(kinds) // 2


def test_cache_init_without_al_writes_the_same_cache():
    rng = np.random.default_rng(5)
    k = wl.round_to_bf16(rng.standard_normal((1, 136, 4, 128)))
    v = wl.round_to_bf16(rng.standard_normal((1, 136, 4, 128)))
    kd, vd = (torch.from_numpy(x).to("cuda", torch.bfloat16) for x in (k, v))
    a = bd.cache_init(kd, vd, 128, 3)
    b = bd.cache_init(kd, vd, 128, 3, with_al=False)
    torch.cuda.synchronize()
    assert "AL" not in b
    for n in ("Kp", "Vp", "Kg", "Vg"):
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("g,d,dtype", [(32, 128, "bf16"), (5, 64, "f32"), (64, 64, "bf16")])
def test_cache_update_then_step(g, d, dtype):
    # Eq. (4): new generation keys/values replace the cached ones; the prompt
    # rows and A_L are untouched, and the next step attends over the new rows.
    b, h, n_prompt, levels = 1, 3, 512, 3
    rng = np.random.default_rng(g * 31 + d)
    rnd = _rounder(dtype)
    arrs = {"Q": rnd(rng.standard_normal((b, h, g, d)) * 1.5),
            "Kp": rnd(rng.standard_normal((b, h, n_prompt, d)) * 1.5),
            "Vp": rnd(rng.standard_normal((b, h, n_prompt, d))),
            "Kg": rnd(rng.standard_normal((b, h, g, d)) * 1.5),
            "Vg": rnd(rng.standard_normal((b, h, g, d)))}
    k_new = rnd(rng.standard_normal((b, g, h, d)) * 1.5)
    v_new = rnd(rng.standard_normal((b, g, h, d)))
    dev = to_device(arrs, dtype)
    al = bd.dwt_lowpass(dev["Kp"], levels)
    kp_before = dev["Kp"].clone()
    dt = torch_dtype(dtype)
    bd.cache_update(torch.from_numpy(k_new).to("cuda", dt), torch.from_numpy(v_new).to("cuda", dt),
                    dev["Kg"], dev["Vg"], n_prompt, levels)
    torch.cuda.synchronize()
    ref = wo.cache_update(k_new[0], v_new[0])
    np.testing.assert_array_equal(dev["Kg"][0].cpu().double().numpy(), ref["Kg"])
    np.testing.assert_array_equal(dev["Vg"][0].cpu().double().numpy(), ref["Vg"])
    assert torch.equal(dev["Kp"], kp_before)
    ks = bd.default_k_per_level(n_prompt, levels, 64)
    o, lse, idx, status = run_step(dev, levels, ks, al=al)
    assert status == 0
    updated = dict(arrs, Kg=ref["Kg"][None], Vg=ref["Vg"][None])
    o, lse, idx = o.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()
    for hi in range(h):
        compare_step_unit(updated, 0, hi, levels, ks, idx[0, hi], o[0, hi], lse[0, hi])


@pytest.mark.parametrize("packed", [False, True])
def test_decode_step_host_matches_device_path(packed):
    # The host-buffer serving step (copies, eq. (4) update, cached step, copy
    # back) on the 4096-token layer: the same O as the device-only calls, bit
    # for bit, and every unit within the step contract for the updated cache.
    cfg = wl.CONFIGS["llada8b_layer"]
    ks = cfg.k_per_level()
    arrs = {n: wl.round_to_bf16(a) for n, a in wl.generate_layer(cfg, 0).items()}
    rng = np.random.default_rng(77)
    b, h, g, d = arrs["Q"].shape
    k_new = wl.round_to_bf16(rng.standard_normal((b, g, h, d)) * 1.5)
    v_new = wl.round_to_bf16(rng.standard_normal((b, g, h, d)))
    k, v = _token_major(arrs)
    kd, vd = (torch.from_numpy(x).to("cuda", torch.bfloat16) for x in (k, v))
    caches = [bd.cache_init(kd, vd, cfg.n_prompt, cfg.levels) for _ in range(2)]
    dims = bd.Dims(b, h, cfg.n_prompt, g, d, cfg.levels, bd.WF_BF16)
    ws = bd.alloc_workspace(dims, ks, kd.device)
    # Device-only path on cache 0.
    q_dev = torch.from_numpy(arrs["Q"]).to("cuda", torch.bfloat16)
    kn_dev = torch.from_numpy(k_new).to("cuda", torch.bfloat16)
    vn_dev = torch.from_numpy(v_new).to("cuda", torch.bfloat16)
    c0 = caches[0]
    bd.cache_update(kn_dev, vn_dev, c0["Kg"], c0["Vg"], cfg.n_prompt, cfg.levels)
    ref = bd.step_cached_al(q_dev, c0["Kp"], c0["Vp"], c0["Kg"], c0["Vg"], c0["AL"], cfg.levels,
                            ks, ws)
    # Host-buffer path on cache 1.
    if packed:  # Q, K, V back to back on both sides: one host-to-device copy
        n_el = q_dev.numel()
        h_pack = torch.empty(3 * n_el, dtype=torch.bfloat16).pin_memory()
        d_pack = torch.empty(3 * n_el, dtype=torch.bfloat16, device="cuda")
        host, stage = {}, {}
        for i, (name, t) in enumerate((("Q", q_dev), ("K", kn_dev), ("V", vn_dev))):
            host[name] = h_pack[i * n_el:(i + 1) * n_el].view(t.shape)
            host[name].copy_(t.cpu())
            stage[name] = d_pack[i * n_el:(i + 1) * n_el].view(t.shape)
    else:
        host = {"Q": q_dev.cpu().pin_memory(), "K": kn_dev.cpu().pin_memory(),
                "V": vn_dev.cpu().pin_memory()}
        stage = {"Q": torch.empty_like(q_dev), "K": torch.empty_like(kn_dev),
                 "V": torch.empty_like(vn_dev)}
    host["O"] = torch.empty((b, h, g, d), dtype=torch.float32).pin_memory()
    stage["O"] = torch.empty_like(ref)
    bd.decode_step_host(dims, host, ks, stage, caches[1], ws)
    torch.cuda.synchronize()
    assert bd.read_device_status(ws) == 0
    assert torch.equal(host["O"], ref.cpu())
    assert torch.equal(caches[1]["Kg"], c0["Kg"]) and torch.equal(caches[1]["Vg"], c0["Vg"])
    upd = wo.cache_update(k_new[0], v_new[0])
    updated = dict(arrs, Kg=upd["Kg"][None], Vg=upd["Vg"][None])
    o = host["O"].numpy()
    idx = torch.empty((b, h, ks[0]), dtype=torch.int32, device="cuda")
    bd.step_cached_al(q_dev, c0["Kp"], c0["Vp"], c0["Kg"], c0["Vg"], c0["AL"], cfg.levels, ks,
                      ws, idx_out=idx)
    idx = idx.cpu().numpy()
    kinds = [compare_step_unit(updated, 0, hi, cfg.levels, ks, idx[0, hi], o[0, hi])
             for hi in range(h)]
    assert kinds.count("exact") >= len(kinds) // 2


def test_cache_init_batched_long_sampled():
    # The largest workload's full launch shape (2 sequences x 32 heads x
    # 131072 + 64 positions, L = 7): token-major K/V of 2.15 GB each, so source
    # and cache byte offsets pass 2^31.  The first and last head of the last
    # sequence carry the workload's generated units and are checked against
    # the oracle; every other head is zero and must stay zero.
    cfg = wl.CONFIGS["batched_long_1pct"]
    b, h, n_p, g, d = cfg.batch, cfg.heads, cfg.n_prompt, cfg.n_gen, cfg.head_dim
    k = torch.zeros((b, n_p + g, h, d), dtype=torch.bfloat16)
    v = torch.zeros((b, n_p + g, h, d), dtype=torch.bfloat16)
    seq, heads = b - 1, (0, h - 1)
    units = {}
    for hi in heads:
        u = wl.generate_unit(cfg, seq, 0, hi)
        units[hi] = (np.concatenate([u["Kp"], u["Kg"]]), np.concatenate([u["Vp"], u["Vg"]]))
        k[seq, :, hi] = torch.from_numpy(units[hi][0]).to(torch.bfloat16)
        v[seq, :, hi] = torch.from_numpy(units[hi][1]).to(torch.bfloat16)
    out = bd.cache_init(k.cuda(), v.cuda(), n_p, cfg.levels)
    del k, v
    torch.cuda.synchronize()
    for hi in heads:
        ku, vu = units[hi]
        ref = wo.cache_init(ku[:, None], vu[:, None], n_p, cfg.levels)
        for n in ("Kp", "Vp", "Kg", "Vg"):
            np.testing.assert_array_equal(out[n][seq, hi].cpu().double().numpy(), ref[n][0],
                                          err_msg=f"{n} head {hi}")
        assert _al_close(out["AL"][seq, hi].cpu().double().numpy(), ref["a_l"][0]), hi
    mask = torch.ones((b, h), dtype=torch.bool)
    for hi in heads:
        mask[seq, hi] = False
    for n in ("Kp", "Vp", "Kg", "Vg", "AL"):
        assert int(torch.count_nonzero(out[n][mask.cuda()])) == 0, n


# ------------------------------------------ eq. (4) over an arbitrary set

def _scatter_positions(rng, b, n_prompt, n_gen, m, with_bad=False):
    """Distinct positions per sequence mixing prompt and generation rows
    (several in one coarse span); optionally one out-of-range entry."""
    pool = np.setdiff1d(np.arange(n_prompt + n_gen), [5, 6])
    # 5 and 6 share a coarse span for every L >= 2
    pos = np.stack([np.r_[5, 6, rng.choice(pool, size=m - 2, replace=False)] for _ in range(b)])
    if with_bad:
        pos[0, -1] = n_prompt + n_gen + 3
    return pos.astype(np.int32)


@pytest.mark.parametrize("name,m", [("tiny", 24), ("llada8b_layer", 48)])
def test_cache_scatter_matches_oracle_and_repairs_al(name, m):
    # Rows bit-exact against the oracle's eq. (4); the repaired A_L equals a
    # fresh wf_dwt_lowpass of the updated prompt keys bit for bit (and the
    # oracle's repair within 1e-3); the cached-A_L step on the updated cache
    # then meets the whole-step contract on every unit.
    cfg = wl.CONFIGS[name]
    ks = cfg.k_per_level()
    rnd = _rounder(cfg.dtype)
    arrs = {k: rnd(v) for k, v in wl.generate_layer(cfg).items()}
    dev = to_device(arrs, cfg.dtype)
    al = bd.dwt_lowpass(dev["Kp"], cfg.levels)
    rng = np.random.default_rng(m)
    b, h, d = cfg.batch, cfg.heads, cfg.head_dim
    pos = _scatter_positions(rng, b, cfg.n_prompt, cfg.n_gen, m)
    nk = rnd(rng.standard_normal((b, m, h, d)) * 1.5)
    nv = rnd(rng.standard_normal((b, m, h, d)))
    cache = {"Kp": dev["Kp"], "Vp": dev["Vp"], "Kg": dev["Kg"], "Vg": dev["Vg"], "AL": al}
    dt = torch_dtype(cfg.dtype)
    ws = bd.alloc_status_workspace("cuda")
    bd.cache_scatter(torch.from_numpy(nk).to("cuda", dt), torch.from_numpy(nv).to("cuda", dt),
                     torch.from_numpy(pos).cuda(), cache, cfg.levels, ws=ws)
    assert bd.read_device_status(ws) == 0
    assert torch.equal(al, bd.dwt_lowpass(dev["Kp"], cfg.levels)), "repair differs from a fresh DWT"
    got = {n: cache[n].cpu().double().numpy() for n in ("Kp", "Vp", "Kg", "Vg", "AL")}
    new = {}
    for bi in range(b):
        ref = wo.cache_scatter(arrs["Kp"][bi], arrs["Vp"][bi], arrs["Kg"][bi], arrs["Vg"][bi],
                               nk[bi], nv[bi], pos[bi])
        for n in ("Kp", "Vp", "Kg", "Vg"):
            np.testing.assert_array_equal(got[n][bi], ref[n], err_msg=f"{n} sequence {bi}")
            new.setdefault(n, []).append(ref[n])
        a0 = np.stack([wo.haar_pyramid(arrs["Kp"][bi, hi], cfg.levels)[cfg.levels]
                       for hi in range(h)])
        rep = wo.al_repair(a0, ref["Kp"], pos[bi], cfg.levels)
        for hi in range(h):
            assert _al_close(got["AL"][bi, hi], rep[hi]), (bi, hi)
    upd = {n: np.stack(v).astype(np.float32) for n, v in new.items()}
    upd["Q"] = arrs["Q"]
    out, lse, idx, status = run_step(dev, cfg.levels, ks, al=al)
    assert status == 0
    out, lse, idx = out.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()
    for bi in range(b):
        for hi in range(h):
            compare_step_unit(upd, bi, hi, cfg.levels, ks, idx[bi, hi], out[bi, hi], lse[bi, hi])


def test_cache_scatter_skips_and_flags_bad_positions():
    cfg = wl.CONFIGS["tiny"]
    arrs = {k: v.astype(np.float32) for k, v in wl.generate_layer(cfg).items()}
    dev = to_device(arrs, cfg.dtype)
    before = {n: dev[n].clone() for n in ("Kp", "Vp", "Kg", "Vg")}
    rng = np.random.default_rng(3)
    pos = _scatter_positions(rng, 1, cfg.n_prompt, cfg.n_gen, 4, with_bad=True)
    nk = rng.standard_normal((1, 4, cfg.heads, cfg.head_dim)).astype(np.float32)
    ws = bd.alloc_status_workspace("cuda")
    cache = {n: dev[n] for n in ("Kp", "Vp", "Kg", "Vg")}
    bd.cache_scatter(torch.from_numpy(nk).cuda(), torch.from_numpy(nk).cuda(),
                     torch.from_numpy(pos).cuda(), cache, cfg.levels, ws=ws)
    assert bd.read_device_status(ws) & bd.DEV_BAD_INDEX
    ref = wo.cache_scatter(arrs["Kp"][0], arrs["Vp"][0], arrs["Kg"][0], arrs["Vg"][0],
                           nk[0, :3], nk[0, :3], pos[0, :3])
    for n in ("Kp", "Vp", "Kg", "Vg"):
        np.testing.assert_array_equal(cache[n][0].cpu().double().numpy(), ref[n])
    assert not torch.equal(cache["Kp"], before["Kp"])
