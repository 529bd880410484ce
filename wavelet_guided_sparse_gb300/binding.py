"""Thin Python binding of ``libwavefilter.so`` (the C ABI in ``include/wavefilter.h``).

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the path runs in the library's CUDA kernels.  If
the library has not been built, :func:`lib` raises; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libwavefilter.so")

WF_OK = 0
WF_BF16, WF_F32 = 0, 1
STATUS_NAMES = {0: "WF_OK", 1: "WF_ERR_NULL", 2: "WF_ERR_SHAPE", 3: "WF_ERR_UNSUPPORTED",
                4: "WF_ERR_WORKSPACE", 5: "WF_ERR_CUDA", 6: "WF_ERR_DEVICE_CHECK",
                7: "WF_ERR_ALIGNMENT"}
DEV_BAD_INDEX, DEV_DUP_INDEX, DEV_WAIT_TIMEOUT = 1, 2, 4
MAX_LEVELS = 12

# Every symbol the header declares (checked by the host tests).
EXPORTS = ("wf_status_string", "wf_last_error_string", "wf_default_k_per_level", "wf_workspace_bytes",
           "wf_step_launch_count", "wf_step_plan", "wf_debug_inject_wait_timeout",
           "wf_clear_device_status", "wf_read_device_status", "wf_dwt_lowpass",
           "wf_score_topk", "wf_recursive_filter", "wf_sparse_gather_attn", "wf_step",
           "wf_step_host", "wf_step_static_scratch", "wf_step_cached_al",
           "wf_cache_init", "wf_cache_update", "wf_cache_scatter", "wf_decode_step_host",
           "wf_daubechies_lowpass", "wf_basis_workspace_bytes", "wf_dwt_lowpass_basis",
           "wf_step_basis")


class WfError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


class Plan(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("final_gather", ctypes.c_int32), ("token_logits", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("filter_stages", ctypes.c_int32),
                ("attend_stages", ctypes.c_int32), ("stream_is_dwt_lowpass", ctypes.c_int32),
                ("al_stages", ctypes.c_int32)]


LOGITS_NAMES = {0: "shared", 1: "workspace", 2: "tensor_memory", 3: "recomputed"}


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("n_prompt", ctypes.c_int32), ("n_gen", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("levels", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_LIB = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i32p = ctypes.POINTER(ctypes.c_int32)
_sz = ctypes.c_size_t
_DIMSP = ctypes.POINTER(Dims)
_f64p = ctypes.POINTER(ctypes.c_double)

_SIGS = {
    "wf_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "wf_last_error_string": (ctypes.c_char_p, []),
    "wf_default_k_per_level": (ctypes.c_int, [_i32, _i32, _i32, _i32p]),
    "wf_workspace_bytes": (ctypes.c_int, [_DIMSP, _i32p, ctypes.POINTER(_sz)]),
    "wf_step_launch_count": (ctypes.c_int, [_DIMSP, _i32p, _i32p]),
    "wf_step_plan": (ctypes.c_int, [_DIMSP, _i32p, ctypes.POINTER(Plan)]),
    "wf_debug_inject_wait_timeout": (ctypes.c_int, [_i32]),
    "wf_clear_device_status": (ctypes.c_int, [_vp, _sz, _vp]),
    "wf_read_device_status": (ctypes.c_int, [_vp, _sz, _vp, _i32p]),
    "wf_dwt_lowpass": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _vp]),
    "wf_score_topk": (ctypes.c_int, [_DIMSP, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "wf_recursive_filter": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _i32p, _vp, _vp, _sz, _vp]),
    "wf_sparse_gather_attn": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                             _vp, _vp, _vp, _sz, _vp]),
    "wf_step": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _vp, _vp, _i32p, _vp, _vp, _vp,
                               _vp, _sz, _vp]),
    "wf_step_host": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _vp, _vp, _i32p, _vp, _vp,
                                    _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "wf_step_static_scratch": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _vp, _vp, _i32p, _vp,
                                              _vp, _vp, _vp]),
    "wf_step_cached_al": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _vp, _vp, _vp, _i32p, _vp, _vp,
                                         _vp, _vp, _sz, _vp]),
    "wf_cache_init": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "wf_cache_update": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _vp, _vp]),
    "wf_cache_scatter": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp,
                                        _vp, _sz, _vp]),
    "wf_decode_step_host": (ctypes.c_int, [_DIMSP, _vp, _vp, _vp, _i32p, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "wf_daubechies_lowpass": (ctypes.c_int, [_i32, _f64p]),
    "wf_basis_workspace_bytes": (ctypes.c_int, [_DIMSP, _i32, _i32p, ctypes.POINTER(_sz)]),
    "wf_dwt_lowpass_basis": (ctypes.c_int, [_DIMSP, _f64p, _i32, _vp, _vp, _vp]),
    "wf_step_basis": (ctypes.c_int, [_DIMSP, _f64p, _i32, _vp, _vp, _vp, _vp, _vp, _i32p, _vp,
                                     _vp, _vp, _vp, _sz, _vp]),
}


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it was not built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(fn: str, status: int) -> None:
    if status != WF_OK:
        err = WfError(fn, status)
        if status == 5:
            err.args = (f"{err.args[0]} ({lib().wf_last_error_string().decode()})",)
        raise err


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _k_array(k: Sequence[int]):
    arr = (ctypes.c_int32 * len(k))(*[int(x) for x in k])
    return arr


def dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return WF_BF16
    if dtype == torch.float32:
        return WF_F32
    raise ValueError(f"unsupported dtype {dtype}")


def make_dims(q: torch.Tensor, kp: torch.Tensor, levels: int) -> Dims:
    """Dims from Q [b, H, G, d] and Kp [b, H, N_p, d]."""
    if q.dim() != 4 or kp.dim() != 4:
        raise ValueError("Q and Kp must be [batch, heads, rows, head_dim]")
    b, h, g, d = q.shape
    if kp.shape[0] != b or kp.shape[1] != h or kp.shape[3] != d:
        raise ValueError("Q and Kp disagree on batch/heads/head_dim")
    return Dims(b, h, kp.shape[2], g, d, levels, dtype_code(kp.dtype))


def _require(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def default_k_per_level(n_prompt: int, levels: int, budget: int) -> list:
    out = (ctypes.c_int32 * (levels + 1))()
    _check("wf_default_k_per_level", lib().wf_default_k_per_level(n_prompt, levels, budget, out))
    return list(out)


def workspace_bytes(dims: Dims, k: Sequence[int]) -> int:
    n = ctypes.c_size_t(0)
    _check("wf_workspace_bytes", lib().wf_workspace_bytes(ctypes.byref(dims), _k_array(k),
                                                          ctypes.byref(n)))
    return n.value


def step_launch_count(dims: Dims, k: Sequence[int]) -> int:
    """Kernel launches one wf_step makes for these sizes (1 fused, else 2)."""
    n = ctypes.c_int32(0)
    _check("wf_step_launch_count", lib().wf_step_launch_count(ctypes.byref(dims), _k_array(k),
                                                              ctypes.byref(n)))
    return n.value


def step_plan(dims: Dims, k: Sequence[int]) -> dict:
    """wf_step's launch plan for these sizes (host only)."""
    p = Plan()
    _check("wf_step_plan", lib().wf_step_plan(ctypes.byref(dims), _k_array(k), ctypes.byref(p)))
    return {"launches": p.launches, "cluster": p.cluster, "final_gather": p.final_gather,
            "token_logits": LOGITS_NAMES.get(p.token_logits, p.token_logits),
            "smem_bytes": p.smem_bytes, "filter_stages": p.filter_stages,
            "attend_stages": p.attend_stages, "stream_is_dwt_lowpass": p.stream_is_dwt_lowpass, "al_stages": p.al_stages}


def inject_wait_timeout(polls: int) -> None:
    """Arms the one-shot wait-timeout injection of the next streaming launch
    (tests of the bounded device waits); 0 disarms."""
    _check("wf_debug_inject_wait_timeout", lib().wf_debug_inject_wait_timeout(int(polls)))


def alloc_workspace(dims: Dims, k: Sequence[int], device) -> torch.Tensor:
    ws = torch.empty(workspace_bytes(dims, k), dtype=torch.uint8, device=device)
    _check("wf_clear_device_status", lib().wf_clear_device_status(_ptr(ws), ws.numel(),
                                                                  _stream()))
    return ws


def alloc_status_workspace(device) -> torch.Tensor:
    """The smallest workspace (status word only): enough for wf_score_topk and
    wf_sparse_gather_attn."""
    return torch.zeros(256, dtype=torch.uint8, device=device)


def read_device_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("wf_read_device_status", lib().wf_read_device_status(_ptr(ws), ws.numel(),
                                                                _stream(stream),
                                                                ctypes.byref(out)))
    return out.value


def clear_device_status(ws: torch.Tensor, stream=None) -> None:
    _check("wf_clear_device_status", lib().wf_clear_device_status(_ptr(ws), ws.numel(),
                                                                  _stream(stream)))


def dwt_lowpass(kp: torch.Tensor, levels: int, all_levels: bool = False, stream=None):
    """A_L [b, H, N_p/2^L, d] fp32 (and, if ``all_levels``, a list of A_1..A_L)."""
    _require(kp, "Kp")
    b, h, n, d = kp.shape
    dims = Dims(b, h, n, 1, d, levels, dtype_code(kp.dtype))
    al = torch.empty((b, h, n >> levels, d), dtype=torch.float32, device=kp.device)
    a_all = None
    if all_levels:
        total = sum(b * h * (n >> j) * d for j in range(1, levels + 1))
        a_all = torch.empty(total, dtype=torch.float32, device=kp.device)
    _check("wf_dwt_lowpass", lib().wf_dwt_lowpass(ctypes.byref(dims), _ptr(kp), _ptr(al),
                                                  _ptr(a_all), _stream(stream)))
    if not all_levels:
        return al
    levels_out, off = [], 0
    for j in range(1, levels + 1):
        size = b * h * (n >> j) * d
        levels_out.append(a_all[off:off + size].view(b, h, n >> j, d))
        off += size
    return al, levels_out


def score_topk(q: torch.Tensor, al: torch.Tensor, n_prompt: int, levels: int, k_l: int,
               ws: torch.Tensor, return_scores: bool = False, stream=None):
    """Coarse Top-K: idx_L [b, H, k_L] int32 ascending (and scores [b, H, P])."""
    _require(q, "Q")
    _require(al, "A_L", torch.float32)
    b, h, g, d = q.shape
    dims = Dims(b, h, n_prompt, g, d, levels, dtype_code(q.dtype))
    idx = torch.empty((b, h, k_l), dtype=torch.int32, device=q.device)
    scores = (torch.empty((b, h, n_prompt >> levels), dtype=torch.float32, device=q.device)
              if return_scores else None)
    _check("wf_score_topk", lib().wf_score_topk(ctypes.byref(dims), _ptr(q), _ptr(al), k_l,
                                                _ptr(idx), _ptr(scores), _ptr(ws), ws.numel(),
                                                _stream(stream)))
    return (idx, scores) if return_scores else idx


def recursive_filter(q: torch.Tensor, kp: torch.Tensor, idx_l: torch.Tensor, levels: int,
                     k_per_level: Sequence[int], ws: torch.Tensor, stream=None):
    """Final token set S [b, H, B] int32 ascending."""
    _require(q, "Q")
    _require(kp, "Kp", q.dtype)
    _require(idx_l, "idx_L", torch.int32)
    dims = make_dims(q, kp, levels)
    b, h = q.shape[:2]
    idx = torch.empty((b, h, int(k_per_level[0])), dtype=torch.int32, device=q.device)
    _check("wf_recursive_filter", lib().wf_recursive_filter(
        ctypes.byref(dims), _ptr(q), _ptr(kp), _ptr(idx_l), _k_array(k_per_level), _ptr(idx),
        _ptr(ws), ws.numel(), _stream(stream)))
    return idx


def sparse_gather_attn(q, kp, vp, kg, vg, idx: Optional[torch.Tensor], levels: int,
                       ws: torch.Tensor, with_lse: bool = False, stream=None):
    """Eq. (3) over Kp/Vp[idx] ∪ Kg/Vg: O [b, H, G, d] fp32 (and lse [b, H, G])."""
    for t, n in ((q, "Q"), (kp, "Kp"), (vp, "Vp"), (kg, "Kg"), (vg, "Vg")):
        _require(t, n, q.dtype)
    budget = 0 if idx is None else idx.shape[-1]
    if idx is not None:
        _require(idx, "idx", torch.int32)
    dims = make_dims(q, kp, levels)
    o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device) if with_lse else None
    _check("wf_sparse_gather_attn", lib().wf_sparse_gather_attn(
        ctypes.byref(dims), _ptr(q), _ptr(kp), _ptr(vp), _ptr(kg), _ptr(vg), _ptr(idx),
        budget, _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return (o, lse) if with_lse else o


def step(q, kp, vp, kg, vg, levels: int, k_per_level: Sequence[int], ws: torch.Tensor,
         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
         idx_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The whole path (steps 1-5) for one layer; returns O [b, H, G, d] fp32."""
    for t, n in ((q, "Q"), (kp, "Kp"), (vp, "Vp"), (kg, "Kg"), (vg, "Vg")):
        _require(t, n, q.dtype)
    dims = make_dims(q, kp, levels)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check("wf_step", lib().wf_step(
        ctypes.byref(dims), _ptr(q), _ptr(kp), _ptr(vp), _ptr(kg), _ptr(vg),
        _k_array(k_per_level), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def step_cached_al(q, kp, vp, kg, vg, al, levels: int, k_per_level: Sequence[int],
                   ws: torch.Tensor, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, idx_out: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
    """Steps 2-5 with A_L [b, H, N_p/2^L, d] fp32 from an earlier dwt_lowpass
    (prompt keys unchanged); returns O [b, H, G, d] fp32."""
    for t, n in ((q, "Q"), (kp, "Kp"), (vp, "Vp"), (kg, "Kg"), (vg, "Vg")):
        _require(t, n, q.dtype)
    _require(al, "AL", torch.float32)
    dims = make_dims(q, kp, levels)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check("wf_step_cached_al", lib().wf_step_cached_al(
        ctypes.byref(dims), _ptr(q), _ptr(kp), _ptr(vp), _ptr(kg), _ptr(vg), _ptr(al),
        _k_array(k_per_level), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def step_host(dims: Dims, host: dict, k_per_level: Sequence[int], dev: dict, ws: torch.Tensor,
              stream=None) -> None:
    """wf_step_host: pinned host inputs/outputs in ``host`` (Q, Kp, Vp, Kg, Vg, O[, lse]),
    device staging buffers of the same names in ``dev``."""
    _check("wf_step_host", lib().wf_step_host(
        ctypes.byref(dims), _ptr(host["Q"]), _ptr(host["Kp"]), _ptr(host["Vp"]),
        _ptr(host["Kg"]), _ptr(host["Vg"]), _k_array(k_per_level), _ptr(host["O"]),
        _ptr(host.get("lse")), _ptr(dev["Q"]), _ptr(dev["Kp"]), _ptr(dev["Vp"]),
        _ptr(dev["Kg"]), _ptr(dev["Vg"]), _ptr(dev["O"]), _ptr(dev.get("lse")), _ptr(ws),
        ws.numel(), _stream(stream)))


def step_static_scratch(q, kp, vp, kg, vg, levels: int, k_per_level: Sequence[int],
                        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                        idx_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """wf_step_static_scratch: the whole path using the library's fixed device
    scratch array instead of a workspace (no device allocation inside the
    call).  Calls that overlap on the GPU share that array and race."""
    for t, n in ((q, "Q"), (kp, "Kp"), (vp, "Vp"), (kg, "Kg"), (vg, "Vg")):
        _require(t, n, q.dtype)
    dims = make_dims(q, kp, levels)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check("wf_step_static_scratch", lib().wf_step_static_scratch(
        ctypes.byref(dims), _ptr(q), _ptr(kp), _ptr(vp), _ptr(kg), _ptr(vg),
        _k_array(k_per_level), _ptr(out), _ptr(lse), _ptr(idx_out), _stream(stream)))
    return out


def cache_init(k: torch.Tensor, v: torch.Tensor, n_prompt: int, levels: int,
               with_al: bool = True, out: Optional[dict] = None, stream=None) -> dict:
    """Eq. (2) cache initialisation from token-major K, V [b, N_p + G, H, d]:
    returns {"Kp", "Vp": [b, H, N_p, d], "Kg", "Vg": [b, H, G, d]} and, if
    ``with_al``, "AL" [b, H, N_p/2^L, d] fp32.  ``out`` may supply the
    destination tensors (same keys)."""
    _require(k, "K")
    _require(v, "V", k.dtype)
    if k.dim() != 4 or v.shape != k.shape:
        raise ValueError("K and V must both be [batch, n_prompt + n_gen, heads, head_dim]")
    b, n, h, d = k.shape
    g = n - n_prompt
    dims = Dims(b, h, n_prompt, g, d, levels, dtype_code(k.dtype))
    o = dict(out or {})
    for name, rows in (("Kp", n_prompt), ("Vp", n_prompt), ("Kg", g), ("Vg", g)):
        if name not in o:
            o[name] = torch.empty((b, h, rows, d), dtype=k.dtype, device=k.device)
        _require(o[name], name, k.dtype)
    if with_al and "AL" not in o:
        o["AL"] = torch.empty((b, h, n_prompt >> levels, d), dtype=torch.float32,
                              device=k.device)
    _check("wf_cache_init", lib().wf_cache_init(
        ctypes.byref(dims), _ptr(k), _ptr(v), _ptr(o["Kp"]), _ptr(o["Vp"]), _ptr(o["Kg"]),
        _ptr(o["Vg"]), _ptr(o.get("AL")) if with_al else None, _stream(stream)))
    return o


def cache_update(k: torch.Tensor, v: torch.Tensor, kg: torch.Tensor, vg: torch.Tensor,
                 n_prompt: int, levels: int, stream=None) -> None:
    """Eq. (4) cache update: token-major K, V [b, G, H, d] into Kg, Vg [b, H, G, d]."""
    for t, name in ((k, "K"), (v, "V"), (kg, "Kg"), (vg, "Vg")):
        _require(t, name, k.dtype)
    b, g, h, d = k.shape
    dims = Dims(b, h, n_prompt, g, d, levels, dtype_code(k.dtype))
    _check("wf_cache_update", lib().wf_cache_update(ctypes.byref(dims), _ptr(k), _ptr(v),
                                                    _ptr(kg), _ptr(vg), _stream(stream)))


def cache_scatter(k: torch.Tensor, v: torch.Tensor, positions: torch.Tensor, cache: dict,
                  levels: int, ws: Optional[torch.Tensor] = None, stream=None) -> None:
    """wf_cache_scatter: token-major new rows K, V [b, M, H, d] at cache
    positions [b, M] (int32) into cache {"Kp", "Vp", "Kg", "Vg"[, "AL"]} in
    place (AL, if present, repaired at the touched coarse positions)."""
    for t, name in ((k, "K"), (v, "V")):
        _require(t, name)
    _require(positions, "positions", torch.int32)
    b, m, h, d = k.shape
    kp = cache["Kp"]
    dims = Dims(b, h, kp.shape[2], cache["Kg"].shape[2], d, levels, dtype_code(k.dtype))
    _check("wf_cache_scatter", lib().wf_cache_scatter(
        ctypes.byref(dims), _ptr(k), _ptr(v), _ptr(positions), m, _ptr(cache["Kp"]),
        _ptr(cache["Vp"]), _ptr(cache["Kg"]), _ptr(cache["Vg"]), _ptr(cache.get("AL")),
        _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def decode_step_host(dims: Dims, host: dict, k_per_level: Sequence[int], stage: dict,
                     cache: dict, ws: torch.Tensor, stream=None) -> None:
    """wf_decode_step_host: pinned host Q [b, H, G, d], new token-major K, V
    [b, G, H, d] and O out (keys Q, K, V, O of ``host``); device staging
    buffers of the same names in ``stage``; the resident cache (Kp, Vp, Kg, Vg,
    AL) in ``cache``, whose Kg/Vg receive the new rows."""
    _check("wf_decode_step_host", lib().wf_decode_step_host(
        ctypes.byref(dims), _ptr(host["Q"]), _ptr(host["K"]), _ptr(host["V"]),
        _k_array(k_per_level), _ptr(host["O"]), _ptr(stage["Q"]), _ptr(stage["K"]),
        _ptr(stage["V"]), _ptr(cache["Kp"]), _ptr(cache["Vp"]), _ptr(cache["Kg"]),
        _ptr(cache["Vg"]), _ptr(cache["AL"]), _ptr(stage["O"]), _ptr(ws), ws.numel(),
        _stream(stream)))


def daubechies_lowpass(n_moments: int) -> list:
    """Extremal-phase Daubechies low-pass filter (2 n_moments taps) from the library."""
    out = (ctypes.c_double * (2 * n_moments))()
    _check("wf_daubechies_lowpass", lib().wf_daubechies_lowpass(n_moments, out))
    return list(out)


def _taps(lowpass: Sequence[float]):
    return (ctypes.c_double * len(lowpass))(*[float(x) for x in lowpass]), len(lowpass)


def basis_workspace_bytes(dims: Dims, lowpass: Sequence[float], k: Sequence[int]) -> int:
    n = ctypes.c_size_t(0)
    _check("wf_basis_workspace_bytes", lib().wf_basis_workspace_bytes(
        ctypes.byref(dims), len(lowpass), _k_array(k), ctypes.byref(n)))
    return n.value


def dwt_lowpass_basis(kp: torch.Tensor, levels: int, lowpass: Sequence[float], stream=None):
    """Levels A_1..A_L [b, H, N_p/2^j, d] fp32 of the basis with low-pass ``lowpass``."""
    _require(kp, "Kp")
    b, h, n, d = kp.shape
    dims = Dims(b, h, n, 1, d, levels, dtype_code(kp.dtype))
    total = sum(b * h * (n >> j) * d for j in range(1, levels + 1))
    a_all = torch.empty(total, dtype=torch.float32, device=kp.device)
    taps, nt = _taps(lowpass)
    _check("wf_dwt_lowpass_basis", lib().wf_dwt_lowpass_basis(
        ctypes.byref(dims), taps, nt, _ptr(kp), _ptr(a_all), _stream(stream)))
    out, off = [], 0
    for j in range(1, levels + 1):
        size = b * h * (n >> j) * d
        out.append(a_all[off:off + size].view(b, h, n >> j, d))
        off += size
    return out


def step_basis(q, kp, vp, kg, vg, levels: int, k_per_level: Sequence[int],
               lowpass: Sequence[float], ws: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               idx_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The whole step with the orthonormal basis of low-pass ``lowpass``;
    returns O [b, H, G, d] fp32.  ``ws`` defaults to a fresh workspace."""
    for t, n in ((q, "Q"), (kp, "Kp"), (vp, "Vp"), (kg, "Kg"), (vg, "Vg")):
        _require(t, n, q.dtype)
    dims = make_dims(q, kp, levels)
    if ws is None:
        ws = torch.zeros(basis_workspace_bytes(dims, lowpass, k_per_level), dtype=torch.uint8,
                         device=q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    taps, nt = _taps(lowpass)
    _check("wf_step_basis", lib().wf_step_basis(
        ctypes.byref(dims), taps, nt, _ptr(q), _ptr(kp), _ptr(vp), _ptr(kg), _ptr(vg),
        _k_array(k_per_level), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def raw_call(name: str, *args) -> int:
    """Calls an entry point with raw ctypes arguments and returns its status
    (used by the host-side validation tests)."""
    return getattr(lib(), name)(*args)
