"""Prof-K top-k selection on GB300: Python binding of libtopk_gb300.so.

Every step of the selection runs in the library's CUDA kernels; this module
only checks tensors, allocates outputs with torch and passes pointers and the
current CUDA stream across the C ABI (include/topk.h).  There is no CPU path:
inputs must be CUDA tensors and the library must be built.

    import top_selection_prof_gb300 as tk
    vals, idx = tk.select(x, k)                  # per row, x: (rows, n) or (n,)
    vals, idx = tk.select_global(acts, K)        # BatchTopK: over the flattened tensor
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (PATH_NAMES, TOPK_BF16, TOPK_F32, TOPK_PATH_AUTO, TOPK_PATH_DIRECT, TOPK_PATH_EXACT,
                   TOPK_PATH_PROFK, TOPK_RULE_ALG1, TOPK_RULE_EXACT, TopkError)

__all__ = ["select", "select_global", "select_ex", "plan", "prof_sample", "prof_filter", "index_bits",
           "options", "TopkError", "TOPK_PATH_AUTO", "TOPK_PATH_DIRECT", "TOPK_PATH_PROFK", "TOPK_PATH_EXACT",
           "TOPK_RULE_EXACT", "TOPK_RULE_ALG1"]


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return TOPK_F32
    if t.dtype == torch.bfloat16:
        return TOPK_BF16
    raise TypeError("top-k takes float32 or bfloat16 tensors, got %s" % t.dtype)


def _check_input(x):
    torch = _torch()
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise TypeError("input must be a CUDA tensor (the engine has no CPU path)")
    if x.dim() not in (1, 2):
        raise ValueError("input must be 1-D (n,) or 2-D (rows, n)")
    if not x.is_contiguous():
        raise ValueError("input must be contiguous")
    return x if x.dim() == 2 else x.view(1, -1)


def _stream_ptr(x, stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    return ctypes.c_void_p(s.cuda_stream)


def options(**kw) -> _lib.TopkOptions:
    """A TopkOptions struct with library defaults, overridden by keyword arguments."""
    opt = _lib.TopkOptions()
    _lib.get().topk_options_init(ctypes.byref(opt))
    for key, val in kw.items():
        if not hasattr(opt, key):
            raise KeyError("unknown option %r" % key)
        setattr(opt, key, val)
    return opt


def _stats_dict(st: _lib.TopkStats) -> dict:
    d = {name: getattr(st, name) for name, _ in st._fields_}
    d["path_name"] = PATH_NAMES.get(st.path, "?")
    return d


def _run(x, k, largest, eps, global_, opt, want_stats, stream):
    torch = _torch()
    x2 = _check_input(x)
    rows, n = x2.shape
    code = _dtype_code(x2)
    out_shape = (k,) if global_ else (rows, k)
    with torch.cuda.device(x2.device):
        vals = torch.empty(out_shape, dtype=x2.dtype, device=x2.device)
        idx = torch.empty(out_shape, dtype=torch.int64, device=x2.device)
        st = _lib.TopkStats() if want_stats else None
        lib = _lib.get()
        sp = _stream_ptr(x2, stream)
        if opt is None and st is None:
            fn = lib.topk_select_global if global_ else lib.topk_select
            rc = fn(x2.data_ptr(), code, rows, n, int(k), int(bool(largest)), float(eps), vals.data_ptr(),
                    idx.data_ptr(), sp)
        else:
            rc = lib.topk_select_ex(x2.data_ptr(), code, rows, n, int(k), int(bool(largest)), float(eps),
                                    vals.data_ptr(), idx.data_ptr(), sp, int(bool(global_)),
                                    ctypes.byref(opt) if opt is not None else None,
                                    ctypes.byref(st) if st is not None else None)
    _lib.check(rc, "topk_select_global" if global_ else "topk_select")
    if x.dim() == 1 and not global_:
        vals, idx = vals[0], idx[0]
    return vals, idx, (_stats_dict(st) if st is not None else None)


def select(x, k: int, largest: bool = True, eps: float = 1e-3, stream=None):
    """Top-k of each row: (values, indices), sorted by (value desc, index asc)."""
    v, i, _ = _run(x, k, largest, eps, False, None, False, stream)
    return v, i


def select_global(x, k: int, largest: bool = True, eps: float = 1e-3, stream=None):
    """Top-k over the whole flattened tensor (BatchTopK): (values[k], flat indices[k])."""
    v, i, _ = _run(x, k, largest, eps, True, None, False, stream)
    return v, i


def select_ex(x, k: int, largest: bool = True, eps: float = 1e-3, global_: bool = False, stats: bool = True,
              stream=None, **opts):
    """select / select_global with library options; returns (values, indices, stats dict or None).

    Requesting stats synchronises the stream."""
    opt = options(**opts) if opts else None
    return _run(x, k, largest, eps, global_, opt, stats, stream)


def plan(n: int, k: int, eps: float = 1e-3, **opts) -> dict:
    """Host-only: the path and (S, t, M) the engine would use for one selection of k out of n."""
    p = _lib.TopkPlan()
    opt = options(**opts) if opts else None
    rc = _lib.get().topk_plan(int(n), int(k), float(eps), ctypes.byref(opt) if opt is not None else None,
                              ctypes.byref(p))
    _lib.check(rc, "topk_plan")
    d = {name: getattr(p, name) for name, _ in p._fields_}
    d["path_name"] = PATH_NAMES.get(p.path, "?")
    return d


def index_bits(length: int) -> int:
    """b of the composite key format for a selection over `length` elements."""
    return int(_lib.get().topk_index_bits(int(length)))


def prof_sample(x, S: int, seed: int, counter: int, global_: bool = False, largest: bool = True, stream=None):
    """Stage 1: composite keys of the S sampled elements per selection, as an int64 tensor of raw bits."""
    torch = _torch()
    x2 = _check_input(x)
    rows, n = x2.shape
    nsel = 1 if global_ else rows
    with torch.cuda.device(x2.device):
        keys = torch.empty((nsel, S), dtype=torch.int64, device=x2.device)
        rc = _lib.get().topk_prof_sample(x2.data_ptr(), _dtype_code(x2), rows, n, int(bool(global_)),
                                         int(bool(largest)), int(S), int(seed), int(counter), keys.data_ptr(),
                                         _stream_ptr(x2, stream))
    _lib.check(rc, "topk_prof_sample")
    return keys


def prof_filter(x, tau, M: int, global_: bool = False, largest: bool = True, stream=None):
    """Stage 3: (buffer[nsel, M] of composite keys as int64 bits, counts[nsel]) for thresholds tau[nsel]."""
    torch = _torch()
    x2 = _check_input(x)
    rows, n = x2.shape
    nsel = 1 if global_ else rows
    tau = tau.to(device=x2.device, dtype=torch.int64).contiguous()
    if tau.numel() != nsel:
        raise ValueError("tau needs one key per selection")
    with torch.cuda.device(x2.device):
        buf = torch.zeros((nsel, M), dtype=torch.int64, device=x2.device)
        counts = torch.empty((nsel,), dtype=torch.int64, device=x2.device)
        rc = _lib.get().topk_prof_filter(x2.data_ptr(), _dtype_code(x2), rows, n, int(bool(global_)),
                                         int(bool(largest)), tau.data_ptr(), int(M), buf.data_ptr(),
                                         counts.data_ptr(), _stream_ptr(x2, stream))
    _lib.check(rc, "topk_prof_filter")
    return buf, counts
