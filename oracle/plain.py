"""Plain top-k by definition, loaded from ``topk_oracle.cpp``.  TEST INFRASTRUCTURE.

Functions (each follows the passage cited in ``topk_oracle.cpp``):
  topk(x, k, largest, global_)        -- exact top-k, (value desc, index asc).
  topk_parallel(x, k, ...)            -- the same answer from all host cores (CPU baseline).
  count_at_or_above(x_row, pivot)     -- R for a threshold element (section 3).
  sample_order_stat(x_row, idx, t)    -- tau = t-th best sampled element.

Pinned by: brute-force rank-by-counting on tiny inputs, the bisection cutoff
identity, the composed stable one-bit split and the lower-bound compaction
identity (tests/test_oracle_pins.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle_topk.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C++ oracle into ``oracle/liboracle_topk.so`` (host code only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", _LIB + ".tmp"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_topk.argtypes = [vp, c_int, i64, i64, i64, c_int, c_int, vp, vp]
        lib.oracle_topk.restype = c_int
        lib.oracle_topk_parallel.argtypes = [vp, c_int, i64, i64, i64, c_int, c_int, c_int, vp, vp]
        lib.oracle_topk_parallel.restype = c_int
        lib.oracle_count_at_or_above.argtypes = [vp, c_int, i64, i64, c_int]
        lib.oracle_count_at_or_above.restype = i64
        lib.oracle_sample_order_stat.argtypes = [vp, c_int, vp, i64, i64, c_int]
        lib.oracle_sample_order_stat.restype = i64
        _lib = lib
    return _lib


def _dtype_code(x: np.ndarray) -> int:
    """0 for float32, 1 for bf16 carried as raw uint16 bits."""
    if x.dtype == np.float32:
        return 0
    if x.dtype == np.uint16:
        return 1
    raise TypeError("oracle takes float32 or bf16 bits as uint16, got %s" % x.dtype)


def topk(x: np.ndarray, k: int, largest: bool = True, global_: bool = False):
    """Exact top-k of each row of ``x`` (2-D), or of the flattened array if ``global_``.

    Returns (values, indices): values carry the input's own bits (same dtype as x),
    indices are int64 (row-local, or flat when ``global_``).  Shapes: (rows, k) or (k,).
    """
    x = np.ascontiguousarray(x)
    if x.ndim == 1:
        x = x[None, :]
    rows, n = x.shape
    code = _dtype_code(x)
    out_rows = 1 if global_ else rows
    vals = np.empty((out_rows, k), dtype=x.dtype)
    idx = np.empty((out_rows, k), dtype=np.int64)
    rc = _load().oracle_topk(x.ctypes.data, code, rows, n, k, int(bool(largest)), int(bool(global_)),
                             vals.ctypes.data, idx.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_topk rejected its arguments (k=%d, shape=%s)" % (k, x.shape))
    if global_:
        return vals[0], idx[0]
    return vals, idx


def topk_parallel(x: np.ndarray, k: int, largest: bool = True, global_: bool = False, threads: int = 0):
    """``topk`` computed by ``threads`` host threads (0 = every core): chunked
    nth_element and a merge.  A multi-threaded CPU baseline; checked against ``topk``."""
    x = np.ascontiguousarray(x)
    if x.ndim == 1:
        x = x[None, :]
    rows, n = x.shape
    threads = threads or os.cpu_count() or 1
    out_rows = 1 if global_ else rows
    vals = np.empty((out_rows, k), dtype=x.dtype)
    idx = np.empty((out_rows, k), dtype=np.int64)
    rc = _load().oracle_topk_parallel(x.ctypes.data, _dtype_code(x), rows, n, k, int(bool(largest)),
                                      int(bool(global_)), int(threads), vals.ctypes.data, idx.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_topk_parallel rejected its arguments (k=%d, shape=%s)" % (k, x.shape))
    if global_:
        return vals[0], idx[0]
    return vals, idx


def count_at_or_above(x_row: np.ndarray, pivot: int, largest: bool = True) -> int:
    """R = number of elements ranking at or above element ``pivot`` (itself included)."""
    x_row = np.ascontiguousarray(x_row).reshape(-1)
    return int(_load().oracle_count_at_or_above(x_row.ctypes.data, _dtype_code(x_row), x_row.size,
                                                int(pivot), int(bool(largest))))


def sample_order_stat(x_row: np.ndarray, idx: np.ndarray, t: int, largest: bool = True) -> int:
    """Index of the t-th best (1-based) sampled element, duplicates counted."""
    x_row = np.ascontiguousarray(x_row).reshape(-1)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    if not 1 <= t <= idx.size:
        raise ValueError("t out of range")
    return int(_load().oracle_sample_order_stat(x_row.ctypes.data, _dtype_code(x_row), idx.ctypes.data,
                                                idx.size, int(t), int(bool(largest))))
