"""Seeded synthetic inputs shaped like the Prof-K paper's workloads.

This module only draws input arrays; it holds none of the selection method's
arithmetic, so that the CUDA path and the CPU oracle can both be fed the same
bytes.  All generators use ``numpy.random.default_rng(seed)``.

Distributions (the paper's synthetic benchmarks use Uniform, Standard Normal
and heavy-tailed Pareto inputs, section 5 "Experimental Setup"; the
BatchTopK application flattens post-ReLU activations of shape B x d_dict,
section 5 "Application: BatchTopK Sparse Autoencoders"; the GPU.js top-k
exercise ranks 65,536 integer-valued scores, "Find the Cutoff Instead"):

  int20            float32(uniform integers in [0, 2^20))
  normal           float32 standard normal
  pareto15         s * U^(-1/1.5), U uniform in (0, 1], s = +-1 (x_m = 1)
  ties1000         float32(uniform integers in [0, 1000))   (massive ties)
  ties1000_sorted  the same values sorted ascending
  relu_normal_bf16 bf16 (round-to-nearest-even) of max(N(0,1), 0), as uint16 bits
  uniform          float32 uniform in [0, 1)
  constant         every element 1.0
  specials         normals with NaN, +-inf, +-0 sprinkled in

bf16 arrays are returned as their raw uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

# The benchmark workloads: (kind, rows, n, k, mode, eps).  mode "row" selects
# per row; "global" selects over the flattened rows*n vector.
WORKLOADS = {
    "single_row_65536_int20_k10": dict(kind="int20", rows=1, n=65536, k=10, mode="row", eps=1e-3),
    "rows1024x32768_normal_k64": dict(kind="normal", rows=1024, n=32768, k=64, mode="row", eps=1e-3),
    "single_row_2p28_pareto15_k1024": dict(kind="pareto15", rows=1, n=1 << 28, k=1024, mode="row",
                                           eps=1e-6),
    "single_row_2p26_ties1000_k10000": dict(kind="ties1000", rows=1, n=1 << 26, k=10000, mode="row",
                                            eps=1e-3),
    "single_row_2p26_ties1000_sorted_k10000": dict(kind="ties1000_sorted", rows=1, n=1 << 26, k=10000,
                                                   mode="row", eps=1e-3),
    "batchtopk_4096x65536_relu_bf16_k131072": dict(kind="relu_normal_bf16", rows=4096, n=65536,
                                                   k=131072, mode="global", eps=1e-3),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def make(kind: str, rows: int, n: int, seed: int) -> np.ndarray:
    """A (rows, n) input array of the given kind, deterministic in ``seed``."""
    rng = np.random.default_rng(seed)
    size = rows * n
    if kind == "int20":
        a = rng.integers(0, 1 << 20, size=size).astype(np.float32)
    elif kind == "normal":
        a = rng.standard_normal(size, dtype=np.float32)
    elif kind == "uniform":
        a = rng.random(size, dtype=np.float32)
    elif kind == "pareto15":
        u = 1.0 - rng.random(size)                       # (0, 1]
        sign = np.where(rng.integers(0, 2, size=size) == 1, 1.0, -1.0)
        a = (sign * u ** (-1.0 / 1.5)).astype(np.float32)
    elif kind == "ties1000":
        a = rng.integers(0, 1000, size=size).astype(np.float32)
    elif kind == "ties1000_sorted":
        a = np.sort(rng.integers(0, 1000, size=size)).astype(np.float32)
    elif kind == "relu_normal_bf16":
        a = f32_to_bf16_bits(np.maximum(rng.standard_normal(size, dtype=np.float32), np.float32(0)))
    elif kind == "constant":
        a = np.ones(size, dtype=np.float32)
    elif kind == "specials":
        a = rng.standard_normal(size, dtype=np.float32)
        pick = rng.integers(0, 8, size=size)
        a[pick == 0] = np.float32(0.0)
        a[pick == 1] = np.float32(-0.0)
        a[pick == 2] = np.float32(np.nan)
        a[pick == 3] = np.float32(np.inf)
        a[pick == 4] = np.float32(-np.inf)
    else:
        raise ValueError("unknown input kind %r" % kind)
    return a.reshape(rows, n)


def is_bf16(kind: str) -> bool:
    return kind.endswith("_bf16")
