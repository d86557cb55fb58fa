"""Bit-exact parity with the CPU oracle at the benchmark configurations' own sizes.

Each case is one of the five workloads at full size, run through the entry
point the benchmark times (topk_select / topk_select_global), and compared
element by element with the oracle's (value desc, index asc) top-k: values
by their bits and indices exactly, tolerance 0 (selection does no
arithmetic).  Prof-K paper, section 3 (problem setup) for what is computed;
"Rank by Counting" (Goal) for the index tie-break.  The oracle needs about
16 bytes of host memory per element (4 GiB for a 2^28-element selection)
and seconds per call, so the inputs are made once per module.
"""
import functools

import numpy as np
import pytest

from oracle import plain
from top_selection_prof_gb300 import workloads

from .gpu_util import assert_same, to_device

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@functools.lru_cache(maxsize=1)
def _input(name, seed):
    cfg = workloads.WORKLOADS[name]
    return workloads.make(cfg["kind"], cfg["rows"], cfg["n"], seed)


def _run(name, largest, seed=0):
    import torch
    import top_selection_prof_gb300 as tk
    cfg = workloads.WORKLOADS[name]
    x = _input(name, seed)
    glob = cfg["mode"] == "global"
    xd = to_device(x)
    if glob:
        v, i = tk.select_global(xd, cfg["k"], largest=largest, eps=cfg["eps"])
    else:
        v, i = tk.select(xd, cfg["k"], largest=largest, eps=cfg["eps"])
    torch.cuda.synchronize()
    lib = tk._lib.get()
    assert lib.topk_last_status(torch.cuda.current_stream().cuda_stream) == 0
    _, _, st = tk.select_ex(xd, cfg["k"], largest=largest, eps=cfg["eps"], global_=glob)
    del xd
    ov, oi = plain.topk(x, cfg["k"], largest=largest, global_=glob)
    assert_same(v, i, ov, oi, "%s largest=%s path=%s" % (name, largest, st["path_name"]))
    return st


@pytest.mark.parametrize("largest", [True, False])
def test_single_row_65536_int20_k10(largest):
    st = _run("single_row_65536_int20_k10", largest)
    assert st["path_name"] == "direct"


@pytest.mark.parametrize("largest", [True, False])
def test_rows_1024x32768_normal_k64(largest):
    st = _run("rows1024x32768_normal_k64", largest)
    assert st["path_name"] == "direct"


@pytest.mark.parametrize("largest", [True, False])
def test_single_row_2p28_pareto15_k1024(largest):
    st = _run("single_row_2p28_pareto15_k1024", largest)
    assert st["path_name"] == "profk" and (st["S"], st["t"], st["M"]) == (86966, 7, 87009)


@pytest.mark.parametrize("largest", [True, False])
def test_single_row_2p26_ties1000_k10000(largest):
    st = _run("single_row_2p26_ties1000_k10000", largest)
    assert st["path_name"] == "profk" and (st["S"], st["t"], st["M"]) == (108655, 32, 33310)


@pytest.mark.parametrize("largest", [True, False])
def test_single_row_2p26_ties1000_sorted_k10000(largest):
    st = _run("single_row_2p26_ties1000_sorted_k10000", largest)
    assert st["path_name"] == "profk"


@pytest.mark.parametrize("largest", [True, False])
def test_batchtopk_4096x65536_relu_bf16_k131072(largest):
    st = _run("batchtopk_4096x65536_relu_bf16_k131072", largest)
    assert st["path_name"] == "profk" and (st["S"], st["t"], st["M"]) == (131072, 93, 262190)


def test_batchtopk_4096x65536_relu_bf16_k131072_unsorted():
    """The unsorted option on the BatchTopK workload at full size: the oracle's
    winners as a set, each returned with the input's own bits at its index
    (the order is left open; the Prof-K paper's BatchTopK application takes
    the set)."""
    import torch
    import top_selection_prof_gb300 as tk
    name = "batchtopk_4096x65536_relu_bf16_k131072"
    cfg = workloads.WORKLOADS[name]
    x = _input(name, 0)
    xd = to_device(x)
    v, i, st = tk.select_ex(xd, cfg["k"], eps=cfg["eps"], global_=True, unsorted=1)
    torch.cuda.synchronize()
    del xd
    assert st["path_name"] == "profk" and st["launches"] == 3, st
    ov, oi = plain.topk(x, cfg["k"], global_=True)
    gi = i.cpu().numpy().reshape(-1)
    assert np.array_equal(np.sort(gi), np.sort(np.asarray(oi).reshape(-1))), "winner set"
    bits = v.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
    assert np.array_equal(bits, x.reshape(-1)[gi].view(np.uint16)), "values are the input's bits at the indices"
