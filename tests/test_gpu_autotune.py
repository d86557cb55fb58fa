"""The measured cost model (Prof-K paper, section 4, "Optimal Sample Size":
tau_B / tau_A estimated by microbenchmarking; Figure 3: the N from which
Prof-K beats a direct method).  topk_autotune times the pipeline's own
stages; plans that ask for the measured ratio (cost_ratio = 0) then take
Algorithm 1's S from Eq. 14 with it, and results stay exact."""
import ctypes

import numpy as np
import pytest

from oracle import params, plain
from top_selection_prof_gb300 import workloads

from .gpu_util import assert_same, to_device

pytestmark = pytest.mark.gpu


def test_autotune_model_and_its_use():
    import torch
    import top_selection_prof_gb300 as tk
    lib = tk._lib.get()
    t = tk._lib.TopkTuning()
    rc = lib.topk_autotune(1024, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(t))
    assert rc == 0
    assert t.tau_a_ns > 0 and t.tau_b_ns > 0
    assert abs(t.cost_ratio - t.tau_b_ns / t.tau_a_ns) <= 1e-9 * t.cost_ratio
    assert t.crossover_k == 1024
    assert t.crossover_n == 0 or (t.crossover_n & (t.crossover_n - 1)) == 0
    t2 = tk._lib.TopkTuning()
    assert lib.topk_tuning(ctypes.byref(t2)) == 0 and t2.cost_ratio == t.cost_ratio
    # Eq. 14 with the measured ratio, as the oracle computes it
    for n, k, eps in [(1 << 28, 1024, 1e-6), (1 << 28, 131072, 1e-3), (1 << 26, 10000, 1e-3)]:
        pl = tk.plan(n, k, eps, cost_ratio=0.0)
        s, tt, m = params.exact(n, k, eps, cost_ratio=t.cost_ratio)
        if pl["path_name"] == "profk":
            assert (pl["S"], pl["t"], pl["M"]) == (s, tt, m)
    # selections with the measured model are exact
    x = workloads.make("pareto15", 1, 1 << 22, seed=51)
    v, i, st = tk.select_ex(to_device(x), 1024, eps=1e-3, cost_ratio=0.0)
    ov, oi = plain.topk(x, 1024)
    assert_same(v, i, ov, oi, "measured cost model")
    h = workloads.make("relu_normal_bf16", 64, 65536, seed=52)
    v, i, st = tk.select_ex(to_device(h), 20000, eps=1e-3, global_=True, cost_ratio=0.0)
    ov, oi = plain.topk(h, 20000, global_=True)
    assert_same(v, i, ov, oi, "measured cost model, bf16 global")
