"""Failure detection without a GPU fault: bounded device waits that run out,
and the routing of misses to the fallback.

The exact fallback (Prof-K paper, section 3 stage 4; Appendix D, "Fallback as
a Safety Mechanism") synchronises its cooperative grid with bounded waits.  A
host-set test knob makes one block leave its first wait without arriving, so
every other block's wait (limited here to 1 ms) runs out: the kernels return,
the call reports TOPK_ETIMEOUT -- with stats, or later through
topk_last_status -- and the next call on the stream is exact again.  Nothing
here faults, traps or spins without a limit.
"""
import ctypes

import numpy as np
import pytest

from oracle import plain
from top_selection_prof_gb300 import workloads

from .gpu_util import assert_same, to_device

pytestmark = pytest.mark.gpu

WAIT_NS = 1_000_000  # 1 ms


def _tk():
    import top_selection_prof_gb300 as tk
    return tk


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


# (kind, rows, n, k, global): the fallback kernel after the filter (k = 1024,
# forced miss), and the fallback inside the grid refinement (k >= 8192)
CASES = [("pareto15", 1, 1 << 22, 1024, False), ("relu_normal_bf16", 64, 65536, 20000, True)]


@pytest.mark.parametrize("kind,rows,n,k,global_", CASES)
def test_timed_out_wait_is_reported_and_the_next_call_is_exact(kind, rows, n, k, global_):
    import torch
    tk = _tk()
    lib = tk._lib.get()
    x = workloads.make(kind, rows, n, seed=31)
    xd = to_device(x)
    ov, oi = plain.topk(x, k, global_=global_)
    # with stats: the call itself reports the timeout
    with pytest.raises(tk.TopkError) as err:
        tk.select_ex(xd, k, eps=1e-3, global_=global_, force_miss=1, inject_wait_timeout=1,
                     wait_limit_ns=WAIT_NS)
    assert err.value.status == tk._lib.TOPK_ETIMEOUT
    # the next call on the stream is exact and clean
    v, i, st = tk.select_ex(xd, k, eps=1e-3, global_=global_)
    assert_same(v, i, ov, oi, "after a timeout")
    assert lib.topk_last_status(_stream()) == tk._lib.TOPK_OK
    # without stats: the call returns at once; topk_last_status reports it
    v, i, _ = tk.select_ex(xd, k, eps=1e-3, global_=global_, stats=False, force_miss=1,
                           inject_wait_timeout=1, wait_limit_ns=WAIT_NS)
    assert lib.topk_last_status(_stream()) == tk._lib.TOPK_ETIMEOUT
    # a forced miss that runs to completion is exact (and its status clean)
    v, i, st = tk.select_ex(xd, k, eps=1e-3, global_=global_, force_miss=1, wait_limit_ns=WAIT_NS * 1000)
    assert st["misses"] == 1
    assert_same(v, i, ov, oi, "forced miss after a timeout")
    v, i = (tk.select_global if global_ else tk.select)(xd, k, eps=1e-3)
    assert lib.topk_last_status(_stream()) == tk._lib.TOPK_OK
    assert_same(v if global_ else v, i, ov, oi, "plain call")
    torch.cuda.synchronize()


def test_last_status_on_a_fresh_stream_is_ok():
    import torch
    tk = _tk()
    s = torch.cuda.Stream()
    assert tk._lib.get().topk_last_status(s.cuda_stream) == tk._lib.TOPK_OK


def test_forced_miss_takes_the_grid_wide_fallback():
    """A miss the caller forces never runs in the refinement's cluster (which
    would stream the whole row from one or two SMs): the fallback kernel is
    launched after the filter, and the result is exact."""
    x = workloads.make("pareto15", 1, 1 << 22, seed=32)
    tk = _tk()
    xd = to_device(x)
    ov, oi = plain.topk(x, 1024)
    v, i, st = tk.select_ex(xd, 1024, eps=1e-6)
    assert st["launches"] == 3                       # no miss expected: the refinement checks
    v, i, st = tk.select_ex(xd, 1024, eps=1e-6, force_miss=1)
    assert st["launches"] == 4 and st["misses"] == 1, st   # + the fallback kernel
    assert_same(v, i, ov, oi, "forced miss")


def test_miss_routing_follows_the_plans_own_miss_probability():
    """Algorithm 1 as printed keeps t = 1 here (the sparse branch), whose recall
    fails often; the plan's own miss probability, not eps, decides that the
    grid-wide fallback is launched."""
    tk = _tk()
    n, k, eps = 1 << 22, 1024, 1e-6
    pl = tk.plan(n, k, eps, rule=tk.TOPK_RULE_ALG1)
    assert pl["t"] == 1 and pl["p_recall_fail"] > 0.01
    x = workloads.make("pareto15", 1, n, seed=33)
    xd = to_device(x)
    ov, oi = plain.topk(x, k)
    v, i, st = tk.select_ex(xd, k, eps=eps, rule=tk.TOPK_RULE_ALG1)
    assert st["launches"] == 4, st
    assert_same(v, i, ov, oi, "Algorithm 1 rule")
