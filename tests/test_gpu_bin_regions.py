"""Bin regions of the filter, and each way out of them, against the oracle.

For one selection with large k the TMA-ring filter keeps each block's
survivors in shared memory and, at the block's end, places them in regions
by their bin of the survivor histogram (2048 bins of (key - tau) >> shift);
the grid refinement and the bin sort then read the regions instead of
partitioning the candidate buffer.  The regions are used only when they are
complete and the bins are a plain digit; otherwise the call takes the
partition of the buffer.  Each input below is built to reach one of those
routes; every output is compared with the oracle bit for bit (values by
their bits, indices exactly), sorted and with the unsorted option (then as a
set, each index holding the input's own bits).  Prof-K paper, section 3
(problem setup) for what is computed.
"""
import numpy as np
import pytest

from oracle import plain
from top_selection_prof_gb300 import workloads

from .gpu_util import assert_same, bits, to_device

pytestmark = pytest.mark.gpu


def _check(x, k, largest=True, global_=False, unsorted=False, eps=1e-3):
    import top_selection_prof_gb300 as tk
    xd = to_device(x)
    v, i, st = tk.select_ex(xd, k, largest=largest, eps=eps, global_=global_, unsorted=int(unsorted))
    assert st["path_name"] == "profk", st
    ov, oi = plain.topk(x, k, largest=largest, global_=global_)
    if not unsorted:
        assert_same(v, i, ov, oi, "k=%d largest=%s" % (k, largest))
        return st
    gi = i.cpu().numpy().reshape(-1)
    assert np.array_equal(np.sort(gi), np.sort(np.asarray(oi).reshape(-1))), "winner set"
    flat = x.reshape(-1)
    want = flat[gi].view(np.uint16) if flat.dtype == np.uint16 else flat[gi].view(np.uint32)
    assert np.array_equal(bits(v).reshape(-1), want), "values are the input's bits at the indices"
    return st


@pytest.mark.parametrize("unsorted", [False, True])
@pytest.mark.parametrize("largest", [True, False])
def test_complete_regions(largest, unsorted):
    # the common route: survivors spread over many bins, none overflowing
    x = workloads.make("relu_normal_bf16", 64, 65536, seed=31)
    _check(x, 20000, largest=largest, global_=True, unsorted=unsorted)
    _check(workloads.make("normal", 1, 1 << 22, seed=32), 30000, largest=largest, unsorted=unsorted)


@pytest.mark.parametrize("unsorted", [False, True])
def test_a_bin_overflows_its_region(unsorted):
    # 1 % of the elements are huge, so the largest sampled key is far above
    # tau and the shift is wide: the ordinary survivors (~1 % of 2^22) all
    # fall in the lowest bin, far more than its region holds
    rng = np.random.default_rng(33)
    n = 1 << 22
    x = rng.standard_normal(n).astype(np.float32)
    far = rng.random(n) < 0.01
    x[far] = (1e30 * (1.0 + rng.random(int(far.sum())))).astype(np.float32)
    x = x.reshape(1, n)
    _check(x, n // 50, unsorted=unsorted)
    _check(-x, n // 50, largest=False, unsorted=unsorted)


@pytest.mark.parametrize("unsorted", [False, True])
def test_survivors_crowd_a_few_blocks(unsorted):
    # ascending input: every survivor lies in the last tiles, so a few filter
    # blocks meet them all and their warps' stages overflow
    # (non-negative bf16 values: ascending bit patterns are ascending values)
    x = np.sort(workloads.make("relu_normal_bf16", 64, 65536, seed=34).reshape(-1)).reshape(64, 65536)
    _check(x, 20000, global_=True, unsorted=unsorted)
    t = workloads.make("ties1000_sorted", 1, 1 << 22, seed=35)
    _check(t, 10000, unsorted=unsorted)


@pytest.mark.parametrize("unsorted", [False, True])
def test_keys_beyond_the_top_bin(unsorted):
    # a heavy tail: survivors far above the largest sampled key land in the
    # top (overflow) bin, whose keys are no plain digit
    x = workloads.make("pareto15", 1, 1 << 22, seed=36)
    _check(x, 65536, unsorted=unsorted)


@pytest.mark.parametrize("unsorted", [False, True])
@pytest.mark.parametrize("kind,k", [("uniform", 3072), ("normal", 4096), ("pareto15", 6000), ("ties1000", 5000)])
def test_mid_k_single_rows(kind, k, unsorted):
    # k from 3072 up to the bin sort's own bound: one aligned row takes the
    # bin regions too (grid refinement + bin sort instead of the cluster)
    x = workloads.make(kind, 1, 1 << 22, seed=37)
    st = _check(x, k, unsorted=unsorted)
    assert st["launches"] == (3 if unsorted else 4), st
    _check(x, k, largest=False, unsorted=unsorted)


@pytest.mark.slow
@pytest.mark.parametrize("largest", [True, False])
@pytest.mark.parametrize("kind,k", [("pareto15", 2048), ("normal", 512)])
def test_refinement_cluster_reads_the_regions(kind, k, largest):
    # k below 3072 and survivors expected beyond one refinement CTA's cache
    # (2^27 elements, eps = 1e-6): CTA 0 of the cluster takes the winners
    # straight from the bin regions
    x = workloads.make(kind, 1, 1 << 27, seed=38)
    st = _check(x, k, largest=largest, eps=1e-6)
    assert st["launches"] == 3, st
