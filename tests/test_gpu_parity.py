"""Parity of the CUDA path with the CPU oracle: bit-exact values and indices.

Sizes are chosen so the oracle finishes in seconds while spanning many filter
tiles and ragged tails.  Every case goes through the C ABI via the binding.
"""
import zlib

import pytest

from oracle import plain
from top_selection_prof_gb300 import workloads

from .gpu_util import assert_same, to_device

pytestmark = pytest.mark.gpu


def _tk():
    import top_selection_prof_gb300 as tk
    return tk


def _check(x, k, largest=True, eps=1e-3, global_=False, expect_path=None, **opts):
    tk = _tk()
    xd = to_device(x)
    v, i, st = tk.select_ex(xd, k, largest=largest, eps=eps, global_=global_, **opts)
    ov, oi = plain.topk(x, k, largest=largest, global_=global_)
    assert_same(v, i, ov, oi, "k=%d largest=%s path=%s" % (k, largest, st["path_name"]))
    if expect_path is not None:
        assert st["path_name"] == expect_path, st
    return st


# (kind, rows, n, k, eps, global, expected path)
CASES = [
    ("int20", 1, 65536, 10, 1e-3, False, "direct"),             # the exercise's own shape
    ("normal", 64, 32768, 64, 1e-3, False, "direct"),
    ("normal", 3, 100_003, 37, 1e-3, False, "profk"),            # ragged rows -> scalar loads
    ("pareto15", 1, 1 << 22, 1024, 1e-6, False, "profk"),
    ("ties1000", 1, 1 << 22, 10000, 1e-3, False, "profk"),
    ("ties1000_sorted", 1, 1 << 22, 10000, 1e-3, False, "profk"),
    ("relu_normal_bf16", 256, 65536, 8192, 1e-3, True, "profk"),
    ("relu_normal_bf16", 256, 65536, 100000, 1e-3, True, "profk"),  # 16-CTA cluster sort
    ("uniform", 1, 1_000_003, 777, 1e-3, False, "profk"),
    ("pareto15", 4, 1 << 21, 100, 1e-3, False, "profk"),          # per-row Prof-K
    ("normal", 1, 1 << 20, 1, 1e-3, False, "profk"),
    ("specials", 1, 1 << 20, 3000, 1e-3, False, "profk"),
    ("specials", 5, 4099, 50, 1e-3, False, "direct"),
    ("constant", 1, 1 << 21, 500, 1e-3, False, "profk"),
    ("relu_normal_bf16", 7, 33_333, 20, 1e-3, False, None),
    ("normal", 1, 1 << 22, 9000, 1e-3, False, "profk"),            # k just above the bin-sort bound
    ("ties1000", 1, 1 << 24, 12000, 1e-3, False, "profk"),         # bin sort with a 2-CTA cluster
    ("uniform", 1, (1 << 22) + 8, 9000, 0.0, False, "exact"),      # exact path, sort after the fallback
    ("ties1000", 5, 1 << 22, 12000, 1e-3, False, "profk"),         # more rows than the grid refinement takes
    ("normal", 4, 1 << 21, 8500, 1e-3, False, "profk"),            # grid refinement over four rows
    ("normal", 1, 1 << 22, 131072, 1e-3, False, "profk"),          # candidates crossing powers of two
]


@pytest.mark.parametrize("kind,rows,n,k,eps,global_,path", CASES)
@pytest.mark.parametrize("largest", [True, False])
def test_parity(kind, rows, n, k, eps, global_, path, largest):
    x = workloads.make(kind, rows, n, seed=zlib.crc32(("%s/%d/%d/%d" % (kind, rows, n, k)).encode()) % 1000)
    _check(x, k, largest=largest, eps=eps, global_=global_, expect_path=path)


@pytest.mark.parametrize("path", [1, 2, 3])   # direct, Prof-K, grid-wide exact
def test_every_path_on_the_same_input(path):
    x = workloads.make("ties1000", 1, 1 << 21, seed=3)
    _check(x, 2500, eps=1e-3 if path == 2 else 0.0, path=path)
    x = workloads.make("relu_normal_bf16", 32, 65536, seed=4)
    _check(x, 3000, eps=1e-3 if path == 2 else 0.0, global_=True, path=path)


def test_forced_miss_takes_the_fallback_and_stays_exact():
    x = workloads.make("pareto15", 1, 1 << 22, seed=5)
    st = _check(x, 1024, eps=1e-3, force_miss=1)
    assert st["misses"] == 1 and st["path_name"] == "profk"


@pytest.mark.parametrize("m_override,t_override", [(1100, 0), (0, 1), (0, 400)])
def test_overflow_and_recall_misses_are_repaired(m_override, t_override):
    # a tiny buffer overflows; t = 1 tends to miss recall; a huge t overflows the buffer
    x = workloads.make("normal", 1, 1 << 22, seed=6)
    st = _check(x, 1000, eps=1e-3, m_override=m_override, t_override=t_override)
    if st["misses"]:
        assert st["R"] < 1000 or st["R"] > st["M"]
    else:
        assert 1000 <= st["R"] <= st["M"]


def test_k_equals_n_and_k_one_direct():
    x = workloads.make("ties1000", 3, 5000, seed=7)
    _check(x, 5000)
    _check(x, 1)


def test_unaligned_input_pointer():
    tk = _tk()
    base = workloads.make("normal", 1, (1 << 21) + 1, seed=8)
    flat = to_device(base.reshape(-1))[1:]         # 4-byte offset: no 16-byte vectors
    assert flat.data_ptr() % 16 != 0
    v, i, st = tk.select_ex(flat, 300, eps=1e-3)
    ov, oi = plain.topk(base.reshape(-1)[1:][None, :], 300)
    assert_same(v[None, :], i[None, :], ov, oi, "unaligned")
    assert st["path_name"] == "profk"


def test_rows_zero_is_a_noop():
    import torch
    tk = _tk()
    x = torch.empty((0, 100), device="cuda")
    v, i = tk.select(x, 5)
    assert v.shape == (0, 5) and i.shape == (0, 5)


def test_maximum_k_cluster_sort():
    tk = _tk()
    kmax = 16 * 11776
    x = workloads.make("normal", 1, 1 << 20, seed=9)
    _check(x, kmax, eps=1e-3)
    with pytest.raises(tk.TopkError):
        tk.select(to_device(x), kmax + 1)


def test_repeated_calls_and_streams():
    import torch
    tk = _tk()
    x = workloads.make("pareto15", 1, 1 << 22, seed=10)
    xd = to_device(x)
    ov, oi = plain.topk(x, 512)
    s = torch.cuda.Stream()
    for rep in range(3):
        with torch.cuda.stream(s):
            v, i = tk.select(xd, 512)
        s.synchronize()
        assert_same(v, i, ov, oi, "rep %d" % rep)


@pytest.mark.parametrize("kind,rows,n,k,eps,global_,expect", [
    ("pareto15", 1, 1 << 22, 1024, 1e-6, False, 3),            # sample + threshold, filter, refinement
    ("relu_normal_bf16", 256, 65536, 100000, 1e-3, True, 4),   # ... grid refinement + bin sort
    # five rows: fallback kernel (a miss in one of five clusters is expected to
    # cost more than the launch), refinement cluster + bin sort
    ("ties1000", 5, 1 << 22, 12000, 1e-3, False, 5),
    ("normal", 64, 32768, 64, 1e-3, False, 1),                 # direct: one kernel
])
def test_launch_count(kind, rows, n, k, eps, global_, expect):
    x = workloads.make(kind, rows, n, seed=11)
    st = _check(x, k, eps=eps, global_=global_)
    assert st["launches"] == expect, st


# Large k on one cooperative grid: the miss check, the fallback and the
# partition of the winners, then the bin sort.
@pytest.mark.parametrize("largest", [True, False])
def test_grid_refinement_forced_miss(largest):
    x = workloads.make("relu_normal_bf16", 64, 65536, seed=12)
    st = _check(x, 20000, largest=largest, eps=1e-3, global_=True, force_miss=1)
    assert st["misses"] == 1 and st["path_name"] == "profk"


def test_grid_refinement_overflow_is_repaired():
    x = workloads.make("ties1000", 1, 1 << 22, seed=13)
    # S = 43088 here: t = 200 keeps ~19,500 candidates (sd ~1,400), far more
    # than the 10,050 the buffer holds
    st = _check(x, 10000, eps=1e-3, m_override=10050, t_override=200)
    assert st["misses"] == 1 and st["R"] > st["M"]


def test_grid_refinement_exact_kth_key():
    # One outlier and a constant row: the first digit below the top varying
    # bit puts every candidate but the outlier in one bin, which holds more
    # than the exchange buffer's 2k places; the k-th key is then found by
    # further digits across the grid and only the winners are placed.
    import numpy as np
    x = np.full((1, 1 << 22), 1.0, dtype=np.float32)
    x[0, 12345] = 3.0e38
    k = 9000
    _check(x, k, eps=1e-3)  # (few candidates: the whole boundary bin fits)
    # S = 41286 for this size: t = 266 keeps about 27,000 candidates (> 2k)
    st = _check(x, k, eps=1e-3, m_override=200000, t_override=266)
    assert st["misses"] == 0 and st["R"] > 2 * k, st


def test_grid_refinement_repeated_calls_alternate_control_words():
    import torch
    tk = _tk()
    x = workloads.make("relu_normal_bf16", 32, 65536, seed=14)
    xd = to_device(x)
    ov, oi = plain.topk(x, 10000, global_=True)
    for rep in range(5):
        v, i = tk.select_global(xd, 10000)
        torch.cuda.synchronize()
        assert_same(v, i, ov, oi, "rep %d" % rep)


@pytest.mark.parametrize("kind,rows,n,k,global_,cluster,launches", [
    ("relu_normal_bf16", 64, 65536, 20000, True, 1, 4),   # one selection, large k: the grid refinement
    ("ties1000", 5, 1 << 22, 12000, False, 2, 5),          # five selections: a refinement cluster per row
])
def test_large_k_refinement_route(kind, rows, n, k, global_, cluster, launches):
    x = workloads.make(kind, rows, n, seed=15)
    st = _check(x, k, eps=1e-3, global_=global_)
    assert st["cluster"] == cluster and st["launches"] == launches, st


def test_grid_refinement_more_rows_after_fewer():
    # The refinement's control words alternate between two copies; a call
    # with four selections after calls with one must find every row clean.
    x4 = workloads.make("normal", 4, 1 << 21, seed=16)
    x1 = workloads.make("relu_normal_bf16", 32, 65536, seed=17)
    for rep in range(2):   # four rows, three single selections, four rows: the first copy again
        _check(x4, 8500, largest=rep == 0)
        _check(x1, 9000, global_=True)
        _check(x1, 9000, global_=True, largest=False)
        _check(x1, 9500, global_=True)
        _check(x4, 8500, largest=rep == 1)


@pytest.mark.parametrize("largest", [True, False])
def test_few_winners_from_many_candidates(largest):
    # k <= 1024 is refined by one CTA; with about 40,000 candidates (S = 32768
    # here, t = 312) they do not fit its shared memory and every pass re-reads
    # them from L2.
    x = workloads.make("normal", 1, 1 << 22, seed=18)
    st = _check(x, 1000, largest=largest, eps=1e-3, t_override=312, m_override=200000)
    assert st["misses"] == 0 and st["R"] > 30000, st


def _check_set(x, k, largest=True, global_=False, **opts):
    """Unsorted output: the oracle's winners as a set, each with its own input bits."""
    import numpy as np
    tk = _tk()
    v, i, st = tk.select_ex(to_device(x), k, largest=largest, eps=1e-3, global_=global_, unsorted=1, **opts)
    ov, oi = plain.topk(x, k, largest=largest, global_=global_)
    rows = 1 if global_ else x.shape[0]
    gi = i.cpu().numpy().reshape(rows, k)
    assert np.array_equal(np.sort(gi, axis=1), np.sort(np.asarray(oi).reshape(rows, k), axis=1)), "winner sets"
    flat = x.reshape(rows, -1)
    bits = (v.view(__import__("torch").int16).cpu().numpy().view(np.uint16) if flat.dtype == np.uint16
            else v.cpu().numpy().view(np.uint32)).reshape(rows, k)
    want = np.take_along_axis(flat, gi, axis=1)
    want = want.view(np.uint16) if flat.dtype == np.uint16 else want.view(np.uint32)
    assert np.array_equal(bits, want), "values are the input's bits at the returned positions"
    return st


@pytest.mark.parametrize("largest", [True, False])
def test_unsorted_output_is_the_exact_set(largest):
    st = _check_set(workloads.make("relu_normal_bf16", 64, 65536, seed=19), 20000, largest=largest, global_=True)
    assert st["launches"] == 3, st          # sample + threshold, filter, grid refinement: no sort
    _check_set(workloads.make("ties1000", 1, 1 << 22, seed=20), 10000, largest=largest)
    _check_set(workloads.make("normal", 4, 1 << 21, seed=21), 8500, largest=largest)


def test_unsorted_output_after_a_miss():
    st = _check_set(workloads.make("relu_normal_bf16", 64, 65536, seed=22), 20000, global_=True, force_miss=1)
    assert st["misses"] == 1


def test_unsorted_request_elsewhere_still_sorts():
    # (k below the grid refinement's range: the option is a permission, the output stays sorted)
    x = workloads.make("pareto15", 1, 1 << 22, seed=23)
    _check(x, 1000, eps=1e-3, unsorted=1)
