"""Host-side tests of the C ABI: the library loads, exports what include/topk.h
declares, rejects bad arguments, and its parameter math matches the oracle.
No CUDA compute is launched here."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import params as oparams

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "topk.h")


@pytest.fixture(scope="module")
def lib():
    from top_selection_prof_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from top_selection_prof_gb300 import build
        build.build()
    return _lib.get()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(topk_\w+)\s*\(", text, flags=re.M)))


def test_header_declarations_match_binding():
    from top_selection_prof_gb300 import _lib
    assert _declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    from top_selection_prof_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(topk_\w+)", out))
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    assert lib.topk_status_str(0) == b"ok"
    assert lib.topk_status_str(-1) == b"invalid argument"
    assert lib.topk_status_str(-4) == b"unsupported size"
    assert lib.topk_status_str(12345) == b"unknown status"
    assert lib.topk_version() >= 200   # topk_options_t with `unsorted`


def test_index_bits(lib):
    for n, b in [(1, 1), (2, 1), (3, 2), (4, 2), (5, 3), (65536, 16), (65537, 17), (1 << 28, 28), (1 << 32, 32)]:
        assert lib.topk_index_bits(n) == b


def test_argument_validation_without_gpu(lib):
    vp = ctypes.c_void_p
    dummy = vp(16)     # never dereferenced: validation rejects before any launch
    sel = lib.topk_select
    assert sel(dummy, 0, 0, 10, 3, 1, 1e-3, dummy, dummy, None) == 0          # rows == 0: no-op
    assert sel(None, 0, 2, 10, 3, 1, 1e-3, dummy, dummy, None) == -1          # null x
    assert sel(dummy, 0, 2, 10, 3, 1, 1e-3, None, dummy, None) == -1          # null out_vals
    assert sel(dummy, 0, 2, 10, 0, 1, 1e-3, dummy, dummy, None) == -1         # k < 1
    assert sel(dummy, 0, 2, 10, 11, 1, 1e-3, dummy, dummy, None) == -1        # k > n
    assert sel(dummy, 0, -1, 10, 3, 1, 1e-3, dummy, dummy, None) == -1        # rows < 0
    assert sel(dummy, 0, 2, 0, 1, 1, 1e-3, dummy, dummy, None) == -1          # n < 1
    assert sel(dummy, 0, 2, 10, 3, 1, 1.0, dummy, dummy, None) == -1          # eps >= 1
    assert sel(dummy, 0, 2, 10, 3, 1, -0.1, dummy, dummy, None) == -1         # eps < 0
    assert sel(dummy, 7, 2, 10, 3, 1, 1e-3, dummy, dummy, None) == -1         # dtype
    assert sel(dummy, 0, 2, 1 << 31, 3, 1, 1e-3, dummy, dummy, None) == -4    # n >= 2^31
    assert sel(dummy, 0, 1, 1 << 20, 200000, 1, 1e-3, dummy, dummy, None) == -4  # k above the cluster sort
    glob = lib.topk_select_global
    assert glob(dummy, 0, 4, 10, 41, 1, 1e-3, dummy, dummy, None) == -1       # k > rows*n
    assert glob(dummy, 0, 1 << 16, 1 << 17, 5, 1, 1e-3, dummy, dummy, None) == -4  # f32 global >= 2^32


def _plan(lib, n, k, eps, rule=0):
    from top_selection_prof_gb300 import _lib
    opt = _lib.TopkOptions()
    lib.topk_options_init(ctypes.byref(opt))
    opt.rule = rule
    p = _lib.TopkPlan()
    assert lib.topk_plan(n, k, eps, ctypes.byref(opt), ctypes.byref(p)) == 0
    return p


CASES = [(1 << 28, 1024, 1e-6), (1 << 26, 10000, 1e-3), (1 << 28, 131072, 1e-3), (1 << 24, 32, 1e-3),
         (1 << 30, 1 << 12, 1e-3), (1 << 22, 1, 1e-3), (1 << 22, 7, 0.05), (50331648, 131072, 1e-3),
         (1 << 29, 64, 1e-3), (3_000_017, 2_500, 1e-4), (1 << 26, 100, 0.3)]


@pytest.mark.parametrize("n,k,eps", CASES)
def test_exact_rule_parity_with_oracle(lib, n, k, eps):
    p = _plan(lib, n, k, eps, rule=0)
    s, t, m = oparams.exact(n, k, eps)
    if p.path == 2:
        assert (p.S, p.t, p.M) == (s, t, m)
        assert abs(p.p_recall_fail - oparams.p_recall_fail(n, k, s, t)) <= 1e-9 * max(1e-300, eps) + 1e-12
        assert abs(p.p_overflow - oparams.p_overflow(n, s, t, m)) <= 1e-9 * max(1e-300, eps) + 1e-12
    else:
        # the engine declined Prof-K: the oracle's parameters must make it inapplicable
        assert 2 * s >= n or 2 * m > n or t == 0


@pytest.mark.parametrize("n,k,eps", CASES)
def test_alg1_rule_parity_with_oracle(lib, n, k, eps):
    p = _plan(lib, n, k, eps, rule=1)
    s, t, m = oparams.alg1(n, k, eps)
    if p.path == 2:
        assert (p.S, p.t, p.M) == (s, t, m)


def test_plan_picks_direct_path_for_small_rows(lib):
    assert _plan(lib, 32768, 64, 1e-3).path == 1     # S would be the whole row
    assert _plan(lib, 65536, 10, 1e-3).path == 1     # S = n/2
    assert _plan(lib, 1 << 28, 1024, 0.0).path == 3  # eps == 0 on a huge row: grid-wide exact select
    assert _plan(lib, 1 << 28, 1024, 1e-6).path == 2


def test_random_plan_grid_parity(lib):
    rng = np.random.default_rng(4)
    for _ in range(40):
        n = int(rng.integers(1 << 18, 1 << 33))
        k = int(rng.integers(1, min(n // 64, 180000)))
        eps = float(10 ** rng.uniform(-8, -1))
        p = _plan(lib, n, k, eps)
        if p.path == 2:
            assert (p.S, p.t, p.M) == oparams.exact(n, k, eps), (n, k, eps)


@pytest.mark.parametrize("n,k,eps,recall", [(1 << 28, 131072, 1e-3, 0.95), (1 << 26, 10000, 1e-3, 0.9),
                                            (1 << 20, 1000, 0.2, 0.9), (1 << 28, 1024, 1e-6, 0.5),
                                            (1 << 24, 100, 1e-3, 0.999)])
def test_relaxed_recall_rule_parity_with_oracle(lib, n, k, eps, recall):
    """Relaxed recall: t for rank ceil(recall*k), M for k (the buffer's size), same S."""
    from top_selection_prof_gb300 import _lib
    opt = _lib.TopkOptions()
    lib.topk_options_init(ctypes.byref(opt))
    opt.recall = recall
    p = _lib.TopkPlan()
    assert lib.topk_plan(n, k, eps, ctypes.byref(opt), ctypes.byref(p)) == 0
    s, t, m = oparams.exact_relaxed(n, k, eps, recall)
    kt = oparams.recall_rank(k, recall)
    assert p.path == 2 and (p.S, p.t, p.M) == (s, t, m)
    # the recall target's failure bound and minimality, and t never above the exact rule's
    assert oparams.p_recall_fail(n, kt, s, t) <= eps / 2
    assert t == 1 or oparams.p_recall_fail(n, kt, s, t - 1) > eps / 2
    assert abs(p.p_recall_fail - oparams.p_recall_fail(n, kt, s, t)) <= 1e-9 * eps + 1e-12
    assert t <= oparams.exact(n, k, eps)[1]


def test_tuning_entry_points_without_gpu(lib):
    from top_selection_prof_gb300 import _lib
    t = _lib.TopkTuning()
    assert lib.topk_autotune(1024, None, None) == -1          # null out
    assert lib.topk_autotune(-1, None, ctypes.byref(t)) == -1 # k outside [0, 65536]
    assert lib.topk_autotune(70000, None, ctypes.byref(t)) == -1
    assert lib.topk_tuning(None) == -1
