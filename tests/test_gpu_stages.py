"""Stage-by-stage parity of the Prof-K pipeline with the oracle.

Stage 1 (sampling): positions drawn on the GPU equal the oracle's Philox
sampler bit for bit.  Stage 2 (threshold): the sampled t-th largest element is
the oracle's order statistic of the same draws.  Stage 3 (filter): the count R
and the buffer contents are the oracle's survivor set.  Fallback: the measured
miss rate follows the exact tails (Theorem 3's budget).
"""
import math

import numpy as np
import pytest

from oracle import params, philox, plain
from top_selection_prof_gb300 import workloads

from .gpu_util import to_device, unpack_keys

pytestmark = pytest.mark.gpu


def _tk():
    import top_selection_prof_gb300 as tk
    return tk


@pytest.mark.parametrize("kind,rows,n,S,global_", [
    ("normal", 1, 1 << 20, 32768, False),
    ("pareto15", 3, 300_007, 10_001, False),
    ("relu_normal_bf16", 64, 65536, 131072, True),
    ("uniform", 1, 12345, 999, False),
])
def test_sampler_positions_match_oracle_philox(kind, rows, n, S, global_):
    tk = _tk()
    x = workloads.make(kind, rows, n, seed=1)
    length = rows * n if global_ else n
    for seed, counter in [(0x243F6A8885A308D3, 0), (12345, 7), ((1 << 64) - 1, (1 << 40) + 3)]:
        keys = tk.prof_sample(to_device(x), S, seed, counter, global_=global_).cpu().numpy()
        vkey, pos = unpack_keys(keys, tk.index_bits(length))
        for r in range(1 if global_ else rows):
            assert np.array_equal(pos[r], philox.sample_positions(length, S, seed, counter, row=r)), (seed, r)


@pytest.mark.parametrize("largest", [True, False])
def test_sample_keys_rank_like_the_oracle(largest):
    tk = _tk()
    x = workloads.make("ties1000", 1, 1 << 18, seed=2)
    S = 5000
    keys = tk.prof_sample(to_device(x), S, 99, 5, largest=largest).cpu().numpy()[0]
    _, pos = unpack_keys(keys[None, :], tk.index_bits(x.size))
    sorted_keys = np.sort(keys.view(np.uint64))[::-1]
    for t in (1, 2, 17, S // 2, S):
        want = plain.sample_order_stat(x[0], pos[0], t, largest=largest)
        _, p = unpack_keys(sorted_keys[t - 1:t].view(np.int64)[None, :], tk.index_bits(x.size))
        assert p[0][0] == want, t


@pytest.mark.parametrize("kind,n,k,eps,global_rows", [
    ("pareto15", 1 << 22, 1024, 1e-6, 0),
    ("ties1000", 1 << 22, 10000, 1e-3, 0),
    ("ties1000_sorted", 1 << 22, 10000, 1e-3, 0),
    ("relu_normal_bf16", 65536, 8192, 1e-3, 256),
    # 32768 draws from 65600 elements: many positions drawn twice, also at
    # the boundary ranks (k = 20: each block keeps its own top t; k = 100:
    # the grid-wide radix select)
    ("uniform", 65600, 20, 1e-3, 0),
    ("uniform", 65600, 100, 1e-3, 0),
])
def test_threshold_and_survivor_count_match_oracle(kind, n, k, eps, global_rows):
    tk = _tk()
    rows = global_rows or 1
    x = workloads.make(kind, rows, n, seed=3)
    flat = x.reshape(-1)
    for counter in (0, 1, 2):
        v, i, st = tk.select_ex(to_device(x), k, eps=eps, global_=bool(global_rows), counter=counter)
        assert st["path_name"] == "profk"
        pos = philox.sample_positions(flat.size, st["S"], st["seed"], counter)
        assert st["tau_index"] == plain.sample_order_stat(flat, pos, st["t"])
        assert st["R"] == plain.count_at_or_above(flat, st["tau_index"])
        ora_s, ora_t, ora_m = params.exact(flat.size, k, eps)
        assert (st["S"], st["t"], st["M"]) == (ora_s, ora_t, ora_m)


@pytest.mark.parametrize("largest", [True, False])
def test_filter_buffer_is_the_survivor_set(largest):
    import torch
    tk = _tk()
    x = workloads.make("normal", 2, 1 << 20, seed=4)
    keys = tk.prof_sample(to_device(x), 4096, 7, 11, largest=largest)
    ib = tk.index_bits(x.shape[1])
    ks = keys.cpu().numpy()
    # per row pick the 40th largest sampled key as tau
    tau = np.array([np.sort(ks[r].view(np.uint64))[::-1][39] for r in range(2)], dtype=np.uint64)
    tau_t = torch.from_numpy(tau.view(np.int64))
    buf, counts = tk.prof_filter(to_device(x), tau_t, 20000, largest=largest)
    counts = counts.cpu().numpy()
    buf = buf.cpu().numpy()
    for r in range(2):
        _, pivot = unpack_keys(tau[r:r + 1].view(np.int64)[None, :], ib)
        R = plain.count_at_or_above(x[r], int(pivot[0][0]), largest=largest)
        assert counts[r] == R
        _, oi = plain.topk(x[r:r + 1], R, largest=largest)
        _, got = unpack_keys(buf[r:r + 1, :R], ib)
        assert sorted(got[0].tolist()) == sorted(oi[0].tolist())
    # a buffer smaller than R keeps counting and stores M distinct survivors
    small, c2 = tk.prof_filter(to_device(x), tau_t, 50, largest=largest)
    assert np.array_equal(c2.cpu().numpy(), counts)
    _, got = unpack_keys(small.cpu().numpy()[0:1], ib)
    _, oi = plain.topk(x[0:1], int(counts[0]), largest=largest)
    assert len(set(got[0].tolist())) == 50 and set(got[0].tolist()) <= set(oi[0].tolist())


@pytest.mark.parametrize("rule", [0, 1])
def test_miss_rate_follows_the_exact_tails(rule):
    """Observed fallback frequency vs P[R<k] + P[R>M] for the (S, t, M) in use."""
    tk = _tk()
    n, k, eps, S = 1 << 20, 100, 0.2, 2048
    x = workloads.make("uniform", 1, n, seed=5)
    xd = to_device(x)
    ov, oi = plain.topk(x, k)
    ovb = ov.view(np.uint32)
    runs, misses = 300, 0
    st = None
    for c in range(runs):
        v, i, st = tk.select_ex(xd, k, eps=eps, counter=c, s_min=S, s_max=S, rule=rule)
        misses += st["misses"]
        # every call is exact, whether or not it took the fallback
        assert np.array_equal(i.cpu().numpy(), oi), (c, st["misses"])
        assert np.array_equal(v.cpu().numpy().view(np.uint32), ovb), (c, st["misses"])
    p = params.p_recall_fail(n, k, st["S"], st["t"]) + params.p_overflow(n, st["S"], st["t"], st["M"])
    if rule == 0:
        assert p <= eps
    sd = math.sqrt(max(p * (1 - p), 1e-4) / runs)
    assert abs(misses / runs - p) < 4.5 * sd, (misses, runs, p)
