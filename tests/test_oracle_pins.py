"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Every test here runs on the CPU.  None retypes the oracle's own code: each
checks it against an independent statement (brute force, an identity from one
of the GPU.js exercises, a closed form, enumeration, or printed numbers).
"""
import itertools
import math
import os

import numpy as np
import pytest

from oracle import params, philox, plain
from top_selection_prof_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                key, value, tol = line.split()
                vals[key] = (float(value), float(tol))
    return vals


# --------------------------------------------------------------------------
# Rank by Counting (top-k task 1): rank_i = #{j : x_j > x_i} + #{j < i : x_j == x_i}
# --------------------------------------------------------------------------

def _ranks_by_counting(x):
    """O(n^2) ranks exactly as the exercise defines them (vectorised over j)."""
    n = x.size
    ranks = np.empty(n, dtype=np.int64)
    idx = np.arange(n)
    for i in range(n):
        ranks[i] = np.count_nonzero(x > x[i]) + np.count_nonzero((x == x[i]) & (idx < i))
    return ranks


@pytest.mark.parametrize("seed,n,hi", [(0, 8, 4), (1, 257, 30), (2, 2048, 1000), (3, 4096, 1000)])
def test_rank_by_counting_matches_oracle_order(seed, n, hi):
    rng = np.random.default_rng(seed)
    x = rng.integers(0, hi, size=n).astype(np.float32)   # scores repeat constantly
    ranks = _ranks_by_counting(x)
    # every rank appears exactly once; the largest score has rank 0
    assert np.array_equal(np.sort(ranks), np.arange(n))
    assert x[np.argmin(ranks)] == x.max()
    # the oracle's full order (k = n) is "sort by counted rank"
    _, idx = plain.topk(x[None, :], n)
    assert np.array_equal(idx[0], np.argsort(ranks))
    for k in (1, 5, n // 2, n):
        v, i = plain.topk(x[None, :], k)
        assert np.array_equal(i[0], np.argsort(ranks)[:k])
        assert np.array_equal(v[0], x[np.argsort(ranks)[:k]])


def test_rank_by_counting_smallest_mode():
    rng = np.random.default_rng(7)
    x = rng.integers(0, 20, size=500).astype(np.float32)
    ranks = _ranks_by_counting(-x)      # smallest first == largest of the negation
    _, idx = plain.topk(x[None, :], 500, largest=False)
    assert np.array_equal(idx[0], np.argsort(ranks))


def test_special_values_reading():
    """NaN above every number and NaNs equal, -0 == +0, infinities ordinary; ties by index."""
    x = np.array([0.0, -0.0, np.nan, 1.0, np.inf, -np.inf, np.nan, -0.0, 0.0, 1.0], dtype=np.float32)

    def rank_class(i):   # independent statement of the reading as a sort key
        v = float(x[i])
        return (0, 0.0, i) if math.isnan(v) else (1, -v, i)

    expect = sorted(range(x.size), key=rank_class)
    v, i = plain.topk(x[None, :], x.size)
    assert list(i[0]) == expect
    # output values are the input's own bits (the sign of zero survives)
    assert np.array_equal(v[0].view(np.uint32), x[expect].view(np.uint32))
    expect_small = sorted(range(x.size), key=lambda j: (1, 0.0, j) if math.isnan(float(x[j]))
                          else (0, float(x[j]), j))
    _, i = plain.topk(x[None, :], x.size, largest=False)
    assert list(i[0]) == expect_small


def test_bf16_is_widened_exactly():
    rng = np.random.default_rng(3)
    f = rng.standard_normal(3000).astype(np.float32)
    h = workloads.f32_to_bf16_bits(f)
    w = workloads.bf16_bits_to_f32(h)
    v16, i16 = plain.topk(h[None, :], 100)
    v32, i32 = plain.topk(w[None, :], 100)
    assert np.array_equal(i16, i32)
    assert np.array_equal(v16, h[i32[0]][None, :])


def test_rows_and_global_agree_with_per_row_loop():
    rng = np.random.default_rng(5)
    x = rng.integers(0, 50, size=(6, 300)).astype(np.float32)
    v, i = plain.topk(x, 17)
    for r in range(6):
        vr, ir = plain.topk(x[r:r + 1], 17)
        assert np.array_equal(ir[0], i[r]) and np.array_equal(vr[0], v[r])
    vg, ig = plain.topk(x, 40, global_=True)
    flat = x.reshape(-1)
    ranks = _ranks_by_counting(flat)
    assert np.array_equal(ig, np.argsort(ranks)[:40])
    assert np.array_equal(vg, flat[ig])


# --------------------------------------------------------------------------
# Find the Cutoff Instead (top-k task 4): bisection on the value axis
# --------------------------------------------------------------------------

def _count_above_strided(values, t, threads):
    """The counting kernel: thread x counts values[i*threads + x] > t; the host totals."""
    partial = np.zeros(threads, dtype=np.int64)
    for x in range(threads):
        partial[x] = np.count_nonzero(values[x::threads] > t)
    return int(partial.sum())


def test_bisection_cutoff_identity():
    g = _golden("prof_k_printed_numbers.txt")
    n, k, threads = int(g["cutoff_scores"][0]), int(g["cutoff_k"][0]), int(g["cutoff_threads"][0])
    for seed in range(3):
        x = workloads.make("int20", 1, n, seed)[0]
        v, _ = plain.topk(x[None, :], k + 1)
        if v[0][k - 1] == v[0][k]:
            continue                       # the exercise requires distinct k-th and (k+1)-th
        lo, hi = float(x.min()) - 1.0, float(x.max())
        steps = 0
        while hi - lo > 0.5:
            mid = (lo + hi) / 2.0
            if _count_above_strided(x, mid, threads) >= k:
                lo = mid
            else:
                hi = mid
            steps += 1
        cutoff = math.floor(lo)
        assert _count_above_strided(x, cutoff, threads) == k
        assert float(v[0][k - 1]) == cutoff + 1        # the k-th value is the cutoff + 1
        _, i = plain.topk(x[None, :], k)
        assert set(i[0].tolist()) == set(np.nonzero(x > cutoff)[0].tolist())
        assert 15 <= steps <= 22                        # "eighteen halvings" for 2^20 values


# --------------------------------------------------------------------------
# One Bit at a Time (radix sort task 2): the stable one-bit split
# --------------------------------------------------------------------------

def _split_low_bit(keys, payload, bit):
    flags = (keys >> bit) & 1
    zeros = int(np.count_nonzero(flags == 0))
    dest = np.empty(keys.size, dtype=np.int64)
    for i in range(keys.size):           # destination by counting earlier equals
        before = int(np.count_nonzero(flags[:i] == flags[i]))
        dest[i] = before if flags[i] == 0 else zeros + before
    out_k = np.empty_like(keys)
    out_p = np.empty_like(payload)
    out_k[dest] = keys
    out_p[dest] = payload
    return out_k, out_p


def test_one_bit_split_is_stable_partition():
    rng = np.random.default_rng(11)
    keys = rng.integers(0, 16, size=64)
    out, pay = _split_low_bit(keys, np.arange(64), 0)
    expect = [i for i in range(64) if keys[i] % 2 == 0] + [i for i in range(64) if keys[i] % 2 == 1]
    assert list(pay) == expect and np.array_equal(out, keys[expect])


def test_composed_splits_reproduce_oracle_order():
    rng = np.random.default_rng(12)
    n, bits = 600, 10
    x = rng.integers(0, 1 << bits, size=n)
    keys = (1 << bits) - 1 - x            # ascending key == descending value
    payload = np.arange(n)
    for b in range(bits):                 # LSD: least significant bit first
        keys, payload = _split_low_bit(keys, payload, b)
    _, idx = plain.topk(x.astype(np.float32)[None, :], n)
    assert np.array_equal(idx[0], payload)


# --------------------------------------------------------------------------
# Find It in log n (stream compaction task 4): lower bound over the running count
# --------------------------------------------------------------------------

def _lower_bound_gather(flags, slots):
    running = np.cumsum(flags)            # offsets[i] + flags[i]
    out = []
    for j in range(slots):
        lo, hi = 0, flags.size
        while lo < hi:
            mid = (lo + hi) // 2
            if running[mid] > j:
                hi = mid
            else:
                lo = mid + 1
        out.append(lo)
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lower_bound_resolves_boundary_ties(seed):
    x = workloads.make("ties1000", 1, 50000, seed)[0]
    k = 777
    v, i = plain.topk(x[None, :], k)
    vk = v[0][-1]
    above = int(np.count_nonzero(x > vk))
    need = k - above
    tied = _lower_bound_gather((x == vk).astype(np.int64), need)
    assert np.array_equal(np.sort(i[0][above:]), np.asarray(tied))
    assert np.array_equal(i[0][above:], np.asarray(tied))   # ascending index order inside the tie


# --------------------------------------------------------------------------
# Prof-K parameters (section 4 and Algorithm 1)
# --------------------------------------------------------------------------

def test_printed_z_and_clamps():
    g = _golden("prof_k_printed_numbers.txt")
    z, tol = g["z_at_eps_1e-3"]
    assert abs(params.z_total(1e-3) - z) <= tol
    assert params.S_MIN_DEFAULT == int(g["s_min"][0]) and params.S_MAX_DEFAULT == int(g["s_max"][0])
    assert int(g["sae_n"][0]) == 4096 * 12288 and int(g["sae_k"][0]) == 4096 * 32


def test_corollary4_equals_eqs_8_and_11():
    """M from Eq. 12 equals ceil(c*k) with c from Eqs. 8 and 11 (z_A = z_B = z/2)."""
    for n, k, eps in [(1 << 28, 1024, 1e-6), (1 << 26, 10000, 1e-3), (10 ** 9, 100, 1e-2)]:
        s, _, m = params.alg1(n, k, eps)
        za = zb = params.z_total(eps) / 2
        alpha, f = k / n, 1 - s / n
        c0 = 1 + za / math.sqrt(s) * math.sqrt((1 - alpha) / alpha * f)
        c = c0 + zb * math.sqrt((1 - alpha) * f / (alpha * s))
        near_integer = abs(c * k - round(c * k)) < 1e-7 * c * k
        assert m == math.ceil(c * k) or near_integer


def test_theorem5_minimises_the_cost_model():
    """S* of Eq. 14 is the minimiser of C = tau_A S + tau_B M(S) log k (numerical search)."""
    for n, k, eps in [(10 ** 9, 100, 1e-3), (1 << 28, 1024, 1e-6), (1 << 30, 1 << 12, 1e-3)]:
        z = params.z_total(eps)
        log_k = math.log2(k)

        def cost(s):
            return s + (k + z * math.sqrt(k * (n - k) / s)) * log_k

        grid = np.exp(np.linspace(math.log(10.0), math.log(1e7), 200001))
        best = grid[np.argmin([cost(s) for s in grid])]
        assert abs(best - params.s_star(n, k, eps)) / best < 1e-3


def test_sample_size_scaling_and_printed_example():
    g = _golden("prof_k_printed_numbers.txt")
    value, tol = g["s_star_n1e9_k100"]
    # the printed S* ~ 4,600 at N = 1e9, k = 100 is the (kN)^(1/3) scaling statement
    assert abs((100 * 1e9) ** (1 / 3) - value) / value < tol
    # S* grows as (kN)^(1/3): multiplying N by 8 at fixed k doubles it (k << N)
    r = params.s_star(8 * 10 ** 12, 64, 1e-3) / params.s_star(10 ** 12, 64, 1e-3)
    assert abs(r - 2.0) < 1e-6
    assert params.sample_size(1 << 20, 10, 1e-3) == params.S_MIN_DEFAULT        # clamp from below
    assert params.sample_size(1 << 34, 1 << 18, 1e-3) == params.S_MAX_DEFAULT   # clamp from above


def test_lemma1_by_enumeration():
    """Eq. 1 and Eq. 2 against every without-replacement sample of a tiny population."""
    n, s = 9, 4
    for t in range(1, s + 1):
        counts = {}
        for subset in itertools.combinations(range(1, n + 1), s):   # ranks, 1 = largest
            r = sorted(subset)[t - 1]
            counts[r] = counts.get(r, 0) + 1
        total = math.comb(n, s)
        mean = sum(r * c for r, c in counts.items()) / total
        var = sum((r - mean) ** 2 * c for r, c in counts.items()) / total
        for r in range(t, n - s + t + 1):
            assert abs(counts.get(r, 0) / total - params.negative_hypergeometric_pmf(n, s, t, r)) < 1e-12
        em, ev = params.negative_hypergeometric_moments(n, s, t)
        assert abs(mean - em) < 1e-12 and abs(var - ev) < 1e-12


@pytest.mark.parametrize("n,s", [(7, 3), (6, 4)])
def test_exact_tails_by_enumeration(n, s):
    """With-replacement sampling: enumerate all N^S draw sequences and compare P[R<k], P[R>M]."""
    seqs = list(itertools.product(range(1, n + 1), repeat=s))      # ranks drawn, 1 = largest
    for k in range(1, n + 1):
        for t in range(1, s + 1):
            rs = [sorted(q)[t - 1] for q in seqs]                  # R = rank of the t-th best draw
            p_fail = sum(r < k for r in rs) / len(seqs)
            assert abs(p_fail - params.p_recall_fail(n, k, s, t)) < 1e-12
            for m in range(k, n + 1):
                p_over = sum(r > m for r in rs) / len(seqs)
                assert abs(p_over - params.p_overflow(n, s, t, m)) < 1e-12


@pytest.mark.parametrize("n,k,eps", [(1 << 28, 1024, 1e-6), (1 << 26, 10000, 1e-3),
                                     (1 << 28, 131072, 1e-3), (1 << 22, 32, 1e-2), (1 << 24, 1, 1e-3)])
def test_exact_rule_is_minimal_and_meets_budget(n, k, eps):
    s, t, m = params.exact(n, k, eps)
    assert params.p_recall_fail(n, k, s, t) <= eps / 2
    assert t == 1 or params.p_recall_fail(n, k, s, t - 1) > eps / 2
    assert params.p_overflow(n, s, t, m) <= eps / 2
    assert m == k or params.p_overflow(n, s, t, m - 1) > eps / 2
    assert params.p_recall_fail(n, k, s, t) + params.p_overflow(n, s, t, m) <= eps   # Theorem 3


def test_alg1_sparse_rule_misses_more_than_its_budget():
    """The printed t = 1 rule fails recall far above eps in the sparse regime (reading of Alg. 1 line 8)."""
    n, k, eps = 1 << 28, 1024, 1e-6
    s, t, _ = params.alg1(n, k, eps)
    assert t == 1
    assert params.p_recall_fail(n, k, s, t) > 0.1


# --------------------------------------------------------------------------
# Philox4x32-10 and the sampler
# --------------------------------------------------------------------------

def test_philox_known_answers():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for row in rows:
        words = [int(w, 16) for w in row]
        out = philox.philox4x32_10(*words[:6])
        assert [int(o) for o in out] == words[6:]


def test_sampler_range_and_uniformity():
    n, s = 1000003, 200000
    pos = philox.sample_positions(n, s, seed=0x1234, counter=5, row=2)
    assert pos.min() >= 0 and pos.max() < n
    hist = np.bincount(pos * 64 // n, minlength=64)
    chi2 = float(((hist - s / 64) ** 2 / (s / 64)).sum())
    assert chi2 < 120            # 63 degrees of freedom; p ~ 1e-5 at 120
    other = philox.sample_positions(n, s, seed=0x1234, counter=6, row=2)
    assert not np.array_equal(pos, other)


def test_sampled_threshold_rank_follows_the_binomial_law():
    """Monte Carlo of stages 1-3 with the oracle's sampler: P[R < k] and E[R] match the exact law."""
    n, k, s, t = 1 << 14, 40, 256, 2
    x = np.random.default_rng(9).permutation(n).astype(np.float32)  # ranks only matter
    runs = 600
    rs = []
    for c in range(runs):
        pos = philox.sample_positions(n, s, seed=77, counter=c)
        piv = plain.sample_order_stat(x, pos, t)
        rs.append(plain.count_at_or_above(x, piv))
    rs = np.asarray(rs)
    p = params.p_recall_fail(n, k, s, t)
    sd = math.sqrt(p * (1 - p) / runs)
    assert abs(np.mean(rs < k) - p) < 4 * sd + 1e-3
    # E[R] under with-replacement draws: sum_r P[R > r] = sum_r P[Bin(S, r/N) <= t-1]
    from scipy import stats
    r_grid = np.arange(0, n)
    mean = float(stats.binom.cdf(t - 1, s, r_grid / n).sum())
    assert abs(rs.mean() - mean) < 4 * rs.std() / math.sqrt(runs)


# --------------------------------------------------------------------------
# The survivor count R and the sampled order statistic (section 3, stages 2-3)
# --------------------------------------------------------------------------

def _ranks_with_reading(x, largest=True):
    """Brute-force 0-based ranks under the special-value reading: NaN ranks
    above every number (below, when smallest first), all NaNs are equal,
    -0 == +0; an equal element outranks you only when its index is lower
    (Rank by Counting, Goal).  Written independently of the C++ comparators."""
    n = x.size
    nan = np.isnan(x)
    idx = np.arange(n)
    ranks = np.empty(n, dtype=np.int64)
    for i in range(n):
        if largest:
            better = (nan & ~nan[i]) | (~nan & ~nan[i] & (x > x[i]))
        else:
            better = (~nan & nan[i]) | (~nan & ~nan[i] & (x < x[i]))
        equal = (nan & nan[i]) | (~nan & ~nan[i] & (x == x[i]))
        ranks[i] = np.count_nonzero(better) + np.count_nonzero(equal & (idx < i))
    return ranks


def _tied_specials(seed, n):
    rng = np.random.default_rng(seed)
    x = rng.integers(0, 6, size=n).astype(np.float32)          # six values: massive ties
    pick = rng.integers(0, 10, size=n)
    x[pick == 0] = np.float32(np.nan)
    x[pick == 1] = np.float32(-0.0)
    x[pick == 2] = np.float32(0.0)
    x[pick == 3] = np.float32(np.inf)
    x[pick == 4] = np.float32(-np.inf)
    return x


@pytest.mark.parametrize("largest", [True, False])
@pytest.mark.parametrize("seed", [0, 1])
def test_count_at_or_above_is_the_pivots_rank_plus_one(seed, largest):
    """R for a threshold element = the elements ranking at or above it, the pivot
    included: rank(pivot) + 1.  Ties at the pivot's value split by index, so an
    excluded pivot or a reversed tie order fails here."""
    x = _tied_specials(seed, 700)
    ranks = _ranks_with_reading(x, largest)
    assert np.array_equal(np.sort(ranks), np.arange(x.size))
    for pivot in range(0, x.size, 7):
        assert plain.count_at_or_above(x, pivot, largest=largest) == ranks[pivot] + 1, pivot
    # bf16 carries the same reading (widened exactly)
    h = workloads.f32_to_bf16_bits(x)
    h[np.isnan(x)] = np.uint16(0x7FC0)
    hr = _ranks_with_reading(workloads.bf16_bits_to_f32(h), largest)
    for pivot in range(3, x.size, 11):
        assert plain.count_at_or_above(h, pivot, largest=largest) == hr[pivot] + 1, pivot


@pytest.mark.parametrize("largest", [True, False])
def test_sample_order_stat_counts_repeated_draws(largest):
    """The t-th best of the sampled positions, a position drawn twice taking two
    places: an independent sort of the drawn (rank, draw) pairs."""
    x = _tied_specials(2, 60)
    ranks = _ranks_with_reading(x, largest)
    rng = np.random.default_rng(3)
    for trial in range(20):
        draws = rng.integers(0, x.size, size=150)              # 150 draws of 60 positions
        order = sorted(range(draws.size), key=lambda j: (ranks[draws[j]], j))
        for t in (1, 2, 3, 37, 75, 149, 150):
            want = int(draws[order[t - 1]])
            assert plain.sample_order_stat(x, draws, t, largest=largest) == want, (trial, t)
    # a position drawn t times in a row is also the t-th best when it is the best
    best = int(np.argmin(ranks))
    draws = np.array([best] * 4 + list(rng.integers(0, x.size, size=10)), dtype=np.int64)
    for t in (1, 2, 3, 4):
        assert plain.sample_order_stat(x, draws, t, largest=largest) == best


# --------------------------------------------------------------------------
# Algorithm 1, dense regime: t is the smallest rank meeting Eq. 5
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n,k,eps", [(1 << 26, 10000, 1e-3), (1 << 28, 131072, 1e-3),
                                     (1 << 24, 4096, 1e-2), (1 << 22, 100000, 1e-4),
                                     (10 ** 8, 50000, 1e-6)])
def test_alg1_t_is_the_smallest_rank_meeting_eq5(n, k, eps):
    """With q = t/S and the substitution the text makes before Eq. 6
    (q(1-q) ~ alpha(1-alpha)), Eq. 5 bounds P(R < k) by
    Phi(-(q - alpha) / sqrt(alpha(1-alpha) f / S)) with eps_A = eps/2.
    Algorithm 1's t (dense branch) must satisfy it and t - 1 must not.
    The normal CDF here is scipy.stats.norm, not the quantile the oracle uses."""
    from scipy import stats
    s, t, _ = params.alg1(n, k, eps)
    alpha, f = k / n, 1.0 - s / n
    assert alpha * s >= -math.log(eps / 2.0)                  # the dense branch applies
    sd = math.sqrt(alpha * (1.0 - alpha) * f / s)

    def p_fail(tt):
        return float(stats.norm.cdf(-((tt / s) - alpha) / sd))

    assert t > 1
    assert p_fail(t) <= eps / 2.0
    assert p_fail(t - 1) > eps / 2.0


@pytest.mark.parametrize("threads", [1, 3, 8])
@pytest.mark.parametrize("largest", [True, False])
def test_parallel_cpu_baseline_equals_the_oracle(threads, largest):
    """The multi-threaded CPU baseline returns exactly the oracle's answer (ties
    straddling chunk borders, special values, per-row and global)."""
    x = _tied_specials(4, 5000).reshape(5, 1000)
    for k in (1, 7, 400, 1000):
        v, i = plain.topk(x, k, largest=largest)
        vp, ip = plain.topk_parallel(x, k, largest=largest, threads=threads)
        assert np.array_equal(ip, i) and np.array_equal(vp.view(np.uint32), v.view(np.uint32))
    v, i = plain.topk(x, 2500, largest=largest, global_=True)
    vp, ip = plain.topk_parallel(x, 2500, largest=largest, global_=True, threads=threads)
    assert np.array_equal(ip, i) and np.array_equal(vp.view(np.uint32), v.view(np.uint32))
    h = workloads.make("relu_normal_bf16", 4, 3000, 6)
    v, i = plain.topk(h, 900, largest=largest, global_=True)
    vp, ip = plain.topk_parallel(h, 900, largest=largest, global_=True, threads=threads)
    assert np.array_equal(ip, i) and np.array_equal(vp, v)
