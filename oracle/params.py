"""Prof-K parameter selection (S, t, M).  TEST INFRASTRUCTURE ONLY.

Source: "Prof-K: Probabilistic One-Pass Filtering for Efficient Top-k
Selection", section 4 (Lemma 1, Eqs. 5-12, Theorem 5 / Eq. 14, the practical
clamp of S) and Algorithm 1 (adaptive parameter selection).

Two rules are written out:

* ``alg1`` -- Algorithm 1 exactly as printed: z = 2 * Phi^{-1}(1 - eps/2),
  S* from Eq. 14 with log base 2 and the cost ratio, S rounded to nearest and
  clamped to [S_min, S_max], f = 1 - S/N, t from Eq. 6 with z/2, M from
  Eq. 12 (Corollary 4), and t = 1 when alpha*S < -ln(eps/2).

* ``exact`` (the engine's default) -- the same S, with t and M chosen from the
  exact tails of the sampling law instead of the normal approximation.  The
  sampler draws S positions independently and uniformly (with replacement).
  Counting as in the proof of Lemma 1: recall fails (R < k) exactly when at
  least t draws land among the top k-1 ranks, and the buffer overflows
  (R > M) exactly when fewer than t draws land among the top M ranks.  These
  counts are Binomial(S, (k-1)/N) and Binomial(S, M/N), so
      t = min{ t >= 1 : P[Bin(S, (k-1)/N) >= t] <= eps/2 }
      M = min{ M >= k : P[Bin(S, M/N) <= t-1] <= eps/2 }
  which meets Theorem 3's total budget eps = eps_A + eps_B with
  eps_A = eps_B = eps/2, without the Gaussian step.

The library routines used as steps are scipy.special.ndtri (Phi^{-1}) and
scipy.stats.binom (binomial tails).  Pinned by: z ~ 6.58 at eps = 1e-3
(Algorithm 1's own annotation), Corollary 4 == Eqs. 8/11 substituted, the
(kN)^{1/3} scaling of Eq. 14, and brute-force enumeration of every sample on
tiny N (tests/test_oracle_pins.py).
"""
from __future__ import annotations

import math

import numpy as np
from scipy import special, stats

S_MIN_DEFAULT = 32768       # section 4, "Optimal Sample Size": S_min = 32768
S_MAX_DEFAULT = 131072      # same passage: S_max = 2^17
COST_RATIO_DEFAULT = 1.0    # tau_B / tau_A, default 1 (same passage)


def z_total(eps: float) -> float:
    """Algorithm 1, line 1: z = Phi^{-1}(1-eps/2) + Phi^{-1}(1-eps/2)."""
    zh = float(special.ndtri(1.0 - eps / 2.0))
    return zh + zh


def s_star(n: int, k: int, eps: float, cost_ratio: float = COST_RATIO_DEFAULT) -> float:
    """Eq. 14 as Algorithm 1 writes it (log base 2, cost ratio tau_B/tau_A)."""
    z = z_total(eps)
    return (z * cost_ratio * math.log2(k) / 2.0) ** (2.0 / 3.0) * (k * (n - k)) ** (1.0 / 3.0)


def sample_size(n: int, k: int, eps: float, s_min: int = S_MIN_DEFAULT, s_max: int = S_MAX_DEFAULT,
                cost_ratio: float = COST_RATIO_DEFAULT) -> int:
    """Algorithm 1: S = min(S_max, max(S_min, round(S*)))."""
    return int(min(s_max, max(s_min, int(math.floor(s_star(n, k, eps, cost_ratio) + 0.5)))))


def alg1(n: int, k: int, eps: float, s_min: int = S_MIN_DEFAULT, s_max: int = S_MAX_DEFAULT,
         cost_ratio: float = COST_RATIO_DEFAULT):
    """Algorithm 1 verbatim.  Returns (S, t, M)."""
    z = z_total(eps)
    alpha = k / n
    s = sample_size(n, k, eps, s_min, s_max, cost_ratio)
    f = 1.0 - s / n
    t = max(1, math.ceil(s * alpha + (z / 2.0) * math.sqrt(s * alpha * (1.0 - alpha) * f)))
    m = math.ceil(k + z * math.sqrt(k * (n - k) / s * f))
    if alpha * s < -math.log(eps / 2.0):
        t = 1
    return s, t, m


def p_recall_fail(n: int, k: int, s: int, t: int) -> float:
    """P[R < k] for the with-replacement sampler: P[Bin(S, (k-1)/N) >= t]."""
    return float(stats.binom.sf(t - 1, s, (k - 1) / n))


def p_overflow(n: int, s: int, t: int, m: int) -> float:
    """P[R > M] for the with-replacement sampler: P[Bin(S, M/N) <= t-1]."""
    return float(stats.binom.cdf(t - 1, s, min(m, n) / n))


def exact_t(n: int, k: int, s: int, eps: float) -> int:
    """Smallest t >= 1 with P[Bin(S, (k-1)/N) >= t] <= eps/2 (0 if none <= S)."""
    ts = np.arange(1, s + 1)
    tails = stats.binom.sf(ts - 1, s, (k - 1) / n)
    ok = np.nonzero(tails <= eps / 2.0)[0]
    return int(ts[ok[0]]) if ok.size else 0


def exact_m(n: int, k: int, s: int, t: int, eps: float) -> int:
    """Smallest M in [k, N] with P[Bin(S, M/N) <= t-1] <= eps/2 (bisection; monotone in M)."""
    lo, hi = k, n
    if p_overflow(n, s, t, lo) <= eps / 2.0:
        return lo
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if p_overflow(n, s, t, mid) <= eps / 2.0:
            hi = mid
        else:
            lo = mid
    return hi


def exact(n: int, k: int, eps: float, s_min: int = S_MIN_DEFAULT, s_max: int = S_MAX_DEFAULT,
          cost_ratio: float = COST_RATIO_DEFAULT):
    """Exact-tail rule (engine default).  Returns (S, t, M); t == 0 means no valid t."""
    s = sample_size(n, k, eps, s_min, s_max, cost_ratio)
    t = exact_t(n, k, s, eps)
    if t == 0:
        return s, 0, n
    return s, t, exact_m(n, k, s, t, eps)


def negative_hypergeometric_pmf(n: int, s: int, t: int, r: int) -> float:
    """Lemma 1, Eq. 1: P(R = r) for the t-th largest of S drawn without replacement."""
    return math.comb(r - 1, t - 1) * math.comb(n - r, s - t) / math.comb(n, s)


def negative_hypergeometric_moments(n: int, s: int, t: int):
    """Lemma 1, Eq. 2: (E[R], Var[R])."""
    mean = (n + 1) / (s + 1) * t
    var = t * (s - t + 1) * (n + 1) * (n - s) / ((s + 1) ** 2 * (s + 2))
    return mean, var


def recall_rank(k: int, recall: float) -> int:
    """The rank the threshold targets under relaxed recall: ceil(recall * k) (k when exact)."""
    if not 0.0 < recall < 1.0:
        return k
    return max(1, min(k, math.ceil(recall * k - 1e-9)))


def exact_relaxed(n: int, k: int, eps: float, recall: float, s_min: int = S_MIN_DEFAULT,
                  s_max: int = S_MAX_DEFAULT, cost_ratio: float = COST_RATIO_DEFAULT):
    """Relaxed recall (Prof-K paper, abstract: recovering e.g. 95% of the true
    top-k): the same S, t chosen so that fewer than ceil(recall*k) survivors
    occur with probability <= eps/2, and M so that the buffer (which must hold
    k) overflows with probability <= eps/2.  Returns (S, t, M)."""
    s = sample_size(n, k, eps, s_min, s_max, cost_ratio)
    t = exact_t(n, recall_rank(k, recall), s, eps)
    if t == 0:
        return s, 0, n
    return s, t, exact_m(n, k, s, t, eps)
