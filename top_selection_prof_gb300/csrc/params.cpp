// Host-side parameter selection for Prof-K: the sample size S, threshold rank t
// and buffer capacity M ("Prof-K: Probabilistic One-Pass Filtering for
// Efficient Top-k Selection", section 4 and Algorithm 1).
//
// S always follows Algorithm 1: S* of Eq. 14 with log base 2 and the cost
// ratio tau_B/tau_A, rounded to nearest and clamped to [S_min, S_max].
//
// Rule 1 (Algorithm 1 as printed): z = 2 Phi^{-1}(1 - eps/2); t from Eq. 6
// with z/2; M from Eq. 12 (Corollary 4); t = 1 when alpha*S < -ln(eps/2).
//
// Rule 0 (default, exact tails): the sampler draws S positions independently
// and uniformly.  Counting as in Lemma 1's proof, R < k happens exactly when at
// least t draws fall among the top k-1 ranks, and R > M exactly when fewer
// than t draws fall among the top M ranks; those counts are Binomial(S,
// (k-1)/N) and Binomial(S, M/N).  t is the smallest rank whose recall-failure
// tail is <= eps/2 and M the smallest capacity whose overflow tail is <= eps/2,
// so the two failure modes together stay within eps (Theorem 3).
//
// Numerics: Phi^{-1} solves 0.5*erfc(x/sqrt 2) = q by safeguarded Newton steps
// on log Q(x); binomial tails sum pmf terms from the tail inwards using
// lgamma/log1p for the first term and the term ratio for the rest.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "engine.h"

namespace tk {

namespace {
constexpr double kSqrt2 = 1.4142135623730950488;
constexpr double kInvSqrt2Pi = 0.39894228040143267794;

double upper_q(double x) { return 0.5 * std::erfc(x / kSqrt2); }

double log_pmf(int64_t s, double p, int64_t j) {
  return std::lgamma(static_cast<double>(s) + 1.0) - std::lgamma(static_cast<double>(j) + 1.0) -
         std::lgamma(static_cast<double>(s - j) + 1.0) + static_cast<double>(j) * std::log(p) +
         static_cast<double>(s - j) * std::log1p(-p);
}

// Sum of pmf(j) for j = t, t+1, ..., s (terms shrink when t > mean).
double sum_up(int64_t s, double p, int64_t t) {
  double term = std::exp(log_pmf(s, p, t));
  double sum = 0.0;
  const double ratio_scale = p / (1.0 - p);
  for (int64_t j = t; j <= s; ++j) {
    sum += term;
    if (term <= sum * 1e-18 && static_cast<double>(j) > static_cast<double>(s) * p) break;
    term *= static_cast<double>(s - j) / static_cast<double>(j + 1) * ratio_scale;
  }
  return sum;
}

// Sum of pmf(j) for j = t, t-1, ..., 0 (terms shrink when t < mean).
double sum_down(int64_t s, double p, int64_t t) {
  double term = std::exp(log_pmf(s, p, t));
  double sum = 0.0;
  const double ratio_scale = (1.0 - p) / p;
  for (int64_t j = t; j >= 0; --j) {
    sum += term;
    if (term <= sum * 1e-18 && static_cast<double>(j) < static_cast<double>(s) * p) break;
    term *= static_cast<double>(j) / static_cast<double>(s - j + 1) * ratio_scale;
  }
  return sum;
}
}  // namespace

double inv_normal_upper(double q) {
  if (!(q > 0.0 && q < 1.0)) return std::nan("");
  double lo = -40.0, hi = 40.0;
  double x = (q < 0.5) ? std::sqrt(-2.0 * std::log(q)) : -std::sqrt(-2.0 * std::log1p(-q));
  for (int it = 0; it < 200; ++it) {
    const double qx = upper_q(x);
    if (qx > q) lo = x; else hi = x;
    const double g = std::log(qx) - std::log(q);
    const double dg = -kInvSqrt2Pi * std::exp(-0.5 * x * x) / qx;
    double xn = x - g / dg;
    if (!(xn > lo && xn < hi) || !std::isfinite(xn)) xn = 0.5 * (lo + hi);
    if (std::fabs(xn - x) <= 1e-15 * std::fmax(1.0, std::fabs(x))) return xn;
    x = xn;
  }
  return x;
}

double binom_upper_tail(int64_t s, double p, int64_t t) {
  if (t <= 0) return 1.0;
  if (t > s) return 0.0;
  if (p <= 0.0) return 0.0;
  if (p >= 1.0) return 1.0;
  const double mean = static_cast<double>(s) * p;
  if (static_cast<double>(t) > mean) return sum_up(s, p, t);
  return 1.0 - sum_down(s, p, t - 1);
}

double binom_lower_tail(int64_t s, double p, int64_t t) {
  if (t < 0) return 0.0;
  if (t >= s) return 1.0;
  if (p <= 0.0) return 1.0;
  if (p >= 1.0) return 0.0;
  const double mean = static_cast<double>(s) * p;
  if (static_cast<double>(t) < mean) return sum_down(s, p, t);
  return 1.0 - sum_up(s, p, t + 1);
}

int64_t alg1_sample_size(int64_t n, int64_t k, double eps, const ParamRule& pr) {
  const double z = 2.0 * inv_normal_upper(eps / 2.0);
  const double kd = static_cast<double>(k), nd = static_cast<double>(n);
  const double s_star = std::pow(z * pr.cost_ratio * std::log2(kd) / 2.0, 2.0 / 3.0) *
                        std::pow(kd * (nd - kd), 1.0 / 3.0);
  double s = std::floor(s_star + 0.5);
  if (s < static_cast<double>(pr.s_min)) s = static_cast<double>(pr.s_min);
  if (s > static_cast<double>(pr.s_max)) s = static_cast<double>(pr.s_max);
  return static_cast<int64_t>(s);
}

int64_t recall_rank(int64_t k, double recall) {
  if (!(recall > 0.0 && recall < 1.0)) return k;
  const int64_t kt = static_cast<int64_t>(std::ceil(recall * static_cast<double>(k) - 1e-9));
  return kt < 1 ? 1 : (kt > k ? k : kt);
}

bool choose_params(int64_t n, int64_t k, double eps, const ParamRule& pr, int64_t* S_out,
                   int64_t* t_out, int64_t* M_out) {
  const int64_t S = alg1_sample_size(n, k, eps, pr);
  const double nd = static_cast<double>(n), kd = static_cast<double>(k);
  // relaxed recall: the threshold rank targets rank ceil(recall * k) instead
  // of k; the buffer still has to hold k
  const double kt = static_cast<double>(recall_rank(k, pr.recall));
  int64_t t = 0, M = 0;
  if (pr.rule == 1) {
    const double z = 2.0 * inv_normal_upper(eps / 2.0);
    const double alpha = kt / nd;
    const double Sd = static_cast<double>(S);
    const double f = 1.0 - Sd / nd;
    double tt = std::ceil(Sd * alpha + (z / 2.0) * std::sqrt(Sd * alpha * (1.0 - alpha) * f));
    t = tt < 1.0 ? 1 : static_cast<int64_t>(tt);
    M = static_cast<int64_t>(std::ceil(kd + z * std::sqrt(kd * (nd - kd) / Sd * f)));
    if (alpha * Sd < -std::log(eps / 2.0)) t = 1;
  } else {
    const double half = eps / 2.0;
    const double p = (kt - 1.0) / nd;
    // smallest t in [1, S] with P[Bin(S, p) >= t] <= eps/2
    if (binom_upper_tail(S, p, S) > half) return false;
    int64_t lo = 0, hi = S;  // invariant: tail(hi) <= half, tail(lo) > half or lo == 0
    while (hi - lo > 1) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (binom_upper_tail(S, p, mid) <= half) hi = mid; else lo = mid;
    }
    t = hi;
    // smallest M in [k, n] with P[Bin(S, M/n) <= t-1] <= eps/2
    if (binom_lower_tail(S, kd / nd, t - 1) <= half) {
      M = k;
    } else {
      int64_t mlo = k, mhi = n;
      while (mhi - mlo > 1) {
        const int64_t mid = mlo + (mhi - mlo) / 2;
        if (binom_lower_tail(S, static_cast<double>(mid) / nd, t - 1) <= half) mhi = mid;
        else mlo = mid;
      }
      M = mhi;
    }
  }
  if (M > n) M = n;
  if (M < k) M = k;
  *S_out = S;
  *t_out = t;
  *M_out = M;
  return true;
}

double plan_miss_probability(int64_t n, int64_t k, int64_t S, int64_t t, int64_t M) {
  const double nd = static_cast<double>(n);
  const double pm = M >= n ? 1.0 : static_cast<double>(M) / nd;
  return binom_upper_tail(S, (static_cast<double>(k) - 1.0) / nd, t) + binom_lower_tail(S, pm, t - 1);
}

bool miss_in_refine(const Problem& p, int64_t k, int64_t t, int64_t S, double p_miss) {
  constexpr double kLaunchUs = 4.0;       // a fallback launch that exits at once
  // ~12 GB/s per SM of the cluster over its passes (a miss of the 1 GiB f32
  // row in a 2-CTA cluster measured ~135 ms)
  constexpr double kSmBytesPerUs = 1.2e4;
  const double row_bytes = static_cast<double>(p.len) * (p.dtype == 0 ? 4.0 : 2.0);  // f32 : bf16
  int64_t g = (k + 11775) / 11776;        // the refinement cluster's size, at least
  const double er = static_cast<double>(t) * (static_cast<double>(p.len) + 1.0) / (static_cast<double>(S) + 1.0);
  const int64_t g_cache = static_cast<int64_t>(1.5 * er / 23552.0) + 1;
  if (g_cache > g) g = g_cache;
  if (g > 16) g = 16;
  const double miss_us = 3.0 * row_bytes / (static_cast<double>(g) * kSmBytesPerUs);
  // probability that some selection of the call misses
  const double p_any = std::min(1.0, p_miss * static_cast<double>(p.nsel));
  return p_any * miss_us < kLaunchUs;
}

bool pdl_edge(unsigned bit) {
  // Programmatic dependent launch per pipeline edge (bits: 1 threshold
  // select, 2 filter, 4 fallback, 8 refinement and bin sort, 16 grid
  // refinement).  On by default for the edges where it shortens the
  // pipeline (1, 2, 8; the filter edge only where the preceding grid leaves
  // the filter's SMs free, see overlap_sms).  The grid refinement's edge
  // gains nothing: a cooperative grid measured to start ~3 us after the
  // filter ends either way.  TOPK_PDL_MASK overrides (0 turns it off).
  static const unsigned mask = [] {
    const char* m = std::getenv("TOPK_PDL_MASK");
    return m ? static_cast<unsigned>(std::strtoul(m, nullptr, 0)) : (kPdlTau | kPdlFilter | kPdlRefine);
  }();
  return (mask & bit) != 0;
}

}  // namespace tk
