/*
 * topk.h -- C ABI of the GB300 Prof-K top-k selection engine (libtopk_gb300.so).
 *
 * The method is Prof-K ("Prof-K: Probabilistic One-Pass Filtering for
 * Efficient Top-k Selection", sections 3-4 and Algorithm 1): draw S uniform
 * positions, take the t-th largest sampled element as a threshold tau, stream
 * the input once keeping every element that ranks at or above tau in a buffer
 * of capacity M, then select the exact top-k of the buffer.  When fewer than k
 * elements survive, or more than M do, the engine falls back to an exact
 * selection over the whole input, so every result is exact.
 *
 * Conventions shared by every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller.  x is
 *     row-major and contiguous, rows x n elements of the given dtype.
 *   - out_vals has the dtype of x and holds the input's own bits at the chosen
 *     positions; out_idx is int64.
 *   - Order: each output row lists the k winners by (value descending, index
 *     ascending) -- equal values go to the lower index, as in "Rank by
 *     Counting" (top-k task 1).  With largest == 0 the value order is reversed
 *     (smallest first) and ties still go to the lower index.  NaN ranks above
 *     every number (so it comes last when largest == 0), all NaNs are equal,
 *     -0 equals +0.
 *   - The call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and does no host synchronisation, except that
 *     topk_select_ex synchronises the stream when `stats` is non-NULL.
 *   - The library keeps a per-(device, stream) workspace for the sample, the
 *     threshold, the candidate buffer and counters (and, for one selection
 *     over 16-byte aligned data with k >= 3072, or with 512 <= k < 3072 and
 *     more expected survivors than one refinement block caches, 32 MiB of
 *     bin regions into which the filter places its survivors); it grows on
 *     demand with stream-ordered allocation and is never shrunk.  Calls that
 *     share a stream are ordered; calls on different streams use different
 *     workspaces.
 *   - Errors are returned as topk_status_t codes; nothing is thrown across the
 *     ABI and no message is printed.
 */
#ifndef TOPK_GB300_H
#define TOPK_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { TOPK_F32 = 0, TOPK_BF16 = 1 } topk_dtype_t;

typedef enum {
  TOPK_OK = 0,
  TOPK_EINVAL = -1,        /* bad argument: null pointer, k < 1, k > n, eps outside [0,1), ... */
  TOPK_ENOMEM = -2,        /* workspace allocation failed */
  TOPK_ECUDA = -3,         /* a CUDA runtime call or kernel launch failed */
  TOPK_EUNSUPPORTED = -4,  /* valid request outside the engine's limits (see topk_select) */
  TOPK_ETIMEOUT = -5       /* a bounded device-side wait gave up (with stats, or from topk_last_status) */
} topk_status_t;

/* Parameter rule for (t, M).  Both use Algorithm 1's sample size S.
 *   TOPK_RULE_EXACT (default): t and M from the exact binomial tails of the
 *     with-replacement sampler, eps/2 for recall failure and eps/2 for
 *     overflow (Theorem 3's split without the normal approximation).
 *   TOPK_RULE_ALG1: t and M as Algorithm 1 prints them (Eq. 6, Eq. 12 and
 *     the t = 1 sparse rule).  Results stay exact; only the miss rate differs. */
typedef enum { TOPK_RULE_EXACT = 0, TOPK_RULE_ALG1 = 1 } topk_rule_t;

/* Which pipeline ran (or is forced).
 *   TOPK_PATH_DIRECT: exact radix select straight over each row (small rows, or
 *     when the sample would be at least half the row).
 *   TOPK_PATH_PROFK:  sample -> threshold -> one-pass filter -> exact refine,
 *     with the full-input fallback on a miss.
 *   TOPK_PATH_EXACT:  the full-input radix select of the fallback, used for
 *     large rows when eps == 0. */
typedef enum {
  TOPK_PATH_AUTO = 0,
  TOPK_PATH_DIRECT = 1,
  TOPK_PATH_PROFK = 2,
  TOPK_PATH_EXACT = 3
} topk_path_t;

/* Tuning and test knobs.  Initialise with topk_options_init(). */
typedef struct {
  int64_t s_min;       /* Algorithm 1 S_min (default 32768) */
  int64_t s_max;       /* Algorithm 1 S_max (default 131072) */
  double cost_ratio;   /* tau_B / tau_A of Eq. 13 (default 1); 0 = as measured on this device by
                          topk_autotune (1 before that), which also applies the measured
                          Prof-K / direct crossover to the automatic path choice */
  int rule;            /* topk_rule_t (default TOPK_RULE_EXACT) */
  int path;            /* topk_path_t; TOPK_PATH_AUTO lets the engine choose */
  uint64_t seed;       /* Philox key for the sampler (default fixed) */
  int64_t counter;     /* Philox call counter; -1 = next value of a per-process counter */
  int force_miss;      /* non-zero: every row takes the fallback (fault injection on the host) */
  int64_t m_override;  /* > 0: use this buffer capacity M instead of the rule's */
  int64_t t_override;  /* > 0: use this threshold rank t instead of the rule's */
  /* Optional cudaEvent_t handles (NULL = none) recorded on `stream` at the
   * stage boundaries of the Prof-K path: [0] before the sample kernel, [1]
   * after it, [2] after the threshold selection, [3] after the filter, [4]
   * after the fallback check, [5] after the final selection.  The caller owns
   * the events; they are only recorded, never created or destroyed here. */
  void* events[6];
  /* Non-zero: the caller needs only the set of winners (BatchTopK keeps the
   * K largest activations, in any order: Prof-K paper, section 5).  For
   * selections refined on the grid (k >= 8192, at most 4 selections) the
   * k winners are then written in no particular order and the final sort
   * is skipped; every other path still sorts.  The set, the values and the
   * positions are exact either way.  Default 0. */
  int unsorted;
  /* > 0: limit in nanoseconds of each grid-wide wait of the exact fallback
   * (default 0 = 2 s).  After it the kernel records a timeout, returns, and
   * the call reports TOPK_ETIMEOUT (with stats, or from topk_last_status). */
  int64_t wait_limit_ns;
  /* Testing only (fault injection on the host's request, no GPU fault): when
   * the fallback runs, one of its blocks leaves its first grid-wide wait
   * without arriving, so every other block's bounded wait runs out.  The
   * call's output is then undefined and its status is TOPK_ETIMEOUT; the next
   * call on the stream starts clean.  Default 0. */
  int inject_wait_timeout;
  /* Relaxed recall (Prof-K paper, abstract: "relaxing the recall target (e.g.,
   * recovering 95% of the true top-k values)").  0 (default) or >= 1: exact.
   * In (0, 1): the threshold rank t is chosen for rank ceil(recall * k)
   * instead of k, so that P[fewer than ceil(recall * k) of the true top-k
   * survive] <= eps/2, and fewer than k survivors no longer take the
   * fallback: when R < k, the first R places of the row hold the exact top-R
   * (all of them true top-k elements), sorted as usual, and places R..k-1
   * hold index -1 and the value -inf (+inf when largest == 0).  A buffer
   * overflow (R > M) still takes the exact fallback.  Applies to the Prof-K
   * path; the direct and exact paths return the exact top-k. */
  double recall;
} topk_options_t;

/* Per-call report (row 0 for the per-row fields). */
typedef struct {
  int path;            /* topk_path_t that ran */
  int index_bits;      /* b of the composite key format below */
  int64_t S, t, M;     /* sample size, threshold rank, buffer capacity (0 on the direct path) */
  int64_t R;           /* row 0: elements that passed the filter (before any fallback) */
  int64_t misses;      /* rows whose filter result missed k <= R <= M and took the fallback */
  uint64_t tau;        /* row 0: composite key of the sampled threshold */
  int64_t tau_index;   /* row 0: position of the element tau was taken from */
  uint64_t seed;       /* Philox key and counter the sampler used */
  int64_t counter;
  int cluster;         /* CTAs per thread-block cluster in the final selection */
  int launches;        /* kernels this call launched on the stream */
  int64_t shortfalls;  /* rows that returned fewer than k winners (relaxed recall only) */
} topk_stats_t;

/* Parameters the engine would use for a selection of k out of n (host only). */
typedef struct {
  int path;            /* topk_path_t the automatic choice resolves to */
  int64_t S, t, M;
  double p_recall_fail;  /* P[R < k] (relaxed recall: P[R < ceil(recall*k)]) under the with-replacement sampler */
  double p_overflow;     /* P[R > M] */
} topk_plan_t;

/* Fills *opt with the defaults above. */
void topk_options_init(topk_options_t* opt);

/*
 * Per-row top-k (section 3: "for batched inputs ... applied in parallel to each
 * batch element").  For each of `rows` rows of n elements, writes the k
 * winners to out_vals[r*k + j] and their row-local positions to
 * out_idx[r*k + j].  eps in [0, 1) is the target probability that a row takes
 * the fallback (Theorem 3); eps == 0 selects exactly without sampling.  The
 * result never depends on eps or on the sampler.
 *   Limits: n < 2^31; k <= 188416 (EUNSUPPORTED beyond); rows == 0 is a no-op.
 *   EINVAL: null pointer (with rows > 0), rows < 0, n < 1, k < 1, k > n,
 *           eps outside [0, 1), unknown dtype.
 */
int topk_select(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                double eps, void* out_vals, int64_t* out_idx, void* stream);

/*
 * Batch-global top-k (BatchTopK, section 5: the B x d_dict activations are
 * flattened into one vector of N = B*d_dict and the K = B*k largest are kept).
 * Treats the rows*n elements as one vector: out_vals[j], out_idx_flat[j] for
 * j < k, with flat positions r*n + c.
 *   Limits: rows*n <= 2^32 for F32 and <= 2^48 for BF16; k <= 188416.
 *   EINVAL as topk_select, with k > rows*n in place of k > n.
 */
int topk_select_global(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                       double eps, void* out_vals, int64_t* out_idx_flat, void* stream);

/*
 * topk_select (global == 0) or topk_select_global (global != 0) with options
 * (NULL = defaults) and an optional report.  When stats is non-NULL the call
 * synchronises `stream` before returning and can return TOPK_ETIMEOUT.
 */
int topk_select_ex(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                   double eps, void* out_vals, int64_t* out_idx, void* stream, int global,
                   const topk_options_t* opt, topk_stats_t* stats);

/* Host-only: the path and (S, t, M) the engine uses for one selection of k out
 * of n elements (n = rows*n for the global variant).  Algorithm 1 and the rule
 * in opt (NULL = defaults).  EINVAL on bad arguments. */
int topk_plan(int64_t n, int64_t k, double eps, const topk_options_t* opt, topk_plan_t* plan);

/*
 * Device-side status of the most recent selection issued on `stream` (of the
 * current device) by topk_select, topk_select_global, topk_select_ex or
 * topk_select_noalloc.  Synchronises `stream` first.  Returns TOPK_OK, or
 * TOPK_ETIMEOUT when one of that call's bounded device waits gave up (its
 * output is then undefined), or TOPK_ECUDA when its kernels found their state
 * inconsistent; CUDA errors of the synchronisation itself map to TOPK_ECUDA.
 * The status words are reset by each call, so this reports the last call
 * only.  The short-row direct path (rows of at most 32768 elements, k <= 1024)
 * keeps a status word only when topk_select_ex is given `stats`; otherwise
 * this returns TOPK_OK for it.  Calls without any selection on `stream`
 * return TOPK_OK.
 */
int topk_last_status(void* stream);

/* Measured cost model of this device (Prof-K paper, section 4, "Optimal
 * Sample Size": the ratio tau_B / tau_A "may be estimated by lightweight
 * microbenchmarking"; Figure 3 for the crossover with a direct method). */
typedef struct {
  double tau_a_ns;      /* sampling and threshold: device time per additional sampled element */
  double tau_b_ns;      /* refinement: device time per additional buffered element, per log2 k */
  double cost_ratio;    /* tau_b_ns / tau_a_ns, the ratio of Eq. 13 and 14 */
  int64_t crossover_n;  /* smallest measured row length from which Prof-K beat the direct path
                           at every larger measured length (0: it never did) */
  int64_t crossover_k;  /* the k the crossover was measured at */
} topk_tuning_t;

/*
 * Measures the cost model on the current device with synthetic uniform f32
 * rows through the selection pipeline itself (CUDA events at its stage
 * boundaries, medians of repeated calls): tau_A from the sampling and
 * threshold stage at S = 32768 and S = 131072; tau_B from the refinement at
 * two survivor counts (k = 1024); the crossover from full selections of k out
 * of n = 2^16 ... 2^24 by the direct path and by Prof-K (eps = 1e-3).  Allocates
 * about 256 MiB of device memory for the duration and synchronises `stream`;
 * takes on the order of a second.  The result is kept for the device and used
 * by calls whose options set cost_ratio = 0.  k: the k of the crossover (0 =
 * 1024).  Errors: TOPK_EINVAL for a null `out` or k outside [0, 65536],
 * TOPK_ENOMEM / TOPK_ECUDA.
 */
int topk_autotune(int64_t k, void* stream, topk_tuning_t* out);

/* The measured cost model of the current device (TOPK_EINVAL when topk_autotune
 * has not run on it). */
int topk_tuning(topk_tuning_t* out);

/* Static text for a status code. */
const char* topk_status_str(int status);

/* Library version: major*10000 + minor*100 + patch.  0.2.0 (200) added the
 * `unsorted` field at the end of topk_options_t; 0.3.0 (300) added
 * `wait_limit_ns`, `inject_wait_timeout` and `recall` after it, `shortfalls`
 * at the end of topk_stats_t, topk_last_status, topk_autotune and topk_tuning
 * (cost_ratio = 0 meaning "measured").
 * Fill the struct with topk_options_init from the same version's library. */
int topk_version(void);

/* ------------------------------------------------------------------------
 * Stage entry points: the individual steps of the Prof-K pipeline, for tests
 * and for callers that want the pieces.
 *
 * Composite key format.  Every element is identified by a 64-bit key whose
 * unsigned order is the selection order:
 *     key = (v << b) | (2^b - 1 - i)
 * where i is the element's position in its selection (row-local, or flat for
 * the global variant), b = topk_index_bits(length of the selection), and v is
 * the order-preserving image of the value: for F32 bits u (BF16 likewise on 16
 * bits), NaN -> all ones, -0 -> +0, then v = u | signbit if u is non-negative,
 * else ~u; with largest == 0, v is complemented.  Larger key = better rank;
 * keys are distinct, so "ranks at or above tau" is simply key >= tau.
 * ------------------------------------------------------------------------ */

/* b for a selection over `len` elements: the bits needed for positions 0..len-1 (at least 1). */
int topk_index_bits(int64_t len);

/*
 * Stage 1 (section 3, sampling): for each selection r, draws S positions with
 * Philox4x32-10 -- draw j uses counter (j/2, r, counter_lo, counter_hi) and key
 * (seed_lo, seed_hi); the even draw takes the 64-bit word (w1<<32 | w0), the
 * odd one (w3<<32 | w2); the position is floor(word * len / 2^64) -- and writes
 * the composite keys of the drawn elements to out_keys[r*S + j].
 * global != 0 treats x as one selection of rows*n elements.
 */
int topk_prof_sample(const void* x, int dtype, int64_t rows, int64_t n, int global, int largest,
                     int64_t S, uint64_t seed, int64_t counter, uint64_t* out_keys, void* stream);

/*
 * Stage 3 (section 3, filtering): for each selection r, streams its elements
 * once and appends the composite key of every element with key >= tau[r] to
 * buf[r*M ...]; counts[r] receives the number R of such elements (it keeps
 * counting past M; only the first M found are stored, in no particular order).
 * tau (device, one key per selection) uses the key format above.
 */
int topk_prof_filter(const void* x, int dtype, int64_t rows, int64_t n, int global, int largest,
                     const uint64_t* tau, int64_t M, uint64_t* buf, uint64_t* counts,
                     void* stream);

/*
 * topk_select_noalloc -- the selection of topk_select (global == 0) or
 * topk_select_global (global != 0) without any device allocation.  The paper
 * has no counterpart of this entry point.
 *
 * For callers that cannot allocate while they run: a process whose device
 * memory belongs to another allocator (a framework caching allocator holding
 * nearly all of HBM, where a hidden cudaMalloc can fail or fragment it), or
 * latency-critical loops that cannot take cudaMalloc's implicit device
 * synchronisation.  All scratch comes from one static device array of 8 MiB
 * inside the library, held by every GPU that loads the library until exit.
 * The selection runs through the same kernels and the same choices of path
 * as topk_select; only the scratch memory differs.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the array and it keeps the last call's
 *     contents; the library clears the words that must start at zero.  Calls
 *     that overlap on the GPU (e.g. unordered streams of one device) race on
 *     the array: order them on one stream.
 *   - A request whose scratch would exceed 8 MiB returns TOPK_EUNSUPPORTED
 *     before anything is launched; use topk_select then.  About 2.2 MiB is a
 *     fixed part; the rest grows with the selections: roughly 8 bytes per
 *     sample (S) and per buffer slot (M), 16 bytes per winner (k), and 1 byte
 *     per 1024 input elements.  The 4096 x 65536 bf16 BatchTopK selection
 *     (K = 131072) fits.
 *   - A bounded device wait that gives up is reported by topk_last_status on
 *     the same stream (this call itself does not synchronise).
 * Arguments, outputs, limits and the other error codes are those of
 * topk_select / topk_select_global.
 */
int topk_select_noalloc(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                        double eps, void* out_vals, int64_t* out_idx, int global, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TOPK_GB300_H */
