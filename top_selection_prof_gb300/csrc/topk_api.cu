// C ABI of the engine (declared in include/topk.h): argument checks, the
// choice of path, the per-(device, stream) workspace and the launch sequence.
//
// Prof-K path (section 3 of "Prof-K: Probabilistic One-Pass Filtering for
// Efficient Top-k Selection"), all on the caller's stream, no host sync:
//   sample_kernel    S Philox draws per selection -> composite keys
//   select_kernel    t-th largest sampled key -> tau             (stage 2)
//   filter_kernel    one pass over x, keys >= tau -> buffer, R    (stage 3)
//   select_kernel    exact top-k of the buffer, sorted -> outputs (stage 4);
//                    on a miss (R < k or R > M) it selects from x instead
// The miss decision is made on the device, by the refinement kernel itself
// or by the grid-wide fallback_kernel launched after the filter (chosen per
// call from the plan's miss probability).  The exact path (no Prof-K) runs
// the grid-wide fallback_kernel and then the same sort.  Scratch memory comes
// from a per-(device, stream) pool, or from a fixed block the caller owns
// (select_with_fixed_scratch, used by topk_select_noalloc).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/topk.h"
#include "common.cuh"
#include "engine.h"

namespace tk {
namespace {

constexpr uint64_t kDefaultSeed = 0x243F6A8885A308D3ull;
constexpr int64_t kDirectMaxLen = int64_t(1) << 22;  // larger single rows use the grid-wide exact path
std::atomic<uint64_t> g_counter{0};

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  ScratchCounters counters;  // pick the alternating zero-kept regions (see the layout below)
};
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

// Returns a device block of at least `bytes` for this (device, stream); grows
// with stream-ordered allocation (the old block is released in stream order).
cudaError_t workspace(cudaStream_t st, size_t bytes, void** out, ScratchCounters** counters = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  Workspace& w = g_ws[std::make_pair(dev, st)];
  if (w.bytes < bytes) {
    size_t grow = bytes + bytes / 4;
    grow = (grow + 0xFFFFF) & ~size_t(0xFFFFF);
    void* p = nullptr;
    e = cudaMallocAsync(&p, grow, st);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p, 0, grow, st);
    if (e != cudaSuccess) return e;
    if (w.ptr) cudaFreeAsync(w.ptr, st);
    w.ptr = p;
    w.bytes = grow;
  }
  *out = w.ptr;
  if (counters) *counters = &w.counters;
  return cudaSuccess;
}

// Where a call's scratch comes from: the per-(device, stream) pool above, or
// a fixed block the caller owns (no allocation; too small -> unsupported).
struct ScratchSource {
  const FixedScratch* fixed = nullptr;
};
constexpr cudaError_t kScratchTooSmall = cudaErrorInvalidValue;  // (mapped to TOPK_EUNSUPPORTED)

cudaError_t acquire(const ScratchSource& src, cudaStream_t st, size_t bytes, void** out,
                    ScratchCounters** counters = nullptr) {
  if (!src.fixed) return workspace(st, bytes, out, counters);
  if (bytes > src.fixed->bytes) return kScratchTooSmall;
  *out = src.fixed->base;
  if (counters) *counters = src.fixed->counters;
  return cudaSuccess;
}

// The device status word of the last call on each (device, stream), or null
// when that call kept none; read back by topk_last_status.
std::map<std::pair<int, cudaStream_t>, int*> g_last_status;
void record_status_word(cudaStream_t st, int* word) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  g_last_status[std::make_pair(dev, st)] = word;
}

// Every workspace starts with the same prefix, whatever the call's layout:
// the device header, two halves of the sample histograms, the fused
// threshold grid's control words and its gather buffer, and two copies of
// the grid refinement's control words.  The halves alternate between Prof-K
// calls: a call's sample kernel counts into one and clears the other for the
// next call, so they stay zero between calls without a memset (the block is
// zeroed once when it is allocated); the threshold grid's control words are
// cleared by each call's refinement; the grid refinement's copies alternate
// like the halves.
size_t align_up(size_t v);
constexpr size_t kHistHalfBytes = sizeof(unsigned) * kSampleHistHalfWords;
size_t ws_hist_offset() { return align_up(sizeof(DevHeader)); }
size_t ws_tau_ctl_offset() { return ws_hist_offset() + 2 * kHistHalfBytes; }
size_t ws_tau_gather_offset() { return align_up(ws_tau_ctl_offset() + sizeof(unsigned) * kTauCtlWords); }
size_t ws_refine_ctl_offset() {
  return align_up(ws_tau_gather_offset() + sizeof(uint64_t) * kTauGather * kSampleHistMaxRows);
}
constexpr size_t kRefineCtlCopyBytes = sizeof(unsigned) * kRefineGridMaxSel * kRefineGridCtlWords;
size_t ws_prefix() { return align_up(ws_refine_ctl_offset() + 2 * kRefineCtlCopyBytes); }

size_t align_up(size_t v) { return (v + 255) & ~size_t(255); }


int index_bits(int64_t len) {
  int b = 1;
  while (b < 63 && (int64_t(1) << b) < len) ++b;
  return b;
}

struct Plan {
  int path;
  int64_t S, t, M;
  double p_miss;  // P[R < k] + P[R > M] per selection for (S, t, M) (Prof-K path)
};


bool relaxed_recall(const topk_options_t* o) { return o && o->recall > 0.0 && o->recall < 1.0; }

// The cost model measured by topk_autotune, per device.
std::mutex g_tune_mu;
std::map<int, topk_tuning_t> g_tuning;
bool tuned_model(topk_tuning_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(g_tune_mu);
  auto it = g_tuning.find(dev);
  if (it == g_tuning.end()) return false;
  *out = it->second;
  return true;
}
// cost_ratio == 0 asks for the measured model
bool wants_tuned(const topk_options_t* o) { return o && o->cost_ratio == 0.0; }

ParamRule rule_of(const topk_options_t* o) {
  ParamRule pr;
  if (o) {
    pr.s_min = o->s_min;
    pr.s_max = o->s_max;
    pr.cost_ratio = o->cost_ratio;
    if (wants_tuned(o)) {
      topk_tuning_t tm;
      pr.cost_ratio = tuned_model(&tm) && tm.cost_ratio > 0.0 ? tm.cost_ratio : 1.0;
    }
    pr.rule = o->rule;
    pr.recall = relaxed_recall(o) ? o->recall : 0.0;
  }
  return pr;
}

// Parameters of recent (len, k, eps, rule) requests: the tail searches cost
// tens of microseconds, a lookup well under one.
struct PlanKey {
  int64_t len, k;
  double eps;
  int64_t s_min, s_max;
  double ratio;
  int rule;
  double recall;
  bool operator<(const PlanKey& o) const {
    if (len != o.len) return len < o.len;
    if (k != o.k) return k < o.k;
    if (eps != o.eps) return eps < o.eps;
    if (s_min != o.s_min) return s_min < o.s_min;
    if (s_max != o.s_max) return s_max < o.s_max;
    if (ratio != o.ratio) return ratio < o.ratio;
    if (recall != o.recall) return recall < o.recall;
    return rule < o.rule;
  }
};
struct PlanVal {
  bool ok;
  int64_t S, t, M;
  double p_miss;
};
std::mutex g_plan_mu;
std::map<PlanKey, PlanVal> g_plans;

// Probability that a selection takes the fallback: P[R < k] + P[R > M], or
// only P[R > M] under relaxed recall (fewer survivors are returned as they are).
double fallback_probability(int64_t len, int64_t k, int64_t S, int64_t t, int64_t M, double recall) {
  if (recall > 0.0 && recall < 1.0) {
    const double pm = M >= len ? 1.0 : static_cast<double>(M) / static_cast<double>(len);
    return binom_lower_tail(S, pm, t - 1);
  }
  return plan_miss_probability(len, k, S, t, M);
}

bool cached_params(int64_t len, int64_t k, double eps, const ParamRule& pr, int64_t* S, int64_t* t,
                   int64_t* M, double* p_miss) {
  const PlanKey key{len, k, eps, pr.s_min, pr.s_max, pr.cost_ratio, pr.rule, pr.recall};
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
      *S = it->second.S;
      *t = it->second.t;
      *M = it->second.M;
      *p_miss = it->second.p_miss;
      return it->second.ok;
    }
  }
  PlanVal v{};
  v.ok = choose_params(len, k, eps, pr, &v.S, &v.t, &v.M);
  v.p_miss = v.ok && v.t >= 1 && v.t <= v.S ? fallback_probability(len, k, v.S, v.t, v.M, pr.recall) : 1.0;
  std::lock_guard<std::mutex> lock(g_plan_mu);
  if (g_plans.size() > 4096) g_plans.clear();
  g_plans[key] = v;
  *S = v.S;
  *t = v.t;
  *M = v.M;
  *p_miss = v.p_miss;
  return v.ok;
}

// Path choice for one selection of k out of len (nsel selections).
int make_plan(int64_t len, int64_t k, double eps, int64_t nsel, bool many_rows,
              const topk_options_t* o, Plan* plan) {
  plan->S = plan->t = plan->M = 0;
  plan->p_miss = 0.0;
  const int forced = o ? o->path : TOPK_PATH_AUTO;
  bool profk_ok = false;
  if (eps > 0.0) {
    const ParamRule pr = rule_of(o);
    if (pr.s_min < 1 || pr.s_max < pr.s_min || !(pr.cost_ratio > 0.0) || (pr.rule != 0 && pr.rule != 1) ||
        (o && o->cost_ratio < 0.0))
      return TOPK_EINVAL;
    int64_t S = 0, t = 0, M = 0;
    double p_miss = 1.0;
    if (cached_params(len, k, eps, pr, &S, &t, &M, &p_miss)) {
      const bool overridden = o && (o->t_override > 0 || o->m_override > 0);
      if (o && o->t_override > 0) t = o->t_override;
      if (o && o->m_override > 0) M = o->m_override;
      if (overridden) p_miss = t >= 1 && t <= S ? fallback_probability(len, k, S, t, M, pr.recall) : 1.0;
      plan->S = S;
      plan->t = t;
      plan->M = M;
      plan->p_miss = p_miss;
      profk_ok = t >= 1 && t <= S && 2 * S < len && 2 * M <= len && M >= k && nsel <= 65535;
    }
  }
  // the measured crossover (cost_ratio = 0): the direct path below it
  if (profk_ok && forced == TOPK_PATH_AUTO && wants_tuned(o) && (len <= kDirectMaxLen || many_rows)) {
    topk_tuning_t tm;
    if (tuned_model(&tm) && (tm.crossover_n == 0 || len < tm.crossover_n)) profk_ok = false;
  }
  switch (forced) {
    case TOPK_PATH_AUTO:
      if (profk_ok) plan->path = TOPK_PATH_PROFK;
      else if (len <= kDirectMaxLen || many_rows) plan->path = TOPK_PATH_DIRECT;
      else plan->path = TOPK_PATH_EXACT;
      break;
    case TOPK_PATH_PROFK:
      if (eps <= 0.0 || plan->t < 1 || plan->t > plan->S || plan->M < k || plan->S >= len ||
          nsel > 65535)
        return TOPK_EUNSUPPORTED;
      plan->path = TOPK_PATH_PROFK;
      break;
    case TOPK_PATH_DIRECT:
    case TOPK_PATH_EXACT:
      plan->path = forced;
      break;
    default:
      return TOPK_EINVAL;
  }
  if (plan->path != TOPK_PATH_PROFK) {
    plan->S = plan->t = plan->M = 0;
    plan->p_miss = 0.0;
  }
  return TOPK_OK;
}

int sm_count_host() {
  static int sms = 0;
  if (sms) return sms;
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  sms = v;
  return sms;
}

int check_common(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, double eps,
                 const void* out_vals, const void* out_idx, bool global) {
  if (dtype != TOPK_F32 && dtype != TOPK_BF16) return TOPK_EINVAL;
  if (rows < 0 || n < 1 || k < 1) return TOPK_EINVAL;
  if (!(eps >= 0.0 && eps < 1.0)) return TOPK_EINVAL;
  if (rows == 0) return TOPK_OK;
  if (!x || !out_vals || !out_idx) return TOPK_EINVAL;
  if (!global) {
    if (k > n) return TOPK_EINVAL;
    if (n >= (int64_t(1) << 31)) return TOPK_EUNSUPPORTED;
  } else {
    if (rows > INT64_MAX / n) return TOPK_EUNSUPPORTED;
    const int64_t len = rows * n;
    if (k > len) return TOPK_EINVAL;
    const int64_t lim = dtype == TOPK_F32 ? (int64_t(1) << 32) : (int64_t(1) << 48);
    if (len > lim) return TOPK_EUNSUPPORTED;
  }
  if (k > select_max_k()) return TOPK_EUNSUPPORTED;
  return TOPK_OK;
}

Problem make_problem(const void* x, int dtype, int64_t rows, int64_t n, int largest, bool global) {
  Problem p;
  p.x = x;
  p.dtype = dtype;
  p.nsel = global ? 1 : rows;
  p.len = global ? rows * n : n;
  p.ib = index_bits(p.len);
  p.flip = largest ? 0u : (dtype == TOPK_F32 ? 0xffffffffu : 0xffffu);
  const int vec = dtype == TOPK_F32 ? 4 : 8;
  p.vec_ok = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (p.len % vec == 0);
  return p;
}

int status_of(cudaError_t e) {
  if (e == cudaSuccess) return TOPK_OK;
  if (e == cudaErrorMemoryAllocation) return TOPK_ENOMEM;
  return TOPK_ECUDA;
}

#define TK_TRY(expr)                         \
  do {                                       \
    const cudaError_t _e = (expr);           \
    if (_e != cudaSuccess) return status_of(_e); \
  } while (0)

int run(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest, double eps,
        void* out_vals, int64_t* out_idx, cudaStream_t st, bool global, const topk_options_t* o,
        topk_stats_t* stats, const ScratchSource& src = ScratchSource{}) {
  int rc = check_common(x, dtype, rows, n, k, eps, out_vals, out_idx, global);
  if (rc != TOPK_OK) return rc;
  if (stats) std::memset(stats, 0, sizeof(*stats));
  if (rows == 0) return TOPK_OK;
  const Problem p = make_problem(x, dtype, rows, n, largest, global);
  const bool many = p.nsel >= sm_count_host();
  Plan plan;
  rc = make_plan(p.len, k, eps, p.nsel, many, o, &plan);
  if (rc != TOPK_OK) return rc;
  if (stats) {
    stats->path = plan.path;
    stats->index_bits = p.ib;
    stats->S = plan.S;
    stats->t = plan.t;
    stats->M = plan.M;
  }
  // (a fixed block that is too small: nothing has been launched yet)
  auto scratch_status = [](cudaError_t e) { return e == kScratchTooSmall ? TOPK_EUNSUPPORTED : status_of(e); };

  int cluster = 0;
  if (plan.path == TOPK_PATH_DIRECT && rows_supported(p, k)) {
    // short rows: one block per row, the row in registers; the status word
    // is only kept when the caller asks for statistics
    int* status = nullptr;
    if (stats) {
      void* ws = nullptr;
      const cudaError_t e = acquire(src, st, ws_prefix(), &ws);
      if (e != cudaSuccess) return scratch_status(e);
      status = &static_cast<DevHeader*>(ws)->status;
      TK_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
    }
    TK_TRY(launch_rows(p, k, out_vals, out_idx, status, st));
    record_status_word(st, status);
    if (stats) {
      stats->launches = 1;
      stats->cluster = 1;
      stats->R = p.len;
      int dstat = 0;
      TK_TRY(cudaMemcpyAsync(&dstat, status, sizeof(int), cudaMemcpyDeviceToHost, st));
      TK_TRY(cudaStreamSynchronize(st));
      if (dstat != kDevOk) return dstat == kDevTimeout ? TOPK_ETIMEOUT : TOPK_ECUDA;
    }
    return TOPK_OK;
  }
  if (plan.path == TOPK_PATH_DIRECT) {
    // the status word and the sort's exchange buffer
    void* ws = nullptr;
    const cudaError_t e = acquire(src, st, ws_prefix() + sizeof(uint64_t) * p.nsel * k, &ws);
    if (e != cudaSuccess) return scratch_status(e);
    DevHeader* hdr = static_cast<DevHeader*>(ws);
    TK_TRY(cudaMemsetAsync(&hdr->status, 0, sizeof(int), st));
    SelectJob job{};
    job.keys = nullptr;
    job.r = k;
    job.want_topk = true;
    job.out_vals = out_vals;
    job.out_idx = out_idx;
    job.status = &hdr->status;
    job.xbuf = reinterpret_cast<uint64_t*>(static_cast<char*>(ws) + ws_prefix());
    int nl = 0;
    job.launch_count = &nl;
    TK_TRY(launch_select(p, job, p.len, &cluster, st));
    record_status_word(st, &hdr->status);
    if (stats) {
      stats->launches = nl;
      stats->cluster = cluster;
      stats->R = p.len;
      int dstat = 0;
      TK_TRY(cudaMemcpyAsync(&dstat, &hdr->status, sizeof(int), cudaMemcpyDeviceToHost, st));
      TK_TRY(cudaStreamSynchronize(st));
      if (dstat != kDevOk) return dstat == kDevTimeout ? TOPK_ETIMEOUT : TOPK_ECUDA;
    }
    return TOPK_OK;
  }

  // one or a few selections: sampling and the threshold in one grid (no
  // threshold launch; the sample and threshold stages then share one event
  // interval), which needs no sample array
  const int64_t nsel = p.nsel;
  const int64_t M = plan.path == TOPK_PATH_PROFK ? plan.M : k;
  const int64_t S = plan.S;
  const bool fused = plan.path == TOPK_PATH_PROFK && nsel <= kSampleHistMaxRows && sample_tau_supported(p, S);

  // workspace layout
  const int64_t ntile = (p.len + kFallbackTile - 1) / kFallbackTile;
  const size_t o_hdr = 0;
  size_t off = ws_prefix();
  const size_t o_counts = off; off = align_up(off + sizeof(unsigned long long) * nsel);
  const size_t o_rseen = off; off = align_up(off + sizeof(unsigned long long) * nsel);
  const size_t o_tau = off; off = align_up(off + sizeof(uint64_t) * nsel);
  const size_t o_taux = off; off = align_up(off + sizeof(uint64_t) * nsel);
  const size_t o_ghist = off; off = align_up(off + sizeof(unsigned) * 8 * 256);
  const size_t o_tiles = off; off = align_up(off + sizeof(unsigned) * ntile);
  const size_t o_samples = off; off = align_up(off + (fused ? 0 : sizeof(uint64_t) * nsel * S));
  // One selection over 16-byte aligned data after the fused sampler: the
  // TMA-ring filter places its survivors in bin regions, from which the grid
  // refinement and the bin sort take them -- also for k below the bin
  // sort's usual bound, from kBinnedMinK (the refinement cluster's radix
  // passes and its 2-CTA collection then go).  Left out when a fixed
  // scratch has no room for the regions.
  // (below kBinnedMinK the refinement cluster reads the regions only when it
  // would otherwise need more than one CTA for the expected survivors, with
  // headroom: one CTA holding them all selects faster from its cache)
  const double expect_r = plan.path == TOPK_PATH_PROFK
                              ? static_cast<double>(plan.t) * (static_cast<double>(p.len) + 1.0) /
                                    (static_cast<double>(S) + 1.0)
                              : 0.0;
  const bool region_route =
      plan.path == TOPK_PATH_PROFK && fused && nsel == 1 && p.vec_ok &&
      (select_binfo_words(k) > 0 || k >= kBinnedMinK ||
       (k >= kBinnedSelMinK && 1.5 * expect_r > static_cast<double>(select_cta_cache())));
  const int64_t binfo_w = region_route ? binfo_words(k) : select_binfo_words(k);
  const int64_t xstride = region_route ? 2 * k : select_xbuf_stride(k);
  const size_t o_buf = off; off = align_up(off + sizeof(uint64_t) * nsel * M);
  const size_t o_xbuf = off; off = align_up(off + sizeof(uint64_t) * nsel * xstride);
  const size_t o_binfo = off; off = align_up(off + sizeof(unsigned) * nsel * binfo_w);
  bool binned = region_route;
  const size_t o_region = off;
  if (binned) {
    const size_t with = align_up(off + sizeof(uint64_t) * kRefineGridBins * kBinRegionCap);
    if (src.fixed && with > src.fixed->bytes) binned = false;
    else off = with;
  }
  void* ws = nullptr;
  ScratchCounters* wcnt = nullptr;
  {
    const cudaError_t e = acquire(src, st, off, &ws, &wcnt);
    if (e != cudaSuccess) return scratch_status(e);
  }
  char* base = static_cast<char*>(ws);
  DevHeader* hdr = reinterpret_cast<DevHeader*>(base + o_hdr);
  auto* counts = reinterpret_cast<unsigned long long*>(base + o_counts);
  auto* r_seen = reinterpret_cast<unsigned long long*>(base + o_rseen);
  auto* tau = reinterpret_cast<uint64_t*>(base + o_tau);
  auto* tau_x = reinterpret_cast<uint64_t*>(base + o_taux);
  auto* ghist = reinterpret_cast<unsigned*>(base + o_ghist);
  auto* tiles = reinterpret_cast<unsigned*>(base + o_tiles);
  auto* samples = reinterpret_cast<uint64_t*>(base + o_samples);
  auto* buf = reinterpret_cast<uint64_t*>(base + o_buf);
  auto* xbuf = reinterpret_cast<uint64_t*>(base + o_xbuf);

  // relaxed recall: fewer than k survivors are returned as they are, padded
  const bool relaxed = plan.path == TOPK_PATH_PROFK && relaxed_recall(o);
  FallbackScratch fs{ghist, tiles, hdr->barrier, &hdr->status, r_seen, &hdr->misses, &hdr->shortfalls, tau_x,
                     relaxed ? tau : nullptr, kWaitLimitNs, -1};
  if (o && o->wait_limit_ns > 0) fs.wait_ns = static_cast<uint64_t>(o->wait_limit_ns);
  if (o && o->inject_wait_timeout) fs.stall_block = 0;
  const uint64_t seed = (o && o->seed) ? o->seed : kDefaultSeed;
  const uint64_t counter = (o && o->counter >= 0) ? static_cast<uint64_t>(o->counter)
                                                  : g_counter.fetch_add(1);
  const int force = (o && o->force_miss) ? 1 : 0;
  // Large k and a few selections: the miss check, the fallback and the
  // partition of the winners run on one cooperative grid over every SM, and
  // the bin sort follows (no refinement cluster).
  const bool grid_refine = (select_binfo_words(k) > 0 || (binned && k >= kBinnedMinK)) && nsel <= kRefineGridMaxSel &&
                           M <= refine_grid_capacity(p);
  // Winners in no particular order (allowed by the caller): the grid
  // refinement writes them itself and no sort follows.
  const bool unsorted_out = grid_refine && o && o->unsorted;

  auto mark = [&](int i) -> cudaError_t {
    if (!o || !o->events[i]) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(o->events[i]), st);
  };
  // The grid refinement's control words: two copies that alternate between
  // its calls (the kernel clears the other one for the next call).  The copy
  // is chosen here because the fused sampler and the filter write into it
  // (the largest sampled key, the survivors' histogram by offset above tau)
  // for the refinement to start from.
  unsigned* refine_ctl = nullptr;
  unsigned* refine_ctl_next = nullptr;
  if (grid_refine || binned) {
    uint64_t parity;
    {
      std::lock_guard<std::mutex> lock(g_ws_mu);
      parity = wcnt->refine_calls++ & 1u;
    }
    char* copies = base + ws_refine_ctl_offset();
    refine_ctl = reinterpret_cast<unsigned*>(copies + parity * kRefineCtlCopyBytes);
    refine_ctl_next = reinterpret_cast<unsigned*>(copies + (parity ^ 1u) * kRefineCtlCopyBytes);
  }
  // (the refinement cluster of one selection reads the histogram only with
  // the bin regions; the grid refinement also without)
  const bool survivor_hist = fused && (grid_refine || binned);
  binned = binned && survivor_hist;
  auto* region = binned ? reinterpret_cast<uint64_t*>(base + o_region) : nullptr;
  bool fallback_launched = false;
  int nl = 0;  // kernels launched
  if (plan.path == TOPK_PATH_PROFK) {
    TK_TRY(mark(0));
    unsigned* hist_add = nullptr;
    unsigned* hist_zero = nullptr;
    if (nsel <= kSampleHistMaxRows) {
      char* halves = base + ws_hist_offset();
      uint64_t parity;
      {
        std::lock_guard<std::mutex> lock(g_ws_mu);
        parity = wcnt->sample_calls++ & 1u;
      }
      hist_add = reinterpret_cast<unsigned*>(halves + parity * kHistHalfBytes);
      hist_zero = reinterpret_cast<unsigned*>(halves + (parity ^ 1u) * kHistHalfBytes);
    }
    if (fused) {
      SampleTauScratch sc{hist_add, hist_zero, reinterpret_cast<unsigned*>(base + ws_tau_ctl_offset()),
                          reinterpret_cast<uint64_t*>(base + ws_tau_gather_offset())};
      sc.refine_ctl = survivor_hist ? refine_ctl : nullptr;

      TK_TRY(launch_sample_tau(p, S, plan.t, seed, counter, counts, hdr, sc, tau, st));
      ++nl;
    } else {
      TK_TRY(launch_sample(p, S, seed, counter, samples, counts, hdr, hist_add, hist_zero, st));
      ++nl;
    }
    TK_TRY(mark(1));
    if (!fused) {
      SelectJob tj{};
      tj.keys = samples;
      tj.key_stride = S;
      tj.r = plan.t;
      tj.want_topk = false;
      tj.tau_out = tau;
      tj.sample_hist = hist_add;
      tj.status = &hdr->status;
      tj.launch_count = &nl;
      int tau_cluster = 0;
      TK_TRY(launch_select(p, tj, S, &tau_cluster, st));
#ifdef TK_PHASE_TIMING
      if (std::getenv("TK_DEBUG_TWICE")) TK_TRY(launch_select(p, tj, S, &tau_cluster, st));
#endif
    }
    TK_TRY(mark(2));
    // The filter may launch while the fused grid finishes (its blocks leave
    // early, one block ranks at the end), not while a 16-CTA threshold
    // cluster runs: that gained nothing.
    // (a fused sampler without grid barriers leaves HBM idle once its draws
    // have landed: the filter's blocks start fetching their tiles into L2)
    const int l2_ahead = fused && sample_tau_local(S, plan.t) &&
                                 p.nsel * p.len * static_cast<int64_t>(p.dtype == kF32 ? 4 : 2) >= kRingL2AheadMinBytes
                             ? kRingL2Ahead
                             : 0;
    TK_TRY(launch_filter(p, tau, M, buf, counts, fused ? 0 : -1, st, survivor_hist ? refine_ctl : nullptr,
                         &hdr->status, region, grid_refine ? nullptr : refine_ctl_next, l2_ahead));
    ++nl;
    TK_TRY(mark(3));
    // Where to handle a miss: inside the refinement kernel (no launch when
    // nothing missed, but on a miss its cluster alone streams x), or in the
    // grid-wide fallback kernel (one launch per call, a fast miss).  The
    // refinement takes it when the expected cost of its slow miss -- the
    // plan's own miss probability times about three passes over a row at
    // ~100 GB/s per SM of the cluster -- is below the launch it saves.  A
    // miss forced by the caller always takes the grid-wide fallback.
    if (!grid_refine && (force || relaxed || !miss_in_refine(p, k, plan.t, plan.S, plan.p_miss))) {
      TK_TRY(launch_fallback(p, k, M, buf, counts, fs, force, st));
      ++nl;
      fallback_launched = true;
    }
    TK_TRY(mark(4));
  } else {  // TOPK_PATH_EXACT
    TK_TRY(cudaMemsetAsync(base, 0, sizeof(DevHeader), st));
    TK_TRY(cudaMemsetAsync(base + o_counts, 0, o_tau - o_counts, st));  // counts, r_seen
    if (!grid_refine) {
      TK_TRY(launch_fallback(p, k, M, buf, counts, fs, 1, st));
      ++nl;
    }
  }
  SelectJob rj{};
  rj.keys = buf;
  rj.key_stride = M;
  rj.counts = counts;
  rj.r = k;
  rj.want_topk = true;
  rj.out_vals = out_vals;
  rj.out_idx = out_idx;
  rj.status = &hdr->status;
  rj.xbuf = xbuf;
  rj.xbuf_stride = grid_refine ? xstride : select_xbuf_stride(k);
  rj.clear_words = reinterpret_cast<unsigned*>(base + ws_tau_ctl_offset());  // the fused threshold grid's
  rj.n_clear = kTauCtlWords;
  rj.launch_count = &nl;
  rj.binfo = (grid_refine || select_binfo_words(k) > 0) && binfo_w ? reinterpret_cast<unsigned*>(base + o_binfo) : nullptr;
  rj.relax_tau = relaxed ? tau_x : nullptr;  // the fallback's per-row padding bound
  if (binned) {  // (the bin sort reads them when the refinement says so)
    rj.fhist = refine_ctl + kRefineGridFilterHist;
    rj.region = region;
    if (!grid_refine) rj.rctl = refine_ctl;  // (the refinement cluster: it checks them itself)
  }
  if (plan.path == TOPK_PATH_PROFK && !fallback_launched) {
    rj.check_miss = true;
    rj.force_miss = force != 0;
    rj.r_seen = r_seen;
    rj.misses = &hdr->misses;
  }
  // expected survivors: E[R] = t (N+1)/(S+1) (Lemma 1, Eq. 2), with
  // headroom.  Only the cluster size depends on it; survivors beyond what the
  // cluster caches are streamed from L2, which a single CTA does slowly.
  int64_t hint = M;
  if (plan.path == TOPK_PATH_PROFK) {
    const double er = static_cast<double>(plan.t) * (static_cast<double>(p.len) + 1.0) /
                      (static_cast<double>(S) + 1.0);
    if (1.5 * er < static_cast<double>(M)) hint = static_cast<int64_t>(1.5 * er);
    if (hint < k) hint = k;
  }
  if (grid_refine) {
    RefineGridScratch rg{};
    rg.ctl = refine_ctl;
    rg.ctl_next = refine_ctl_next;
    rg.tau = survivor_hist ? tau : nullptr;
    rg.region = region;
    rg.xbuf = xbuf;
    rg.xstride = rj.xbuf_stride;
    rg.binfo = rj.binfo;
    rg.clear_words = rj.clear_words;
    rg.n_clear = rj.n_clear;
    rg.unsorted = unsorted_out ? 1 : 0;
    rg.out_vals = out_vals;
    rg.out_idx = out_idx;
    const int fforce = plan.path == TOPK_PATH_PROFK ? force : 1;
    TK_TRY(launch_refine_grid(p, k, M, buf, counts, fs, fforce, rg, st));
    ++nl;
    if (!unsorted_out) TK_TRY(launch_bin_sort(p, rj, st));
    cluster = 1;
  } else {
    TK_TRY(launch_select(p, rj, hint, &cluster, st));
#ifdef TK_PHASE_TIMING
    if (std::getenv("TK_DEBUG_TWICE")) TK_TRY(launch_select(p, rj, hint, &cluster, st));
#endif
  }
  if (plan.path == TOPK_PATH_PROFK) TK_TRY(mark(5));
  record_status_word(st, &hdr->status);

  if (stats) {
    DevHeader h;
    unsigned long long r0 = 0;
    uint64_t tau0 = 0;
    TK_TRY(cudaMemcpyAsync(&h, hdr, sizeof(h), cudaMemcpyDeviceToHost, st));
    TK_TRY(cudaMemcpyAsync(&r0, r_seen, sizeof(r0), cudaMemcpyDeviceToHost, st));
    if (plan.path == TOPK_PATH_PROFK)
      TK_TRY(cudaMemcpyAsync(&tau0, tau, sizeof(tau0), cudaMemcpyDeviceToHost, st));
    TK_TRY(cudaStreamSynchronize(st));
    stats->R = static_cast<int64_t>(r0);
    stats->misses = static_cast<int64_t>(h.misses);
    stats->tau = tau0;
    stats->tau_index = plan.path == TOPK_PATH_PROFK ? static_cast<int64_t>(position_of(tau0, p.ib)) : -1;
    stats->seed = seed;
    stats->counter = static_cast<int64_t>(counter);
    stats->cluster = cluster;
    stats->launches = nl;
    stats->shortfalls = static_cast<int64_t>(h.shortfalls);
    if (h.status != kDevOk) return h.status == kDevTimeout ? TOPK_ETIMEOUT : TOPK_ECUDA;
  }
  return TOPK_OK;
}

}  // namespace

int select_with_fixed_scratch(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                              double eps, void* out_vals, int64_t* out_idx, cudaStream_t st, bool global,
                              const FixedScratch& fs) {
  ScratchSource src;
  src.fixed = &fs;
  return run(x, dtype, rows, n, k, largest, eps, out_vals, out_idx, st, global, nullptr, nullptr, src);
}

namespace {

// Synthetic uniform values in [0, 1) from a counter hash (the tuning input).
__global__ void tune_fill_kernel(float* x, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    uint64_t h = static_cast<uint64_t>(i) * 0x9E3779B97F4A7C15ull;
    h ^= h >> 31;
    h *= 0xBF58476D1CE4E5B9ull;
    h ^= h >> 29;
    x[i] = static_cast<float>(h >> 40) * (1.0f / 16777216.0f);
  }
}

struct StageTimer {
  cudaEvent_t ev[6] = {};
  bool ok = true;
  StageTimer() {
    for (auto& e : ev) ok = ok && cudaEventCreate(&e) == cudaSuccess;
  }
  ~StageTimer() {
    for (auto& e : ev)
      if (e) cudaEventDestroy(e);
  }
};

double median(std::vector<double> v) {
  std::sort(v.begin(), v.end());
  return v.empty() ? 0.0 : v[v.size() / 2];
}

// Median device time (us) between stage events e0 and e1 over `reps` calls of
// one selection of k out of n with the given options (events filled in).
int time_stage(const float* x, int64_t n, int64_t k, double eps, topk_options_t opt, int e0, int e1, int reps,
               float* vals, int64_t* idx, cudaStream_t st, StageTimer& tm, double* us, int64_t* r_out) {
  for (int i = 0; i < 6; ++i) opt.events[i] = tm.ev[i];
  std::vector<double> t;
  for (int rep = -2; rep < reps; ++rep) {
    topk_stats_t stats;
    const int rc = run(x, TOPK_F32, 1, n, k, 1, eps, vals, idx, st, false, &opt, &stats);
    if (rc != TOPK_OK) return rc;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, tm.ev[e0], tm.ev[e1]) != cudaSuccess) return TOPK_ECUDA;
    if (rep >= 0) t.push_back(1e3 * ms);
    if (r_out) *r_out = stats.R;
  }
  *us = median(t);
  return TOPK_OK;
}

// Median time (us) of whole selections through one forced path.
int time_call(const float* x, int64_t n, int64_t k, int path, int reps, float* vals, int64_t* idx, cudaStream_t st,
              StageTimer& tm, double* us) {
  topk_options_t opt;
  topk_options_init(&opt);
  opt.path = path;
  std::vector<double> t;
  for (int rep = -2; rep < reps; ++rep) {
    if (cudaEventRecord(tm.ev[0], st) != cudaSuccess) return TOPK_ECUDA;
    const int rc = run(x, TOPK_F32, 1, n, k, 1, 1e-3, vals, idx, st, false, &opt, nullptr);
    if (rc != TOPK_OK) return rc;
    if (cudaEventRecord(tm.ev[1], st) != cudaSuccess || cudaEventSynchronize(tm.ev[1]) != cudaSuccess)
      return TOPK_ECUDA;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, tm.ev[0], tm.ev[1]) != cudaSuccess) return TOPK_ECUDA;
    if (rep >= 0) t.push_back(1e3 * ms);
  }
  *us = median(t);
  return TOPK_OK;
}

int autotune(int64_t k_cross, cudaStream_t st, topk_tuning_t* out) {
  constexpr int64_t kN = int64_t(1) << 26;  // 256 MiB of f32: larger than L2
  constexpr int64_t kMaxK = 65536;
  constexpr int kReps = 15;
  float* x = nullptr;
  float* vals = nullptr;
  int64_t* idx = nullptr;
  StageTimer tm;
  if (!tm.ok) return TOPK_ECUDA;
  cudaError_t e = cudaMalloc(&x, sizeof(float) * kN);
  if (e == cudaSuccess) e = cudaMalloc(&vals, sizeof(float) * kMaxK);
  if (e == cudaSuccess) e = cudaMalloc(&idx, sizeof(int64_t) * kMaxK);
  int rc = status_of(e);
  if (rc == TOPK_OK) {
    tune_fill_kernel<<<1216, 256, 0, st>>>(x, kN);
    rc = status_of(cudaGetLastError());
  }
  topk_tuning_t r{};
  r.crossover_k = k_cross;
  // tau_A: the sampling and threshold stage (events 0 -> 2) at two sample sizes
  double ta1 = 0, ta2 = 0;
  const int64_t s1 = 32768, s2 = 131072;
  topk_options_t o;
  topk_options_init(&o);
  if (rc == TOPK_OK) {
    o.s_min = o.s_max = s1;
    rc = time_stage(x, kN, 1024, 1e-3, o, 0, 2, kReps, vals, idx, st, tm, &ta1, nullptr);
  }
  if (rc == TOPK_OK) {
    o.s_min = o.s_max = s2;
    rc = time_stage(x, kN, 1024, 1e-3, o, 0, 2, kReps, vals, idx, st, tm, &ta2, nullptr);
  }
  // tau_B: the refinement (events 4 -> 5) at two survivor counts (S fixed,
  // t raised; the buffer sized for the larger count), per log2 k
  double tb1 = 0, tb2 = 0;
  int64_t r1 = 0, r2 = 0;
  if (rc == TOPK_OK) {
    topk_options_init(&o);
    o.s_min = o.s_max = s1;
    o.t_override = 8;
    o.m_override = 1 << 17;
    rc = time_stage(x, kN, 1024, 1e-3, o, 4, 5, kReps, vals, idx, st, tm, &tb1, &r1);
  }
  if (rc == TOPK_OK) {
    o.t_override = 32;
    rc = time_stage(x, kN, 1024, 1e-3, o, 4, 5, kReps, vals, idx, st, tm, &tb2, &r2);
  }
  if (rc == TOPK_OK) {
    r.tau_a_ns = std::max(1e-6, 1e3 * (ta2 - ta1) / static_cast<double>(s2 - s1));
    r.tau_b_ns = std::max(1e-6, r2 > r1 ? 1e3 * (tb2 - tb1) / static_cast<double>(r2 - r1) / std::log2(1024.0) : 0.0);
    r.cost_ratio = r.tau_b_ns / r.tau_a_ns;
    // the crossover: forced Prof-K against the direct path, n = 2^16 .. 2^24
    int64_t cross = 0;
    bool beaten_since = false;
    for (int lg = 16; lg <= 24 && rc == TOPK_OK; ++lg) {
      const int64_t n = int64_t(1) << lg;
      if (k_cross * 8 > n) continue;
      Plan pl;
      topk_options_t po;
      topk_options_init(&po);
      po.path = TOPK_PATH_PROFK;
      if (make_plan(n, k_cross, 1e-3, 1, false, &po, &pl) != TOPK_OK) {  // Prof-K not applicable here
        beaten_since = false;
        continue;
      }
      double td = 0, tp = 0;
      rc = time_call(x, n, k_cross, TOPK_PATH_DIRECT, kReps, vals, idx, st, tm, &td);
      if (rc == TOPK_OK) rc = time_call(x, n, k_cross, TOPK_PATH_PROFK, kReps, vals, idx, st, tm, &tp);
      if (rc != TOPK_OK) break;
      if (tp < td) {
        if (!beaten_since) cross = n;
        beaten_since = true;
      } else {
        beaten_since = false;
        cross = 0;
      }
    }
    r.crossover_n = cross;
  }
  if (x) cudaFree(x);
  if (vals) cudaFree(vals);
  if (idx) cudaFree(idx);
  if (rc != TOPK_OK) return rc;
  int dev = 0;
  TK_TRY(cudaGetDevice(&dev));
  {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    g_tuning[dev] = r;
  }
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    g_plans.clear();  // plans that asked for the measured ratio are recomputed
  }
  *out = r;
  return TOPK_OK;
}

}  // namespace

}  // namespace tk

using namespace tk;

extern "C" {

void topk_options_init(topk_options_t* opt) {
  if (!opt) return;
  std::memset(opt, 0, sizeof(*opt));
  opt->s_min = 32768;
  opt->s_max = 131072;
  opt->cost_ratio = 1.0;
  opt->rule = TOPK_RULE_EXACT;
  opt->path = TOPK_PATH_AUTO;
  opt->seed = kDefaultSeed;
  opt->counter = -1;
  opt->wait_limit_ns = 0;
  opt->inject_wait_timeout = 0;
  opt->recall = 0.0;
}

int topk_select(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest, double eps,
                void* out_vals, int64_t* out_idx, void* stream) {
  return run(x, dtype, rows, n, k, largest, eps, out_vals, out_idx,
             static_cast<cudaStream_t>(stream), false, nullptr, nullptr);
}

int topk_select_global(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                       double eps, void* out_vals, int64_t* out_idx_flat, void* stream) {
  return run(x, dtype, rows, n, k, largest, eps, out_vals, out_idx_flat,
             static_cast<cudaStream_t>(stream), true, nullptr, nullptr);
}

int topk_select_ex(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                   double eps, void* out_vals, int64_t* out_idx, void* stream, int global,
                   const topk_options_t* opt, topk_stats_t* stats) {
  return run(x, dtype, rows, n, k, largest, eps, out_vals, out_idx,
             static_cast<cudaStream_t>(stream), global != 0, opt, stats);
}

int topk_plan(int64_t n, int64_t k, double eps, const topk_options_t* opt, topk_plan_t* plan) {
  if (!plan || n < 1 || k < 1 || k > n || !(eps >= 0.0 && eps < 1.0)) return TOPK_EINVAL;
  Plan pl;
  const int rc = make_plan(n, k, eps, 1, false, opt, &pl);
  if (rc != TOPK_OK) return rc;
  plan->path = pl.path;
  plan->S = pl.S;
  plan->t = pl.t;
  plan->M = pl.M;
  plan->p_recall_fail = 0.0;
  plan->p_overflow = 0.0;
  if (pl.path == TOPK_PATH_PROFK) {
    const double nd = static_cast<double>(n);
    const int64_t kt = recall_rank(k, relaxed_recall(opt) ? opt->recall : 0.0);
    plan->p_recall_fail = binom_upper_tail(pl.S, (static_cast<double>(kt) - 1.0) / nd, pl.t);
    plan->p_overflow = binom_lower_tail(pl.S, static_cast<double>(pl.M) / nd, pl.t - 1);
  }
  return TOPK_OK;
}

int topk_autotune(int64_t k, void* stream, topk_tuning_t* out) {
  if (!out || k < 0 || k > 65536) return TOPK_EINVAL;
  return autotune(k ? k : 1024, static_cast<cudaStream_t>(stream), out);
}

int topk_tuning(topk_tuning_t* out) {
  if (!out) return TOPK_EINVAL;
  return tuned_model(out) ? TOPK_OK : TOPK_EINVAL;
}

int topk_last_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0;
  TK_TRY(cudaGetDevice(&dev));
  int* word = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    auto it = g_last_status.find(std::make_pair(dev, st));
    if (it != g_last_status.end()) word = it->second;
  }
  TK_TRY(cudaStreamSynchronize(st));
  if (!word) return TOPK_OK;
  int dstat = 0;
  TK_TRY(cudaMemcpy(&dstat, word, sizeof(int), cudaMemcpyDeviceToHost));
  if (dstat == kDevOk) return TOPK_OK;
  return dstat == kDevTimeout ? TOPK_ETIMEOUT : TOPK_ECUDA;
}

const char* topk_status_str(int status) {
  switch (status) {
    case TOPK_OK: return "ok";
    case TOPK_EINVAL: return "invalid argument";
    case TOPK_ENOMEM: return "out of device memory";
    case TOPK_ECUDA: return "CUDA error";
    case TOPK_EUNSUPPORTED: return "unsupported size";
    case TOPK_ETIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

// 0.2.0: topk_options_t gained `unsorted` (a caller built against 0.1 passes a shorter struct).
// 0.3.0: topk_options_t gained `wait_limit_ns` and `inject_wait_timeout`; topk_last_status.
int topk_version(void) { return 300; }

#ifdef TK_PHASE_TIMING
int topk_debug_phase_ns(unsigned long long* out) { return tk::debug_phase_ns(out); }
int topk_debug_rows_ns(unsigned long long* out) { return tk::debug_rows_ns(out); }
int topk_debug_binsort_ns(unsigned long long* out) { return tk::debug_binsort_ns(out); }
int topk_debug_sample_tau_ns(unsigned long long* out) { return tk::debug_sample_tau_ns(out); }
int topk_debug_refine_grid_ns(unsigned long long* out) { return tk::debug_refine_grid_ns(out); }
int topk_debug_timeline(unsigned long long* out, int reset) {
  unsigned long long a[16], b[16], c[16], d[16];
  if (tk::debug_timeline_select(a, reset) || tk::debug_timeline_filter(b, reset) ||
      tk::debug_timeline_sample(c, reset) || tk::debug_timeline_fallback(d, reset))
    return -3;
  if (reset) return 0;
  for (int i = 0; i < 8; ++i) {
    unsigned long long s0 = a[2 * i], e0 = a[2 * i + 1];
    s0 = b[2 * i] < s0 ? b[2 * i] : s0;
    s0 = c[2 * i] < s0 ? c[2 * i] : s0;
    s0 = d[2 * i] < s0 ? d[2 * i] : s0;
    e0 = b[2 * i + 1] > e0 ? b[2 * i + 1] : e0;
    e0 = c[2 * i + 1] > e0 ? c[2 * i + 1] : e0;
    e0 = d[2 * i + 1] > e0 ? d[2 * i + 1] : e0;
    out[2 * i] = s0;
    out[2 * i + 1] = e0;
  }
  return 0;
}
#endif

int topk_index_bits(int64_t len) { return len < 1 ? 1 : index_bits(len); }

int topk_prof_sample(const void* x, int dtype, int64_t rows, int64_t n, int global, int largest,
                     int64_t S, uint64_t seed, int64_t counter, uint64_t* out_keys, void* stream) {
  if (dtype != TOPK_F32 && dtype != TOPK_BF16) return TOPK_EINVAL;
  if (rows < 0 || n < 1 || S < 1 || counter < 0) return TOPK_EINVAL;
  if (rows == 0) return TOPK_OK;
  if (!x || !out_keys) return TOPK_EINVAL;
  const Problem p = make_problem(x, dtype, rows, n, largest, global != 0);
  if (p.nsel > 65535) return TOPK_EUNSUPPORTED;
  const cudaError_t e = launch_sample(p, S, seed, static_cast<uint64_t>(counter), out_keys, nullptr,
                                      nullptr, nullptr, nullptr, static_cast<cudaStream_t>(stream));
  return status_of(e);
}

int topk_prof_filter(const void* x, int dtype, int64_t rows, int64_t n, int global, int largest,
                     const uint64_t* tau, int64_t M, uint64_t* buf, uint64_t* counts, void* stream) {
  if (dtype != TOPK_F32 && dtype != TOPK_BF16) return TOPK_EINVAL;
  if (rows < 0 || n < 1 || M < 1) return TOPK_EINVAL;
  if (rows == 0) return TOPK_OK;
  if (!x || !tau || !buf || !counts) return TOPK_EINVAL;
  const Problem p = make_problem(x, dtype, rows, n, largest, global != 0);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(uint64_t) * p.nsel, st);
  if (e != cudaSuccess) return status_of(e);
  e = launch_filter(p, tau, M, buf, reinterpret_cast<unsigned long long*>(counts), 0, st);
  return status_of(e);
}

}  // extern "C"
