// Internal interface between the C ABI (topk_api.cu) and the kernel
// translation units: host declarations, constants, and a few functions both
// sides use.  No torch types anywhere.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

// Functions both the host and the kernels use (this header is also compiled
// by the host compiler, which knows no CUDA qualifiers).
#ifdef __CUDACC__
#define TK_HOST_DEVICE __host__ __device__
#else
#define TK_HOST_DEVICE
#endif

namespace tk {

// One "selection problem" is a row (per-row variant) or the whole flattened
// input (global variant).  `len` elements each, problems laid out back to back.
struct Problem {
  const void* x;
  int dtype;       // kF32 / kBF16
  int64_t nsel;    // number of selections
  int64_t len;     // elements per selection
  int ib;          // index bits of the composite key
  uint32_t flip;   // 0 for largest, value-key mask for smallest
  bool vec_ok;     // 16-byte vector loads are legal (alignment and len % vec)
};

// ---- parameters (params.cpp) -------------------------------------------------
// Whether the refinement kernel should handle a miss itself (no launch when
// nothing misses, but its cluster alone streams x on a miss) rather than the
// grid-wide fallback kernel: true when the miss probability of the plan in
// use (P[R < k] + P[R > M] for its S, t and M, per selection) times the
// expected cost of that slow miss is below the cost of the launch it saves.
bool miss_in_refine(const Problem& p, int64_t k, int64_t t, int64_t S, double p_miss);
// P[R < k] + P[R > M] for one selection of k out of n with (S, t, M) under the
// with-replacement sampler (the exact tails of Lemma 1's counting argument).
double plan_miss_probability(int64_t n, int64_t k, int64_t S, int64_t t, int64_t M);
// Programmatic dependent launch for one pipeline edge (see params.cpp).
constexpr unsigned kPdlTau = 1, kPdlFilter = 2, kPdlFallback = 4, kPdlRefine = 8, kPdlGridRefine = 16;
bool pdl_edge(unsigned bit);
struct ParamRule {
  int64_t s_min = 32768, s_max = 131072;
  double cost_ratio = 1.0;
  int rule = 0;  // 0 exact tails, 1 Algorithm 1 as printed
  double recall = 0.0;  // in (0, 1): t is chosen for rank ceil(recall * k) (relaxed recall)
};
// The rank the threshold is chosen for: k, or ceil(recall * k) under relaxed recall.
int64_t recall_rank(int64_t k, double recall);
double inv_normal_upper(double q);  // x with P[Z > x] = q
double binom_upper_tail(int64_t s, double p, int64_t t);  // P[Bin(s,p) >= t]
double binom_lower_tail(int64_t s, double p, int64_t t);  // P[Bin(s,p) <= t]
int64_t alg1_sample_size(int64_t n, int64_t k, double eps, const ParamRule& pr);
// Returns false when no valid t exists (the caller takes an exact path).
bool choose_params(int64_t n, int64_t k, double eps, const ParamRule& pr, int64_t* S, int64_t* t,
                   int64_t* M);

// Per-call device words shared by the pipeline's kernels.
struct DevHeader {
  unsigned barrier[2];         // grid barrier of the fallback: arrivals, generation
  int status;                  // kDevOk / kDevTimeout / kDevBadState
  unsigned shortfalls;         // selections that returned fewer than k winners (relaxed recall)
  unsigned long long misses;   // selections that took the fallback
};

// ---- sample (kernels_sample.cu) ----------------------------------------------
// Also resets counts[0..nsel) and the header (arrivals, status, misses) when
// those pointers are non-null, so the filter and fallback start clean.
// hist_add / hist_zero (nullable, each kSampleHistHalfWords counters): the
// sampled keys are counted by their leading kSampleHistBits bits into level 0
// of hist_add (row-major, kSampleHistBins per selection; bin =
// kSampleHistBins - 1 - digit, largest keys first), and the whole of
// hist_zero is cleared for the next call.  Both must be zero-initialised
// once; they then alternate between calls.
constexpr int kSampleHistBits = 11;
constexpr int kSampleHistBins = 1 << kSampleHistBits;
constexpr int64_t kSampleHistMaxRows = 16;  // selections with a sample histogram
constexpr int kSampleHistLevels = 6;        // 11-bit digits of a key of up to 64 bits
// One histogram half: kSampleHistLevels levels of kSampleHistMaxRows rows.
constexpr int64_t kSampleHistHalfWords = int64_t(kSampleHistLevels) * kSampleHistMaxRows * kSampleHistBins;
cudaError_t launch_sample(const Problem& p, int64_t S, uint64_t seed, uint64_t counter,
                          uint64_t* keys, unsigned long long* counts_to_zero, DevHeader* hdr,
                          unsigned* hist_add, unsigned* hist_zero, cudaStream_t st);

// Sampling and the threshold in one cooperative grid (kernels_sample.cu): the
// t-th largest sampled key of each selection is found by a radix select over
// the grid (11-bit digits counted into hist level by level, a grid barrier
// per digit) until its bin holds at most kTauGather keys; those are gathered
// and the last block of the selection ranks them.  When blocks x t <=
// kTauGather, each block instead keeps its own t largest keys and the last
// block ranks their union (no grid barrier).  hist / hist_zero are
// histogram halves as above (hist counted into, hist_zero cleared); ctl holds
// kTauCtlWords words and gather kTauGather keys per selection.  ctl must be
// zero on entry; the kernel leaves its grid barrier and counters as it found
// them except after a timeout, so the refinement clears ctl every call.
// refine_ctl (nullable): the grid refinement's control words of this call
// (kRefineGridCtlWords per selection, zero on entry); the largest sampled key
// of each selection is recorded there (atomic max at kRefineGridKmaxWord).
constexpr int kTauGather = 2048;
constexpr int kTauCtlWords = 2 + 2 * static_cast<int>(kSampleHistMaxRows);
struct SampleTauScratch {
  unsigned* hist;
  unsigned* hist_zero;
  unsigned* ctl;
  uint64_t* gather;
  unsigned* refine_ctl = nullptr;
};
// Whether the fused grid fits on the device at once (else launch_sample and
// a threshold select are used).
bool sample_tau_supported(const Problem& p, int64_t S);
// Whether the fused grid ranks without a grid barrier: every block keeps its
// own t largest draws and the last block ranks their union.
bool sample_tau_local(int64_t S, int64_t t);
cudaError_t launch_sample_tau(const Problem& p, int64_t S, int64_t t, uint64_t seed, uint64_t counter,
                              unsigned long long* counts_to_zero, DevHeader* hdr, const SampleTauScratch& sc,
                              uint64_t* tau_out, cudaStream_t st);

// ---- filter (kernels_filter.cu) and fallback (kernels_fallback.cu) ----------
// SMs a threshold select of nsel clusters of G blocks holds while the filter
// launches, or -1 when it spans too many SMs to overlap.
inline int overlap_sms(int G, int64_t nsel) {
  const int64_t held = static_cast<int64_t>(G) * nsel;
  return held <= 16 ? static_cast<int>(held) : -1;
}

struct FallbackScratch {
  unsigned* ghist;        // 8 passes x 256 counters
  unsigned* tile_counts;  // ceil(len / kFallbackTile) counters
  unsigned* barrier;      // [0] arrivals, [1] generation
  int* status;
  unsigned long long* r_seen;  // per selection: R as the filter left it
  unsigned long long* misses;  // number of selections that fell back
  unsigned* shortfalls;        // number of selections returned short (relaxed recall)
  uint64_t* tau_exact;         // per selection: exact k-th key written on a miss; under relaxed
                               // recall also the bound below which keys are padding (0: none)
  // Relaxed recall (nullable): the sampled tau per selection.  A selection
  // with R < k survivors (and R within the buffer) then takes no fallback:
  // slots R..k-1 of its buffer receive the sentinel keys tau - 1 - j, which
  // rank below every survivor and are written out as padding.
  const uint64_t* relax_tau;
  uint64_t wait_ns;            // limit of each grid-wide wait (kWaitLimitNs unless a caller sets it)
  int stall_block;             // testing: this block leaves its first grid-wide wait without
                               // arriving, so the others' bounded wait runs out (-1: none)
};
constexpr int64_t kFallbackTile = 4096;
// reserved_sms: SMs the preceding grid (the threshold select) holds; the
// launch may overlap that grid only when it is >= 0.
// refine_ctl (nullable): the grid refinement's control words of this call,
// holding each selection's largest sampled key (from the fused sampler); the
// survivors are then also counted into the histogram at
// kRefineGridFilterHist, 2048 bins of their offset above tau: bin = 2047 -
// ((key - tau) >> shift), or 0 when that exceeds 2046, with shift =
// survivor_shift(tau, largest sampled key) (filter_core.cuh).
// region (nullable; one selection with refine_ctl only): each filter block
// also places its survivors in bin regions of kBinRegionCap keys at its end
// (kRefineGridBinnedWord of refine_ctl set when they do not fit).
// refine_ctl_next (with region, nullable): the other copy of the control
// words, cleared by the filter's blocks for the next call (when no grid
// refinement, which clears it otherwise, follows).
// l2_ahead (one selection over 16-byte aligned data): tiles past the first
// ring stages that each block of the TMA-ring filter asks L2 to fetch before
// tau is known -- for a preceding grid that leaves HBM idle (0: none).
cudaError_t launch_filter(const Problem& p, const uint64_t* tau, int64_t cap, uint64_t* buf,
                          unsigned long long* counts, int reserved_sms, cudaStream_t st,
                          unsigned* refine_ctl = nullptr, int* status = nullptr, uint64_t* region = nullptr,
                          unsigned* refine_ctl_next = nullptr, int l2_ahead = 0);
// Tiles (16 KB) each of the ring filter's blocks asks L2 to fetch while the
// fused sampler ranks in its local mode (no grid barrier: it waits on L2
// atomics of no other block, and its draws have landed), at most half of a
// block's tiles, and the smallest input (bytes) that gains from it.  On a
// GB300, single f32 rows with k = 1024 back to back: 2^28 175.3 -> 169.4 us,
// 2^26 69.8 -> 66.5, 2^25 51.6 -> 48.3 (13 tiles); 2^24 unchanged; 32 tiles
// lost 2.5 us at 2^25 and 2^26.
constexpr int kRingL2Ahead = 24;
constexpr int64_t kRingL2AheadMinBytes = int64_t{1} << 27;
// force: 0 = only rows that missed, 1 = every row (fault injection / exact path).
cudaError_t launch_fallback(const Problem& p, int64_t k, int64_t cap, uint64_t* buf,
                            unsigned long long* counts, const FallbackScratch& fs, int force,
                            cudaStream_t st);

// Refinement of a few selections with large k on one cooperative grid
// (kernels_fallback.cu): the miss check and, on a miss, the fallback above,
// then the exact partition of each selection's candidates into 2048 equal
// slices of their key range (the first 11-bit digit of key - smallest key)
// in the exchange buffer, published for the bin sort (launch_bin_sort) in the
// bin-info format of the refinement cluster.
constexpr int kRefineGridBins = 2048;          // first-digit bins (the bin sort's)
constexpr int kRefineGridLevels = 6;           // 11-bit digits of a key of up to 64 bits
constexpr int64_t kRefineGridMaxSel = 4;       // selections one grid refines
// Control words per selection: NOT of the smallest and the largest key (2 x
// 64 bits), the boundary bin's placed winners, the blocks done placing
// (kRefineGridTicketWord), the largest sampled key (64 bits at
// kRefineGridKmaxWord), then one counter per bin and digit level, then the
// filter's survivor histogram (kRefineGridFilterHist), then a word the
// filter sets when its bin regions are incomplete (kRefineGridBinnedWord).
constexpr int64_t kRefineGridTicketWord = 5;
constexpr int64_t kRefineGridKmaxWord = 6;
constexpr int64_t kRefineGridFilterHist = 8 + int64_t(kRefineGridLevels) * kRefineGridBins;
constexpr int64_t kRefineGridBinnedWord = kRefineGridFilterHist + kRefineGridBins;
constexpr int64_t kRefineGridCtlWords = kRefineGridBinnedWord + 4;
// Bin regions (one selection): the filter may also place its survivors by
// the bin of the survivor histogram, kBinRegionCap keys a bin, bin b's keys
// at [b * kBinRegionCap, ...) in no particular order.
constexpr int64_t kBinRegionCap = 2048;
// Smallest k that takes the bin regions (one selection): below it the
// refinement cluster stays, faster there (measured on single f32 rows of
// 2^22 to 2^28: k = 512 and 1024 lose 1-6 us on the bin regions, k = 2048
// wins or loses up to 3 us by size, k = 3072 gains 3-6 us from 2^24 on,
// k = 4096 gains 4-8 us).
constexpr int64_t kBinnedMinK = 3072;
// Smallest k whose refinement cluster reads the bin regions (one selection;
// below kBinnedMinK: CTA 0 takes the winners from the regions), when the
// expected survivors would need more than one CTA of it (measured on f32
// rows at k = 512..2048: 3.5-4.5 us faster at 2^28 elements, where the
// cluster takes two CTAs, 3-5 us slower at 2^24-2^26, where one CTA holds
// every survivor).
constexpr int64_t kBinnedSelMinK = 512;
// Most keys the top (overflow) bin may hold for the bin sort to take the
// bin regions (it never cuts that bin by digits).
constexpr unsigned long long kBinnedTopMax = 512;
struct RefineGridScratch {
  unsigned* ctl;          // this call's control words: kRefineGridCtlWords per selection, zero on entry
  unsigned* ctl_next;     // the other copy (kRefineGridMaxSel selections), cleared here for the next call
  uint64_t* xbuf;         // exchange buffer, xstride keys per selection
  int64_t xstride;        // >= 2k
  unsigned* binfo;        // select_binfo_words(k) words per selection
  unsigned* clear_words;  // nullable: words of an earlier grid zeroed once that grid has finished
  int n_clear;
  // unsorted != 0: find the exact k-th key and write the k winners straight
  // to out_vals / out_idx (k per selection, in no particular order); no bin
  // sort follows.  (Inside the kernel: 1 = f32 output, 2 = bf16.)
  int unsorted = 0;
  void* out_vals = nullptr;
  int64_t* out_idx = nullptr;
  // Non-null when the filter counted its survivors into the histogram at
  // kRefineGridFilterHist of ctl (and the sampler recorded the largest
  // sampled key at kRefineGridKmaxWord): the sampled tau per selection.  The
  // partition then takes the bin totals from that histogram (no min / max
  // pass, no grid barrier) when no selection missed, the top bin is empty
  // and the boundary bin fits the exchange buffer.
  const uint64_t* tau = nullptr;
  // Non-null when the filter also placed its survivors in bin regions (one
  // selection, kBinRegionCap keys a bin): with the histogram usable and the
  // regions complete, the winners are copied from them in place order.
  const uint64_t* region = nullptr;
};
// The padding of relaxed recall for one output element: value bits of -inf
// (+inf when the smallest are selected), as f32 or bf16 bits.
inline uint32_t pad_bits(int dtype, bool largest) {
  return dtype == 0 ? (largest ? 0xFF800000u : 0x7F800000u) : (largest ? 0xFF80u : 0x7F80u);
}
// Largest buffer capacity (keys per selection) the grid refinement takes, or
// 0 when it does not apply (too many selections).
int64_t refine_grid_capacity(const Problem& p);
cudaError_t launch_refine_grid(const Problem& p, int64_t k, int64_t cap, uint64_t* buf,
                               unsigned long long* counts, const FallbackScratch& fs, int force,
                               const RefineGridScratch& rg, cudaStream_t st);

// ---- direct path for many short rows (kernels_rows.cu) -----------------------
// One block per selection, the row in registers: len <= 32768, k <= 1024.
bool rows_supported(const Problem& p, int64_t k);
cudaError_t launch_rows(const Problem& p, int64_t k, void* out_vals, int64_t* out_idx, int* status,
                        cudaStream_t st);

// ---- final selection (kernels_select.cu) -------------------------------------
struct SelectJob {
  // source: either composite keys (keys != nullptr) or the raw input (p.x)
  const uint64_t* keys;
  int64_t key_stride;                  // keys per selection in `keys`
  const unsigned long long* counts;    // valid keys per selection (clamped to key_stride); may be null
  int64_t r;                           // rank to find (1-based)
  bool want_topk;                      // true: sort and write the r winners; false: write tau
  uint64_t* tau_out;                   // per selection (want_topk == false)
  void* out_vals;                      // want_topk
  int64_t* out_idx;
  int* status;                         // device status word (kDevBadState on inconsistency)
  uint64_t* xbuf = nullptr;            // want_topk across CTAs: xbuf_stride keys per selection (L2 exchange)
  int64_t xbuf_stride = 0;             // keys per selection in xbuf; at least r (0: r)
  const unsigned* sample_hist = nullptr;  // !want_topk: counts of the keys' leading bits (launch_sample)
  // refinement of the Prof-K buffer: check for a miss (counts[row] < r or >
  // key_stride, or force_miss) and then select from the whole row of x
  bool check_miss = false;
  bool force_miss = false;
  unsigned long long* r_seen = nullptr;   // per selection: R as the filter left it
  unsigned long long* misses = nullptr;   // incremented once per missed selection
  // large k: per selection select_binfo_words(k) words; then the winners are
  // sorted by a second grid of small blocks instead of the cluster alone
  unsigned* binfo = nullptr;
  unsigned* clear_words = nullptr;  // want_topk: n_clear words zeroed after the earlier grids finish
  int n_clear = 0;
  int* launch_count = nullptr;      // nullable: incremented once per kernel launched
  // relaxed recall (nullable): per selection the bound below which keys are
  // the fallback's padding sentinels (the fallback's tau_exact words), written
  // as index -1 and -inf (+inf)
  const uint64_t* relax_tau = nullptr;
  // bin sort, one selection (nullable): the filter's survivor histogram and
  // its bin regions, read when the refinement found them complete (the bin
  // information's header says so) instead of the exchange buffer
  const unsigned* fhist = nullptr;
  const uint64_t* region = nullptr;
  // refinement cluster of one selection whose filter placed its survivors
  // in bin regions (nullable): this call's control words
  const unsigned* rctl = nullptr;
};
int64_t select_binfo_words(int64_t k);  // 0 when k is too small for the bin sort
int64_t select_cta_cache();              // candidates one refinement CTA holds in shared memory
// Output places one bin-sort block owns, and the words of bin information
// per selection (bin starts, a header describing the digit, one descriptor
// per chunk: binfo.cuh).
constexpr int64_t kBinSortChunk = 512;
constexpr int kBinfoHeaderWords = 12;
TK_HOST_DEVICE inline int64_t binfo_words(int64_t k) {
  return kRefineGridBins + kBinfoHeaderWords + 6 * ((k + kBinSortChunk - 1) / kBinSortChunk);
}
// The bin sort alone (job: r = k, xbuf, xbuf_stride, binfo, status, outputs),
// after the grid refinement has partitioned the winners.
cudaError_t launch_bin_sort(const Problem& p, const SelectJob& job, cudaStream_t st);
// Keys per selection the exchange buffer should hold for rank k (2k with the
// bin sort: room to place the boundary's whole first-pass bin).
int64_t select_xbuf_stride(int64_t k);
// Returns the cluster size used via *cluster (may be null).
cudaError_t launch_select(const Problem& p, const SelectJob& job, int64_t source_bound, int* cluster,
                          cudaStream_t st);
int64_t select_max_k();

// ---- the C ABI's pipeline on caller-provided scratch (topk_api.cu) -----------
// Counters that pick which copy of the alternating zero-kept regions a call
// uses (see the workspace layout in topk_api.cu); one set per scratch block.
struct ScratchCounters {
  uint64_t sample_calls = 0;
  uint64_t refine_calls = 0;
};
// A fixed device block used instead of the per-stream pool: zero-initialised
// once, 256-byte aligned, owned by the caller for the life of the process.
struct FixedScratch {
  void* base;
  size_t bytes;
  ScratchCounters* counters;
};
// topk_select (global == false) / topk_select_global with every piece of
// scratch taken from `fs`; TOPK_EUNSUPPORTED, before anything is launched,
// when the call's layout needs more than fs.bytes.
int select_with_fixed_scratch(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                              double eps, void* out_vals, int64_t* out_idx, cudaStream_t st, bool global,
                              const FixedScratch& fs);
#ifdef TK_PHASE_TIMING
int debug_phase_ns(unsigned long long* out);  // debug builds: per-phase timer stamps
int debug_rows_ns(unsigned long long* out);   // debug builds: stamps of the short-row kernel
// debug builds: kernel start / end times, one table per translation unit
int debug_timeline_select(unsigned long long* out, int reset);
int debug_binsort_ns(unsigned long long* out);
int debug_timeline_filter(unsigned long long* out, int reset);
int debug_timeline_fallback(unsigned long long* out, int reset);
int debug_timeline_sample(unsigned long long* out, int reset);
int debug_sample_tau_ns(unsigned long long* out);  // debug builds: stamps of the fused threshold grid
int debug_refine_grid_ns(unsigned long long* out);  // debug builds: stamps of the grid refinement's block 0
#endif

}  // namespace tk
