// Exact selection on one thread-block cluster per selection problem.
//
// Used for three steps of the pipeline:
//   * threshold estimation (section 3, stage 2): the t-th largest of the S
//     sampled composite keys -> tau;
//   * refinement (section 3, stage 4): the exact top-k of the candidate buffer;
//   * the direct path: the exact top-k of the row itself.
//
// Select: radix select ("count elements into buckets and recurse into the
// bucket that contains the boundary", Find the Cutoff Instead) with 11-bit
// digits (2048 bins; 8-bit in the 256-thread variant), starting below the
// most significant bit on which the keys differ.  Each CTA histograms its
// slice of the source into shared memory; the cluster's CTAs read one
// another's counters through distributed shared memory, so every CTA finds
// the same boundary bin with one cluster barrier per digit (the counters are
// double-buffered).  Slices are cached in shared memory when they fit.  When
// the boundary bucket is small it is gathered into CTA 0 and ranked by
// counting ("Rank by Counting": rank = number of larger keys; the composite
// keys are distinct, ties by position being built into them).
//
// Sort (top-k only): the first digit's bins partition the k winners.  Every
// CTA writes its winners into their bins' segments of an L2-resident
// exchange buffer (offsets from the exchanged counts), then owns k/G output
// places.  It reads the bins that overlap its places; a bin at either end
// that would overflow shared memory is cut down, by further digits, to the
// sub-bin holding the boundary place.  The keys in between are ranked by
// counting inside groups of equal leading bits (a stable LSD radix sort if a
// group is too large) and written to their places.  The composite key encodes
// (value descending, index ascending), so that is the output order.
#include <cooperative_groups.h>

#include "binfo.cuh"
#include "common.cuh"
#include "engine.h"
#include "rank.cuh"

namespace cg = cooperative_groups;

namespace tk {

namespace {

constexpr int kMaxCluster = 16;

#ifdef TK_PHASE_TIMING
// Debug builds only: globaltimer stamps of the first cluster's CTA 0.
__device__ unsigned long long g_phase_ns[2][48];
__device__ unsigned long long g_cta_ns[2][16][8];  // per CTA of the first cluster: debug stamps
#define TK_STAMP(i)                                                                         \
  do {                                                                                      \
    if (blockIdx.x == 0 && threadIdx.x == 0) g_phase_ns[a.want_topk][(i)] = globaltimer_ns(); \
  } while (0)
#define TK_CTA(slot, v)                                                                    \
  do {                                                                                     \
    if (blockIdx.x < 16 && threadIdx.x == 0) g_cta_ns[a.want_topk][blockIdx.x][(slot)] = (v); \
  } while (0)
#define TK_DBG(slot, v) (g_cta_ns[1][15][(slot)] = (v))
__device__ unsigned long long g_bs_ns[1024][8];  // debug: per-block phase stamps of the bin sort
#define TK_BSP(i) \
  do { if (threadIdx.x == 0 && blockIdx.x < 1024) g_bs_ns[blockIdx.x][(i)] = globaltimer_ns(); } while (0)
#else
#define TK_BSP(i) \
  do {            \
  } while (0)
#define TK_DBG(slot, v) \
  do {                  \
  } while (0)
#define TK_STAMP(i) \
  do {              \
  } while (0)
#define TK_CTA(slot, v) \
  do {                  \
  } while (0)
#endif

struct SelParams {
  const uint64_t* keys;               // key source (SRC 0, or 3 unless the selection missed)
  int64_t key_stride;
  const unsigned long long* counts;   // valid keys per selection (nullable)
  const void* x;                      // the input (SRC 1 / 2, after a miss, and for output values)
  int64_t len;                        // elements per selection of x
  int ib;
  uint32_t flip;
  int key_bits;                       // value-key bits (32 or 16)
  int key_vec;                        // key rows allow 16-byte loads
  int src_vec;                        // x rows allow 16-byte loads
  int64_t r;                          // rank sought (1-based)
  int want_topk;
  uint64_t* tau_out;
  void* out_vals;
  int64_t* out_idx;
  int* status;
  uint64_t* xbuf;                     // xstride keys per selection: the L2 exchange of the sort
  int64_t xstride;                    // >= r
  const unsigned* shist;              // tau only: first-digit counts of the samples (nullable)
  // refinement of a candidate buffer: when R < r or R > key_stride (a miss;
  // or force), select from x instead (source 1 = f32, 2 = bf16; 0 = no check)
  int miss_src;
  int force;
  unsigned long long* r_seen;         // per selection: R as the filter left it
  unsigned long long* misses;         // selections that missed
  // large k: stop after partitioning the winners and publish the first-digit
  // bins (kBinInfoWords words per selection) for the grid-wide bin sort
  unsigned* binfo;
  int handoff;
  unsigned* clear_words;              // nullable: zeroed once every earlier grid has finished
  int n_clear;
  // relaxed recall (nullable): per selection the bound below which keys are
  // padding sentinels (index -1, value -inf / +inf); a selection returned
  // short holds them in its buffer up to slot r
  const uint64_t* relax_tau;
  // bin sort of one selection (nullable): the filter's survivor histogram
  // and its bin regions, read instead of the exchange buffer when the bin
  // information's header says the refinement left the keys there
  const unsigned* fhist;
  const uint64_t* region;
  // refinement of one selection whose filter placed its survivors in bin
  // regions (nullable): this call's control words (the survivor histogram,
  // the "incomplete" flag)
  const unsigned* rctl;
};

// Published per selection for the bin sort: NB bin starts, then the
// first-digit prefix, mask and shift, the end of the keys placed in the
// exchange buffer (r when only winners were placed, else the end of the
// boundary bin), and a base the digits are taken relative to (digits,
// prefixes and masks describe key - base; 0 from the refinement cluster).
constexpr int kBinInfoBins = 2048;
constexpr int kBinInfoWords = kBinInfoBins + kBinfoHeaderWords;

// Source of the refinement kernel (template source 3), chosen at run time:
// 0 = the candidate buffer, or after a miss 1 / 2 = x as f32 / bf16; and the
// count R its prologue read (the body uses it instead of reading it again).
__shared__ int s_source;
__shared__ unsigned long long s_prologue_r;

// Eight consecutive source elements i0 .. i0+7 (i0 a multiple of 8) as
// composite keys.  Only elements in [lo, hi) are meaningful; vector loads may
// also read neighbours that lie inside the same row.
template <int SRC>
__device__ __forceinline__ void load8(const SelParams& a, int64_t row, int64_t i0, int64_t lo, int64_t hi,
                                      uint64_t (&k)[8]);

template <int SRC>
__device__ __forceinline__ void load8(const SelParams& a, int64_t row, int64_t i0, int64_t lo, int64_t hi,
                                      uint64_t (&k)[8]) {
  if (SRC == 3) {
    const int src = s_source;
    if (src == 0) load8<0>(a, row, i0, lo, hi, k);
    else if (src == 1) load8<1>(a, row, i0, lo, hi, k);
    else load8<2>(a, row, i0, lo, hi, k);
    return;
  }
  if (SRC == 0) {
    const uint64_t* base = a.keys + row * a.key_stride;
    if (a.key_vec && i0 + 8 <= a.key_stride) {
      const uint4* p = reinterpret_cast<const uint4*>(base + i0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldcg(p + q);
        k[2 * q] = (static_cast<uint64_t>(v.y) << 32) | v.x;
        k[2 * q + 1] = (static_cast<uint64_t>(v.w) << 32) | v.z;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) k[j] = (i0 + j >= lo && i0 + j < hi) ? __ldcg(base + i0 + j) : 0ull;
    }
  } else {
    uint32_t u[8];
    if (SRC == 1) {
      const uint32_t* xr = static_cast<const uint32_t*>(a.x) + row * a.len;
      if (a.src_vec && i0 + 8 <= a.len) {
        const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(xr + i0));
        const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(xr + i0) + 1);
        u[0] = v0.x; u[1] = v0.y; u[2] = v0.z; u[3] = v0.w;
        u[4] = v1.x; u[5] = v1.y; u[6] = v1.z; u[7] = v1.w;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = (i0 + j >= lo && i0 + j < hi) ? __ldg(xr + i0 + j) : 0u;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        k[j] = compose(order_key_f32(u[j]) ^ a.flip, static_cast<uint64_t>(i0 + j), a.ib);
    } else {
      const uint16_t* xr = static_cast<const uint16_t*>(a.x) + row * a.len;
      if (a.src_vec && i0 + 8 <= a.len) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + i0));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = (w[j >> 1] >> ((j & 1) * 16)) & 0xffffu;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = (i0 + j >= lo && i0 + j < hi) ? __ldg(xr + i0 + j) : 0u;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        k[j] = compose(order_key_bf16(u[j]) ^ a.flip, static_cast<uint64_t>(i0 + j), a.ib);
    }
  }
}

// Calls f(key, in_range) for every element of the 8-aligned chunks covering
// [lo, hi) of this row, eight keys per thread and iteration.  The trip count
// is the same for the 32 lanes of a warp, so f may use full-warp intrinsics.
template <int SRC, int BLOCK, typename F>
__device__ __forceinline__ void for_slice(const SelParams& a, int64_t row, int64_t lo, int64_t hi, F&& f) {
  const int64_t c0 = lo >> 3, c1 = (hi + 7) >> 3;
  const int lane = threadIdx.x & 31;
  for (int64_t cw = c0 + (threadIdx.x & ~31u); cw < c1; cw += BLOCK) {
    const int64_t c = cw + lane;
    uint64_t k[8];
    if (c < c1) {
      load8<SRC>(a, row, c << 3, lo, hi, k);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) k[j] = 0ull;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t i = (c << 3) + j;
      f(k[j], c < c1 && i >= lo && i < hi);
    }
  }
}

// Calls f(cache[i], valid) for i < n, with a warp-uniform trip count.
template <int BLOCK, typename F>
__device__ __forceinline__ void for_cache(const uint64_t* cache, unsigned n, F&& f) {
  const unsigned lane = threadIdx.x & 31;
#pragma unroll 4
  for (unsigned iw = threadIdx.x & ~31u; iw < n; iw += BLOCK) {
    const unsigned i = iw + lane;
    f(i < n ? cache[i] : 0ull, i < n);
  }
}

// Appends the cached keys that satisfy pred: write(key, slot) with slots
// from *counter (shared memory) onwards, in no particular order.  Four keys
// per thread and round, so each warp issues one atomic and one broadcast per
// 128 keys instead of per 32 (the rounds are a chain of dependent steps).
template <int BLOCK, typename P, typename W>
__device__ __forceinline__ void cache_append(const uint64_t* cache, unsigned n, unsigned* counter, P&& pred,
                                             W&& write) {
  const unsigned lane = threadIdx.x & 31, lt = lanemask_lt();
  for (unsigned c0 = 0; c0 < n; c0 += 4 * BLOCK) {
    uint64_t k[4];
    unsigned m[4], tot = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const unsigned i = c0 + j * BLOCK + threadIdx.x;
      k[j] = i < n ? cache[i] : 0ull;
      m[j] = __ballot_sync(kFull, i < n && pred(k[j]));
      tot += __popc(m[j]);
    }
    if (tot == 0) continue;  // (the same for every lane)
    unsigned b = 0;
    if (lane == 0) b = atomicAdd(counter, tot);
    b = __shfl_sync(kFull, b, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((m[j] >> lane) & 1u) write(k[j], b + __popc(m[j] & lt));
      b += __popc(m[j]);
    }
  }
}


// 16-byte global -> shared copies that bypass registers (cp.async, L2 only).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}


template <int BLOCK>
constexpr int min_blocks() { return BLOCK >= 512 ? 1 : 4; }

// Writes out_vals / out_idx for one winner key at output place `place`.
__device__ __forceinline__ void write_out(const SelParams& a, int64_t row, int64_t k, int64_t place,
                                          uint64_t key) {
  const int64_t oi = row * k + place;
  if (a.relax_tau && key < __ldg(a.relax_tau + row)) {  // padding of relaxed recall
    a.out_idx[oi] = -1;
    if (a.key_bits == 32) static_cast<uint32_t*>(a.out_vals)[oi] = a.flip ? 0x7F800000u : 0xFF800000u;
    else static_cast<uint16_t*>(a.out_vals)[oi] = static_cast<uint16_t>(a.flip ? 0x7F80u : 0xFF80u);
    return;
  }
  const uint64_t pos = position_of(key, a.ib);
  a.out_idx[oi] = static_cast<int64_t>(pos);
  const uint32_t vk = vkey_of(key, a.ib) ^ a.flip;
  if (a.key_bits == 32) {
    static_cast<uint32_t*>(a.out_vals)[oi] =
        (vk == Dt<kF32>::kZeroKey || vk == Dt<kF32>::kNanKey)
            ? __ldg(static_cast<const uint32_t*>(a.x) + row * a.len + pos)
            : value_bits_f32(vk);
  } else {
    static_cast<uint16_t*>(a.out_vals)[oi] =
        (vk == Dt<kBF16>::kZeroKey || vk == Dt<kBF16>::kNanKey)
            ? __ldg(static_cast<const uint16_t*>(a.x) + row * a.len + pos)
            : static_cast<uint16_t>(value_bits_bf16(vk));
  }
}


// Beyond this many compares per key on average, ranking inside groups by
// counting gives way to the LSD radix sort.
constexpr unsigned long long kMaxComparesPerKey = 24;

// Places keys by counting ("Rank by Counting": a key's place is the number
// of keys that outrank it; the keys are distinct, so places form a
// permutation).  The n keys of src are first grouped, largest group first,
// by their offset above the smallest key kmin, cut to its leading log2(NB)
// bits (NB equal slices of the range [kmin, kmax]), so a key only compares
// against its own group.  Slicing the range rather than taking the leading
// varying bits keeps groups small where keys straddle a carry (two adjacent
// values such as ...0111 and ...1000 vary in many bits but span a short
// range).  The keys are then ranked in grouped order,
// so the lanes of a warp mostly share a group: they read each group member
// once (a broadcast) and run the same number of steps.  Only groups starting
// in [split0, split1) are ranked here (how CTAs share the work); keys whose
// place base_place + rank lies in [w0, w1) are written out.  Returns false
// without writing when the largest group exceeds max_group, or when the
// groups are so uneven that counting would cost more than a radix sort.
template <int BLOCK, int NB>
__device__ bool place_by_groups(const uint64_t* src, int n, uint64_t kmin, uint64_t kmax, unsigned split0,
                                unsigned split1, uint64_t* grp, unsigned* gcount, unsigned* gstart,
                                unsigned* gcur, unsigned long long* s_tmp, unsigned max_group,
                                const SelParams& a, int64_t row, int64_t kout, int64_t base_place, int64_t w0,
                                int64_t w1) {
  static_assert(NB % BLOCK == 0, "whole groups per thread");
  static_assert(NB == 256 || NB == 512 || NB == 1024 || NB == 2048 || NB == 4096, "8 to 12 leading bits");
  constexpr int kBits = NB == 4096 ? 12 : (NB == 2048 ? 11 : (NB == 1024 ? 10 : (NB == 512 ? 9 : 8)));
  constexpr int kPer = NB / BLOCK;
  __shared__ unsigned s_gmax;
  __shared__ unsigned long long s_cost;
  const int tid = threadIdx.x;
  const uint64_t span = kmax - kmin;
  const int hb = span ? 63 - __clzll(static_cast<long long>(span)) : 0;
  const int dsh = hb >= kBits - 1 ? hb - (kBits - 1) : 0;  // (span >> dsh) < NB
  const unsigned mask = NB - 1;
  auto group = [&](uint64_t key) { return mask - static_cast<unsigned>((key - kmin) >> dsh); };
  for (int i = tid; i < NB; i += BLOCK) { gcount[i] = 0u; gcur[i] = 0u; }
  if (tid == 0) s_gmax = 0u;
  __syncthreads();
  for (int i = tid; i < n; i += BLOCK) atomicAdd(&gcount[group(src[i])], 1u);
  __syncthreads();
  TK_STAMP(22);
  if constexpr (NB == 1024) TK_BSP(4);  // (the bin sort's group count)
  unsigned c[kPer];
  unsigned long long sum = 0, sq = 0;
  unsigned mx = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    c[q] = gcount[tid * kPer + q];
    sum += c[q];
    sq += static_cast<unsigned long long>(c[q]) * c[q];
    mx = c[q] > mx ? c[q] : mx;
  }
  const unsigned long long incl = block_scan_incl(sum, s_tmp);
  unsigned run = static_cast<unsigned>(incl - sum);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    gstart[tid * kPer + q] = run;
    run += c[q];
  }
  // the counting costs sum(group size^2) compares: with a few large groups
  // (keys differing only in a few low value bits and the position) that
  // exceeds a radix sort's cost, and the caller sorts instead
  const unsigned long long compares = block_scan_incl(sq, s_tmp);
  if (tid == BLOCK - 1) s_cost = compares;
  mx = __reduce_max_sync(kFull, mx);  // one shared atomic per warp
  if ((threadIdx.x & 31) == 0) atomicMax(&s_gmax, mx);
  __syncthreads();
  TK_STAMP(23);
  if constexpr (NB == 1024) TK_BSP(5);  // (the bin sort's group count)
  if (blockIdx.x == 0 && threadIdx.x == 0) TK_DBG(0, s_gmax);
  if (s_gmax > max_group || s_cost > kMaxComparesPerKey * static_cast<unsigned long long>(n)) return false;
  for (int i = tid; i < n; i += BLOCK) {
    const uint64_t key = src[i];
    const unsigned g = group(key);
    grp[gstart[g] + atomicAdd(&gcur[g], 1u)] = key;
  }
  __syncthreads();
  TK_STAMP(25);
  if constexpr (NB == 1024) TK_BSP(6);  // (the bin sort's group count)
  for (int i = tid; i < n; i += BLOCK) {
    const uint64_t v = grp[i];
    const unsigned g = group(v);
    const unsigned g0 = gstart[g];
    if (g0 < split0 || g0 >= split1) continue;
    const unsigned g1 = g0 + gcount[g];
    const unsigned r = count_above(grp, g0, g1, v);
    const int64_t place = base_place + g0 + r;
    if (place >= w0 && place < w1) write_out(a, row, kout, place, v);
  }
#ifdef TK_PHASE_TIMING
  __syncthreads();
  TK_STAMP(26);
#endif
  return true;
}

// OR, AND, smallest and largest of src[0..n) over the block (n >= 1).
struct KeySpan {
  unsigned long long all_or, all_and;
  uint64_t kmin, kmax;
};
// Warp reductions of 64-bit values with the 32-bit redux instruction: OR and
// AND per half; the minimum (maximum) as the extreme high half, then the
// extreme low half among the lanes holding it.
__device__ __forceinline__ unsigned long long warp_or64(unsigned long long v) {
  return (static_cast<unsigned long long>(__reduce_or_sync(kFull, static_cast<unsigned>(v >> 32))) << 32) |
         __reduce_or_sync(kFull, static_cast<unsigned>(v));
}
__device__ __forceinline__ unsigned long long warp_and64(unsigned long long v) {
  return (static_cast<unsigned long long>(__reduce_and_sync(kFull, static_cast<unsigned>(v >> 32))) << 32) |
         __reduce_and_sync(kFull, static_cast<unsigned>(v));
}
__device__ __forceinline__ unsigned long long warp_min64(unsigned long long v) {
  const unsigned hi = __reduce_min_sync(kFull, static_cast<unsigned>(v >> 32));
  const unsigned lo = __reduce_min_sync(kFull, static_cast<unsigned>(v >> 32) == hi ? static_cast<unsigned>(v) : ~0u);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}
__device__ __forceinline__ unsigned long long warp_max64(unsigned long long v) {
  const unsigned hi = __reduce_max_sync(kFull, static_cast<unsigned>(v >> 32));
  const unsigned lo = __reduce_max_sync(kFull, static_cast<unsigned>(v >> 32) == hi ? static_cast<unsigned>(v) : 0u);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}
template <int BLOCK>
__device__ KeySpan block_span(const uint64_t* src, int n) {
  __shared__ unsigned long long s_span[4];
  unsigned long long o = 0, d = ~0ull, lo = ~0ull, hi = 0ull;
  for (int i = threadIdx.x; i < n; i += BLOCK) {
    const unsigned long long v = src[i];
    o |= v;
    d &= v;
    lo = v < lo ? v : lo;
    hi = v > hi ? v : hi;
  }
  if (threadIdx.x == 0) {
    s_span[0] = 0ull;
    s_span[1] = ~0ull;
    s_span[2] = ~0ull;
    s_span[3] = 0ull;
  }
  o = warp_or64(o);
  d = warp_and64(d);
  lo = warp_min64(lo);
  hi = warp_max64(hi);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {  // one shared atomic per warp and quantity
    atomicOr(&s_span[0], o);
    atomicAnd(&s_span[1], d);
    atomicMin(&s_span[2], lo);
    atomicMax(&s_span[3], hi);
  }
  __syncthreads();
  const KeySpan r{s_span[0], s_span[1], s_span[2], s_span[3]};
  __syncthreads();
  return r;
}

// Stable LSD radix sort of src[0..n) into descending key order, one 8-bit
// digit per pass, skipping digits on which all keys agree (bits of `vary`
// clear).  Each warp ranks a contiguous segment stably (lanes with equal
// digits found with one ballot per digit bit), per-warp counts are scanned
// per digit, and keys are scattered to the other buffer.  `scratch` holds kWarps*256 + 2*256 + kQuarters*256
// counters.  Returns the buffer holding the result.
template <int BLOCK, int P>
__device__ __noinline__ uint64_t* lsd_sort(uint64_t* src, uint64_t* dst, int n, unsigned long long vary, unsigned* scratch) {
  constexpr int kWarps = BLOCK / 32;
  constexpr int kQuarters = BLOCK / 256;
  constexpr int kWarpsPerQuarter = kWarps / kQuarters;
  constexpr int kItems = (P + BLOCK - 1) / BLOCK;
  __shared__ unsigned long long s_scan[32];
  unsigned* whist = scratch;
  unsigned* hist = whist + kWarps * 256;
  unsigned* gbase = hist + 256;
  unsigned* part = gbase + 256;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ipw = (n + kWarps - 1) / kWarps;  // items per warp segment
  const int seg0 = warp * ipw;
  const int seg1 = (seg0 + ipw < n) ? seg0 + ipw : n;
  const unsigned lt = lanemask_lt();
  for (int shift = 0; shift < 64; shift += 8) {
    if (((vary >> shift) & 0xffull) == 0) continue;  // uniform over the block
    for (int i = tid; i < kWarps * 256; i += BLOCK) whist[i] = 0u;
    __syncthreads();
    unsigned* wh = whist + warp * 256;
    uint64_t key[kItems];
    unsigned dig[kItems], wr[kItems];
    const int nj = (seg1 - seg0 + 31) >> 5;  // items per lane, uniform in the warp
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      if (j >= nj) break;
      const int i = seg0 + j * 32 + lane;
      const bool v = i < seg1;
      key[j] = v ? src[i] : 0ull;
      dig[j] = v ? 255u - static_cast<unsigned>((key[j] >> shift) & 255u) : 256u;
      // lanes with the same digit: one ballot per digit bit (cheaper here
      // than __match_any_sync); the lanes without a key share digit 256
      unsigned peers = kFull;
#pragma unroll
      for (int bit = 0; bit < 9; ++bit) {
        const bool set = (dig[j] >> bit) & 1u;
        const unsigned bal = __ballot_sync(kFull, set);
        peers &= set ? bal : ~bal;
      }
      const unsigned before = __popc(peers & lt);
      const unsigned b = v ? wh[dig[j]] : 0u;
      __syncwarp();
      if (v && before == 0) wh[dig[j]] = b + __popc(peers);
      __syncwarp();
      wr[j] = b + before;
    }
    __syncthreads();
    // exclusive prefix of the per-warp counts over warps, per digit, within
    // groups of warps and then across groups
    {
      const int d = tid & 255, q = tid >> 8;
      unsigned run = 0;
      for (int w = q * kWarpsPerQuarter; w < (q + 1) * kWarpsPerQuarter; ++w) {
        const unsigned t = whist[w * 256 + d];
        whist[w * 256 + d] = run;
        run += t;
      }
      part[q * 256 + d] = run;
      __syncthreads();
      unsigned qbase = 0;
      for (int q2 = 0; q2 < q; ++q2) qbase += part[q2 * 256 + d];
      if (qbase)
        for (int w = q * kWarpsPerQuarter; w < (q + 1) * kWarpsPerQuarter; ++w) whist[w * 256 + d] += qbase;
      if (q == kQuarters - 1) hist[d] = qbase + run;
    }
    __syncthreads();
    const unsigned long long tot = tid < 256 ? hist[tid] : 0ull;
    const unsigned long long incl = block_scan_incl(tot, s_scan);
    if (tid < 256) gbase[tid] = static_cast<unsigned>(incl - tot);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      if (j >= nj) break;
      const int i = seg0 + j * 32 + lane;
      if (i < seg1) dst[gbase[dig[j]] + wh[dig[j]] + wr[j]] = key[j];
    }
    __syncthreads();
    uint64_t* t = src;
    src = dst;
    dst = t;
  }
  return src;
}

template <int BLOCK, int P, int CB, int NB>
struct Layout {
  static constexpr int kWarps = BLOCK / 32;
  static constexpr int kQuarters = BLOCK / 256;          // thread groups of 256 (one per 8-bit digit)
  static constexpr int kDigitBits = NB == 2048 ? 11 : 8;
  static constexpr int kPer = NB / BLOCK;                // bins per thread in the scans
  // scratch of the local LSD sort: per-warp counters, totals, bases, partials
  static constexpr int kLsdWords = kWarps * 256 + 2 * 256 + kQuarters * 256;
  static constexpr int kWorkWords = (3 * NB > kLsdWords - 2 * NB) ? 3 * NB : kLsdWords - 2 * NB;
  static constexpr unsigned kGather = NB / 2 < 1024 ? NB / 2 : 1024;  // keys gathered into CTA 0
  static constexpr size_t kBufA = 0;
  static constexpr size_t kBufB = kBufA + sizeof(uint64_t) * P;
  static constexpr size_t kH2 = kBufB + sizeof(uint64_t) * CB;     // 2 x NB counters (cluster-visible)
  static constexpr size_t kWork = kH2 + sizeof(unsigned) * 2 * NB;  // kWorkWords counters
  static constexpr size_t kGorg = kWork + sizeof(unsigned) * kWorkWords;
  static constexpr size_t kXch = (kGorg + kGather + 15) / 16 * 16;
  // exchange words: 0-1 this CTA's OR / AND, 3 tau, 4 winner offset,
  // 8.. per-CTA counts (in CTA 0), 24.. every CTA's OR / AND (pushed)
  static constexpr int kXchWords = 24 + 2 * kMaxCluster;
  static constexpr size_t kBytes = kXch + sizeof(unsigned long long) * kXchWords;
  static_assert(CB >= P, "the second buffer holds a full local set");
  static_assert(BLOCK % 256 == 0, "one thread per 8-bit digit in each group of 256");
  static_assert(NB % BLOCK == 0, "whole bins per thread");
};


template <int BLOCK, int P, int CB, int NB, int SRC>
__device__ __forceinline__ void select_body(const SelParams& a) {
  using L = Layout<BLOCK, P, CB, NB>;
  constexpr int DB = L::kDigitBits;
  constexpr unsigned DM = NB - 1;
  constexpr int kPer = L::kPer;
  constexpr unsigned kGatherMax = L::kGather;
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* bufA = reinterpret_cast<uint64_t*>(smem + L::kBufA);
  uint64_t* bufB = reinterpret_cast<uint64_t*>(smem + L::kBufB);
  unsigned* h2 = reinterpret_cast<unsigned*>(smem + L::kH2);
  unsigned* work = reinterpret_cast<unsigned*>(smem + L::kWork);
  unsigned char* gorg = smem + L::kGorg;
  unsigned long long* xch = reinterpret_cast<unsigned long long*>(smem + L::kXch);
  __shared__ unsigned long long s_tmp[32];
  __shared__ unsigned long long s_info[6];
  __shared__ unsigned s_cnt;
  __shared__ unsigned s_gcount;
  __shared__ unsigned s_gbase;
  __shared__ unsigned s_wcnt[kMaxCluster];

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned G = cluster.num_blocks();
  const unsigned crank = cluster.block_rank();
  const int64_t row = blockIdx.x / G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Shared memory of another CTA may be used only once that CTA runs: arrive
  // now, wait before the first remote access.  The gather counter is cleared
  // first and released by the arrival, so no remote atomic precedes it.
  if (threadIdx.x == 0) s_gcount = 0u;
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  bool cluster_started = false;
  auto await_cluster = [&]() {
    if (!cluster_started) {
      asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
      cluster_started = true;
    }
  };
  auto gsync = [&]() {
    await_cluster();
    if (G > 1) cluster.sync(); else __syncthreads();
  };

  const bool from_buf = SRC == 0 || (SRC == 3 && s_source == 0);
  int64_t valid = from_buf ? a.key_stride : a.len;
  if (from_buf && a.counts) {
    const unsigned long long c = SRC == 3 ? s_prologue_r : __ldcg(a.counts + row);
    if (c < static_cast<unsigned long long>(valid)) valid = static_cast<int64_t>(c);
    // (relaxed recall: a row returned short holds padding sentinels up to slot r)
    if (a.relax_tau && valid < a.r && a.r <= a.key_stride) valid = a.r;
  }
  // slices start at even positions so key slices can be copied in 16-byte units
  const int64_t sb = (valid * crank / G) & ~int64_t(1);
  const int64_t se = (crank + 1 == G) ? valid : ((valid * (crank + 1) / G) & ~int64_t(1));
  if (tid == 0) s_cnt = 0u;
  if (tid < kMaxCluster) s_wcnt[tid] = 0u;
  TK_STAMP(0);
  TK_CTA(4, globaltimer_ns());

  // ------------------------------------------------------------------ load
  // The cache is the whole key buffer (both halves).  Whether the slices fit
  // is decided from sizes every CTA of the cluster sees alike.
  uint64_t* cache = bufA;
  const int64_t cache_cap = P + CB;
  // tau from the sample histogram: the first digit is already counted, and
  // only the boundary bucket's keys are read (streamed; cached if small)
  const bool from_hist = NB == 2048 && !a.want_topk && a.shist != nullptr;
  const bool fits = (valid + G - 1) / G + 2 <= cache_cap;
  bool cached = false;
  unsigned cache_n = 0;
  __syncthreads();
  if (fits) {
    const unsigned n = static_cast<unsigned>(se - sb);
    if (from_buf) {
      const uint64_t* from = a.keys + row * a.key_stride + sb;
      if (a.key_vec) {
        for (unsigned i = 2 * tid; i + 1 < n; i += 2 * BLOCK) cp_async16(cache + i, from + i);
        if ((n & 1u) && tid == 0) cache[n - 1] = __ldcg(from + n - 1);
        cp_async_wait_all();
      } else {
        for (unsigned i = tid; i < n; i += BLOCK) cache[i] = __ldcg(from + i);
      }
    } else {
      for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t k, bool in) {
        const unsigned slot = warp_append_slot(&s_cnt, in);
        if (in) cache[slot] = k;
      });
    }
    cached = true;
    cache_n = n;
    __syncthreads();
  }
  TK_STAMP(1);
  TK_CTA(0, globaltimer_ns());

  // ------------------------------------------------------------------ varying bits
  // Bits on which all keys agree are skipped: the first digit is the 11 (or
  // 8) bits below the most significant varying bit.  Streamed slices skip
  // this exchange and start at the top of the key.
  const int kb = a.key_bits + a.ib;
  unsigned long long all_or = (kb >= 64) ? ~0ull : ((1ull << kb) - 1ull), all_and = 0ull;
  if (fits && !from_hist) {
    // warp-reduce, then one shared atomic per warp; the CTA's result is
    // published in xch[0..1] and read by every CTA of the cluster
    if (tid == 0) { xch[0] = 0ull; xch[1] = ~0ull; }
    unsigned long long o = 0, d = ~0ull;
    for (unsigned i = tid; i < cache_n; i += BLOCK) { o |= cache[i]; d &= cache[i]; }
    TK_STAMP(19);
    TK_CTA(1, globaltimer_ns());
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      o |= __shfl_xor_sync(kFull, o, m);
      d &= __shfl_xor_sync(kFull, d, m);
    }
    __syncthreads();
    if (lane == 0 && static_cast<unsigned>(tid) < cache_n) {  // the warp holds keys
      atomicOr(&xch[0], o);
      atomicAnd(&xch[1], d);
    }
    __syncthreads();
    await_cluster();
    if (G == 1) {  // one CTA: its own result is the answer
      all_or = xch[0];
      all_and = xch[1];
    } else {
      // push this CTA's result into every CTA (remote stores need no reply)
      if (warp == 0 && static_cast<unsigned>(lane) < G) {
        unsigned long long* rx = cluster.map_shared_rank(xch, static_cast<unsigned>(lane));
        rx[24 + 2 * crank] = xch[0];
        rx[25 + 2 * crank] = xch[1];
      }
      TK_STAMP(20);
      gsync();  // every CTA's OR / AND has arrived
      TK_STAMP(21);
      TK_CTA(2, globaltimer_ns());
      all_or = 0ull;
      all_and = ~0ull;
      for (unsigned c = 0; c < G; ++c) {
        all_or |= xch[24 + 2 * c];
        all_and &= xch[25 + 2 * c];
      }
    }
  }
  TK_STAMP(2);

  // ------------------------------------------------------------------ select
  // Radix select of the r-th largest key with NB-bin digits.  Bins are
  // indexed in descending key order (bin = DM - digit), so places run with
  // the bin index.  The first pass's per-bin totals and this CTA's offsets
  // inside each bin are kept: they partition the winners later.
  const unsigned long long vary = all_or ^ all_and;
  const int hb = vary ? 63 - __clzll(static_cast<long long>(vary)) : 0;
  uint64_t pmask = (hb >= 63) ? 0ull : (~0ull << (hb + 1));
  uint64_t prefix = all_and & pmask;
  int shift = hb >= DB - 1 ? hb - (DB - 1) : 0;
  const int shift1 = shift;
  const uint64_t prefix1 = prefix, pmask1 = pmask;
  unsigned long long rank = static_cast<unsigned long long>(a.r);
  unsigned long long above_b1 = 0;   // this CTA's keys of the first-pass bin above the bucket
  unsigned long long above_all = 0;  // this CTA's keys above the bucket
  unsigned long long bucket_tot = 0, bucket_mine = static_cast<unsigned long long>(se - sb);
  unsigned long long bucket_before = 0;  // keys of the CTAs before this one in the bucket
  bool counted = false;                  // (a cluster pass counted the bucket per CTA)
  unsigned b1 = 0;
  unsigned* bst = work;           // first place of each first-pass bin
  unsigned* off = work + NB;      // this CTA's first place inside each first-pass bin
  unsigned* cur = work + 2 * NB;  // fill cursors
  int pass = 0;
  bool failed = false;
  // Large k with the bin sort to follow: when the whole first-pass bin of the
  // boundary fits the exchange buffer after the bins above it, every key of
  // those bins is placed and the bin sort takes the first r places of their
  // sorted order.  The exact r-th key is then never needed here: no further
  // passes and no gather.
  bool whole_bin = false;
  const bool whole_bin_ok = NB == kBinInfoBins && a.want_topk && a.handoff && G > 1;
  // Few winners (at most NB: h2's 2 x NB words hold them) and several CTAs:
  // the winners are collected in CTA 0, which sorts them all (see below).
  const bool collect = a.want_topk && G > 1 && !a.handoff && a.r <= static_cast<int64_t>(NB);
  unsigned long long b1_end = 0;  // end of the first-pass bin of the boundary
  // keys a CTA would cache for the remaining passes: in tau mode the bucket
  // only, otherwise the bucket and everything above it
  unsigned long long cache_need = bucket_mine;
  bool run_passes = true;
  if (from_hist) {
    // The sample kernel counted the keys by their leading DB bits (bins in
    // descending order); every CTA finds the same boundary bin from them.
    shift = kb - DB;
    pmask = (kb >= 64) ? 0ull : (~0ull << kb);
    prefix = 0ull;
    const unsigned* h = a.shist + row * NB;
    unsigned tt[kPer];
    unsigned long long tsum = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) { tt[q] = __ldcg(h + tid * kPer + q); tsum += tt[q]; }
    if (tid == 0) s_info[0] = ~0ull;
    const unsigned long long tincl = block_scan_incl(tsum, s_tmp);
    unsigned long long trun = tincl - tsum;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      if (trun < rank && rank <= trun + tt[q]) {
        s_info[0] = static_cast<unsigned long long>(tid * kPer + q);
        s_info[1] = trun;
        s_info[2] = tt[q];
      }
      trun += tt[q];
    }
    __syncthreads();
    if (s_info[0] == ~0ull) {
      failed = true;
      run_passes = false;
    } else {
      prefix |= static_cast<uint64_t>(DM - static_cast<unsigned>(s_info[0])) << shift;
      pmask |= static_cast<uint64_t>(DM) << shift;
      rank -= s_info[1];
      bucket_tot = s_info[2];
      cache_need = bucket_tot;  // an upper bound of every CTA's share
      run_passes = bucket_tot > kGatherMax && shift > 0;
      if (run_passes) shift = shift >= DB ? shift - DB : 0;
    }
    __syncthreads();
  }
  for (; run_passes; ++pass) {
    unsigned* hc = h2 + (pass & 1) * NB;
    const bool will_cache = !cached && cache_need <= static_cast<unsigned long long>(cache_cap);
    for (int i = tid; i < NB; i += BLOCK) hc[i] = 0u;
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    // (plain shared atomics: merging equal bins of a warp with
    // __match_any_sync first measured several times slower)
    auto count = [&](uint64_t k, bool in) {
      if (in && (k & pmask) == prefix) atomicAdd(&hc[DM - static_cast<unsigned>((k >> shift) & DM)], 1u);
    };
    if (cached) {
      for_cache<BLOCK>(cache, cache_n, count);
    } else {
      for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t k, bool in) {
        count(k, in);
        if (will_cache) {
          const bool want = in && (a.want_topk ? k >= prefix : (k & pmask) == prefix);
          const unsigned slot = warp_append_slot(&s_cnt, want);
          if (want && slot < static_cast<unsigned>(cache_cap)) cache[slot] = k;
        }
      });
    }
    if (tid == 0) s_info[0] = ~0ull;
    if (pass == 0) TK_STAMP(15);
    if (pass == 0) TK_CTA(3, globaltimer_ns());
    gsync();  // every CTA's counts of this pass are complete
    if (pass == 0) TK_STAMP(16);
    if (will_cache) {
      cached = true;
      cache_n = s_cnt;
    }
    // totals over the cluster, this CTA's counts, and the counts of the CTAs
    // before it, for this thread's kPer consecutive bins
    // (remote loads are issued eight CTAs at a time, before any is used;
    // CTAs start at different ranks so no CTA's counters are read by all at
    // once; the loops run to G, not to the largest cluster)
    unsigned tt[kPer], mm[kPer], bf[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) { tt[q] = 0u; bf[q] = 0u; mm[q] = hc[tid * kPer + q]; }
    for (unsigned c0 = 0; c0 < G; c0 += 8) {
      const unsigned nb = G - c0 < 8u ? G - c0 : 8u;
      unsigned rv[8][kPer];
      unsigned src = crank + c0;
      if (src >= G) src -= G;
#pragma unroll
      for (unsigned j = 0; j < 8; ++j) {
        if (j < nb) {
          const unsigned* r = cluster.map_shared_rank(hc, src) + tid * kPer;
          if constexpr (kPer == 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(r);
            rv[j][0] = v.x;
            rv[j][1] = v.y;
          } else if constexpr (kPer == 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(r);
            rv[j][0] = v.x;
            rv[j][1] = v.y;
            rv[j][2] = v.z;
            rv[j][3] = v.w;
          } else {
#pragma unroll
            for (int q = 0; q < kPer; ++q) rv[j][q] = r[q];
          }
          if (++src == G) src = 0;
        }
      }
      src = crank + c0;
      if (src >= G) src -= G;
#pragma unroll
      for (unsigned j = 0; j < 8; ++j) {
        if (j < nb) {
#pragma unroll
          for (int q = 0; q < kPer; ++q) {
            tt[q] += rv[j][q];
            if (src < crank) bf[q] += rv[j][q];
          }
          if (++src == G) src = 0;
        }
      }
    }
    if (pass == 0) TK_STAMP(17);
    unsigned long long tsum = 0, msum = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) { tsum += tt[q]; msum += mm[q]; }
    const unsigned long long tincl = block_scan_incl(tsum, s_tmp);
    const unsigned long long mincl = block_scan_incl(msum, s_tmp);
    unsigned long long trun = tincl - tsum, mrun = mincl - msum;
    if (pass == 0) TK_STAMP(18);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int b = tid * kPer + q;
      if (pass == 0 && a.want_topk && G > 1) {
        // this CTA's keys of bin b go to places trun + bf[q] + j; cur[b]
        // starts at their place among this CTA's own keys (mrun), so that
        // off[b] + (mrun + j) is the place (unsigned arithmetic wraps)
        bst[b] = static_cast<unsigned>(trun);
        off[b] = static_cast<unsigned>(trun) + bf[q] - static_cast<unsigned>(mrun);
        cur[b] = static_cast<unsigned>(mrun);
      }
      if (trun < rank && rank <= trun + tt[q]) {
        s_info[0] = static_cast<unsigned long long>(b);
        s_info[1] = trun;
        s_info[2] = tt[q];
        s_info[3] = mrun;   // this CTA's keys in the bins above
        s_info[4] = mm[q];
        s_info[5] = bf[q];  // keys of the CTAs before this one in the bucket
      }
      trun += tt[q];
      mrun += mm[q];
    }
    __syncthreads();
    if (s_info[0] == ~0ull) { failed = true; break; }
    const unsigned bin = static_cast<unsigned>(s_info[0]);
    prefix |= static_cast<uint64_t>(DM - bin) << shift;
    pmask |= static_cast<uint64_t>(DM) << shift;
    rank -= s_info[1];
    bucket_tot = s_info[2];
    above_all += s_info[3];
    if (pass == 0) { b1 = bin; b1_end = s_info[1] + s_info[2]; } else above_b1 += s_info[3];
    bucket_mine = s_info[4];
    bucket_before = s_info[5];
    counted = true;
    cache_need = a.want_topk ? above_all + bucket_mine : bucket_mine;
    TK_STAMP(3 + (pass < 6 ? pass : 6));
    __syncthreads();  // s_info is rewritten by the next pass
    if (whole_bin_ok && pass == 0 && b1_end <= static_cast<unsigned long long>(a.xstride)) {
      whole_bin = true;  // (the same totals in every CTA: the same choice)
      break;
    }
    if (bucket_tot <= kGatherMax || shift == 0) break;
    shift = shift >= DB ? shift - DB : 0;
  }
  if (failed) {
    if (tid == 0 && crank == 0) atomicCAS(a.status, kDevOk, kDevBadState);
    gsync();  // no CTA leaves while another may still read its counters
    return;
  }

  // ------------------------------------------------------------------ gather
  // The boundary bucket (at most kGather keys) is gathered into CTA 0, in the
  // half of its counter area the last pass did not use, and ranked by
  // counting ("Rank by Counting").  Each key carries the CTA it came from,
  // so CTA 0 also counts every CTA's winners inside the first-pass bin.
  await_cluster();  // (when no pass ran) CTA 0 must be running before it is written
  if (!whole_bin) {
    // Each CTA writes its bucket keys to its own range of CTA 0's buffer: the
    // range starts after the keys of the CTAs before it, known from the last
    // pass's counts or, when no pass ran, reserved with one remote atomic per
    // CTA (one per warp on a single counter serialised on CTA 0).
    uint64_t* gb0 = cluster.map_shared_rank(reinterpret_cast<uint64_t*>(h2 + ((pass + 1) & 1) * NB), 0);
    unsigned* gc0 = cluster.map_shared_rank(&s_gcount, 0);
    unsigned char* go0 = cluster.map_shared_rank(gorg, 0);
    auto each = [&](auto&& f) {
      if (cached) {
        for_cache<BLOCK>(cache, cache_n, f);
      } else {
        for_slice<SRC, BLOCK>(a, row, sb, se, f);
      }
    };
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    TK_STAMP(32);
    if (!counted) {
      each([&](uint64_t k, bool in) {
        const unsigned m = __ballot_sync(kFull, in && (k & pmask) == prefix);
        if (lane == 0 && m) atomicAdd(&s_cnt, static_cast<unsigned>(__popc(m)));
      });
      __syncthreads();
      TK_STAMP(33);
      if (tid == 0) {
        s_gbase = atomicAdd(gc0, s_cnt);
        s_cnt = 0u;
      }
      __syncthreads();
      TK_STAMP(34);
    }
    const unsigned gbase = counted ? static_cast<unsigned>(bucket_before) : s_gbase;
    if (cached) {
      cache_append<BLOCK>(cache, cache_n, &s_cnt, [&](uint64_t k) { return (k & pmask) == prefix; },
                          [&](uint64_t k, unsigned slot) {
                            if (gbase + slot < kGatherMax) {
                              gb0[gbase + slot] = k;
                              go0[gbase + slot] = static_cast<unsigned char>(crank);
                            }
                          });
    } else {
      for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t k, bool in) {
        const bool want = in && (k & pmask) == prefix;
        const unsigned slot = gbase + warp_append_slot(&s_cnt, want);
        if (want && slot < kGatherMax) {
          gb0[slot] = k;
          go0[slot] = static_cast<unsigned char>(crank);
        }
      });
    }
    // (collecting: this CTA's winners above the bucket, so that CTA 0 hands
    // every CTA the first place of its winners)
    if (tid == 0) cluster.map_shared_rank(xch, 0)[8 + crank] = collect ? above_all : above_b1;
    TK_STAMP(35);
  }
  TK_CTA(5, globaltimer_ns());
  if (!whole_bin) gsync();  // the bucket is in CTA 0
  TK_CTA(6, globaltimer_ns());
  TK_STAMP(36);
  if (crank == 0 && !whole_bin) {
    const uint64_t* g = reinterpret_cast<const uint64_t*>(h2 + ((pass + 1) & 1) * NB);
    const unsigned long long gn = counted ? bucket_tot : static_cast<unsigned long long>(s_gcount);
    const unsigned n = gn < kGatherMax ? static_cast<unsigned>(gn) : kGatherMax;
    if (tid == 0) xch[3] = 0ull;
    if (tid == 0 && gn > kGatherMax) atomicCAS(a.status, kDevOk, kDevBadState);
    // Local radix passes (8-bit digits, below the keys' highest varying bit)
    // narrow the bucket to at most 32 keys, which are then ranked by
    // counting: counting all of up to kGather keys against each other would
    // cost n^2 / 32 shared-memory wavefronts.  The counters of the last
    // cluster pass (h2's other half) are free here.
    bucket_kth<BLOCK>(g, n, rank, h2 + (pass & 1) * NB, s_tmp, s_info, &s_cnt, reinterpret_cast<uint64_t*>(&xch[3]));
    __syncthreads();
    const uint64_t tau = xch[3];
    if (!a.want_topk) {
      if (tid == 0) a.tau_out[row] = tau;
    } else {
      for (unsigned i = tid; i < n; i += BLOCK)
        if (g[i] >= tau) atomicAdd(&s_wcnt[gorg[i]], 1u);
      __syncthreads();
      if (tid == 0) {
        unsigned long long run = 0;
        for (unsigned c = 0; c < G; ++c) {
          unsigned long long* rx = cluster.map_shared_rank(xch, c);
          rx[3] = tau;
          rx[4] = run;  // winners of the first-pass bin (collecting: all winners) of the CTAs before c
          run += xch[8 + c] + s_wcnt[c];
        }
      }
    }
  }
  TK_STAMP(10);
  if (!a.want_topk) return;  // nothing reads another CTA's shared memory any more
  if (!whole_bin) gsync();  // tau and the offsets are delivered
  // whole-bin mode: every key of the bins down to the boundary's is placed
  const uint64_t tau = whole_bin ? (prefix1 | (static_cast<uint64_t>(DM - b1) << shift1)) : xch[3];
  const int64_t k = a.r;

  int n_c = 0;
  int64_t place0 = 0, my0 = 0, my1 = k;
  if (G == 1) {
    // One CTA holds every winner: compact them to the front of the cache
    // (each chunk is read into registers before any of it is overwritten).
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    if (cached && k <= static_cast<int64_t>(NB)) {
      // Few winners: appended to the counters' space (free once tau is
      // known; NB keys fit), so no chunk of the cache has to be held in
      // registers while the front of it is overwritten; then copied to the
      // front of the cache.
      uint64_t* win = reinterpret_cast<uint64_t*>(h2);
      for (unsigned base = 0; base < cache_n; base += 8 * BLOCK) {
        uint64_t kk[8];
        unsigned wm = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const unsigned i = base + j * BLOCK + tid;
          kk[j] = i < cache_n ? cache[i] : 0ull;
          wm |= (i < cache_n && kk[j] >= tau ? 1u : 0u) << j;
        }
        const unsigned c = __popc(wm);
        unsigned incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += y;
        }
        unsigned wbase = 0;
        if (lane == 31 && incl) wbase = atomicAdd(&s_cnt, incl);
        wbase = __shfl_sync(kFull, wbase, 31);
        unsigned slot = wbase + incl - c;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if ((wm >> j) & 1u) {
            if (slot < static_cast<unsigned>(k)) win[slot] = kk[j];
            ++slot;
          }
      }
      __syncthreads();
      for (int i = tid; i < static_cast<int>(k); i += BLOCK) bufA[i] = win[i];
    } else if (cached) {
      for (unsigned base = 0; base < cache_n; base += 8 * BLOCK) {
        uint64_t kk[8];
        unsigned wm = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const unsigned i = base + j * BLOCK + tid;
          kk[j] = i < cache_n ? cache[i] : 0ull;
          wm |= (i < cache_n && kk[j] >= tau ? 1u : 0u) << j;
        }
        // this thread's winners go to consecutive slots: a warp scan of the
        // counts and one shared atomic per warp
        const unsigned c = __popc(wm);
        unsigned incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += y;
        }
        unsigned wbase = 0;
        if (lane == 31 && incl) wbase = atomicAdd(&s_cnt, incl);
        wbase = __shfl_sync(kFull, wbase, 31);
        __syncthreads();  // the whole chunk is in registers before any slot is written
        unsigned slot = wbase + incl - c;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if ((wm >> j) & 1u) {
            if (slot < static_cast<unsigned>(P)) bufA[slot] = kk[j];
            ++slot;
          }
        __syncthreads();
      }
    } else {
      for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t key, bool in) {
        const bool w = in && key >= tau;
        const unsigned slot = warp_append_slot(&s_cnt, w);
        if (w && slot < static_cast<unsigned>(P)) bufA[slot] = key;
      });
    }
    __syncthreads();
    if (s_cnt != static_cast<unsigned>(k)) {
      if (tid == 0) atomicCAS(a.status, kDevOk, kDevBadState);
      return;
    }
    n_c = static_cast<int>(k);
  } else if (collect) {
    // ------------------------------------------------------------------ collect
    // Every CTA sends its winners to CTA 0, from the first place CTA 0 handed
    // it (xch[4]); CTA 0 sorts all of them.  No exchange through global
    // memory, and no CTA ranks keys that belong to another CTA's places.
    uint64_t* col0 = cluster.map_shared_rank(reinterpret_cast<uint64_t*>(h2), 0);
    const unsigned cbase = static_cast<unsigned>(xch[4]);
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    if (cached) {
      cache_append<BLOCK>(cache, cache_n, &s_cnt, [&](uint64_t key) { return key >= tau; },
                          [&](uint64_t key, unsigned slot) {
                            if (cbase + slot < static_cast<unsigned>(k)) col0[cbase + slot] = key;
                          });
    } else {
      for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t key, bool in) {
        const bool w = in && key >= tau;
        const unsigned slot = cbase + warp_append_slot(&s_cnt, w);
        if (w && slot < static_cast<unsigned>(k)) col0[slot] = key;
      });
    }
    gsync();  // every winner is in CTA 0
    if (crank != 0) return;
    const uint64_t* col = reinterpret_cast<const uint64_t*>(h2);
    for (int i = tid; i < static_cast<int>(k); i += BLOCK) bufA[i] = col[i];
    n_c = static_cast<int>(k);
  } else {
    // ------------------------------------------------------------------ partition
    // Every winner (key >= tau) goes to its first-pass bin's segment of the
    // exchange buffer (bins in descending order: the bins' places).  Inside
    // the first-pass bin of the boundary, this CTA's winners start after those
    // of the CTAs before it.
    // (whole-bin mode: the boundary bin too is split by CTA as the others)
    uint64_t* xb = a.xbuf + row * a.xstride;
    const unsigned long long xend = whole_bin ? b1_end : static_cast<unsigned long long>(k);
    if (tid == 0 && !whole_bin) off[b1] = bst[b1] + static_cast<unsigned>(xch[4]) - cur[b1];
    __syncthreads();
    {
      auto bin_of = [&](uint64_t key) { return DM - static_cast<unsigned>((key >> shift1) & DM); };
      auto put = [&](uint64_t key) {
        const unsigned b = bin_of(key);
        const unsigned pos = off[b] + atomicAdd(&cur[b], 1u);
        if (pos < xend) xb[pos] = key;
      };
      if (cached && cache_n <= static_cast<unsigned>(P)) {
        // Staged: the winners are first sorted by bin inside this CTA (the
        // second buffer is free while the cache fits the first), at their
        // places among this CTA's keys, which are dense from 0; each then
        // goes to off[bin] + its staged index, so consecutive threads write
        // consecutive places of a bin (scattered 8-byte stores cost one
        // memory transaction each).
        uint64_t* stage = bufB;
#pragma unroll 4
        for (unsigned i = tid; i < cache_n; i += BLOCK) {
          const uint64_t key = cache[i];
          if (key >= tau) stage[atomicAdd(&cur[bin_of(key)], 1u)] = key;
        }
        __syncthreads();
        const unsigned nst = cur[b1];
#pragma unroll 4
        for (unsigned i = tid; i < nst && i < static_cast<unsigned>(CB); i += BLOCK) {
          const uint64_t key = stage[i];
          const unsigned pos = off[bin_of(key)] + i;
          if (pos < xend) xb[pos] = key;
        }
      } else if (cached) {
        for (unsigned i = tid; i < cache_n; i += BLOCK)
          if (cache[i] >= tau) put(cache[i]);
      } else {
        for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t key, bool in) {
          if (in && key >= tau) put(key);
        });
      }
    }
    gsync();  // all winners are in the exchange buffer
    TK_STAMP(11);
    if constexpr (NB == kBinInfoBins) {
      if (a.handoff) {
        // the bin sort grid takes over from here: publish the bins
        if (crank == 0) {
          unsigned* bo = a.binfo + row * binfo_words(k);
          for (int i = tid; i < NB; i += BLOCK) bo[i] = bst[i];
          publish_chunks(bst, static_cast<unsigned>(xend), k, bo + NB + kBinfoHeaderWords, tid, BLOCK);
          if (tid == 0) {
            bo[NB] = static_cast<unsigned>(prefix1);
            bo[NB + 1] = static_cast<unsigned>(prefix1 >> 32);
            bo[NB + 2] = static_cast<unsigned>(pmask1);
            bo[NB + 3] = static_cast<unsigned>(pmask1 >> 32);
            bo[NB + 4] = static_cast<unsigned>(shift1);
            bo[NB + 5] = static_cast<unsigned>(xend);
            bo[NB + 6] = 0u;  // digits of the keys themselves (no base)
            bo[NB + 7] = 0u;
            bo[NB + 8] = 0u;  // the keys are in the exchange buffer
          }
        }
        return;
      }
    }

    // ------------------------------------------------------------------ local sort
    // CTA c owns the places [my0, my1).  It takes the first-pass bins that
    // overlap them; a bin at either end that would overflow shared memory is
    // cut, by further digits read from the exchange buffer, down to the
    // sub-bin holding the boundary place.  The keys between the two cuts are a
    // contiguous key range, sorted here.
    const int64_t pe = (k + G - 1) / G;
    my0 = static_cast<int64_t>(crank) * pe;
    if (my0 >= k) return;
    my1 = my0 + pe < k ? my0 + pe : k;
    auto bin_end = [&](unsigned b) -> int64_t {
      const int64_t e = (b + 1 < static_cast<unsigned>(NB)) ? static_cast<int64_t>(bst[b + 1]) : k;
      return e < k ? e : k;
    };
    // bins holding places my0 and my1 - 1
    if (tid == 0) { s_info[0] = 0; s_info[1] = 0; }
    __syncthreads();
  #pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const unsigned b = tid * kPer + q;
      const int64_t s = bst[b], e = bin_end(b);
      if (s <= my0 && my0 < e) s_info[0] = b;
      if (s <= my1 - 1 && my1 - 1 < e) s_info[1] = b;
    }
    __syncthreads();
    const unsigned bfirst = static_cast<unsigned>(s_info[0]), blast = static_cast<unsigned>(s_info[1]);
    __syncthreads();
    const int64_t r0 = bst[bfirst], r1 = bin_end(blast);  // the exchange-buffer range to read
    uint64_t hi_key = ~0ull, lo_key = 0ull;               // key range of the local set
    place0 = r0;                                          // its places
    int64_t place1 = r1;
    if (r1 - r0 > P) {
      const int64_t lim = (P - (my1 - my0)) / 2;
      unsigned* lh = h2;  // free now: no CTA reads counters any more
      // cut bin b down to the sub-bin holding place p; returns its key prefix,
      // mask and place range
      auto cut = [&](unsigned b, int64_t p, uint64_t& pre, uint64_t& msk, int64_t& s0, int64_t& s1) -> bool {
        pre = prefix1 | (static_cast<uint64_t>(DM - b) << shift1);
        msk = pmask1 | (static_cast<uint64_t>(DM) << shift1);
        const int64_t s = bst[b], e = bin_end(b);
        s0 = s;
        s1 = e;
        int sh = shift1;
        while (s1 - s0 > lim && sh > 0) {
          const int sh2 = sh >= DB ? sh - DB : 0;
          for (int i = tid; i < NB; i += BLOCK) lh[i] = 0u;
          if (tid == 0) s_info[2] = ~0ull;
          __syncthreads();
          for (int64_t i = s + tid; i < e; i += BLOCK) {
            const uint64_t key = __ldcg(xb + i);
            if ((key & msk) == pre) atomicAdd(&lh[DM - static_cast<unsigned>((key >> sh2) & DM)], 1u);
          }
          __syncthreads();
          unsigned cc[kPer];
          unsigned long long csum = 0;
  #pragma unroll
          for (int q = 0; q < kPer; ++q) { cc[q] = lh[tid * kPer + q]; csum += cc[q]; }
          const unsigned long long cincl = block_scan_incl(csum, s_tmp);
          unsigned long long crun = static_cast<unsigned long long>(s0) + cincl - csum;
  #pragma unroll
          for (int q = 0; q < kPer; ++q) {
            if (crun <= static_cast<unsigned long long>(p) && static_cast<unsigned long long>(p) < crun + cc[q]) {
              s_info[2] = static_cast<unsigned long long>(tid * kPer + q);
              s_info[3] = crun;
              s_info[4] = cc[q];
            }
            crun += cc[q];
          }
          __syncthreads();
          if (s_info[2] == ~0ull) return false;
          pre |= static_cast<uint64_t>(DM - static_cast<unsigned>(s_info[2])) << sh2;
          msk |= static_cast<uint64_t>(DM) << sh2;
          s0 = static_cast<int64_t>(s_info[3]);
          s1 = s0 + static_cast<int64_t>(s_info[4]);
          sh = sh2;
          __syncthreads();
        }
        return true;
      };
      uint64_t pre, msk;
      int64_t s0, s1;
      bool ok = cut(bfirst, my0, pre, msk, s0, s1);
      hi_key = pre | ~msk;
      place0 = s0;
      ok = ok && cut(blast, my1 - 1, pre, msk, s0, s1);
      lo_key = pre;
      place1 = s1;
      if (!ok || place1 - place0 > P) {
        if (tid == 0) atomicCAS(a.status, kDevOk, kDevBadState);
        return;
      }
    }
    n_c = static_cast<int>(place1 - place0);
    if (r1 - r0 <= P) {
      for (int i = tid; i < n_c; i += BLOCK) bufA[i] = __ldcg(xb + r0 + i);
    } else {
      if (tid == 0) s_cnt = 0u;
      __syncthreads();
      const unsigned lane_u = static_cast<unsigned>(lane);
      for (int64_t iw = r0 + (tid & ~31); iw < r1; iw += BLOCK) {
        const int64_t i = iw + lane_u;
        const uint64_t key = i < r1 ? __ldcg(xb + i) : 0ull;
        const bool want = i < r1 && key <= hi_key && key >= lo_key;
        const unsigned slot = warp_append_slot(&s_cnt, want);
        if (want && slot < static_cast<unsigned>(P)) bufA[slot] = key;
      }
      __syncthreads();
      if (s_cnt != static_cast<unsigned>(n_c)) {
        if (tid == 0) atomicCAS(a.status, kDevOk, kDevBadState);
        return;
      }
    }
  }
  __syncthreads();
  TK_STAMP(12);
  {
    const KeySpan sp = block_span<BLOCK>(bufA, n_c);
    // (up to 1024 keys: 512 groups, a quarter of the counters to clear and
    // scan, still ~2 keys a group)
    constexpr int kFewGroups = NB > 512 && BLOCK <= 512 ? 512 : NB;
    const bool placed =
        n_c <= 1024 ? place_by_groups<BLOCK, kFewGroups>(bufA, n_c, sp.kmin, sp.kmax, 0u, ~0u, bufB, work,
                                                         work + kFewGroups, work + 2 * kFewGroups, s_tmp, 512u, a,
                                                         row, k, place0, my0, my1)
                    : place_by_groups<BLOCK, NB>(bufA, n_c, sp.kmin, sp.kmax, 0u, ~0u, bufB, work, work + NB,
                                                 work + 2 * NB, s_tmp, 512u, a, row, k, place0, my0, my1);
    if (placed) {
      TK_STAMP(13);
      return;
    }
    // a group too large to rank by counting: stable LSD radix sort, one
    // 8-bit digit per pass, of the digits on which the local keys differ
    const uint64_t* sorted = lsd_sort<BLOCK, P>(bufA, bufB, n_c, sp.all_or ^ sp.all_and, h2);
    for (int i = tid; i < n_c; i += BLOCK) {
      const int64_t place = place0 + i;
      if (place >= my0 && place < my1) write_out(a, row, k, place, sorted[i]);
    }
    TK_STAMP(14);
  }
}

// Refinement of one selection whose filter left its survivors in bin regions
// (2048 bins of the survivors' offset above tau, kBinRegionCap keys a bin):
// the k winners are the keys of the bins above the boundary bin and the top
// of that bin, read straight from the regions by CTA 0 -- no pass over the
// candidate buffer, no exchange between the cluster's CTAs.  Every CTA reads
// the same words and the same histogram, so all take the same decision;
// false (everywhere) when the regions cannot serve: incomplete, or more keys
// down to the boundary bin than the first buffer holds.  The caller then
// selects from the buffer as usual.  No miss (checked by the caller).
template <int BLOCK, int P, int CB, int NB>
__device__ bool select_from_regions(const SelParams& a) {
  if constexpr (NB != kBinInfoBins) {
    return false;
  } else {
    using L = Layout<BLOCK, P, CB, NB>;
    constexpr int kPer = NB / BLOCK;
    static_assert(kPer == 4, "one 16-byte load of counters a thread");
    extern __shared__ __align__(16) unsigned char smem[];
    uint64_t* bufA = reinterpret_cast<uint64_t*>(smem + L::kBufA);
    uint64_t* bufB = reinterpret_cast<uint64_t*>(smem + L::kBufB);
    unsigned* h2 = reinterpret_cast<unsigned*>(smem + L::kH2);
    unsigned* work = reinterpret_cast<unsigned*>(smem + L::kWork);
    unsigned* bst = work;  // every bin's first place (NB words)
    __shared__ unsigned long long r_tmp[32];
    __shared__ unsigned long long r_info[6];
    __shared__ unsigned r_cnt;
    __shared__ uint64_t r_kappa;
    __shared__ unsigned long long r_words[2];
    const int tid = threadIdx.x;
    const int64_t k = a.r;
    const int64_t row = 0;
    if (tid == 0) {
      r_words[0] = __ldcg(a.rctl + kRefineGridBinnedWord);  // 0: the regions are complete
      r_info[0] = ~0ull;
    }
    const uint4 hc = ldcg_u4(a.rctl + kRefineGridFilterHist + tid * kPer);
    const unsigned c[kPer] = {hc.x, hc.y, hc.z, hc.w};
    unsigned long long sum = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) sum += c[q];
    const unsigned long long incl = block_scan_incl(sum, r_tmp);  // (synchronises the block)
    unsigned run = static_cast<unsigned>(incl - sum);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const unsigned b = tid * kPer + q;
      bst[b] = run;
      if (run < static_cast<unsigned long long>(k) && static_cast<unsigned long long>(k) <= run + static_cast<unsigned long long>(c[q])) {
        r_info[0] = b;
        r_info[1] = run;
        r_info[2] = c[q];
      }
      run += c[q];
    }
    __syncthreads();
    const unsigned bb = static_cast<unsigned>(r_info[0]);
    const unsigned bb_start = static_cast<unsigned>(r_info[1]), bb_tot = static_cast<unsigned>(r_info[2]);
    // (the top bin -- keys beyond 2047 << shift, no plain digit -- needs no
    // care here: its keys are ranked and sorted as keys, like any other)
    const bool ok = r_words[0] == 0ull && r_info[0] != ~0ull &&
                    static_cast<int64_t>(bb_start) + bb_tot <= static_cast<int64_t>(P);
    if (!ok) {
      __syncthreads();  // (bst and the words are rewritten by the usual selection)
      return false;
    }
    cg::cluster_group cluster = cg::this_cluster();
    if (cluster.block_rank() != 0) return true;
    TK_STAMP(37);
    // the keys of bins 0..bb, in place order: each place's bin by a search
    // of the bin starts in a fixed number of steps, four places of a thread
    // at once so that their searches and loads overlap
    const unsigned n = bb_start + bb_tot;
    constexpr int kJ = 4;
    for (unsigned base = 0; base < n; base += kJ * BLOCK) {
      unsigned pl[kJ], bl[kJ];
      uint64_t key[kJ];
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        pl[j] = base + j * BLOCK + tid;
        bl[j] = 0u;
      }
#pragma unroll
      for (unsigned stp = NB / 2; stp > 0; stp >>= 1)
#pragma unroll
        for (int j = 0; j < kJ; ++j)
          if (bl[j] + stp <= bb && bst[bl[j] + stp] <= pl[j]) bl[j] += stp;
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        key[j] = pl[j] < n ? __ldcg(a.region + static_cast<int64_t>(bl[j]) * kBinRegionCap + (pl[j] - bst[bl[j]]))
                           : 0ull;
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        if (pl[j] < n) bufA[pl[j]] = key[j];
    }
    __syncthreads();
    TK_STAMP(38);
    // the boundary bin's top (k - bb_start) keys: its key of that rank, then
    // those at or above it (distinct keys: exactly that many) after the bins
    // above, through the second buffer
    const unsigned r = static_cast<unsigned>(k) - bb_start;
    bucket_kth<BLOCK>(bufA + bb_start, bb_tot, r, h2, r_tmp, r_info, &r_cnt, &r_kappa);
    __syncthreads();
    TK_STAMP(39);
    const uint64_t kap = r_kappa;
    if (tid == 0) r_cnt = 0u;
    __syncthreads();
    for (unsigned b0 = 0; b0 < bb_tot; b0 += BLOCK) {
      const unsigned i = b0 + tid;
      const uint64_t key = i < bb_tot ? bufA[bb_start + i] : 0ull;
      const bool w = i < bb_tot && key >= kap;
      const unsigned slot = warp_append_slot(&r_cnt, w);
      if (w && slot < r) bufB[slot] = key;
    }
    __syncthreads();
    if (r_cnt != r) {
      if (tid == 0) atomicCAS(a.status, kDevOk, kDevBadState);
      return true;
    }
    for (unsigned i = tid; i < r; i += BLOCK) bufA[bb_start + i] = bufB[i];
    __syncthreads();
    TK_STAMP(40);
    // the k winners sorted and written (as the selection below does)
    const int n_c = static_cast<int>(k);
    const KeySpan sp = block_span<BLOCK>(bufA, n_c);
    constexpr int kFewGroups = NB > 512 && BLOCK <= 512 ? 512 : NB;
    const bool placed =
        n_c <= 1024 ? place_by_groups<BLOCK, kFewGroups>(bufA, n_c, sp.kmin, sp.kmax, 0u, ~0u, bufB, work,
                                                         work + kFewGroups, work + 2 * kFewGroups, r_tmp, 512u, a,
                                                         row, k, 0, 0, k)
                    : place_by_groups<BLOCK, NB>(bufA, n_c, sp.kmin, sp.kmax, 0u, ~0u, bufB, work, work + NB,
                                                 work + 2 * NB, r_tmp, 512u, a, row, k, 0, 0, k);
    if (placed) {
      TK_STAMP(41);
      return true;
    }
    const uint64_t* sorted = lsd_sort<BLOCK, P>(bufA, bufB, n_c, sp.all_or ^ sp.all_and, h2);
    for (int i = tid; i < n_c; i += BLOCK) write_out(a, row, k, i, sorted[i]);
    TK_STAMP(42);
    return true;
  }
}

template <int BLOCK, int P, int CB, int NB, int SRC>
__global__ void __launch_bounds__(BLOCK, min_blocks<BLOCK>()) select_kernel(SelParams a) {
#ifdef TK_PHASE_TIMING
  if (blockIdx.x == 0 && threadIdx.x == 0) g_phase_ns[a.want_topk][27] = globaltimer_ns();
#endif
  TK_TL_BEGIN(a.want_topk ? 3 : 1);
  // programmatic dependent launch: everything below may read what earlier
  // grids wrote, so wait for them; the next grid may begin launching now
  grid_dependency_wait();
#ifdef TK_PHASE_TIMING
  if (blockIdx.x == 0 && threadIdx.x == 0) g_phase_ns[a.want_topk][28] = globaltimer_ns();
#endif
  grid_launch_dependents();
  if (a.clear_words && blockIdx.x == 0)  // control words of an earlier grid, ready for the next call
    for (int i = threadIdx.x; i < a.n_clear; i += BLOCK) a.clear_words[i] = 0u;
  if constexpr (SRC == 3) {
    // The miss check of the refinement (section 4): with fewer than r
    // survivors, or more than the buffer holds, the candidates cannot give
    // the exact answer, and the whole row of x is the source instead.  Every
    // CTA of the cluster reads the same count, so all take the same branch.
    cg::cluster_group cluster = cg::this_cluster();
    const int64_t row = blockIdx.x / cluster.num_blocks();
    if (threadIdx.x == 0) {
      const unsigned long long R = __ldcg(a.counts + row);
      const bool miss = a.force || R < static_cast<unsigned long long>(a.r) ||
                        R > static_cast<unsigned long long>(a.key_stride);
      s_source = miss ? a.miss_src : 0;
      s_prologue_r = R;
      if (cluster.block_rank() == 0) {
        a.r_seen[row] = R;
        if (miss) atomicAdd(a.misses, 1ull);
      }
    }
    __syncthreads();
    if (a.rctl && a.want_topk && s_source == 0 && select_from_regions<BLOCK, P, CB, NB>(a)) {
      TK_TL_END(a.want_topk ? 3 : 1);
      return;
    }
  }
  select_body<BLOCK, P, CB, NB, SRC>(a);
  TK_TL_END(a.want_topk ? 3 : 1);
}

// ---------------------------------------------------------------------------
// Bin sort (large k).  The refinement cluster has partitioned the k winners
// of each selection by their first digit: bin b's winners sit at places
// [bst[b], min(bst[b + 1], k)) of the exchange buffer, bins in descending key
// order.  Each block of this grid owns kBinSortPlaces output places: it cuts
// the bins at either end of its places by further 8-bit digits down to the
// sub-bin holding the boundary place, collects the keys in between (a
// contiguous key range) and ranks them by counting inside groups of equal
// leading bits.  Many small blocks share the sort that one cluster would
// otherwise do alone.
constexpr int kBinSortBlock = 256;
constexpr int kBinSortPlaces = static_cast<int>(kBinSortChunk);
constexpr int kBinSortCap = 2048;  // keys one block sorts
constexpr int kBinSortGroups = 1024;  // slices of the block's key range: ~2 keys each for 2048 keys
constexpr int kBinSortScratch = 3 * kBinSortGroups;  // (also covers the LSD sort's counters)
static_assert(kBinSortScratch >= (kBinSortBlock / 32) * 256 + 2 * 256 + (kBinSortBlock / 256) * 256, "lsd");
constexpr size_t kBinSortSmem = 2 * sizeof(uint64_t) * kBinSortCap + sizeof(unsigned) * kBinSortScratch;

struct BinSortParams {
  SelParams a;  // the refinement's parameters: r = k, xbuf, binfo, outputs
  int q;        // blocks per selection
};

__device__ __forceinline__ void bin_sort_body(const BinSortParams& bp, uint64_t* hbar, int* hcopy);
cudaError_t launch_bin_sort_a(const SelParams& a, int64_t nsel, int* launch_count, cudaStream_t st);
static_assert(kBinInfoBins == kRefineGridBins, "the grid refinement publishes the bin sort's bins");

#ifdef TK_PHASE_TIMING
__device__ unsigned g_bs_info[1024][4];          // debug: set size, cut iterations, max group, lsd
#define TK_BS(i, v) \
  do { if (threadIdx.x == 0 && blockIdx.x < 1024) g_bs_info[blockIdx.x][(i)] = (v); } while (0)
#else
#define TK_BS(i, v) \
  do {              \
  } while (0)
#endif

__global__ void __launch_bounds__(kBinSortBlock) bin_sort_kernel(BinSortParams bp) {
  // a bulk copy of the filter's histogram, issued before the block knows
  // whether it needs it: in flight (hcopy) until waited for, here at the end
  // at the latest, since it writes this block's shared memory
  __shared__ __align__(8) uint64_t s_hbar;
  __shared__ int s_hcopy;
  TK_TL_BEGIN(4);
#ifdef TK_PHASE_TIMING
  grid_dependency_wait();
  TK_BSP(0);
#endif
  if (threadIdx.x == 0) s_hcopy = 0;
  __syncthreads();
  bin_sort_body(bp, &s_hbar, &s_hcopy);
  __syncthreads();
  if (s_hcopy) {
    const bool landed = mbar_wait(&s_hbar, 0u);
    if (threadIdx.x == 0 && !landed) {
      atomicCAS(bp.a.status, kDevOk, kDevTimeout);
      mbar_wait(&s_hbar, 0u);
    }
    __syncthreads();
  }
  TK_TL_END(4);
#ifdef TK_PHASE_TIMING
  TK_BSP(7);
#endif
}

__device__ __forceinline__ void bin_sort_body(const BinSortParams& bp, uint64_t* hbar, int* hcopy) {
  constexpr int BLOCK = kBinSortBlock;
  constexpr int NB = kBinInfoBins;
  constexpr unsigned DM = 255u;  // 8-bit sub-digits
  const SelParams& a = bp.a;
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* bufA = reinterpret_cast<uint64_t*>(smem);
  uint64_t* bufB = bufA + kBinSortCap;
  unsigned* scr = reinterpret_cast<unsigned*>(bufB + kBinSortCap);
  __shared__ unsigned long long s_tmp[32];
  __shared__ unsigned long long s_info[5];
  __shared__ unsigned s_cnt;
  grid_dependency_wait();  // the partition comes from the previous grid
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x / bp.q;
  const int64_t k = a.r;
  const int64_t my0 = static_cast<int64_t>(blockIdx.x % bp.q) * kBinSortPlaces;
  if (my0 >= k) return;
  const int64_t my1 = my0 + kBinSortPlaces < k ? my0 + kBinSortPlaces : k;
  const unsigned* bi = a.binfo + row * binfo_words(k);
  // one round of loads, one word per thread, shared through shared memory:
  // the status word, the digit description and this block's chunk
  // descriptor (its first and last bins with their bounds); with bin regions
  // also the filter's histogram, two 16-byte loads a thread
  constexpr int kHw = 9;  // header words read
  __shared__ unsigned s_words[1 + kHw + kChunkWords];
  __shared__ __align__(16) unsigned s_bst[NB];  // bin regions: the histogram, then every bin's first place
  __shared__ unsigned s_total;
  static_assert(NB == 8 * BLOCK, "eight bins a thread");
  if (tid == 0) s_words[0] = static_cast<unsigned>(__ldcg(a.status));
  else if (tid <= kHw) s_words[tid] = __ldcg(bi + NB + (tid - 1));
  else if (tid <= kHw + kChunkWords)
    s_words[tid] = __ldcg(bi + NB + kBinfoHeaderWords + (blockIdx.x % bp.q) * kChunkWords + (tid - 1 - kHw));
  // the histogram (bin regions) comes in one bulk copy, issued with the
  // words above before it is known to be needed (every block reads these
  // 8 KB, and 16-byte loads by every thread would queue ~2000 requests on
  // each of its L2 lines); it is waited for only when used, else at the end
  if (a.fhist && tid == 0) {
    fence_proxy_async_all();  // (the histogram is the earlier grids' writes)
    mbar_init(hbar, 1u);
    mbar_expect_tx(hbar, static_cast<unsigned>(sizeof(unsigned) * NB));
    bulk_copy_g2s(s_bst, a.fhist, static_cast<unsigned>(sizeof(unsigned) * NB), hbar);
    *hcopy = 1;
  }
  __syncthreads();
  if (s_words[0] != static_cast<unsigned>(kDevOk)) return;  // the refinement failed
  unsigned hw[kHw], cd[kChunkWords];
#pragma unroll
  for (int q = 0; q < kHw; ++q) hw[q] = s_words[1 + q];
#pragma unroll
  for (int q = 0; q < kChunkWords; ++q) cd[q] = s_words[1 + kHw + q];
  const bool binned = a.fhist && a.region && hw[8] == 1u;
  if (binned) {
    const bool landed = mbar_wait(hbar, 0u);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) atomicCAS(a.status, kDevOk, kDevTimeout);
      return;  // (the kernel waits for the copy once more before leaving)
    }
    if (tid == 0) *hcopy = 0;
    // The refinement left the keys in the filter's bin regions: every bin's
    // first place from its histogram (an exclusive scan), the end of the
    // boundary bin and this block's chunk descriptor, as the refinement
    // would have published them.
    unsigned c[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) c[q] = s_bst[tid * 8 + q];
    unsigned long long sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) sum += c[q];
    const unsigned long long incl = block_scan_incl(sum, s_tmp);
    unsigned run = static_cast<unsigned>(incl - sum);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      s_bst[tid * 8 + q] = run;
      run += c[q];
    }
    if (tid == BLOCK - 1) s_total = run;
    __syncthreads();
    auto find = [&](unsigned p) {  // the last bin starting at or before place p
      unsigned b = 0;
#pragma unroll
      for (unsigned stp = NB / 2; stp > 0; stp >>= 1)
        if (s_bst[b + stp] <= p) b += stp;
      return b;
    };
    const unsigned bk = find(static_cast<unsigned>(k - 1));  // the boundary bin
    hw[5] = bk + 1 < static_cast<unsigned>(NB) ? s_bst[bk + 1] : s_total;  // the end of the placed keys
    auto bin_end = [&](unsigned b) -> unsigned {
      const unsigned e = b + 1 < static_cast<unsigned>(NB) ? s_bst[b + 1] : s_total;
      return e < hw[5] ? e : hw[5];
    };
    cd[0] = find(static_cast<unsigned>(my0));
    cd[1] = find(static_cast<unsigned>(my1 - 1));
    cd[2] = s_bst[cd[0]];
    cd[3] = bin_end(cd[0]);
    cd[4] = s_bst[cd[1]];
    cd[5] = bin_end(cd[1]);
  }
  const uint64_t prefix1 = static_cast<uint64_t>(hw[0]) | (static_cast<uint64_t>(hw[1]) << 32);
  const uint64_t pmask1 = static_cast<uint64_t>(hw[2]) | (static_cast<uint64_t>(hw[3]) << 32);
  const int shift1 = static_cast<int>(hw[4]);
  // digits, prefixes and masks are of key - kbase
  const uint64_t kbase = static_cast<uint64_t>(hw[6]) | (static_cast<uint64_t>(hw[7]) << 32);
  const uint64_t* xb = a.xbuf + row * a.xstride;
  // the first-digit bins holding places my0 and my1 - 1, and their bounds
  const unsigned bfirst = cd[0], blast = cd[1];
  const int64_t first_s = cd[2], first_e = cd[3], last_s = cd[4], last_e = cd[5];
  // key at place p of bin b (the exchange buffer, or bin b's region)
  auto bin_key = [&](unsigned b, int64_t p) -> uint64_t {
    return binned ? __ldcg(a.region + static_cast<int64_t>(b) * kBinRegionCap + (p - s_bst[b])) : __ldcg(xb + p);
  };
  // key at place p (bin regions: the bin holding it, among bfirst..blast,
  // by a search in a fixed number of steps, so a thread's searches overlap)
  auto place_key = [&](int64_t p) -> uint64_t {
    if (!binned) return __ldcg(xb + p);
    unsigned b = bfirst;
#pragma unroll
    for (unsigned stp = NB / 2; stp > 0; stp >>= 1)
      if (b + stp <= blast && s_bst[b + stp] <= p) b += stp;
    return __ldcg(a.region + static_cast<int64_t>(b) * kBinRegionCap + (p - s_bst[b]));
  };
  TK_BSP(1);
  const int64_t r0 = first_s < k ? first_s : k, r1 = last_e;
  uint64_t hi_key = ~0ull, lo_key = 0ull;
  int64_t place0 = r0, place1 = r1;
  unsigned cut_iters = 0;
  if (r1 - r0 > kBinSortCap) {
    const int64_t lim = (kBinSortCap - (my1 - my0)) / 2;
    unsigned* lh = scr;  // 256 counters
    // cut bin b down to the 8-bit sub-bin (and so on) holding place p
    auto cut = [&](unsigned b, int64_t bs, int64_t be, int64_t p, uint64_t& pre, uint64_t& msk, int64_t& s0,
                   int64_t& s1) -> bool {
      pre = prefix1 | (static_cast<uint64_t>(2047u - b) << shift1);
      msk = pmask1 | (2047ull << shift1);
      s0 = bs;
      s1 = be;
      int sh = shift1;
      while (s1 - s0 > lim && sh > 0) {
        const int sh2 = sh >= 8 ? sh - 8 : 0;
        lh[tid] = 0u;  // (BLOCK == 256 counters)
        if (tid == 0) s_info[2] = ~0ull;
        __syncthreads();
        for (int64_t i = bs + tid; i < be; i += BLOCK) {
          const uint64_t key = bin_key(b, i) - kbase;
          if ((key & msk) == pre) atomicAdd(&lh[DM - static_cast<unsigned>((key >> sh2) & DM)], 1u);
        }
        __syncthreads();
        const unsigned long long c = lh[tid];
        const unsigned long long incl = block_scan_incl(c, s_tmp);
        const unsigned long long run = static_cast<unsigned long long>(s0) + incl - c;
        if (run <= static_cast<unsigned long long>(p) && static_cast<unsigned long long>(p) < run + c) {
          s_info[2] = static_cast<unsigned long long>(tid);
          s_info[3] = run;
          s_info[4] = c;
        }
        __syncthreads();
        if (s_info[2] == ~0ull) return false;
        pre |= static_cast<uint64_t>(DM - static_cast<unsigned>(s_info[2])) << sh2;
        msk |= static_cast<uint64_t>(DM) << sh2;
        s0 = static_cast<int64_t>(s_info[3]);
        s1 = s0 + static_cast<int64_t>(s_info[4]);
        sh = sh2;
        ++cut_iters;
        __syncthreads();
      }
      return true;
    };
    uint64_t pre, msk;
    int64_t s0, s1;
    // (a bin taken whole bounds nothing: its keys are exactly those of its
    // places, which is what keeps the top bin of bin regions -- not a plain
    // digit, and never cut -- whole)
    bool ok = cut(bfirst, first_s, first_e, my0, pre, msk, s0, s1);
    hi_key = (s0 == first_s && s1 == first_e) ? ~0ull : (pre | ~msk);
    place0 = s0;
    ok = ok && cut(blast, last_s, last_e, my1 - 1, pre, msk, s0, s1);
    lo_key = (s0 == last_s && s1 == last_e) ? 0ull : pre;
    place1 = s1;
    TK_BS(1, cut_iters | (static_cast<unsigned>(first_s < k ? first_e - first_s : 0) << 8));
    if (!ok || place1 - place0 > kBinSortCap || place1 < place0) {
      if (tid == 0) atomicCAS(a.status, kDevOk, kDevBadState);
      return;
    }
  }
  const int n_c = static_cast<int>(place1 - place0);
  if (r1 - r0 <= kBinSortCap) {
    // every load of the thread in flight at once (n_c <= kBinSortCap)
    constexpr int kLoads = kBinSortCap / BLOCK;
    uint64_t kv[kLoads];
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      const int i = tid + q * BLOCK;
      kv[q] = i < n_c ? place_key(r0 + i) : 0ull;
    }
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      const int i = tid + q * BLOCK;
      if (i < n_c) bufA[i] = kv[q];
    }
  } else {
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    for (int64_t iw = r0 + (tid & ~31); iw < r1; iw += BLOCK) {
      const int64_t i = iw + (tid & 31);
      const uint64_t key = i < r1 ? place_key(i) : 0ull;
      const bool want = i < r1 && key - kbase <= hi_key && key - kbase >= lo_key;
      const unsigned slot = warp_append_slot(&s_cnt, want);
      if (want && slot < static_cast<unsigned>(kBinSortCap)) bufA[slot] = key;
    }
    __syncthreads();
    if (s_cnt != static_cast<unsigned>(n_c)) {
      if (tid == 0) atomicCAS(a.status, kDevOk, kDevBadState);
      return;
    }
  }
  __syncthreads();
  TK_BSP(2);
  const KeySpan sp = block_span<BLOCK>(bufA, n_c);
  TK_BSP(3);
  TK_BS(0, static_cast<unsigned>(n_c));
  if (place_by_groups<BLOCK, kBinSortGroups>(bufA, n_c, sp.kmin, sp.kmax, 0u, ~0u, bufB, scr, scr + kBinSortGroups,
                                             scr + 2 * kBinSortGroups, s_tmp, 512u, a, row, k, place0, my0, my1))
    return;
  TK_BS(3, 1u);
  const uint64_t* sorted = lsd_sort<BLOCK, kBinSortCap>(bufA, bufB, n_c, sp.all_or ^ sp.all_and, scr);
  for (int i = tid; i < n_c; i += BLOCK) {
    const int64_t place = place0 + i;
    if (place >= my0 && place < my1) write_out(a, row, k, place, sorted[i]);
  }
}

// Kernel variants: (block, sort positions per CTA, cache/second buffer).
constexpr int kSmallBlock = 256, kSmallP = 1024, kSmallCB = 2048, kSmallNB = 256;
constexpr int kBigBlock = 512, kBigP = 11776, kBigCB = 11776, kBigNB = 2048;
constexpr int64_t kTauSlice = 8192;
constexpr int64_t kBinSortMinK = 8192;  // k from which the winners are sorted by the bin-sort grid  // samples streamed per CTA when tau starts from the histogram

template <int BLOCK, int P, int CB, int NB, int SRC>
cudaError_t configure(int* max_g) {
  using L = Layout<BLOCK, P, CB, NB>;
  auto kern = select_kernel<BLOCK, P, CB, NB, SRC>;
  static int cached = 0;  // largest cluster size the device can schedule for this variant
  if (!cached) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::kBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    int g = kMaxCluster;
    for (; g > 1; g >>= 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(g), 1, 1);
      cfg.blockDim = dim3(BLOCK, 1, 1);
      cfg.dynamicSmemBytes = L::kBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(g);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0) break;
      cudaGetLastError();  // clear a refused query
    }
    cached = g;
  }
  *max_g = cached;
  return cudaSuccess;
}

template <int BLOCK, int P, int CB, int NB, int SRC>
cudaError_t launch_variant(const SelParams& a, int64_t nsel, int G, int* used, cudaStream_t st) {
  using L = Layout<BLOCK, P, CB, NB>;
  int max_g = 1;
  cudaError_t e = configure<BLOCK, P, CB, NB, SRC>(&max_g);
  if (e != cudaSuccess) return e;
  if (G > max_g) G = max_g;
  const int64_t sort_k = a.want_topk ? a.r : 1;
  if (sort_k > static_cast<int64_t>(G) * P) return cudaErrorInvalidConfiguration;
  if (a.want_topk && a.xbuf == nullptr) return cudaErrorInvalidValue;
  *used = G;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nsel * G), 1, 1);
  cfg.blockDim = dim3(BLOCK, 1, 1);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(G);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_edge(a.want_topk ? (a.keys ? kPdlRefine : 0u) : kPdlTau) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, select_kernel<BLOCK, P, CB, NB, SRC>, a);
}

template <int BLOCK, int P, int CB, int NB>
cudaError_t launch_src(const SelParams& a, int src, int64_t nsel, int G, int* used, cudaStream_t st) {
  if (src == 0) return launch_variant<BLOCK, P, CB, NB, 0>(a, nsel, G, used, st);
  if (src == 1) return launch_variant<BLOCK, P, CB, NB, 1>(a, nsel, G, used, st);
  if (src == 2) return launch_variant<BLOCK, P, CB, NB, 2>(a, nsel, G, used, st);
  return launch_variant<BLOCK, P, CB, NB, 3>(a, nsel, G, used, st);
}


int pow2_at_least(int64_t v) {
  int g = 1;
  while (g < v && g < kMaxCluster) g <<= 1;
  return g;
}

int sm_count() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  return sms;
}

}  // namespace

int64_t select_max_k() { return static_cast<int64_t>(kMaxCluster) * kBigP; }
int64_t select_binfo_words(int64_t k) { return k >= kBinSortMinK ? binfo_words(k) : 0; }
int64_t select_cta_cache() { return kBigP + kBigCB; }
int64_t select_xbuf_stride(int64_t k) { return k >= kBinSortMinK ? 2 * k : k; }

#ifdef TK_PHASE_TIMING
TK_TIMELINE_ACCESSOR(debug_timeline_select)
int debug_binsort_ns(unsigned long long* out) {
  if (cudaMemcpyFromSymbol(out, g_bs_ns, sizeof(g_bs_ns)) != cudaSuccess) return -3;
  return cudaMemcpyFromSymbol(out + 8192, g_bs_info, sizeof(g_bs_info)) == cudaSuccess ? 0 : -3;
}
int debug_phase_ns(unsigned long long* out) {
  if (cudaMemcpyFromSymbol(out, g_phase_ns, sizeof(g_phase_ns)) != cudaSuccess) return -3;
  return cudaMemcpyFromSymbol(out + 96, g_cta_ns, sizeof(g_cta_ns)) == cudaSuccess ? 0 : -3;  // 2*16*8
}
#endif

cudaError_t launch_select(const Problem& p, const SelectJob& job, int64_t source_hint, int* cluster,
                          cudaStream_t st) {
  SelParams a{};
  a.keys = job.keys;
  a.key_stride = job.key_stride;
  a.counts = job.counts;
  a.x = p.x;
  a.len = p.len;
  a.ib = p.ib;
  a.flip = p.flip;
  a.key_bits = p.dtype == kF32 ? 32 : 16;
  a.key_vec = job.keys && (reinterpret_cast<uintptr_t>(job.keys) % 16 == 0) &&
              (job.key_stride % 2 == 0 || p.nsel == 1);
  a.src_vec = p.vec_ok;
  a.r = job.r;
  a.want_topk = job.want_topk ? 1 : 0;
  a.tau_out = job.tau_out;
  a.out_vals = job.out_vals;
  a.out_idx = job.out_idx;
  a.status = job.status;
  a.xbuf = job.xbuf;
  a.clear_words = job.clear_words;
  a.n_clear = job.n_clear;
  a.relax_tau = job.relax_tau;
  a.xstride = job.xbuf_stride > job.r ? job.xbuf_stride : job.r;
  a.shist = job.want_topk ? nullptr : job.sample_hist;
  if (job.want_topk && job.rctl && job.region && p.nsel == 1) {
    a.rctl = job.rctl;
    a.region = job.region;
  }
  if (job.want_topk && job.keys && job.check_miss) {
    a.miss_src = p.dtype == kF32 ? 1 : 2;
    a.force = job.force_miss ? 1 : 0;
    a.r_seen = job.r_seen;
    a.misses = job.misses;
  }
  const int src = job.keys ? (a.miss_src ? 3 : 0) : (p.dtype == kF32 ? 1 : 2);
  const bool many = p.nsel >= sm_count();
  constexpr int64_t kBigCache = kBigP + kBigCB;
  int G;
  bool small;
  if (!job.want_topk && job.sample_hist) {
    // tau from the sample histogram: one streaming pass for the bucket
    small = false;
    G = pow2_at_least((source_hint + kTauSlice - 1) / kTauSlice);
  } else if (!job.want_topk) {
    // tau: every CTA caches its whole slice of the samples
    small = false;
    G = pow2_at_least((source_hint + kBigCache - 1) / kBigCache);
  } else if (many && job.r <= kSmallP) {
    small = true;
    G = 1;
  } else {
    // each CTA sorts at most P places; prefer slices that fit the cache
    small = false;
    const int64_t g_min = (job.r + kBigP - 1) / kBigP;
    const int64_t g_cache = (source_hint + kBigCache - 1) / kBigCache;
    G = many ? pow2_at_least(g_min) : pow2_at_least(g_min > g_cache ? g_min : g_cache);
  }
  // large k: the cluster stops after partitioning the winners, and a grid of
  // small blocks sorts them
  if (!small) {  // the cluster size the device can schedule (as launch_variant clamps it)
    int max_g = 1;
    const cudaError_t ce = configure<kBigBlock, kBigP, kBigCB, kBigNB, 0>(&max_g);
    if (ce != cudaSuccess) return ce;
    if (G > max_g) G = max_g;
  }
  // (a one-CTA cluster sorts its winners in place and never partitions them)
  const bool handoff = job.want_topk && job.binfo && !small && job.r >= kBinSortMinK && G > 1;
  a.binfo = handoff ? job.binfo : nullptr;
  a.handoff = handoff ? 1 : 0;
  int used = G;
  cudaError_t e = small ? launch_src<kSmallBlock, kSmallP, kSmallCB, kSmallNB>(a, src, p.nsel, G, &used, st)
                        : launch_src<kBigBlock, kBigP, kBigCB, kBigNB>(a, src, p.nsel, G, &used, st);
  if (cluster) *cluster = used;
  if (e == cudaSuccess && job.launch_count) ++*job.launch_count;
  if (e != cudaSuccess || !handoff) return e;
  return launch_bin_sort_a(a, p.nsel, job.launch_count, st);
}

cudaError_t launch_bin_sort(const Problem& p, const SelectJob& job, cudaStream_t st) {
  if (!job.binfo || !job.xbuf || job.xbuf_stride < job.r || job.r < 1) return cudaErrorInvalidValue;
  SelParams a{};
  a.x = p.x;
  a.len = p.len;
  a.ib = p.ib;
  a.flip = p.flip;
  a.key_bits = p.dtype == kF32 ? 32 : 16;
  a.r = job.r;
  a.want_topk = 1;
  a.out_vals = job.out_vals;
  a.out_idx = job.out_idx;
  a.status = job.status;
  a.xbuf = job.xbuf;
  a.xstride = job.xbuf_stride;
  a.binfo = job.binfo;
  a.handoff = 1;
  a.relax_tau = job.relax_tau;
  a.fhist = job.fhist;
  a.region = job.region;
  return launch_bin_sort_a(a, p.nsel, job.launch_count, st);
}

namespace {

cudaError_t launch_bin_sort_a(const SelParams& a, int64_t nsel, int* launch_count, cudaStream_t st) {
  static bool configured = false;
  cudaError_t e;
  if (!configured) {
    e = cudaFuncSetAttribute(bin_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kBinSortSmem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  BinSortParams bp{a, static_cast<int>((a.r + kBinSortPlaces - 1) / kBinSortPlaces)};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nsel * bp.q), 1, 1);
  cfg.blockDim = dim3(kBinSortBlock, 1, 1);
  cfg.dynamicSmemBytes = kBinSortSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_edge(kPdlRefine) ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, bin_sort_kernel, bp);
  if (e == cudaSuccess && launch_count) ++*launch_count;
  return e;
}

}  // namespace

}  // namespace tk
