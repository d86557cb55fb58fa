// The filter's tile loop and its helpers, shared by the filter kernel
// (kernels_filter.cu) and the fallback's re-filter (kernels_fallback.cu):
// the survivor test of a 16-byte group against tau, the exact composite-key
// test, the warp stages and their flush.  Device code only; each translation
// unit that includes it gets its own copy (anonymous namespace).
#pragma once

#include "common.cuh"
#include "engine.h"
#include "rank.cuh"

namespace tk {

namespace {

constexpr int kFilterBlock = 256;
constexpr int kFilterUnroll = 4;
constexpr int kWarpStage = 256;  // survivors staged per warp before a flush

// Division by the invariant tiles-per-row count without a divide instruction
// (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", the round-up multiplier of their section 4): with
// l = ceil(log2 d) and m = floor(2^64 (2^l - d) / d) + 1,
// n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0) where t = mulhi(m, n).
struct Divider {
  uint64_t m;
  uint32_t s1, s2;
};

Divider make_divider(uint64_t d) {
  int l = 0;
  while (l < 63 && (1ull << l) < d) ++l;
  const unsigned __int128 two64 = static_cast<unsigned __int128>(1) << 64;
  const uint64_t m = static_cast<uint64_t>(two64 * ((1ull << l) - d) / d + 1);
  return Divider{m, static_cast<uint32_t>(l < 1 ? l : 1), static_cast<uint32_t>(l > 1 ? l - 1 : 0)};
}

__device__ __forceinline__ uint64_t divide(uint64_t n, const Divider& dv) {
  const uint64_t t = __umul64hi(dv.m, n);
  return (t + ((n - t) >> dv.s1)) >> dv.s2;
}

struct FilterParams {
  const void* x;
  int64_t nsel, len;
  int ib;
  uint32_t flip;
  const uint64_t* tau;
  int64_t cap;
  uint64_t* buf;
  unsigned long long* counts;
  Divider tiles_per_row;  // set by the launcher for its tile size
  // survivor histogram (HIST variants): the grid refinement's control words
  // (kRefineGridCtlWords per selection) hold the largest sampled key and
  // receive the counts
  unsigned* refine_ctl = nullptr;
  int* status = nullptr;  // nullable: the call's device status word (a wait that gave up)
  // nullable (one selection, with refine_ctl): the survivors stay in the
  // warps' stages until the block ends, which places them in bin regions
  // of kBinRegionCap keys (the filter_ring_kernel's end)
  uint64_t* region = nullptr;
  unsigned* refine_ctl_next = nullptr;  // (with region, nullable) cleared by the blocks for the next call
  // (TMA-ring filter) tiles past its first ring stages that each block asks
  // L2 to fetch before tau is known
  int l2_ahead = 0;
};

// (with bin regions) set when some survivors of this block left its stages;
// initialised by the filter kernel that bins
__shared__ int s_filter_block_bad;

// The word a filter block sets when its survivors did not all stay in its
// stages or a bin region overflowed: the regions are then incomplete.
__device__ __forceinline__ unsigned* binned_bad_word(const FilterParams& fp, int64_t row) {
  return fp.refine_ctl + row * kRefineGridCtlWords + kRefineGridBinnedWord;
}

__device__ __forceinline__ unsigned long long sampled_kmax(const unsigned* refine_ctl, int64_t row) {
  return __ldcg(reinterpret_cast<const unsigned long long*>(refine_ctl + row * kRefineGridCtlWords +
                                                            kRefineGridKmaxWord));
}

// Bins of a survivor's offset above tau for the grid refinement: 2048 bins in
// descending key order, bin = 2047 - ((key - tau) >> shift) while the offset
// is below 2047 << shift, bin 0 above that.  The shift makes the span from
// tau to the largest sampled key cover fewer than 1024 bins, so the keys
// above the largest sampled one (about N / S of them) still have room.
__host__ __device__ __forceinline__ int survivor_shift(uint64_t tau, uint64_t kmax) {
  const uint64_t span = kmax > tau ? kmax - tau : 0ull;
  int bits = 0;
  while (bits < 64 && (span >> bits) != 0ull) ++bits;
  return bits > 10 ? bits - 10 : 0;
}
__device__ __forceinline__ unsigned survivor_bin(uint64_t key, uint64_t tau, int shift) {
  const uint64_t d = (key - tau) >> shift;  // key >= tau
  return d >= static_cast<uint64_t>(kRefineGridBins - 1) ? 0u
                                                          : static_cast<unsigned>(kRefineGridBins - 1) - static_cast<unsigned>(d);
}

// Element e of a packed group of raw words (VEC elements).
template <int DT, int VEC>
__device__ __forceinline__ uint32_t elem(const uint4& v, int e) {
  const uint32_t w = (e >> (DT == kF32 ? 0 : 1)) == 0 ? v.x
                     : (e >> (DT == kF32 ? 0 : 1)) == 1 ? v.y
                     : (e >> (DT == kF32 ? 0 : 1)) == 2 ? v.z : v.w;
  if (DT == kF32) return w;
  return (VEC == 1) ? (w & 0xffffu) : ((w >> ((e & 1) * 16)) & 0xffffu);
}

// The input is read exactly once: its L2 lines are marked evict-first, so
// the stream leaves the next kernels' code, keys and buffers in L2.
constexpr bool kStreamEvictFirst = true;

template <int DT, int VEC>
__device__ __forceinline__ uint4 load_group(const typename Dt<DT>::storage* p, uint64_t policy) {
  if (VEC == 1) return make_uint4(static_cast<uint32_t>(__ldg(p)), 0u, 0u, 0u);
  if (kStreamEvictFirst) return ld_stream_v4(p, policy);
  return ld_stream_v4(p);
}

// NaN-propagating max / min (PTX max.NaN / min.NaN).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bmin2_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Packed bf16x2 compares: each 16-bit half of the result is all ones where the
// compare holds.  gtu holds for NaN too; lt and eq do not.
__device__ __forceinline__ uint32_t bset_gtu(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.gtu.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bset_lt(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.lt.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bset_eq(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.eq.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Eight per-element compare results of a bf16 group (four packed words, each
// half 0xffff or 0) -> an 8-bit mask, bit e for element e.
__device__ __forceinline__ uint32_t halves_to_mask(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
  // one byte per element (0xff or 0): the high byte of each half
  const uint32_t lo = __byte_perm(a0, a1, 0x7531);  // elements 0..3
  const uint32_t hi = __byte_perm(a2, a3, 0x7531);  // elements 4..7
  // keep bit e in byte e of lo and bit e+4 in byte e of hi, then add the bytes
  const uint32_t b = (lo & 0x08040201u) | (hi & 0x80402010u);
  return (b * 0x01010101u) >> 24;
}

// Superset test for a group: does any element rank at or above tau's value?
// One NaN-propagating max (largest) or min (smallest) over the group and one
// compare; NaN elements always pass here (the exact test sorts them out).
template <int DT, bool LARGEST, int VEC>
__device__ __forceinline__ bool group_candidate(const uint4& v, float tv) {
  float m;
  if (DT == kF32) {
    if (VEC == 1) {
      m = __uint_as_float(v.x);
    } else if (LARGEST) {
      m = fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                   fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    } else {
      m = fmin_nan(fmin_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                   fmin_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
  } else {
    if (VEC == 1) {
      m = __uint_as_float(v.x << 16);
    } else {
      const uint32_t c = LARGEST ? bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w))
                                 : bmin2_nan(bmin2_nan(v.x, v.y), bmin2_nan(v.z, v.w));
      const float lo = __uint_as_float(c << 16), hi = __uint_as_float(c & 0xffff0000u);
      m = LARGEST ? fmax_nan(lo, hi) : fmin_nan(lo, hi);
    }
  }
  return LARGEST ? !(m < tv) : !(m > tv);
}

// Per-row threshold in the forms the filter tests against.
struct RowTau {
  uint64_t key;   // composite key
  uint64_t pos;   // position of the element it came from
  float value;    // its value (0 for the zero key)
  uint32_t v2;    // bf16: the value's bits in both halves of a word
  bool nan;       // tau's value is NaN: fall back to composite-key compares
  int hshift;     // survivor histogram: survivor_shift(tau, largest sampled key)
};

template <int DT>
__device__ __forceinline__ RowTau row_tau(uint64_t tau, int ib, uint32_t flip) {
  RowTau r;
  r.key = tau;
  r.pos = position_of(tau, ib);
  const uint32_t k = vkey_of(tau, ib) ^ flip;
  r.nan = (k == Dt<DT>::kNanKey);
  r.value = (k == Dt<DT>::kZeroKey || r.nan) ? 0.0f : Dt<DT>::to_float(Dt<DT>::bits(k));
  const uint32_t b16 = __float_as_uint(r.value) >> 16;  // exact for a bf16 value
  r.v2 = (b16 << 16) | b16;
  return r;
}

// A warp's survivor stage: slots in shared memory and a fill counter that the
// warp's lanes advance with shared atomics.
struct Stage {
  uint64_t* s;
  unsigned* n;
};

// Moves the stage to the candidate buffer: one global atomic reserves the
// slots (the counter keeps counting past the capacity, so R stays exact; only
// slots below the capacity are written).  Called by the whole warp.
__device__ __forceinline__ void stage_flush(const Stage& st, int64_t row, int64_t cap, uint64_t* buf,
                                            unsigned long long* counts) {
  __syncwarp();
  const unsigned filled = *st.n;
  const unsigned n = filled < static_cast<unsigned>(kWarpStage) ? filled : static_cast<unsigned>(kWarpStage);
  if (n) {
    const int lane = threadIdx.x & 31;
    unsigned long long base = 0;
    if (lane == 0) base = atomicAdd(counts + row, static_cast<unsigned long long>(n));
    base = __shfl_sync(kFull, base, 0);
    uint64_t* dst = buf + row * cap;
    for (unsigned j = lane; j < n; j += 32) {
      const unsigned long long pos = base + j;
      if (pos < static_cast<unsigned long long>(cap)) dst[pos] = st.s[j];
    }
  }
  __syncwarp();
  if ((threadIdx.x & 31) == 0) *st.n = 0u;
  __syncwarp();
}

// Exact test of one group: bit e is set when element e ranks at or above
// tau, i.e. its value ranks strictly above tau's value, or equals it at a
// position <= tau's (the composite-key order).  Packed compares give the
// "above" and "equal" masks; the position test runs only for ties.
template <int DT, bool LARGEST, int VEC>
__device__ __forceinline__ uint32_t exact_mask(const uint4& v, int64_t pos, const RowTau& t, int ib,
                                               uint32_t flip) {
  uint32_t above = 0, equal = 0;
  if (t.nan) {  // only NaN keys tie with tau: compare composite keys
#pragma unroll
    for (int e = 0; e < VEC; ++e)
      above |= static_cast<uint32_t>(compose(Dt<DT>::key(elem<DT, VEC>(v, e)) ^ flip,
                                             static_cast<uint64_t>(pos + e), ib) >= t.key) << e;
    return above;
  }
  if (DT == kBF16 && VEC == 8) {
    const uint32_t tv = t.v2;
    above = LARGEST ? halves_to_mask(bset_gtu(v.x, tv), bset_gtu(v.y, tv), bset_gtu(v.z, tv), bset_gtu(v.w, tv))
                    : halves_to_mask(bset_lt(v.x, tv), bset_lt(v.y, tv), bset_lt(v.z, tv), bset_lt(v.w, tv));
    equal = halves_to_mask(bset_eq(v.x, tv), bset_eq(v.y, tv), bset_eq(v.z, tv), bset_eq(v.w, tv));
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const float f = Dt<DT>::to_float(elem<DT, VEC>(v, e));
      above |= static_cast<uint32_t>(LARGEST ? !(f <= t.value) : (f < t.value)) << e;
      equal |= static_cast<uint32_t>(f == t.value) << e;
    }
  }
  while (equal) {  // ties with tau's value: the lower position ranks higher
    const int e = __ffs(equal) - 1;
    equal &= equal - 1;
    if (static_cast<uint64_t>(pos + e) <= t.pos) above |= 1u << e;
  }
  return above;
}

// Appends the elements of `mask` to the warp's stage with one shared atomic;
// what does not fit is appended to the buffer directly (and, when the block
// bins its survivors, marks the bin regions incomplete).  HIST: each
// survivor is also counted into the block's histogram of its offset above tau.
template <int DT, int VEC, bool HIST>
__device__ __forceinline__ void lane_append(uint32_t mask, const uint4& v, int64_t pos, const FilterParams& fp,
                                            const Stage& st, int64_t row, const RowTau& t, unsigned* sh_hist) {
  const int ib = fp.ib;
  const uint32_t flip = fp.flip;
  const int64_t cap = fp.cap;
  uint64_t* buf = fp.buf;
  const unsigned n = __popc(mask);
  const unsigned slot = atomicAdd(st.n, n);
  const unsigned fit = slot >= static_cast<unsigned>(kWarpStage)
                           ? 0u
                           : (slot + n <= static_cast<unsigned>(kWarpStage) ? n : kWarpStage - slot);
  unsigned long long gbase = 0;
  if (fit < n) {
    gbase = atomicAdd(fp.counts + row, static_cast<unsigned long long>(n - fit));
    if (fp.region) {
      *binned_bad_word(fp, row) = 1u;
      s_filter_block_bad = 1;
    }
  }
  unsigned j = 0;
  while (mask) {
    const int e = __ffs(mask) - 1;
    mask &= mask - 1;
    const uint64_t key = compose(Dt<DT>::key(elem<DT, VEC>(v, e)) ^ flip, static_cast<uint64_t>(pos + e), ib);
    if (HIST) atomicAdd(&sh_hist[survivor_bin(key, t.key, t.hshift)], 1u);
    if (j < fit) {
      st.s[slot + j] = key;
    } else {
      const unsigned long long q = gbase + (j - fit);
      if (q < static_cast<unsigned long long>(cap)) buf[row * cap + q] = key;
    }
    ++j;
  }
}

// Adds the block's survivor histogram of one selection to the global one and
// clears it.  Called by the whole block at the same point.
__device__ __forceinline__ void hist_flush(unsigned* sh_hist, const FilterParams& fp, int64_t row) {
  __syncthreads();
  unsigned* g = fp.refine_ctl + row * kRefineGridCtlWords + kRefineGridFilterHist;
  for (int i = threadIdx.x; i < kRefineGridBins; i += blockDim.x) {
    const unsigned c = sh_hist[i];
    if (c) {
      atomicAdd(g + i, c);
      sh_hist[i] = 0u;
    }
  }
  __syncthreads();
}

// Returns whether the group held survivors (appended to the stage).
template <int DT, bool LARGEST, int VEC, bool HIST>
__device__ __forceinline__ bool test_group(const uint4& v, int64_t pos, const RowTau& t, const FilterParams& fp,
                                           const Stage& st, int64_t row, unsigned* sh_hist) {
  if (group_candidate<DT, LARGEST, VEC>(v, t.value) || t.nan) {
    const uint32_t mask = exact_mask<DT, LARGEST, VEC>(v, pos, t, fp.ib, fp.flip);
    if (mask) {
      lane_append<DT, VEC, HIST>(mask, v, pos, fp, st, row, t, sh_hist);
      return true;
    }
  }
  return false;
}

// Candidate groups (a 16-byte group with some element at or above tau's
// value) are queued per warp and tested 32 at a time, one per lane, instead
// of in a branch where the whole warp waits for one lane: with ~0.1 % of the
// elements surviving, a fifth of a warp's steps would hold a candidate.
constexpr int kGroupQueue = 64;  // entries per warp (at most 63 between drains)
struct GroupQueue {
  uint4* v;        // kGroupQueue groups
  int64_t* pos;    // their first element's position
};

// Tests `n` (<= 32) queued groups [first, first + n), one per lane.  Called
// by the whole warp.
template <int DT, bool LARGEST, int VEC, bool HIST>
__device__ __forceinline__ void drain_groups(const GroupQueue& q, unsigned first, unsigned n, const RowTau& t,
                                             const FilterParams& fp, const Stage& st, int64_t row,
                                             unsigned* sh_hist) {
  const unsigned lane = threadIdx.x & 31;
  if (lane < n) {
    const uint4 v = q.v[first + lane];
    const int64_t pos = q.pos[first + lane];
    const uint32_t mask = exact_mask<DT, LARGEST, VEC>(v, pos, t, fp.ib, fp.flip);
    if (mask) lane_append<DT, VEC, HIST>(mask, v, pos, fp, st, row, t, sh_hist);
  }
  __syncwarp();
}

// Queues this lane's group when it is a candidate (qn: the warp's queue
// fill, the same in every lane) and tests 32 queued groups once the queue
// holds that many.
template <int DT, bool LARGEST, int VEC, bool HIST>
__device__ __forceinline__ void queue_group(bool cand, const uint4& v, int64_t pos, const GroupQueue& q,
                                            unsigned& qn, const RowTau& t, const FilterParams& fp,
                                            const Stage& st, int64_t row, unsigned* sh_hist) {
  const unsigned m = __ballot_sync(kFull, cand);
  if (m == 0u) return;
  if (cand) {
    const unsigned slot = qn + __popc(m & lanemask_lt());
    q.v[slot] = v;
    q.pos[slot] = pos;
  }
  qn += __popc(m);
  if (qn >= 32u) {
    __syncwarp();
    qn -= 32u;
    drain_groups<DT, LARGEST, VEC, HIST>(q, qn, 32u, t, fp, st, row, sh_hist);
  }
}

// The common path of one full tile of a single selection: this thread's
// kFilterUnroll groups (group u at position base + u * kFilterBlock * VEC)
// are tested against tau's value, candidate groups queued, and the warp's
// stage moved out once it is half full.  Called by the whole warp.
template <int DT, bool LARGEST, int VEC, bool HIST>
__device__ __forceinline__ void single_tile_groups(const uint4 (&v)[kFilterUnroll], int64_t base, const RowTau& t,
                                                   const FilterParams& fp, const Stage& st, unsigned* sh_hist,
                                                   const GroupQueue& q, unsigned& qn) {
  bool cand[kFilterUnroll];
  bool any = false;
#pragma unroll
  for (int u = 0; u < kFilterUnroll; ++u) {
    cand[u] = group_candidate<DT, LARGEST, VEC>(v[u], t.value) || t.nan;
    any |= cand[u];
  }
  if (__any_sync(kFull, any)) {
#pragma unroll
    for (int u = 0; u < kFilterUnroll; ++u)
      queue_group<DT, LARGEST, VEC, HIST>(cand[u], v[u], base + u * kFilterBlock * VEC, q, qn, t, fp, st, 0,
                                          sh_hist);
    // a warp-uniform point: move the stage out once it is half full; when
    // the block bins its survivors at its end they stay, unless the stage
    // is three quarters full (a crowded stretch of the input, as a sorted
    // one): then it is moved out and the bin regions marked incomplete
    const unsigned fill = __shfl_sync(kFull, *st.n, 0);
    if (fill >= static_cast<unsigned>(fp.region ? kWarpStage * 3 / 4 : kWarpStage / 2)) {
      if (fp.region && (threadIdx.x & 31) == 0) {
        *binned_bad_word(fp, 0) = 1u;
        s_filter_block_bad = 1;  // (this block then skips its own placement)
      }
      stage_flush(st, 0, fp.cap, fp.buf, fp.counts);
    }
  }
}

// Tile loop of a single selection (the whole input is one row): no row
// arithmetic per tile, one pointer step, candidate groups queued.  Covers the
// full tiles [tile_begin, tile_end) with stride tile_step; `t` is the row's
// tau.  (Issuing the next tile's loads before testing the current one was
// measured slower: the extra registers cost a block per SM.)
template <int DT, bool LARGEST, int VEC, bool HIST>
__device__ __forceinline__ void filter_full_tiles_single(const FilterParams& fp, int64_t tile_begin, int64_t tile_end,
                                                         int64_t tile_step, const Stage& st, unsigned* sh_hist,
                                                         const RowTau& t, uint64_t pol, const GroupQueue& q) {
  using T = typename Dt<DT>::storage;
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  const T* p = static_cast<const T*>(fp.x) + tile_begin * kTile + threadIdx.x * VEC;
  const int64_t pstep = tile_step * kTile;
  unsigned qn = 0;
  for (int64_t tile = tile_begin; tile < tile_end; tile += tile_step) {
    uint4 v[kFilterUnroll];
#pragma unroll
    for (int u = 0; u < kFilterUnroll; ++u) v[u] = load_group<DT, VEC>(p + u * kFilterBlock * VEC, pol);
    single_tile_groups<DT, LARGEST, VEC, HIST>(v, tile * kTile + threadIdx.x * VEC, t, fp, st, sh_hist, q, qn);
    p += pstep;
  }
  if (qn) drain_groups<DT, LARGEST, VEC, HIST>(q, 0u, qn, t, fp, st, 0, sh_hist);
}

template <int DT, bool LARGEST, int VEC, bool HIST = false>
__device__ void filter_tiles(const FilterParams& fp, int64_t tile_begin, int64_t tile_end,
                             int64_t tile_step, const Stage& st, unsigned* sh_hist = nullptr,
                             const GroupQueue* queue = nullptr) {
  using T = typename Dt<DT>::storage;
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  const int64_t tiles_per_row = (fp.len + kTile - 1) / kTile;
  const uint64_t pol = l2_evict_first_policy();
  // tau (and the largest sampled key) of the current selection: one thread
  // loads them and the block reads shared memory -- a load by every thread of
  // every block would queue thousands of requests on the same L2 line
  __shared__ uint64_t s_row_words[2];
  int64_t cur_row = -1;
  RowTau t{};
  if (fp.nsel == 1) {
    // one selection: the full tiles by the single-row loop, then at most one partial tile below
    if (threadIdx.x == 0) {
      s_row_words[0] = __ldcg(fp.tau);
      if (HIST) s_row_words[1] = sampled_kmax(fp.refine_ctl, 0);
    }
    __syncthreads();
    t = row_tau<DT>(s_row_words[0], fp.ib, fp.flip);
    t.hshift = HIST ? survivor_shift(t.key, s_row_words[1]) : 0;
    cur_row = 0;
    const int64_t full = fp.len / kTile;  // tiles lying wholly inside the row
    int64_t fend = tile_end < full ? tile_end : full;
    if (queue) {
      filter_full_tiles_single<DT, LARGEST, VEC, HIST>(fp, tile_begin, fend, tile_step, st, sh_hist, t, pol, *queue);
    } else {
      // (no queue: the generic loop below takes every tile)
      fend = tile_begin;
    }
    // continue with the tiles from `fend` on (the partial one), by the generic loop
    if (tile_begin < fend) tile_begin += ((fend - tile_begin + tile_step - 1) / tile_step) * tile_step;
  }
  for (int64_t tile = tile_begin; tile < tile_end; tile += tile_step) {
    const int64_t row = static_cast<int64_t>(divide(static_cast<uint64_t>(tile), fp.tiles_per_row));
    const int64_t base = (tile - row * tiles_per_row) * kTile;
    if (row != cur_row) {
      if (cur_row >= 0) {
        stage_flush(st, cur_row, fp.cap, fp.buf, fp.counts);
        if (HIST) hist_flush(sh_hist, fp, cur_row);
      }
      cur_row = row;
      if (threadIdx.x == 0) {
        s_row_words[0] = __ldcg(fp.tau + row);
        if (HIST) s_row_words[1] = sampled_kmax(fp.refine_ctl, row);
      }
      __syncthreads();
      t = row_tau<DT>(s_row_words[0], fp.ib, fp.flip);
      t.hshift = HIST ? survivor_shift(t.key, s_row_words[1]) : 0;
      __syncthreads();  // (the words are rewritten at the next selection)
    }
    const T* xr = static_cast<const T*>(fp.x) + row * fp.len;
    uint4 v[kFilterUnroll];
    if (base + kTile <= fp.len) {
#pragma unroll
      for (int u = 0; u < kFilterUnroll; ++u)
        v[u] = load_group<DT, VEC>(xr + base + (u * kFilterBlock + threadIdx.x) * VEC, pol);
#pragma unroll
      for (int u = 0; u < kFilterUnroll; ++u)
        test_group<DT, LARGEST, VEC, HIST>(v[u], base + (u * kFilterBlock + threadIdx.x) * VEC, t, fp, st, row,
                                           sh_hist);
    } else {  // the last, partial tile of a selection
#pragma unroll
      for (int u = 0; u < kFilterUnroll; ++u) {
        const int64_t pos = base + (u * kFilterBlock + threadIdx.x) * VEC;
        if (pos < fp.len) {
          v[u] = load_group<DT, VEC>(xr + pos, pol);
          test_group<DT, LARGEST, VEC, HIST>(v[u], pos, t, fp, st, row, sh_hist);
        }
      }
    }
    // a warp-uniform point: move the stage out once it is half full
    __syncwarp();
    if (__shfl_sync(kFull, *st.n, 0) >= static_cast<unsigned>(kWarpStage / 2))
      stage_flush(st, row, fp.cap, fp.buf, fp.counts);
  }
  if (cur_row >= 0) {
    stage_flush(st, cur_row, fp.cap, fp.buf, fp.counts);
    if (HIST) hist_flush(sh_hist, fp, cur_row);
  }
}

}  // namespace

}  // namespace tk
