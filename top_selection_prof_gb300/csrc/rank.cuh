// Ranking helpers shared by the threshold and refinement kernels: a
// block-wide scan, counting the keys above a key ("Rank by Counting", Find the
// Cutoff Instead), and the key of a given rank among a few hundred keys.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace tk {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Appends key to dst[*counter ...] for lanes with want set: one atomic per
// warp (shared or global).  Returns the slot of this lane's key (meaningless when !want).
// Called by all 32 lanes of the warp.
__device__ __forceinline__ unsigned warp_append_slot(unsigned* counter, bool want) {
  const unsigned m = __ballot_sync(kFull, want);
  if (m == 0) return 0u;
  const int leader = __ffs(m) - 1;
  unsigned base = 0;
  if (static_cast<int>(threadIdx.x & 31) == leader) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(kFull, base, leader);
  return base + __popc(m & lanemask_lt());
}

// Block-wide inclusive scan of one 64-bit value per thread.  `tmp` holds 32
// entries.  Ends with a barrier, so `tmp` may be reused at once.
__device__ __forceinline__ unsigned long long block_scan_incl(unsigned long long v,
                                                              unsigned long long* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long s = lane < nwarps ? tmp[lane] : 0ull;
    unsigned long long si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, si, o);
      if (lane >= o) si += y;
    }
    if (lane < nwarps) tmp[lane] = si - s;
  }
  __syncthreads();
  v += tmp[warp];
  __syncthreads();
  return v;
}

// Number of keys in src[j0, j1) greater than v.  Rounds of eight
// independent, predicated loads (a slot past j1 reads as key 0, which is
// never greater): the loop is bound by shared-memory latency, not by the
// compares, so no round may wait on the previous one.
__device__ __forceinline__ unsigned count_above(const uint64_t* src, unsigned j0, unsigned j1, uint64_t v) {
  unsigned r = 0;
  for (unsigned j = j0; j < j1; j += 8) {
    uint64_t t[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) t[q] = j + q < j1 ? src[j + q] : 0ull;
#pragma unroll
    for (int q = 0; q < 8; ++q) r += t[q] > v ? 1u : 0u;
  }
  return r;
}

// 0-based rank of slot i among src[0, n): the keys greater than src[i], plus
// the equal keys in earlier slots, so that equal keys (the same position
// drawn twice by the sampler) take consecutive ranks in slot order.  Rounds
// of eight independent loads, as count_above.
__device__ __forceinline__ unsigned rank_in_slots(const uint64_t* src, unsigned n, unsigned i) {
  const uint64_t v = src[i];
  unsigned r = 0;
  for (unsigned j = 0; j < n; j += 8) {
    uint64_t t[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) t[q] = j + q < n ? src[j + q] : 0ull;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      r += (j + q < n && (t[q] > v || (t[q] == v && j + q < i))) ? 1u : 0u;
  }
  return r;
}

// rank_in_slots counted over the slots [j0, j1) only.
__device__ __forceinline__ unsigned rank_in_slot_range(const uint64_t* src, unsigned j0, unsigned j1, unsigned i) {
  const uint64_t v = src[i];
  unsigned r = 0;
  for (unsigned j = j0; j < j1; j += 8) {
    uint64_t t[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) t[q] = j + q < j1 ? src[j + q] : 0ull;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      r += (j + q < j1 && (t[q] > v || (t[q] == v && j + q < i))) ? 1u : 0u;
  }
  return r;
}

// The key of 1-based descending rank `rank` among g[0..n) (in shared or
// global memory; equal keys count once each, ranked in slot order); the
// thread that finds it writes it to *out (the caller synchronises before
// reading).  Few keys (up to 128) are ranked by counting directly, each key
// by a group of p consecutive lanes that count a slice of the slots each
// (p as large as the block allows, at most 32).  More keys are first
// narrowed by 8-bit radix passes below their highest varying bit to at most
// 32, since counting all n keys against each other costs n^2 compares on
// the block's few busy warps (measured: 152 keys ranked directly by one
// thread each 5 us, narrowed first 1.5 us).  lh holds 256 counters; s_tmp 32
// words; s_info 3.  Every thread of the block calls it.
template <int BLOCK>
__device__ void bucket_kth(const uint64_t* g, unsigned n, unsigned long long rank, unsigned* lh,
                           unsigned long long* s_tmp, unsigned long long* s_info, unsigned* s_cnt, uint64_t* out) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (n <= 128u) {
    __syncthreads();
    unsigned p = 1;
    while (p < 32u && 2u * p * n <= static_cast<unsigned>(BLOCK)) p *= 2u;
    const unsigned i = static_cast<unsigned>(tid) / p, part = static_cast<unsigned>(tid) % p;
    unsigned r = 0;
    if (i < n) {
      const unsigned per = (n + p - 1u) / p;
      const unsigned j0 = part * per < n ? part * per : n;
      const unsigned j1 = j0 + per < n ? j0 + per : n;
      r = rank_in_slot_range(g, j0, j1, i);
    }
    // (p divides 32: a key's group of lanes lies inside one warp)
    for (unsigned o = 1; o < p; o <<= 1) r += __shfl_xor_sync(kFull, r, o);
    if (i < n && part == 0u && r == rank - 1) *out = g[i];
    return;
  }
  uint64_t* small = reinterpret_cast<uint64_t*>(s_tmp);  // <= 32 keys (the scans are done by then)
  {
    unsigned long long o = 0, d = ~0ull;
    for (unsigned i = tid; i < n; i += BLOCK) { o |= g[i]; d &= g[i]; }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      o |= __shfl_xor_sync(kFull, o, m);
      d &= __shfl_xor_sync(kFull, d, m);
    }
    if (tid == 0) { s_info[0] = 0ull; s_info[1] = ~0ull; }
    __syncthreads();
    if (lane == 0) { atomicOr(&s_info[0], o); atomicAnd(&s_info[1], d); }
    __syncthreads();
  }
  const unsigned long long gv = s_info[0] ^ s_info[1];
  __syncthreads();
  int lsh = gv ? 63 - __clzll(static_cast<long long>(gv)) : 0;
  lsh = lsh >= 7 ? lsh - 7 : 0;
  uint64_t lpre = 0, lmsk = 0;
  unsigned long long lrank = rank, lcnt = n;
#pragma unroll 1
  while (lcnt > 32) {
    for (int i = tid; i < 256; i += BLOCK) lh[i] = 0u;
    __syncthreads();
    for (unsigned i = tid; i < n; i += BLOCK)
      if ((g[i] & lmsk) == lpre) atomicAdd(&lh[255u - static_cast<unsigned>((g[i] >> lsh) & 255u)], 1u);
    __syncthreads();
    const unsigned long long c = tid < 256 ? lh[tid] : 0ull;
    const unsigned long long incl = block_scan_incl(c, s_tmp);
    if (tid < 256 && incl - c < lrank && lrank <= incl) {
      s_info[0] = static_cast<unsigned long long>(tid);
      s_info[1] = incl - c;
      s_info[2] = c;
    }
    __syncthreads();
    lpre |= static_cast<uint64_t>(255u - static_cast<unsigned>(s_info[0])) << lsh;
    lmsk |= 255ull << lsh;
    lrank -= s_info[1];
    lcnt = s_info[2];
    __syncthreads();
    if (lsh == 0) break;
    lsh = lsh >= 8 ? lsh - 8 : 0;
  }
  if (tid == 0) *s_cnt = 0u;
  __syncthreads();
  for (unsigned i = tid; i < n; i += BLOCK)
    if ((g[i] & lmsk) == lpre) {
      const unsigned slot = atomicAdd(s_cnt, 1u);
      if (slot < 32u) small[slot] = g[i];
    }
  __syncthreads();
  const unsigned ns = *s_cnt < 32u ? *s_cnt : 32u;
  if (static_cast<unsigned>(tid) < ns &&
      rank_in_slots(small, ns, tid) == lrank - 1)
    *out = small[tid];
}

// ---------------------------------------------------------------------------
// The t largest of a block's keys for small t (t <= kSmallTopT), with
// multiplicity (equal keys -- a position drawn twice -- count once each):
// every lane sorts its few keys, each warp pops its t largest by t rounds of
// a warp maximum (the lowest lane holding it advances), and warp 0 does the
// same over the warps' lists.  A handful of instructions per round instead
// of radix passes with a block barrier each.
constexpr int kSmallTopT = 32;

// Sorts v[0..MAXK) descending (a compile-time exchange network).
template <int MAXK>
__device__ __forceinline__ void sort_desc(uint64_t (&v)[MAXK]) {
#pragma unroll
  for (int i = 0; i < MAXK; ++i)
#pragma unroll
    for (int j = 0; j + 1 < MAXK - i; ++j)
      if (v[j] < v[j + 1]) {
        const uint64_t w = v[j];
        v[j] = v[j + 1];
        v[j + 1] = w;
      }
}

// The lanes hold v[0..c) sorted descending.  Pops the warp's t largest
// (t <= 32); lane r returns the r-th (0-based) in *out and the function
// returns how many were popped (fewer when the warp holds fewer keys).
template <int MAXK>
__device__ __forceinline__ int warp_pop_top(uint64_t (&v)[MAXK], int c, int t, uint64_t* out) {
  const int lane = threadIdx.x & 31;
  int popped = 0;
  for (int r = 0; r < t; ++r) {
    const bool has = c > 0;
    const uint64_t head = v[0];
    const unsigned hi = __reduce_max_sync(kFull, has ? static_cast<unsigned>(head >> 32) : 0u);
    const unsigned lo =
        __reduce_max_sync(kFull, (has && static_cast<unsigned>(head >> 32) == hi) ? static_cast<unsigned>(head) : 0u);
    const uint64_t m = (static_cast<uint64_t>(hi) << 32) | lo;
    const unsigned wins = __ballot_sync(kFull, has && head == m);
    if (wins == 0u) break;  // (warp-uniform)
    if (lane == r) *out = m;
    if (lane == __ffs(wins) - 1) {
#pragma unroll
      for (int j = 0; j + 1 < MAXK; ++j) v[j] = v[j + 1];
      --c;
    }
    ++popped;
  }
  return popped;
}

// The block's t largest keys (t <= kSmallTopT), from v[0..c) per thread (any
// order; slots >= c ignored), into top[0..n) in descending order; returns n =
// min(t, keys held).  lists: (BLOCK / 32) * 32 keys of shared memory;
// counts: BLOCK / 32 words; top: kSmallTopT keys; s_n: one word.  Every
// thread of the block calls it; top and the result are valid on return.
template <int BLOCK, int MAXK>
__device__ int block_top_small(uint64_t (&v)[MAXK], int c, int t, uint64_t* lists, unsigned* counts,
                               uint64_t* top, unsigned* s_n) {
  static_assert(BLOCK / 32 <= 8, "warp 0 merges at most eight warps' lists (8 keys a lane)");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < MAXK; ++j)
    if (j >= c) v[j] = 0ull;
  sort_desc(v);
  uint64_t mine = 0ull;
  const int np = warp_pop_top(v, c, t, &mine);
  if (lane < np) lists[warp * 32 + lane] = mine;
  if (lane == 0) counts[warp] = static_cast<unsigned>(np);
  __syncthreads();
  if (warp == 0) {
    // lane l takes eight consecutive entries of one warp's (sorted) list
    constexpr int kW = BLOCK / 32;
    uint64_t u[8];
    int cu = 0;
    const int w = lane / 4, r0 = (lane % 4) * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool ok = w < kW && r0 + j < static_cast<int>(counts[w < kW ? w : 0]);
      u[j] = ok ? lists[w * 32 + r0 + j] : 0ull;
      cu += ok ? 1 : 0;
    }
    uint64_t best = 0ull;
    const int n = warp_pop_top(u, cu, t, &best);
    if (lane < n) top[lane] = best;
    if (lane == 0) *s_n = static_cast<unsigned>(n);
  }
  __syncthreads();
  return static_cast<int>(*s_n);
}

}  // namespace
}  // namespace tk
