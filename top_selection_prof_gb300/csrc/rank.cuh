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

// The key of 1-based descending rank `rank` among g[0..n) (in shared or
// global memory; equal keys count once each, ranked in slot order); the
// thread that finds it writes it to *out (the caller synchronises before
// reading).  Few keys are ranked by counting
// directly (up to 128); more are first narrowed by 8-bit radix passes below
// their highest varying bit to at most 32, since counting all n keys against
// each other costs n^2 compares on the block's few busy warps (measured: 152
// keys ranked directly 5 us, narrowed first 1.5 us).  lh holds 256 counters;
// s_tmp 32 words; s_info 3.  Every thread of the block calls it.
template <int BLOCK>
__device__ void bucket_kth(const uint64_t* g, unsigned n, unsigned long long rank, unsigned* lh,
                           unsigned long long* s_tmp, unsigned long long* s_info, unsigned* s_cnt, uint64_t* out) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (n <= 128u) {
    __syncthreads();
    for (unsigned i = tid; i < n; i += BLOCK)
      if (rank_in_slots(g, n, i) == rank - 1) *out = g[i];
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

}  // namespace
}  // namespace tk
