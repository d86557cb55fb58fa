// Exact selection on one thread-block cluster per selection problem.
//
// Used for three steps of the pipeline:
//   * threshold estimation (section 3, stage 2): the t-th largest of the S
//     sampled composite keys -> tau;
//   * refinement (section 3, stage 4): the exact top-k of the candidate buffer;
//   * the direct path for small rows: the exact top-k of the row itself.
//
// Select: radix select from the most significant 8-bit digit of the composite
// key ("count elements into buckets and recurse into the bucket that contains
// the boundary", Find the Cutoff Instead).  Each CTA histograms its slice of
// the source into per-warp shared-memory counters (warp-aggregated with
// __match_any_sync, so equal digits never serialise on one address); the
// cluster's CTAs read one another's histograms through distributed shared
// memory, so every CTA finds the same boundary digit without global memory.
// Slices are read with 16-byte loads, eight keys per thread in flight.  Once a
// CTA's elements at or above the current prefix fit in shared memory it caches
// them and stops re-reading the source.  When the boundary bucket holds at
// most kGather keys, they are gathered into CTA 0 and ranked by counting
// ("Rank by Counting": rank = number of larger keys, ties by position), which
// ends the select without further digit passes.
//
// Sort (top-k only): the k winners (keys >= the k-th key; keys are distinct)
// are sorted by a stable LSD radix sort, descending, one 8-bit digit per pass,
// skipping digits on which all winners agree.  If the winners fit in one CTA
// they are gathered into CTA 0 and sorted there with block barriers only;
// otherwise they are spread evenly over the cluster and every pass ranks a
// CTA's items stably per warp, exchanges per-digit counts over DSMEM and
// scatters each key straight into its destination CTA's shared memory.  The
// composite key encodes (value descending, index ascending), so that is the
// output order.
#include <cooperative_groups.h>

#include "common.cuh"
#include "engine.h"

namespace cg = cooperative_groups;

namespace tk {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned kGather = 256;  // bucket size at which the select finishes by ranking
constexpr int64_t kRankMax = 4096;  // winners sorted by counting ranks instead of radix passes

#ifdef TK_PHASE_TIMING
// Debug builds only: globaltimer stamps of the first cluster's CTA 0.
__device__ unsigned long long g_phase_ns[2][32];
__device__ unsigned long long g_cta_ns[2][16][8];  // per CTA of the first cluster: debug stamps
#define TK_STAMP(i)                                                                         \
  do {                                                                                      \
    if (blockIdx.x == 0 && threadIdx.x == 0) g_phase_ns[a.want_topk][(i)] = globaltimer_ns(); \
  } while (0)
#define TK_CTA(slot, v)                                                                    \
  do {                                                                                     \
    if (blockIdx.x < 16 && threadIdx.x == 0) g_cta_ns[a.want_topk][blockIdx.x][(slot)] = (v); \
  } while (0)
#else
#define TK_STAMP(i) \
  do {              \
  } while (0)
#define TK_CTA(slot, v) \
  do {                  \
  } while (0)
#endif

struct SelParams {
  const uint64_t* keys;               // key source (SRC == 0)
  int64_t key_stride;
  const unsigned long long* counts;   // valid keys per selection (nullable)
  const void* x;                      // the input (SRC != 0, and for output values)
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
  uint64_t* xbuf;                     // 2*r keys per selection: the L2 exchange of the sort
};

template <int BLOCK, int P, int CB>
struct Layout {
  static constexpr int kWarps = BLOCK / 32;
  static constexpr int kItems = (P + BLOCK - 1) / BLOCK;
  static constexpr int kQuarters = BLOCK / 256;          // thread groups of 256 (one per digit)
  static constexpr int kWarpsPerQuarter = kWarps / kQuarters;
  static constexpr size_t kBufA = 0;
  static constexpr size_t kBufB = kBufA + sizeof(uint64_t) * P;
  static constexpr size_t kWhist = kBufB + sizeof(uint64_t) * CB;
  static constexpr size_t kHist = kWhist + sizeof(unsigned) * kWarps * 256;
  static constexpr size_t kGbase = kHist + sizeof(unsigned) * 256;
  static constexpr size_t kPart = kGbase + sizeof(unsigned) * 256;
  static constexpr size_t kXch = kPart + sizeof(unsigned) * kQuarters * 256;
  static constexpr size_t kBytes = kXch + sizeof(unsigned long long) * 4;
  static_assert(CB >= P, "cache buffer doubles as the second sort buffer");
  static_assert(BLOCK % 256 == 0, "one thread per digit in each group of 256");
  static_assert(kWarps * 256 * sizeof(unsigned) >= kGather * sizeof(uint64_t), "gather buffer");
};

// Eight consecutive source elements i0 .. i0+7 (i0 a multiple of 8) as
// composite keys.  Only elements in [lo, hi) are meaningful; vector loads may
// also read neighbours that lie inside the same row.
template <int SRC>
__device__ __forceinline__ void load8(const SelParams& a, int64_t row, int64_t i0, int64_t lo, int64_t hi,
                                      uint64_t (&k)[8]) {
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
  for (unsigned iw = threadIdx.x & ~31u; iw < n; iw += BLOCK) {
    const unsigned i = iw + lane;
    f(i < n ? cache[i] : 0ull, i < n);
  }
}

// Adds one to this warp's counter for `digit` (256 = nothing to count).
// Lanes holding the same digit are merged with __match_any_sync and only the
// lowest of them writes, so there is no atomic and no same-address conflict.
// Called by all 32 lanes of the warp.
__device__ __forceinline__ void warp_hist_add(unsigned* wh, unsigned digit) {
  const unsigned peers = __match_any_sync(kFull, digit);
  if (digit < 256u && (peers & lanemask_lt()) == 0) wh[digit] += __popc(peers);
  __syncwarp();
}

// Appends key to dst[*counter ...] for lanes with want set: one shared atomic
// per warp.  Returns the slot of this lane's key (meaningless when !want).
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

// 16-byte global -> shared copies that bypass registers (cp.async, L2 only).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
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

__device__ __forceinline__ unsigned long long block_sum(unsigned long long v, unsigned long long* tmp) {
  __shared__ unsigned long long s_tot;
  const unsigned long long inc = block_scan_incl(v, tmp);
  if (threadIdx.x == blockDim.x - 1) s_tot = inc;
  __syncthreads();
  const unsigned long long r = s_tot;
  __syncthreads();
  return r;
}

template <int BLOCK>
constexpr int min_blocks() { return BLOCK >= 1024 ? 1 : 4; }

// Writes out_vals / out_idx for one winner key at output place `place`.
__device__ __forceinline__ void write_out(const SelParams& a, int64_t row, int64_t k, int64_t place,
                                          uint64_t key) {
  const int64_t oi = row * k + place;
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

// Places keys by counting ("Rank by Counting": a key's place is the number
// of keys that outrank it; the keys are distinct, so places form a
// permutation).  The n keys of src are first grouped, largest group first, by
// the NB-bucket digit of their most significant varying bits, so a key only
// compares against its own group.  The keys are then ranked in grouped order,
// so the lanes of a warp mostly share a group: they read each group member
// once (a broadcast) and run the same number of steps.  Only groups starting
// in [split0, split1) are ranked here (how CTAs share the work); keys whose
// place base_place + rank lies in [w0, w1) are written out.  Returns false
// without writing when the largest group exceeds max_group.
template <int BLOCK, int NB>
__device__ bool place_by_groups(const uint64_t* src, int n, unsigned long long vary, unsigned split0,
                                unsigned split1, uint64_t* grp, unsigned* gcount, unsigned* gstart,
                                unsigned* gcur, unsigned long long* s_tmp, unsigned max_group,
                                const SelParams& a, int64_t row, int64_t kout, int64_t base_place, int64_t w0,
                                int64_t w1) {
  static_assert(NB % BLOCK == 0, "whole groups per thread");
  constexpr int kBits = NB == 2048 ? 11 : 8;
  constexpr int kPer = NB / BLOCK;
  __shared__ unsigned s_gmax;
  const int tid = threadIdx.x;
  const int hb = vary ? 63 - __clzll(static_cast<long long>(vary)) : 0;
  const int dsh = hb >= kBits - 1 ? hb - (kBits - 1) : 0;
  const unsigned mask = NB - 1;
  for (int i = tid; i < NB; i += BLOCK) { gcount[i] = 0u; gcur[i] = 0u; }
  if (tid == 0) s_gmax = 0u;
  __syncthreads();
  for (int i = tid; i < n; i += BLOCK) atomicAdd(&gcount[mask - static_cast<unsigned>((src[i] >> dsh) & mask)], 1u);
  __syncthreads();
  unsigned c[kPer];
  unsigned long long sum = 0;
  unsigned mx = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    c[q] = gcount[tid * kPer + q];
    sum += c[q];
    mx = c[q] > mx ? c[q] : mx;
  }
  const unsigned long long incl = block_scan_incl(sum, s_tmp);
  unsigned run = static_cast<unsigned>(incl - sum);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    gstart[tid * kPer + q] = run;
    run += c[q];
  }
  atomicMax(&s_gmax, mx);
  __syncthreads();
  if (s_gmax > max_group) return false;
  for (int i = tid; i < n; i += BLOCK) {
    const uint64_t key = src[i];
    const unsigned g = mask - static_cast<unsigned>((key >> dsh) & mask);
    grp[gstart[g] + atomicAdd(&gcur[g], 1u)] = key;
  }
  __syncthreads();
  for (int i = tid; i < n; i += BLOCK) {
    const uint64_t v = grp[i];
    const unsigned g = mask - static_cast<unsigned>((v >> dsh) & mask);
    const unsigned g0 = gstart[g];
    if (g0 < split0 || g0 >= split1) continue;
    const unsigned g1 = g0 + gcount[g];
    unsigned r0 = 0, r1 = 0;
    unsigned j = g0;
    for (; j + 1 < g1; j += 2) {
      r0 += grp[j] > v ? 1u : 0u;
      r1 += grp[j + 1] > v ? 1u : 0u;
    }
    if (j < g1) r0 += grp[j] > v ? 1u : 0u;
    const int64_t place = base_place + g0 + r0 + r1;
    if (place >= w0 && place < w1) write_out(a, row, kout, place, v);
  }
  return true;
}

// OR and AND of src[0..n) over the block.
template <int BLOCK>
__device__ void block_or_and(const uint64_t* src, int n, unsigned long long* out_or, unsigned long long* out_and) {
  __shared__ unsigned long long s_or[32], s_and[32];
  unsigned long long o = 0, d = ~0ull;
  for (int i = threadIdx.x; i < n; i += BLOCK) { o |= src[i]; d &= src[i]; }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    o |= __shfl_xor_sync(kFull, o, m);
    d &= __shfl_xor_sync(kFull, d, m);
  }
  if ((threadIdx.x & 31) == 0) { s_or[threadIdx.x >> 5] = o; s_and[threadIdx.x >> 5] = d; }
  __syncthreads();
  o = 0;
  d = ~0ull;
  for (int w = 0; w < BLOCK / 32; ++w) { o |= s_or[w]; d &= s_and[w]; }
  *out_or = o;
  *out_and = d;
  __syncthreads();
}

template <int BLOCK, int P, int CB, int SRC>
__global__ void __launch_bounds__(BLOCK, min_blocks<BLOCK>()) select_kernel(SelParams a) {
  using L = Layout<BLOCK, P, CB>;
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* bufA = reinterpret_cast<uint64_t*>(smem + L::kBufA);
  uint64_t* bufB = reinterpret_cast<uint64_t*>(smem + L::kBufB);
  unsigned* whist = reinterpret_cast<unsigned*>(smem + L::kWhist);
  unsigned* hist = reinterpret_cast<unsigned*>(smem + L::kHist);
  unsigned* gbase = reinterpret_cast<unsigned*>(smem + L::kGbase);
  unsigned* part = reinterpret_cast<unsigned*>(smem + L::kPart);
  unsigned long long* xch = reinterpret_cast<unsigned long long*>(smem + L::kXch);
  __shared__ unsigned long long s_tmp[32];
  __shared__ unsigned long long s_info[5];
  __shared__ unsigned s_cnt;
  __shared__ unsigned s_gcount;
  __shared__ int s_over;

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned G = cluster.num_blocks();
  const unsigned crank = cluster.block_rank();
  const int64_t row = blockIdx.x / G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // programmatic dependent launch: everything below may read what earlier
  // grids wrote, so wait for them; the next grid may begin launching now
  grid_dependency_wait();
  grid_launch_dependents();

  int64_t valid = (SRC == 0) ? a.key_stride : a.len;
  if (SRC == 0 && a.counts) {
    const unsigned long long c = __ldcg(a.counts + row);
    if (c < static_cast<unsigned long long>(valid)) valid = static_cast<int64_t>(c);
  }
  // slices start at even positions so key slices can be copied in 16-byte units
  const int64_t sb = (valid * crank / G) & ~int64_t(1);
  const int64_t se = (crank + 1 == G) ? valid : ((valid * (crank + 1) / G) & ~int64_t(1));
  if (tid == 0) s_gcount = 0u;
  TK_STAMP(0);
  TK_CTA(0, globaltimer_ns());

  // The cache is the whole buffer (both halves): the winners later leave
  // through the L2 exchange buffer, so nothing else is written here meanwhile.
  uint64_t* cache = bufA;
  const unsigned long long cache_cap = P + CB;
  bool cached = false;
  unsigned cache_n = 0;
  if (SRC == 0 && static_cast<unsigned long long>(se - sb) <= cache_cap) {
    // the whole slice fits: copy it in with cp.async, no registers involved
    const uint64_t* from = a.keys + row * a.key_stride + sb;
    const unsigned n = static_cast<unsigned>(se - sb);
    if (a.key_vec) {
      for (unsigned i = 2 * tid; i + 1 < n; i += 2 * BLOCK) cp_async16(cache + i, from + i);
      if ((n & 1u) && tid == 0) cache[n - 1] = __ldcg(from + n - 1);
      cp_async_wait_all();
    } else {
      for (unsigned i = tid; i < n; i += BLOCK) cache[i] = __ldcg(from + i);
    }
    cached = true;
    cache_n = n;
    __syncthreads();
  }
  TK_STAMP(1);

  // ------------------------------------------------------------------ select
  const int kb = a.key_bits + a.ib;
  uint64_t prefix = 0, pmask = 0;
  unsigned long long rank = static_cast<unsigned long long>(a.r);
  unsigned long long local_above = 0, local_bucket = static_cast<unsigned long long>(se - sb);
  bool failed = false;
  for (int shift = ((kb - 1) / 8) * 8; shift >= 0; shift -= 8) {
    const bool will_cache = !cached && (local_above + local_bucket) <= cache_cap;
    for (int i = tid; i < L::kWarps * 256; i += BLOCK) whist[i] = 0u;
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    unsigned* wh = whist + warp * 256;
    if (cached) {
      for (unsigned i = 2 * tid; i < cache_n; i += 2 * BLOCK) {
        const uint64_t k0 = cache[i];
        if ((k0 & pmask) == prefix) atomicAdd(&wh[(k0 >> shift) & 255u], 1u);
        if (i + 1 < cache_n) {
          const uint64_t k1 = cache[i + 1];
          if ((k1 & pmask) == prefix) atomicAdd(&wh[(k1 >> shift) & 255u], 1u);
        }
      }
    } else {
      for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t k, bool in) {
        warp_hist_add(wh, (in && (k & pmask) == prefix) ? static_cast<unsigned>((k >> shift) & 255u) : 256u);
        if (will_cache) {
          const bool want = in && k >= prefix;
          const unsigned slot = warp_append_slot(&s_cnt, want);
          if (want) cache[slot] = k;
        }
      });
    }
    __syncthreads();
    if (shift == ((kb - 1) / 8) * 8) TK_STAMP(25);
    {
      // per-digit sum over the warps' counters: each group of 256 threads
      // sums a quarter of the warps, then the quarters are added
      const int dq = tid & 255, q = tid >> 8;
      unsigned sq = 0;
      for (int w = q * L::kWarpsPerQuarter; w < (q + 1) * L::kWarpsPerQuarter; ++w) sq += whist[w * 256 + dq];
      part[q * 256 + dq] = sq;
      __syncthreads();
      if (tid < 256) {
        unsigned sd = 0;
        for (int q2 = 0; q2 < L::kQuarters; ++q2) sd += part[q2 * 256 + tid];
        hist[tid] = sd;
      }
    }
    if (will_cache) {
      cache_n = s_cnt;
      cached = true;
    }
    if (tid == 0) s_info[0] = ~0ull;
    if (shift == ((kb - 1) / 8) * 8) TK_STAMP(26);
    cluster.sync();
    if (shift == ((kb - 1) / 8) * 8) TK_STAMP(27);
    // digit 255 - tid; inclusive scans from the top digit downwards of the
    // cluster totals and of this CTA's own counts
    unsigned long long tot = 0, mine = 0;
    const int d = 255 - tid;
    if (tid < 256) {
      for (unsigned c = 0; c < G; ++c) tot += cluster.map_shared_rank(hist, c)[d];
      mine = hist[d];
    }
    const unsigned long long incl = block_scan_incl(tot, s_tmp);
    const unsigned long long mine_incl = block_scan_incl(mine, s_tmp);
    if (shift == ((kb - 1) / 8) * 8) TK_STAMP(28);
    if (tid < 256) {
      const unsigned long long excl = incl - tot;
      if (excl < rank && rank <= incl) {
        s_info[0] = static_cast<unsigned long long>(d);
        s_info[1] = excl;
        s_info[2] = mine;
        s_info[3] = mine_incl - mine;  // this CTA's keys in digits above d
        s_info[4] = tot;
      }
    }
    cluster.sync();
    TK_STAMP(2 + (shift >> 3));
    if (s_info[0] == ~0ull) { failed = true; break; }
    prefix |= s_info[0] << shift;
    pmask |= 0xffull << shift;
    rank -= s_info[1];
    local_above += s_info[3];
    local_bucket = s_info[2];
    if (shift > 0 && s_info[4] <= kGather) {
      // Gather the boundary bucket into CTA 0 and rank it by counting.
      unsigned* g_cnt = cluster.map_shared_rank(&s_gcount, 0);
      uint64_t* g_buf = cluster.map_shared_rank(reinterpret_cast<uint64_t*>(whist), 0);
      if (cached) {
        for (unsigned i = tid; i < cache_n; i += BLOCK) {
          const uint64_t k = cache[i];
          if ((k & pmask) == prefix) g_buf[atomicAdd(g_cnt, 1u)] = k;
        }
      } else {
        for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t k, bool in) {
          if (in && (k & pmask) == prefix) g_buf[atomicAdd(g_cnt, 1u)] = k;
        });
      }
      cluster.sync();
      if (crank == 0) {
        const unsigned n = s_gcount;
        const uint64_t* g = reinterpret_cast<const uint64_t*>(whist);
        if (static_cast<unsigned>(tid) < n) {
          const uint64_t mine = g[tid];
          unsigned long long above = 0;
          for (unsigned j = 0; j < n; ++j) {
            const uint64_t o = g[j];
            above += (o > mine || (o == mine && j < static_cast<unsigned>(tid))) ? 1ull : 0ull;
          }
          if (above == rank - 1)
            for (unsigned c = 0; c < G; ++c) cluster.map_shared_rank(xch, c)[3] = mine;
        }
      }
      cluster.sync();
      TK_STAMP(12);
      prefix = xch[3];
      pmask = ~0ull;
      break;
    }
  }
  if (failed) {
    if (tid == 0 && crank == 0) atomicCAS(a.status, kDevOk, kDevBadState);
    return;
  }
  const uint64_t tau = prefix;  // the r-th largest key
  if (!a.want_topk) {
    if (tid == 0 && crank == 0) a.tau_out[row] = tau;
    return;
  }

  // ------------------------------------------------------------------ winners
  TK_STAMP(13);
  const int64_t k = a.r;
  {
    unsigned long long cnt = 0, orm = 0, andm = ~0ull;
    if (tid == 0) {
      s_cnt = 0u;
      s_over = 0;
      xch[1] = 0ull;
      xch[2] = ~0ull;
    }
    __syncthreads();
    if (cached) {
      for (unsigned i = tid; i < cache_n; i += BLOCK) {
        const uint64_t key = cache[i];
        if (key >= tau) { ++cnt; orm |= key; andm &= key; }
      }
    } else {
      for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t key, bool in) {
        const bool w = in && key >= tau;
        if (w) { ++cnt; orm |= key; andm &= key; }
        const unsigned slot = warp_append_slot(&s_cnt, w);
        if (w) {
          if (slot < static_cast<unsigned>(CB)) bufB[slot] = key; else s_over = 1;
        }
      });
    }
    const unsigned long long total = block_sum(cnt, s_tmp);
    TK_STAMP(15);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      orm |= __shfl_xor_sync(kFull, orm, o);
      andm &= __shfl_xor_sync(kFull, andm, o);
    }
    if (lane == 0) {
      atomicOr(&xch[1], orm);
      atomicAnd(&xch[2], andm);
    }
    if (tid == 0) xch[0] = total;
  }
  cluster.sync();
  unsigned long long base = 0, all_or = 0, all_and = ~0ull, all_cnt = 0;
  for (unsigned c = 0; c < G; ++c) {
    const unsigned long long* rx = cluster.map_shared_rank(xch, c);
    if (c < crank) base += rx[0];
    all_cnt += rx[0];
    all_or |= rx[1];
    all_and &= rx[2];
  }
  if (all_cnt != static_cast<unsigned long long>(k)) {
    if (tid == 0 && crank == 0) atomicCAS(a.status, kDevOk, kDevBadState);
    cluster.sync();
    return;
  }
  TK_STAMP(29);
  // Place the winners: position base + local sequence, in an L2-resident
  // exchange buffer (plain global stores; each CTA then reads back what it
  // needs), which costs far less than scattering single keys into other CTAs'
  // shared memory.
  uint64_t* xb = a.xbuf + row * 2 * k;
  int xsel = 0;  // which half of the exchange buffer the next exchange uses
  {
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    auto place = [&](uint64_t key, bool want) {
      const unsigned slot = warp_append_slot(&s_cnt, want);
      if (want) {
        xb[static_cast<unsigned>(base) + slot] = key;
      }
    };
    if (cached || !s_over) {
      const unsigned n = cached ? cache_n : static_cast<unsigned>(xch[0]);
      const uint64_t* from = cached ? cache : bufB;
      for_cache<BLOCK>(from, n, [&](uint64_t key, bool in) { place(key, in && (!cached || key >= tau)); });
    } else {
      for_slice<SRC, BLOCK>(a, row, sb, se, [&](uint64_t key, bool in) { place(key, in && key >= tau); });
    }
  }
  TK_STAMP(30);
  cluster.sync();
  TK_STAMP(14);
  if (k <= kRankMax) {
    // Every CTA holds all k winners (read from the exchange buffer, in the
    // same order everywhere) and places its 1/G share of them.
    for (int i = tid; i < k; i += BLOCK) bufA[i] = __ldcg(xb + i);
    // CTA c ranks the groups that start in its 1/G of the places
    const unsigned kc = static_cast<unsigned>((k + G - 1) / G);
    const unsigned lo = crank * kc, hi = crank + 1 == G ? static_cast<unsigned>(k) : lo + kc;
    if constexpr (BLOCK >= 1024)
      place_by_groups<BLOCK, 2048>(bufA, static_cast<int>(k), all_or ^ all_and, lo, hi, bufB, whist,
                                   whist + 2048, whist + 4096, s_tmp, ~0u, a, row, k, 0, 0, k);
    else
      place_by_groups<BLOCK, 256>(bufA, static_cast<int>(k), all_or ^ all_and, lo, hi, bufB, hist, gbase,
                                  part, s_tmp, ~0u, a, row, k, 0, 0, k);
    TK_STAMP(24);
    return;
  }

  // ------------------------------------------------------------------ large k
  // Each CTA owns the output places [my0, my0 + n_mine).  The winners are
  // partitioned once by their 11 most significant varying bits: exact bin
  // counts are exchanged over DSMEM, every key is written to its bin's
  // segment of the exchange buffer, and each CTA then sorts only the bins
  // that overlap its places, locally.  If some CTA's bins do not fit in its
  // shared memory (a pathological bin), the cluster falls back to an LSD
  // radix sort over evenly split chunks.
  const unsigned long long vary = all_or ^ all_and;
  const int hb = vary ? 63 - __clzll(static_cast<long long>(vary)) : 0;
  const int64_t pe = (k + G - 1) / G;
  const int64_t my0 = static_cast<int64_t>(crank) * pe;
  const int n_mine = static_cast<int>(my0 >= k ? 0 : (k - my0 < pe ? k - my0 : pe));
  for (int i = tid; i < n_mine; i += BLOCK) bufA[i] = __ldcg(xb + my0 + i);
  __syncthreads();
  bool local_sort = (G == 1);
  int64_t ext0 = my0;
  int n_c = n_mine;
  if (G > 1 && BLOCK == 1024) {
    const int psh = hb >= 10 ? hb - 10 : 0;
    unsigned* lh = whist;           // local count per bin (read by the other CTAs)
    unsigned* bst = whist + 2048;   // first place of each bin (the end of the last one is k)
    unsigned* off = whist + 4096;   // this CTA's first place inside each bin
    unsigned* cur = whist + 6144;   // fill cursors
    for (int i = tid; i < 2048; i += BLOCK) { lh[i] = 0u; cur[i] = 0u; }
    __syncthreads();
    for (int i = tid; i < n_mine; i += BLOCK) atomicAdd(&lh[2047u - ((bufA[i] >> psh) & 2047u)], 1u);
    cluster.sync();
    {
      unsigned tt[2], bm[2];
      unsigned long long tsum = 0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int b = tid * 2 + q;
        unsigned t = 0, before = 0;
        for (unsigned c = 0; c < G; ++c) {
          const unsigned h = cluster.map_shared_rank(lh, c)[b];
          t += h;
          if (c < crank) before += h;
        }
        tt[q] = t;
        bm[q] = before;
        tsum += t;
      }
      const unsigned long long incl = block_scan_incl(tsum, s_tmp);
      unsigned run = static_cast<unsigned>(incl - tsum);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int b = tid * 2 + q;
        bst[b] = run;
        off[b] = run + bm[q];
        run += tt[q];
      }
    }
    cluster.sync();  // every CTA has read the others' counts
    uint64_t* xb1 = xb + k;
    for (int i = tid; i < n_mine; i += BLOCK) {
      const uint64_t key = bufA[i];
      const unsigned bi = 2047u - static_cast<unsigned>((key >> psh) & 2047u);
      xb1[off[bi] + atomicAdd(&cur[bi], 1u)] = key;
    }
    // extended range of every CTA: from the start of the bin holding its
    // first place to the end of the bin holding its last place
    __shared__ unsigned s_ext[2 * 16];
    __shared__ int s_fit;
    if (tid == 0) s_fit = 1;
    __syncthreads();
    if (tid < static_cast<int>(G)) {
      const int64_t c0 = static_cast<int64_t>(tid) * pe;
      const int64_t c1 = c0 + pe < k ? c0 + pe : k;
      unsigned e0 = 0, e1 = 0;
      if (c0 < k) {
        // bin holding place p: the last b with bst[b] <= p (empty bins have
        // no place, so the first b with bst[b] > p follows the right one)
        auto bin_of = [&](unsigned p) {
          int lo2 = 0, hi2 = 2048;
          while (lo2 < hi2) {
            const int mid = (lo2 + hi2) >> 1;
            if (bst[mid] <= p) lo2 = mid + 1; else hi2 = mid;
          }
          return lo2 - 1;
        };
        e0 = bst[bin_of(static_cast<unsigned>(c0))];
        const int b1 = bin_of(static_cast<unsigned>(c1 - 1)) + 1;
        e1 = b1 < 2048 ? bst[b1] : static_cast<unsigned>(k);
      }
      s_ext[2 * tid] = e0;
      s_ext[2 * tid + 1] = e1;
      if (e1 - e0 > static_cast<unsigned>(P)) atomicAnd(&s_fit, 0);
    }
    cluster.sync();  // the bins are complete in the exchange buffer
    if (s_fit) {
      local_sort = true;
      ext0 = s_ext[2 * crank];
      n_c = static_cast<int>(s_ext[2 * crank + 1] - s_ext[2 * crank]);
      for (int i = tid; i < n_c; i += BLOCK) bufA[i] = __ldcg(xb1 + ext0 + i);
      __syncthreads();
    }
  }
  TK_STAMP(15);
  TK_CTA(1, globaltimer_ns());
  if constexpr (BLOCK >= 1024) if (local_sort) {
    unsigned long long lo_or, lo_and;
    block_or_and<BLOCK>(bufA, n_c, &lo_or, &lo_and);
    if (place_by_groups<BLOCK, 2048>(bufA, n_c, lo_or ^ lo_and, 0u, ~0u, bufB, whist, whist + 2048,
                                     whist + 4096, s_tmp, 512u, a, row, k, ext0, my0, my0 + n_mine)) {
      TK_STAMP(24);
      TK_CTA(2, globaltimer_ns());
      TK_CTA(3, 1ull);
      return;
    }
  }
  const unsigned sortG = local_sort ? 1u : G;  // CTAs taking part in each sort pass

  // ------------------------------------------------------------------ sort
  uint64_t* src = bufA;
  uint64_t* dst = bufB;
  const int ipw = (n_c + L::kWarps - 1) / L::kWarps;  // items per warp segment
  const int seg0 = warp * ipw;
  const int seg1 = (seg0 + ipw < n_c) ? seg0 + ipw : n_c;
  const unsigned lt = lanemask_lt();
  auto gsync = [&]() {
    if (sortG > 1) cluster.sync(); else __syncthreads();
  };
  for (int shift = 0; shift < 64; shift += 8) {
    if (((vary >> shift) & 0xffull) == 0) continue;  // uniform over the sorting CTAs
    for (int i = tid; i < L::kWarps * 256; i += BLOCK) whist[i] = 0u;
    __syncthreads();
    unsigned* wh = whist + warp * 256;
    uint64_t key[L::kItems];
    unsigned dig[L::kItems], wr[L::kItems];
    const int nj = (seg1 - seg0 + 31) >> 5;  // items per lane, uniform in the warp
#pragma unroll
    for (int j = 0; j < L::kItems; ++j) {
      if (j >= nj) break;
      const int i = seg0 + j * 32 + lane;
      const bool v = i < seg1;
      key[j] = v ? src[i] : 0ull;
      dig[j] = v ? 255u - static_cast<unsigned>((key[j] >> shift) & 255u) : 256u + lane;
      const unsigned peers = __match_any_sync(kFull, dig[j]);
      const unsigned before = __popc(peers & lt);
      const unsigned b = v ? wh[dig[j]] : 0u;
      __syncwarp();
      if (v && before == 0) wh[dig[j]] = b + __popc(peers);
      __syncwarp();
      wr[j] = b + before;
    }
    __syncthreads();
    TK_STAMP(10);
    // exclusive prefix of the per-warp counts over warps, per digit, in two
    // steps: within groups of warps, then across groups
    {
      const int d = tid & 255, q = tid >> 8;
      unsigned run = 0;
      for (int w = q * L::kWarpsPerQuarter; w < (q + 1) * L::kWarpsPerQuarter; ++w) {
        const unsigned t = whist[w * 256 + d];
        whist[w * 256 + d] = run;
        run += t;
      }
      part[q * 256 + d] = run;
      __syncthreads();
      unsigned qbase = 0;
      for (int q2 = 0; q2 < q; ++q2) qbase += part[q2 * 256 + d];
      if (qbase)
        for (int w = q * L::kWarpsPerQuarter; w < (q + 1) * L::kWarpsPerQuarter; ++w) whist[w * 256 + d] += qbase;
      if (q == L::kQuarters - 1) hist[d] = qbase + run;
    }
    TK_STAMP(11);
    gsync();
    TK_STAMP(31);
    unsigned long long tot = 0, before_me = 0;
    if (tid < 256) {
      if (sortG == 1) {
        tot = hist[tid];  // this CTA sorts alone
      } else {
        for (unsigned c = 0; c < sortG; ++c) {
          const unsigned h = cluster.map_shared_rank(hist, c)[tid];
          tot += h;
          if (c < crank) before_me += h;
        }
      }
    }
    const unsigned long long incl = block_scan_incl(tot, s_tmp);
    if (tid < 256) gbase[tid] = static_cast<unsigned>(incl - tot + before_me);
    gsync();
    TK_STAMP(23);
#pragma unroll
    for (int j = 0; j < L::kItems; ++j) {
      if (j >= nj) break;
      const int i = seg0 + j * 32 + lane;
      if (i < seg1) {
        const unsigned pos = gbase[dig[j]] + wh[dig[j]] + wr[j];
        if (sortG == 1) dst[pos] = key[j]; else xb[xsel * k + pos] = key[j];
      }
    }
    TK_STAMP(22);
    gsync();
    TK_STAMP(21);
    if (sortG == 1) {
      uint64_t* t = src; src = dst; dst = t;
    } else {
      // read back this CTA's range; the next exchange uses the other half, so
      // no CTA can overwrite what another is still reading
      const uint64_t* from = xb + xsel * k + my0;
      for (int i = tid; i < n_c; i += BLOCK) src[i] = __ldcg(from + i);
      xsel ^= 1;
      __syncthreads();
    }
    TK_STAMP(16 + (shift >> 3));
  }

  // ------------------------------------------------------------------ output
  TK_STAMP(24);
  // local index i holds place ext0 + i; this CTA writes the places it owns
  for (int i = tid; i < n_c; i += BLOCK) {
    const int64_t place = ext0 + i;
    if (place >= my0 && place < my0 + n_mine) write_out(a, row, k, place, src[i]);
  }
  TK_CTA(2, globaltimer_ns());
  TK_CTA(3, 2ull + static_cast<unsigned long long>(n_c));
}

// Kernel variants: (block, sort positions per CTA, cache/second buffer).
constexpr int kSmallBlock = 256, kSmallP = 1024, kSmallCB = 2048;
constexpr int kBigBlock = 1024, kBigP = 12000, kBigCB = 12000;
constexpr int kMaxCluster = 16;

template <int BLOCK, int P, int CB, int SRC>
cudaError_t configure(int* max_g) {
  using L = Layout<BLOCK, P, CB>;
  auto kern = select_kernel<BLOCK, P, CB, SRC>;
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

template <int BLOCK, int P, int CB, int SRC>
cudaError_t launch_variant(const SelParams& a, int64_t nsel, int G, int* used, cudaStream_t st) {
  using L = Layout<BLOCK, P, CB>;
  int max_g = 1;
  cudaError_t e = configure<BLOCK, P, CB, SRC>(&max_g);
  if (e != cudaSuccess) return e;
  if (G > max_g) G = max_g;
  const int64_t sort_k = a.want_topk ? a.r : 1;
  if (sort_k > static_cast<int64_t>(G) * P) return cudaErrorInvalidConfiguration;
  if (a.want_topk && G > 1 && a.xbuf == nullptr) return cudaErrorInvalidValue;
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
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, select_kernel<BLOCK, P, CB, SRC>, a);
}

template <int BLOCK, int P, int CB>
cudaError_t launch_src(const SelParams& a, int src, int64_t nsel, int G, int* used, cudaStream_t st) {
  if (src == 0) return launch_variant<BLOCK, P, CB, 0>(a, nsel, G, used, st);
  if (src == 1) return launch_variant<BLOCK, P, CB, 1>(a, nsel, G, used, st);
  return launch_variant<BLOCK, P, CB, 2>(a, nsel, G, used, st);
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

#ifdef TK_PHASE_TIMING
int debug_phase_ns(unsigned long long* out) {
  if (cudaMemcpyFromSymbol(out, g_phase_ns, sizeof(g_phase_ns)) != cudaSuccess) return -3;
  return cudaMemcpyFromSymbol(out + 64, g_cta_ns, sizeof(g_cta_ns)) == cudaSuccess ? 0 : -3;  // 2*16*8
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
  const int src = job.keys ? 0 : (p.dtype == kF32 ? 1 : 2);
  const bool many = p.nsel >= sm_count();
  int G;
  bool small;
  if (!job.want_topk) {
    // tau: cache every key of the slice; the whole buffer is the cache
    small = false;
    G = pow2_at_least((source_hint + kBigP + kBigCB - 1) / (kBigP + kBigCB));
  } else if (many && job.r <= kSmallP) {
    small = true;
    G = 1;
  } else {
    small = false;
    const int64_t g_min = (job.r + kBigP - 1) / kBigP;
    const int64_t g_cache = (source_hint + kBigCB - 1) / kBigCB;
    G = many ? pow2_at_least(g_min) : pow2_at_least(g_min > g_cache ? g_min : g_cache);
  }
  int used = G;
  const cudaError_t e = small ? launch_src<kSmallBlock, kSmallP, kSmallCB>(a, src, p.nsel, G, &used, st)
                              : launch_src<kBigBlock, kBigP, kBigCB>(a, src, p.nsel, G, &used, st);
  if (cluster) *cluster = used;
  return e;
}

}  // namespace tk
