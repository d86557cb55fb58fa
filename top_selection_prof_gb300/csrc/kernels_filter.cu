// Stage 3 of Prof-K (section 3, "Filtering") and the exact fallback
// (section 3, stage 4, and Appendix D "Fallback as a Safety Mechanism").
//
// filter_kernel streams every selection once and appends the composite key of
// each element ranking at or above tau to the candidate buffer.  It is the
// HBM-bound hot loop: a persistent grid walks 16 KB tiles with 16-byte
// read-only loads; one NaN-propagating max (min) per 16 bytes and a float
// compare against tau's value is the common-path test.  Only a lane whose
// group holds a candidate builds exact composite keys, and it appends its
// survivors to its warp's shared-memory stage with one shared atomic; the
// stage is flushed at tile ends with one global atomicAdd per flush.  The
// counter keeps counting past the capacity M so R is exact; only slots < M are
// written.
//
// fallback_kernel is a cooperative launch.  For every selection whose filter
// result missed k <= R <= M (or every selection when forced) it finds the
// k-th largest element exactly by radix select on the value key (8-bit digits,
// one grid-wide histogram per digit), resolves ties at that value by index --
// per-tile counts of the tied value, a scan and a lower bound over the running
// count ("Find It in log n"), then an ordered scan of one tile -- and re-runs
// the filter with that exact threshold, which keeps exactly k elements.
// Grid-wide steps use a bounded barrier that reports a timeout instead of
// hanging.
#include <cooperative_groups.h>

#include "common.cuh"
#include "engine.h"

namespace tk {

namespace {

constexpr int kFilterBlock = 256;
constexpr int kFilterUnroll = 4;
constexpr int kWarpStage = 256;  // survivors staged per warp before a flush
constexpr unsigned kFull = 0xffffffffu;

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
};

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
// what does not fit is appended to the buffer directly.
template <int DT, int VEC>
__device__ __forceinline__ void lane_append(uint32_t mask, const uint4& v, int64_t pos, int ib, uint32_t flip,
                                            const Stage& st, int64_t row, int64_t cap, uint64_t* buf,
                                            unsigned long long* counts) {
  const unsigned n = __popc(mask);
  const unsigned slot = atomicAdd(st.n, n);
  const unsigned fit = slot >= static_cast<unsigned>(kWarpStage)
                           ? 0u
                           : (slot + n <= static_cast<unsigned>(kWarpStage) ? n : kWarpStage - slot);
  unsigned long long gbase = 0;
  if (fit < n) gbase = atomicAdd(counts + row, static_cast<unsigned long long>(n - fit));
  unsigned j = 0;
  while (mask) {
    const int e = __ffs(mask) - 1;
    mask &= mask - 1;
    const uint64_t key = compose(Dt<DT>::key(elem<DT, VEC>(v, e)) ^ flip, static_cast<uint64_t>(pos + e), ib);
    if (j < fit) {
      st.s[slot + j] = key;
    } else {
      const unsigned long long q = gbase + (j - fit);
      if (q < static_cast<unsigned long long>(cap)) buf[row * cap + q] = key;
    }
    ++j;
  }
}

template <int DT, bool LARGEST, int VEC>
__device__ __forceinline__ void test_group(const uint4& v, int64_t pos, const RowTau& t, const FilterParams& fp,
                                           const Stage& st, int64_t row) {
  if (group_candidate<DT, LARGEST, VEC>(v, t.value) || t.nan) {
    const uint32_t mask = exact_mask<DT, LARGEST, VEC>(v, pos, t, fp.ib, fp.flip);
    if (mask) lane_append<DT, VEC>(mask, v, pos, fp.ib, fp.flip, st, row, fp.cap, fp.buf, fp.counts);
  }
}

// Filter the tiles [tile_begin, tile_end) (stride tile_step) of the flattened
// tile space (selection-major).  Used by the filter kernel and the fallback.
template <int DT, bool LARGEST, int VEC>
__device__ void filter_tiles(const FilterParams& fp, int64_t tile_begin, int64_t tile_end,
                             int64_t tile_step, const Stage& st) {
  using T = typename Dt<DT>::storage;
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  const int64_t tiles_per_row = (fp.len + kTile - 1) / kTile;
  const uint64_t pol = l2_evict_first_policy();
  int64_t cur_row = -1;
  RowTau t{};
  for (int64_t tile = tile_begin; tile < tile_end; tile += tile_step) {
    const int64_t row = static_cast<int64_t>(divide(static_cast<uint64_t>(tile), fp.tiles_per_row));
    const int64_t base = (tile - row * tiles_per_row) * kTile;
    if (row != cur_row) {
      if (cur_row >= 0) stage_flush(st, cur_row, fp.cap, fp.buf, fp.counts);
      cur_row = row;
      t = row_tau<DT>(__ldcg(fp.tau + row), fp.ib, fp.flip);
    }
    const T* xr = static_cast<const T*>(fp.x) + row * fp.len;
    uint4 v[kFilterUnroll];
    if (base + kTile <= fp.len) {
#pragma unroll
      for (int u = 0; u < kFilterUnroll; ++u)
        v[u] = load_group<DT, VEC>(xr + base + (u * kFilterBlock + threadIdx.x) * VEC, pol);
#pragma unroll
      for (int u = 0; u < kFilterUnroll; ++u)
        test_group<DT, LARGEST, VEC>(v[u], base + (u * kFilterBlock + threadIdx.x) * VEC, t, fp, st, row);
    } else {  // the last, partial tile of a selection
#pragma unroll
      for (int u = 0; u < kFilterUnroll; ++u) {
        const int64_t pos = base + (u * kFilterBlock + threadIdx.x) * VEC;
        if (pos < fp.len) {
          v[u] = load_group<DT, VEC>(xr + pos, pol);
          test_group<DT, LARGEST, VEC>(v[u], pos, t, fp, st, row);
        }
      }
    }
    // a warp-uniform point: move the stage out once it is half full
    __syncwarp();
    if (__shfl_sync(kFull, *st.n, 0) >= static_cast<unsigned>(kWarpStage / 2))
      stage_flush(st, row, fp.cap, fp.buf, fp.counts);
  }
  if (cur_row >= 0) stage_flush(st, cur_row, fp.cap, fp.buf, fp.counts);
}

// ---------------------------------------------------------------------------
// Fallback
// ---------------------------------------------------------------------------

struct FallbackParams {
  FilterParams fp;
  int64_t k;
  int force;
  FallbackScratch fs;
};

// Grid-wide barrier for a cooperative launch.  Gives up after kWaitLimitNs and
// records kDevTimeout in the status word; returns false then (and when another
// block already reported an error).
__device__ bool grid_barrier(unsigned* bar, int* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned gen = ld_acquire_u32(bar + 1);
    __threadfence();
    const unsigned arrived = atomicAdd(bar, 1u) + 1u;
    if (arrived == gridDim.x) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u32(bar + 1) == gen) {
        if (*reinterpret_cast<volatile int*>(status) != kDevOk ||
            globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicCAS(status, kDevOk, kDevTimeout);
          ok = 0;
          break;
        }
        __nanosleep(128);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Block-wide exclusive scan of one unsigned per thread (blockDim.x <= 1024).
__device__ unsigned block_exclusive_scan(unsigned v, unsigned* warp_sums, unsigned* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  unsigned inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += y;
  }
  __syncthreads();
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    unsigned s = lane < nwarps ? warp_sums[lane] : 0u;
    unsigned si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(kFull, si, o);
      if (lane >= o) si += y;
    }
    if (lane < nwarps) warp_sums[lane] = si - s;
    if (lane == 31) *total = si;
  }
  __syncthreads();
  return inc - v + warp_sums[warp];
}

// The miss check and the exact fallback (section 4): every block of a
// cooperative grid runs this after the survivor counts are final.  `stage`
// and `stage_n` are the caller's per-warp survivor stages.
#ifdef TK_PHASE_TIMING
__device__ unsigned long long g_fb_ns[16];  // debug: phase stamps of the fallback's block 0
#define TK_FB(i) \
  do { if (blockIdx.x == 0 && threadIdx.x == 0) g_fb_ns[(i)] = globaltimer_ns(); } while (0)
#else
#define TK_FB(i) \
  do {           \
  } while (0)
#endif

// Visits every element of one row across the whole grid, f(raw bits): VEC
// elements per 16-byte load and four loads in flight per thread (VEC == 1:
// four scalar loads), so a full pass runs near the HBM rate.  VEC > 1
// requires len % VEC == 0 and a 16-byte aligned row (the launcher's rule).
template <int DT, int VEC, typename F>
__device__ __forceinline__ void grid_elems(const typename Dt<DT>::storage* xr, int64_t len, int64_t gtid,
                                           int64_t nthreads, uint64_t policy, F&& f) {
  constexpr int U = 4;
  const int64_t ng = len / VEC;
  int64_t g = gtid;
  for (; g + (U - 1) * nthreads < ng; g += U * nthreads) {
    uint4 w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) w[u] = load_group<DT, VEC>(xr + (g + u * nthreads) * VEC, policy);
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int e = 0; e < VEC; ++e) f(elem<DT, VEC>(w[u], e));
  }
  for (; g < ng; g += nthreads) {
    const uint4 w = load_group<DT, VEC>(xr + g * VEC, policy);
#pragma unroll
    for (int e = 0; e < VEC; ++e) f(elem<DT, VEC>(w, e));
  }
}

// Returns 1 when some selection missed (its buffer was rebuilt), 0 when none
// did, -1 when a grid barrier gave up or the state was inconsistent.
template <int DT, bool LARGEST, int VEC>
__device__ int fallback_body(const FallbackParams& a, uint64_t (*stage)[kWarpStage],
                                           unsigned* stage_n) {
  using T = typename Dt<DT>::storage;
  constexpr int kVKB = Dt<DT>::kKeyBits;
  __shared__ unsigned shist[kFilterBlock / 32][256];
  __shared__ unsigned scan_tmp[32];
  __shared__ unsigned s_total;
  __shared__ unsigned long long s_bucket_info[2];
  __shared__ int s_tile_found;
  __shared__ unsigned long long s_found_pos;

  // the re-filter compares against the exact threshold found here
  FilterParams fp = a.fp;
  fp.tau = a.fs.tau_exact;
  const FallbackScratch& fs = a.fs;
  const int warp = threadIdx.x >> 5;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint64_t policy = l2_evict_first_policy();

  int missed = 0;
  for (int64_t row = 0; row < fp.nsel; ++row) {
    const unsigned long long R = __ldcg(fp.counts + row);
    const bool miss = a.force || R < static_cast<unsigned long long>(a.k) ||
                      R > static_cast<unsigned long long>(fp.cap);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      fs.r_seen[row] = R;
      if (miss) atomicAdd(fs.misses, 1ull);
    }
    if (!miss) continue;
    missed = 1;
    const T* xr = static_cast<const T*>(fp.x) + row * fp.len;

    // -- zero the per-digit histograms
    TK_FB(0);
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) fs.ghist[i] = 0u;
    if (!grid_barrier(fs.barrier, fs.status)) return -1;
    TK_FB(1);

    // -- phase A: radix select of the k-th largest value key
    uint32_t vprefix = 0, vmask = 0;
    unsigned long long rank = static_cast<unsigned long long>(a.k);
    int pass = 0;
    for (int shift = kVKB - 8; shift >= 0; shift -= 8, ++pass) {
      for (int i = threadIdx.x; i < (kFilterBlock / 32) * 256; i += blockDim.x) (&shist[0][0])[i] = 0u;
      __syncthreads();
      grid_elems<DT, VEC>(xr, fp.len, gtid, nthreads, policy, [&](uint32_t raw) {
        const uint32_t vk = Dt<DT>::key(raw) ^ fp.flip;
        if ((vk & vmask) == vprefix) atomicAdd(&shist[warp][(vk >> shift) & 255u], 1u);
      });
      __syncthreads();
      for (int d = threadIdx.x; d < 256; d += blockDim.x) {
        unsigned s = 0;
        for (int wv = 0; wv < kFilterBlock / 32; ++wv) s += shist[wv][d];
        if (s) atomicAdd(&fs.ghist[pass * 256 + d], s);
      }
      TK_FB(2 + 2 * pass);
      if (!grid_barrier(fs.barrier, fs.status)) return -1;
      TK_FB(3 + 2 * pass);
      // every block finds the digit holding the rank-th largest (same answer
      // everywhere); thread j looks at digit 255 - j (kFilterBlock == 256)
      {
        const int d = 255 - static_cast<int>(threadIdx.x);
        const unsigned c = ld_acquire_u32(&fs.ghist[pass * 256 + d]);
        unsigned v = c;
        const int lane = threadIdx.x & 31, wv = threadIdx.x >> 5;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(kFull, v, o);
          if (lane >= o) v += y;
        }
        if (lane == 31) scan_tmp[wv] = v;
        __syncthreads();
        unsigned before = 0;
        for (int q = 0; q < wv; ++q) before += scan_tmp[q];
        const unsigned long long incl = static_cast<unsigned long long>(before) + v;
        const unsigned long long excl = incl - c;
        if (excl < rank && rank <= incl) {
          s_bucket_info[0] = static_cast<unsigned long long>(d);
          s_bucket_info[1] = excl;
        }
      }
      __syncthreads();
      vprefix |= static_cast<uint32_t>(s_bucket_info[0]) << shift;
      vmask |= 255u << shift;
      rank -= s_bucket_info[1];
      __syncthreads();
    }
    // vprefix is the k-th largest value key; `rank` is its place (1-based)
    // among the elements holding that value, in index order.

    TK_FB(10);
    // -- phase B: count the tied value per tile
    const int64_t ntile = (fp.len + kFallbackTile - 1) / kFallbackTile;
    for (int64_t tile = blockIdx.x; tile < ntile; tile += gridDim.x) {
      unsigned c = 0;
      const int64_t end = (tile + 1) * kFallbackTile < fp.len ? (tile + 1) * kFallbackTile : fp.len;
      // (a tile starts at a multiple of VEC; with VEC > 1 so does its end)
#pragma unroll 4
      for (int64_t g = tile * kFallbackTile / VEC + threadIdx.x; g < end / VEC; g += blockDim.x) {
        const uint4 w = load_group<DT, VEC>(xr + g * VEC, policy);
#pragma unroll
        for (int e = 0; e < VEC; ++e) c += ((Dt<DT>::key(elem<DT, VEC>(w, e)) ^ fp.flip) == vprefix) ? 1u : 0u;
      }
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
      if ((threadIdx.x & 31) == 0) scan_tmp[warp] = c;
      __syncthreads();
      if (threadIdx.x == 0) {
        unsigned s = 0;
        for (int q = 0; q < kFilterBlock / 32; ++q) s += scan_tmp[q];
        fs.tile_counts[tile] = s;
      }
      __syncthreads();
    }
    TK_FB(11);
    if (!grid_barrier(fs.barrier, fs.status)) return -1;
    TK_FB(12);

    if (blockIdx.x == 0) {
      // lower bound over the running count of the tied value: the first tile
      // whose inclusive count reaches `rank`.
      const int64_t per = (ntile + blockDim.x - 1) / blockDim.x;
      const int64_t lo = threadIdx.x * per, hi = lo + per < ntile ? lo + per : ntile;
      unsigned mine = 0;
      for (int64_t j = lo; j < hi; ++j) mine += ld_acquire_u32(&fs.tile_counts[j]);
      const unsigned before = block_exclusive_scan(mine, scan_tmp, &s_total);
      if (threadIdx.x == 0) s_tile_found = -1;
      __syncthreads();
      if (before < rank && rank <= static_cast<unsigned long long>(before) + mine) {
        unsigned run = before;
        for (int64_t j = lo; j < hi; ++j) {
          const unsigned c = ld_acquire_u32(&fs.tile_counts[j]);
          if (rank <= static_cast<unsigned long long>(run) + c) {
            s_found_pos = static_cast<unsigned long long>(j);
            s_bucket_info[1] = run;  // tied elements before this tile
            s_tile_found = 1;
            break;
          }
          run += c;
        }
      }
      __syncthreads();
      if (s_tile_found != 1) {
        if (threadIdx.x == 0) atomicCAS(fs.status, kDevOk, kDevBadState);
      } else {
        // ordered scan inside the tile: the (rank - before)-th tied element
        const int64_t tile = static_cast<int64_t>(s_found_pos);
        unsigned long long need = rank - s_bucket_info[1];
        const int64_t end = (tile + 1) * kFallbackTile < fp.len ? (tile + 1) * kFallbackTile : fp.len;
        for (int64_t start = tile * kFallbackTile; start < end; start += blockDim.x) {
          const int64_t i = start + threadIdx.x;
          const unsigned f = (i < end && ((Dt<DT>::key(static_cast<uint32_t>(xr[i])) ^ fp.flip) == vprefix))
                                 ? 1u : 0u;
          const unsigned ex = block_exclusive_scan(f, scan_tmp, &s_total);
          if (f && ex + 1 == need) s_found_pos = static_cast<unsigned long long>(i);
          __syncthreads();
          if (s_total >= need) break;   // block-uniform
          need -= s_total;
          __syncthreads();
        }
        if (threadIdx.x == 0) {
          fs.tau_exact[row] = compose(vprefix, s_found_pos, fp.ib);
          fp.counts[row] = 0ull;
        }
      }
    }
    TK_FB(13);
    if (!grid_barrier(fs.barrier, fs.status)) return -1;
    if (*reinterpret_cast<volatile int*>(fs.status) != kDevOk) return -1;
    TK_FB(14);

    // -- phase C: filter the selection again with the exact threshold
    constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
    const int64_t tiles_per_row = (fp.len + kTile - 1) / kTile;
    if ((threadIdx.x & 31) == 0) stage_n[threadIdx.x >> 5] = 0u;
    __syncwarp();
    const Stage st{stage[threadIdx.x >> 5], &stage_n[threadIdx.x >> 5]};
    filter_tiles<DT, LARGEST, VEC>(fp, row * tiles_per_row + blockIdx.x, (row + 1) * tiles_per_row,
                                   gridDim.x, st);
    TK_FB(15);
  }
  return missed;
}

template <int DT, bool LARGEST, int VEC>
__global__ void __launch_bounds__(kFilterBlock) fallback_kernel(FallbackParams a) {
  __shared__ uint64_t stage[kFilterBlock / 32][kWarpStage];
  __shared__ unsigned stage_n[kFilterBlock / 32];
  TK_TL_BEGIN(5);
  grid_dependency_wait();    // the survivor counts come from the filter
  grid_launch_dependents();  // the final selection may start launching
  fallback_body<DT, LARGEST, VEC>(a, stage, stage_n);
  TK_TL_END(5);
}

template <int DT, bool LARGEST, int VEC>
__global__ void __launch_bounds__(kFilterBlock) filter_kernel(FilterParams fp) {
  __shared__ uint64_t stage[kFilterBlock / 32][kWarpStage];
  __shared__ unsigned stage_n[kFilterBlock / 32];
  TK_TL_BEGIN(2);
  grid_dependency_wait();  // tau and the zeroed counters come from the previous grid
  if ((threadIdx.x & 31) == 0) stage_n[threadIdx.x >> 5] = 0u;
  __syncwarp();
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  const int64_t ntiles = fp.nsel * ((fp.len + kTile - 1) / kTile);
  const Stage st{stage[threadIdx.x >> 5], &stage_n[threadIdx.x >> 5]};
  filter_tiles<DT, LARGEST, VEC>(fp, blockIdx.x, ntiles, gridDim.x, st);
  TK_TL_END(2);
}

// One full wave: SMs x resident blocks per SM, less the SMs held by the
// preceding grid when this launch may overlap it (programmatic dependent
// launch): the tiles are dealt out by block index, so every block must start
// at once.
template <int DT, bool LARGEST, int VEC>
int filter_grid_size(int reserved_sms) {
  static int sms = 0, per_sm = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, filter_kernel<DT, LARGEST, VEC>, kFilterBlock, 0);
    if (per_sm < 1) per_sm = 1;
  }
  const int usable = sms - reserved_sms > sms / 2 ? sms - reserved_sms : sms / 2;
  return usable * per_sm;
}

template <int DT, bool LARGEST, int VEC>
cudaError_t launch_filter_t(const FilterParams& fp, int reserved_sms, cudaStream_t st) {
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  const int64_t ntiles = fp.nsel * ((fp.len + kTile - 1) / kTile);
  FilterParams args = fp;
  args.tiles_per_row = make_divider(static_cast<uint64_t>((fp.len + kTile - 1) / kTile));
  const bool pdl = reserved_sms >= 0 && pdl_edge(kPdlFilter);
  int64_t grid = filter_grid_size<DT, LARGEST, VEC>(pdl ? reserved_sms : 0);
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kFilterBlock, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, filter_kernel<DT, LARGEST, VEC>, args);
}

template <int DT, bool LARGEST, int VEC>
cudaError_t launch_fallback_t(const FallbackParams& a, cudaStream_t st) {
  static unsigned grid = 0;  // co-resident blocks: one full wave of the device
  if (!grid) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, fallback_kernel<DT, LARGEST, VEC>, kFilterBlock, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (per_sm > 2) per_sm = 2;  // enough for the rare full passes, cheap when nothing missed
    grid = static_cast<unsigned>(sms * per_sm);
  }
  FallbackParams args = a;
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  args.fp.tiles_per_row = make_divider(static_cast<uint64_t>((a.fp.len + kTile - 1) / kTile));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kFilterBlock, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every block resident
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_edge(kPdlFallback) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fallback_kernel<DT, LARGEST, VEC>, args);
}

// ---------------------------------------------------------------------------
// Grid refinement (large k)
// ---------------------------------------------------------------------------
// Stage 4 for a few selections with many winners, on every SM at once: the
// miss check and fallback above, then the candidates of each selection are
// partitioned into 2048 equal slices of their key range ("count into
// buckets", Find the Cutoff Instead): the first 11-bit digit of key - kmin.
// Each block caches its slice of the buffer, the slices' minima and maxima
// give the range, one histogram per block is added into a grid-wide one (the
// returned old count is the block's offset inside each bin), and after a
// grid barrier
// every block scans the same totals and knows every bin's first place.  When
// the bin holding rank k fits the exchange buffer after the bins above it,
// every key of those bins is placed and the bin sort keeps the first k
// places; otherwise further digits inside that bin, one grid-wide histogram
// each, find the exact k-th key and only the winners are placed.  Keys are
// staged by bin in shared memory first, so a warp writes consecutive places.
constexpr unsigned kPartDM = kRefineGridBins - 1;
constexpr int kPartDigit = 11;
constexpr int kPartCache = (kFilterBlock / 32) * kWarpStage;  // keys a block holds: the fallback's stages
constexpr int kPartPer = kRefineGridBins / kFilterBlock;      // bins per thread in the scans
constexpr size_t kPartDynBytes = sizeof(unsigned) * 3 * kRefineGridBins + sizeof(uint64_t) * kPartCache;
static_assert(kRefineGridBins == (1 << kPartDigit) && kRefineGridBins % kFilterBlock == 0, "bins");

#ifdef TK_PHASE_TIMING
__device__ unsigned long long g_rg_ns[16];  // debug: phase stamps of block 0
#define TK_RG(i) \
  do { if (blockIdx.x == 0 && threadIdx.x == 0) g_rg_ns[(i)] = globaltimer_ns(); } while (0)
#else
#define TK_RG(i) \
  do {           \
  } while (0)
#endif

struct RefineGridParams {
  FallbackParams fb;  // fb.fp: the candidate buffer (buf, cap, counts)
  RefineGridScratch rg;
};

// Every block scans the kRefineGridBins counters g[] (bins in descending key
// order) and finds the bin holding rank `rank` (1-based): *bin, the keys
// before it and its count; `starts` (nullable) receives every bin's first place.
// Returns false when the counts do not reach `rank`.
__device__ bool find_rank_bin(const unsigned* g, unsigned long long rank, unsigned* starts, unsigned* warp_sums,
                              unsigned* info) {
  __shared__ unsigned s_total;
  unsigned c[kPartPer], sum = 0;
#pragma unroll
  for (int q = 0; q < kPartPer; ++q) {
    c[q] = __ldcg(g + threadIdx.x * kPartPer + q);
    sum += c[q];
  }
  if (threadIdx.x == 0) info[0] = ~0u;
  unsigned run = block_exclusive_scan(sum, warp_sums, &s_total);
#pragma unroll
  for (int q = 0; q < kPartPer; ++q) {
    const unsigned b = threadIdx.x * kPartPer + q;
    if (starts) starts[b] = run;
    if (run < rank && rank <= static_cast<unsigned long long>(run) + c[q]) {
      info[0] = b;
      info[1] = run;
      info[2] = c[q];
    }
    run += c[q];
  }
  __syncthreads();
  return info[0] != ~0u;
}

__device__ bool partition_row(const RefineGridParams& a, int64_t row, uint64_t* cache, unsigned char* dsm) {
  const FilterParams& fp = a.fb.fp;
  const FallbackScratch& fs = a.fb.fs;
  const RefineGridScratch& rg = a.rg;
  const unsigned long long k = static_cast<unsigned long long>(a.fb.k);
  unsigned* mine = reinterpret_cast<unsigned*>(dsm);  // this block's count, then its place offset, per bin
  unsigned* bst = mine + kRefineGridBins;             // first place of each bin
  unsigned* cur = bst + kRefineGridBins;              // this block's offset inside each bin; staging cursors
  uint64_t* stg = reinterpret_cast<uint64_t*>(cur + kRefineGridBins);  // keys staged by bin
  __shared__ unsigned s_ws[32];
  __shared__ unsigned s_info[4];
  __shared__ unsigned s_total;
  __shared__ unsigned long long s_nmin, s_max;
  __shared__ unsigned s_w;
  unsigned* ctl = rg.ctl + row * kRefineGridCtlWords;
  unsigned long long* g_nmin = reinterpret_cast<unsigned long long*>(ctl);  // NOT of the smallest key
  unsigned long long* g_max = g_nmin + 1;
  unsigned* g_win = ctl + 4;
  unsigned* g_lev = ctl + 8;
  const int tid = threadIdx.x;

  // ---- the block's slice, cached; the smallest and largest key over the grid
  const unsigned long long R = __ldcg(fp.counts + row);
  const int64_t n = R < static_cast<unsigned long long>(fp.cap) ? static_cast<int64_t>(R) : fp.cap;
  const int64_t sb = n * blockIdx.x / gridDim.x, se = n * (blockIdx.x + 1) / gridDim.x;
  const int cn = static_cast<int>(se - sb);  // <= kPartCache: the host checks n <= gridDim.x * kPartCache
  const uint64_t* src = fp.buf + row * fp.cap + sb;
  unsigned long long mn = ~0ull, mx = 0ull;
  for (int i = tid; i < cn; i += kFilterBlock) {
    const uint64_t key = __ldcg(src + i);
    cache[i] = key;
    mn = key < mn ? key : mn;
    mx = key > mx ? key : mx;
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    const unsigned long long a = __shfl_xor_sync(kFull, mn, m), b = __shfl_xor_sync(kFull, mx, m);
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  if (tid == 0) { s_nmin = 0ull; s_max = 0ull; }
  __syncthreads();
  if ((tid & 31) == 0) { atomicMax(&s_nmin, ~mn); atomicMax(&s_max, mx); }
  __syncthreads();
  if (tid == 0 && cn > 0) { atomicMax(g_nmin, s_nmin); atomicMax(g_max, s_max); }
  TK_RG(3);
  if (!grid_barrier(fs.barrier, fs.status)) return false;
  TK_RG(4);
  // Digits are taken of key - kmin: 2048 equal slices of the keys' range.
  // (Digits of the keys themselves below their top varying bit leave only a
  // few non-empty bins when the candidates' values cross a power of two.)
  // The cache holds key - kmin from here on; the order is the same.
  const uint64_t kmin = ~__ldcg(g_nmin), kmax = __ldcg(g_max);
  const uint64_t span = kmax - kmin;
  const int hb = span ? 63 - __clzll(static_cast<long long>(span)) : 0;
  const uint64_t pmask1 = hb >= 63 ? 0ull : (~0ull << (hb + 1));
  const uint64_t prefix1 = 0ull;
  const int shift1 = hb >= kPartDigit - 1 ? hb - (kPartDigit - 1) : 0;
  for (int i = tid; i < cn; i += kFilterBlock) cache[i] -= kmin;
  __syncthreads();
  auto bin_of = [&](uint64_t key) { return kPartDM - static_cast<unsigned>((key >> shift1) & kPartDM); };

  // ---- first digit: this block's histogram, its range inside each bin
  for (int i = tid; i < kRefineGridBins; i += kFilterBlock) mine[i] = 0u;
  __syncthreads();
  for (int i = tid; i < cn; i += kFilterBlock) atomicAdd(&mine[bin_of(cache[i])], 1u);
  __syncthreads();
  for (int i = tid; i < kRefineGridBins; i += kFilterBlock) {
    const unsigned c = mine[i];
    cur[i] = c ? atomicAdd(g_lev + i, c) : 0u;
  }
  TK_RG(5);
  if (!grid_barrier(fs.barrier, fs.status)) return false;
  TK_RG(6);
  if (!find_rank_bin(g_lev, k, bst, s_ws, s_info)) {
    if (tid == 0) atomicCAS(fs.status, kDevOk, kDevBadState);
    return false;
  }
  TK_RG(7);
  const unsigned bb = s_info[0], bb_start = s_info[1], bb_tot = s_info[2];
  const bool whole = static_cast<int64_t>(bb_start) + bb_tot <= rg.xstride;
  uint64_t kappa = 0ull;
  if (!whole) {
    // ---- the exact k-th key: further digits inside the boundary bin
    uint64_t prefix = prefix1 | (static_cast<uint64_t>(kPartDM - bb) << shift1);
    uint64_t pmask = pmask1 | (static_cast<uint64_t>(kPartDM) << shift1);
    unsigned long long rank = k - bb_start;
    int shift = shift1;
    unsigned* lh = reinterpret_cast<unsigned*>(stg);
    for (int level = 1; shift > 0; ++level) {
      if (level >= kRefineGridLevels) {
        if (tid == 0) atomicCAS(fs.status, kDevOk, kDevBadState);
        return false;
      }
      shift = shift >= kPartDigit ? shift - kPartDigit : 0;
      for (int i = tid; i < kRefineGridBins; i += kFilterBlock) lh[i] = 0u;
      __syncthreads();
      for (int i = tid; i < cn; i += kFilterBlock) {
        const uint64_t key = cache[i];
        if ((key & pmask) == prefix) atomicAdd(&lh[kPartDM - static_cast<unsigned>((key >> shift) & kPartDM)], 1u);
      }
      __syncthreads();
      unsigned* gl = g_lev + level * kRefineGridBins;
      for (int i = tid; i < kRefineGridBins; i += kFilterBlock)
        if (lh[i]) atomicAdd(gl + i, lh[i]);
      if (!grid_barrier(fs.barrier, fs.status)) return false;
      if (!find_rank_bin(gl, rank, nullptr, s_ws, s_info)) {
        if (tid == 0) atomicCAS(fs.status, kDevOk, kDevBadState);
        return false;
      }
      prefix |= static_cast<uint64_t>(kPartDM - s_info[0]) << shift;
      pmask |= static_cast<uint64_t>(kPartDM) << shift;
      rank -= s_info[1];
      __syncthreads();  // s_info is rewritten by the next level
    }
    kappa = prefix;  // every bit fixed: the k-th largest key (less kmin)
    // this block's winners inside the boundary bin, and where they start
    unsigned w = 0;
    for (int i = tid; i < cn; i += kFilterBlock) {
      const uint64_t key = cache[i];
      w += (bin_of(key) == bb && key >= kappa) ? 1u : 0u;
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) w += __shfl_xor_sync(kFull, w, m);
    if (tid == 0) s_w = 0u;
    __syncthreads();
    if ((tid & 31) == 0 && w) atomicAdd(&s_w, w);
    __syncthreads();
    if (tid == 0) {
      cur[bb] = s_w ? atomicAdd(g_win, s_w) : 0u;
      mine[bb] = s_w;
    }
    __syncthreads();
  }

  TK_RG(8);
  // ---- placement: stage this block's winners by bin, then write them out
  {
    unsigned m[kPartPer], sum = 0;
#pragma unroll
    for (int q = 0; q < kPartPer; ++q) {
      const unsigned b = tid * kPartPer + q;
      m[q] = b <= bb ? mine[b] : 0u;
      sum += m[q];
    }
    unsigned run = block_exclusive_scan(sum, s_ws, &s_total);
#pragma unroll
    for (int q = 0; q < kPartPer; ++q) {
      const unsigned b = tid * kPartPer + q;
      // staged index i of bin b goes to place bst[b] + cur[b] + (i - run)
      // (unsigned arithmetic wraps)
      mine[b] = bst[b] + cur[b] - run;
      cur[b] = run;
      run += m[q];
    }
    __syncthreads();
  }
  for (int i = tid; i < cn; i += kFilterBlock) {
    const uint64_t key = cache[i];
    const unsigned b = bin_of(key);
    if (b < bb || (b == bb && (whole || key >= kappa))) stg[atomicAdd(&cur[b], 1u)] = key;
  }
  __syncthreads();
  const unsigned nst = s_total;
  const unsigned xend = whole ? bb_start + bb_tot : static_cast<unsigned>(k);
  uint64_t* xb = rg.xbuf + row * rg.xstride;
  for (unsigned i = tid; i < nst; i += kFilterBlock) {
    const uint64_t key = stg[i];
    const unsigned pos = mine[bin_of(key)] + i;
    if (pos < xend) xb[pos] = key + kmin;
  }
  if (blockIdx.x == 0) {
    // the bin sort's view of the partition
    unsigned* bo = rg.binfo + row * (kRefineGridBins + 8);
    for (int i = tid; i < kRefineGridBins; i += kFilterBlock) bo[i] = bst[i];
    if (tid == 0) {
      bo[kRefineGridBins] = static_cast<unsigned>(prefix1);
      bo[kRefineGridBins + 1] = static_cast<unsigned>(prefix1 >> 32);
      bo[kRefineGridBins + 2] = static_cast<unsigned>(pmask1);
      bo[kRefineGridBins + 3] = static_cast<unsigned>(pmask1 >> 32);
      bo[kRefineGridBins + 4] = static_cast<unsigned>(shift1);
      bo[kRefineGridBins + 5] = xend;
      bo[kRefineGridBins + 6] = static_cast<unsigned>(kmin);  // digits are of key - kmin
      bo[kRefineGridBins + 7] = static_cast<unsigned>(kmin >> 32);
    }
  }
  __syncthreads();  // the shared arrays are reused by the next selection
  TK_RG(9);
  return true;
}

template <int DT, bool LARGEST, int VEC>
__global__ void __launch_bounds__(kFilterBlock, 2) refine_grid_kernel(RefineGridParams a) {
  __shared__ uint64_t stage[kFilterBlock / 32][kWarpStage];
  __shared__ unsigned stage_n[kFilterBlock / 32];
  extern __shared__ __align__(16) unsigned char part_smem[];
  TK_TL_BEGIN(3);
  TK_RG(0);
  grid_dependency_wait();    // the buffer and its counts come from the filter
  grid_launch_dependents();  // the bin sort may start launching
  const RefineGridScratch& rg = a.rg;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // The next call's control words, first of all (a call that gives up leaves
  // only its own copy unclean, and the next call clears that one); the whole
  // copy, since the next call may refine more selections than this one.
  for (int64_t i = gtid; i < kRefineGridMaxSel * kRefineGridCtlWords; i += nthreads) rg.ctl_next[i] = 0u;
  if (rg.clear_words && blockIdx.x == 0)
    for (int i = threadIdx.x; i < rg.n_clear; i += blockDim.x) rg.clear_words[i] = 0u;
  TK_RG(1);
  const int missed = fallback_body<DT, LARGEST, VEC>(a.fb, stage, stage_n);
  TK_RG(2);
  if (missed < 0) return;
  // a rebuilt buffer is complete once every block has filtered its tiles
  if (missed > 0 && !grid_barrier(a.fb.fs.barrier, a.fb.fs.status)) return;
  uint64_t* cache = &stage[0][0];
  for (int64_t row = 0; row < a.fb.fp.nsel; ++row)
    if (!partition_row(a, row, cache, part_smem)) return;
  TK_TL_END(3);
}

template <int DT, bool LARGEST, int VEC>
unsigned refine_grid_blocks() {
  static unsigned grid = 0;  // co-resident blocks: one full wave, two blocks per SM at most
  if (!grid) {
    int dev = 0, sms = 0, per_sm = 0;
    // (static and dynamic shared memory together exceed the default 48 KB)
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(refine_grid_kernel<DT, LARGEST, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPartDynBytes)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, refine_grid_kernel<DT, LARGEST, VEC>, kFilterBlock,
                                                      kPartDynBytes) != cudaSuccess)
      return 0;
    if (per_sm > 2) per_sm = 2;
    grid = per_sm > 0 ? static_cast<unsigned>(sms * per_sm) : 0u;
  }
  return grid;
}

template <int DT, bool LARGEST, int VEC>
cudaError_t launch_refine_grid_t(const RefineGridParams& a, cudaStream_t st) {
  const unsigned grid = refine_grid_blocks<DT, LARGEST, VEC>();
  if (!grid) return cudaErrorInvalidConfiguration;
  RefineGridParams args = a;
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  args.fb.fp.tiles_per_row = make_divider(static_cast<uint64_t>((a.fb.fp.len + kTile - 1) / kTile));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kFilterBlock, 1, 1);
  cfg.dynamicSmemBytes = kPartDynBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every block resident
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_edge(kPdlFallback) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, refine_grid_kernel<DT, LARGEST, VEC>, args);
}

template <int DT, bool LARGEST, int VEC>
int64_t refine_grid_capacity_t() {
  return static_cast<int64_t>(refine_grid_blocks<DT, LARGEST, VEC>()) * kPartCache;
}

}  // namespace

cudaError_t launch_filter(const Problem& p, const uint64_t* tau, int64_t cap, uint64_t* buf,
                          unsigned long long* counts, int reserved_sms, cudaStream_t st) {
  const FilterParams fp{p.x, p.nsel, p.len, p.ib, p.flip, tau, cap, buf, counts, Divider{}};
  const bool largest = p.flip == 0;
  if (p.dtype == kF32) {
    if (p.vec_ok) return largest ? launch_filter_t<kF32, true, 4>(fp, reserved_sms, st)
                                 : launch_filter_t<kF32, false, 4>(fp, reserved_sms, st);
    return largest ? launch_filter_t<kF32, true, 1>(fp, reserved_sms, st)
                   : launch_filter_t<kF32, false, 1>(fp, reserved_sms, st);
  }
  if (p.vec_ok) return largest ? launch_filter_t<kBF16, true, 8>(fp, reserved_sms, st)
                               : launch_filter_t<kBF16, false, 8>(fp, reserved_sms, st);
  return largest ? launch_filter_t<kBF16, true, 1>(fp, reserved_sms, st)
                 : launch_filter_t<kBF16, false, 1>(fp, reserved_sms, st);
}

cudaError_t launch_fallback(const Problem& p, int64_t k, int64_t cap, uint64_t* buf,
                            unsigned long long* counts, const FallbackScratch& fs, int force,
                            cudaStream_t st) {
  // the re-filter reads the exact threshold the fallback itself writes
  FallbackParams a{{p.x, p.nsel, p.len, p.ib, p.flip, fs.tau_exact, cap, buf, counts, Divider{}}, k, force, fs};
  const bool largest = p.flip == 0;
  if (p.dtype == kF32) {
    if (p.vec_ok) return largest ? launch_fallback_t<kF32, true, 4>(a, st) : launch_fallback_t<kF32, false, 4>(a, st);
    return largest ? launch_fallback_t<kF32, true, 1>(a, st) : launch_fallback_t<kF32, false, 1>(a, st);
  }
  if (p.vec_ok) return largest ? launch_fallback_t<kBF16, true, 8>(a, st) : launch_fallback_t<kBF16, false, 8>(a, st);
  return largest ? launch_fallback_t<kBF16, true, 1>(a, st) : launch_fallback_t<kBF16, false, 1>(a, st);
}

int64_t refine_grid_capacity(const Problem& p) {
  if (p.nsel > kRefineGridMaxSel) return 0;
  const bool largest = p.flip == 0;
  if (p.dtype == kF32) {
    if (p.vec_ok) return largest ? refine_grid_capacity_t<kF32, true, 4>() : refine_grid_capacity_t<kF32, false, 4>();
    return largest ? refine_grid_capacity_t<kF32, true, 1>() : refine_grid_capacity_t<kF32, false, 1>();
  }
  if (p.vec_ok) return largest ? refine_grid_capacity_t<kBF16, true, 8>() : refine_grid_capacity_t<kBF16, false, 8>();
  return largest ? refine_grid_capacity_t<kBF16, true, 1>() : refine_grid_capacity_t<kBF16, false, 1>();
}

cudaError_t launch_refine_grid(const Problem& p, int64_t k, int64_t cap, uint64_t* buf,
                               unsigned long long* counts, const FallbackScratch& fs, int force,
                               const RefineGridScratch& rg, cudaStream_t st) {
  if (p.nsel > kRefineGridMaxSel || cap > refine_grid_capacity(p) || rg.xstride < 2 * k)
    return cudaErrorInvalidValue;
  const RefineGridParams a{{{p.x, p.nsel, p.len, p.ib, p.flip, fs.tau_exact, cap, buf, counts, Divider{}}, k, force, fs},
                           rg};
  const bool largest = p.flip == 0;
  if (p.dtype == kF32) {
    if (p.vec_ok) return largest ? launch_refine_grid_t<kF32, true, 4>(a, st) : launch_refine_grid_t<kF32, false, 4>(a, st);
    return largest ? launch_refine_grid_t<kF32, true, 1>(a, st) : launch_refine_grid_t<kF32, false, 1>(a, st);
  }
  if (p.vec_ok) return largest ? launch_refine_grid_t<kBF16, true, 8>(a, st) : launch_refine_grid_t<kBF16, false, 8>(a, st);
  return largest ? launch_refine_grid_t<kBF16, true, 1>(a, st) : launch_refine_grid_t<kBF16, false, 1>(a, st);
}

#ifdef TK_PHASE_TIMING
TK_TIMELINE_ACCESSOR(debug_timeline_filter)
int debug_refine_grid_ns(unsigned long long* out) {
  if (cudaMemcpyFromSymbol(out, g_rg_ns, sizeof(g_rg_ns)) != cudaSuccess) return -3;
  return cudaMemcpyFromSymbol(out + 16, g_fb_ns, sizeof(g_fb_ns)) == cudaSuccess ? 0 : -3;
}
#endif

}  // namespace tk
