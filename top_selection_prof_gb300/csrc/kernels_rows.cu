// Direct path for many short rows: one 1024-thread CTA per selection holds the
// whole row in registers (up to 32 elements per thread, so rows of at most
// 32768 elements) and returns its exact top-k (k <= 1024), sorted.
//
// Common case ("Prof-K" applied inside one CTA, with the per-thread maxima as
// the sample): the k-th largest of the 1024 per-thread maxima, L, is found by
// a radix select over one value per thread.  At least k elements are >= L (k
// threads have a maximum >= L), and every element >= L belongs to one of the
// threads whose maximum is >= L, so there are at most 32 per such thread.
// When those candidates fit in shared memory they are gathered as composite
// keys (value key, complemented position) and each one's place is its rank by
// counting among them ("Rank by Counting"); places below k are the output.
// Otherwise (many equal values) the exact k-th largest value is found by a
// radix select over every element, ties at that value are taken in position
// order with block-wide scans, and the k winners are ranked the same way.
//
// The row is read once from HBM; a persistent grid of one block per SM walks
// the rows, and one thread has the TMA engine copy the next row into shared
// memory (cp.async.bulk completing on an mbarrier) while the current one is
// selected from registers.
#include <cooperative_groups.h>

#include "common.cuh"
#include "engine.h"

namespace tk {

namespace {

constexpr int kRowBlock = 1024;
constexpr int kRowElems = 32;                      // elements per thread
constexpr int64_t kRowMaxLen = int64_t(kRowBlock) * kRowElems;
constexpr int64_t kRowMaxK = 1024;
constexpr int kRowCap = 2048;                      // candidates ranked by counting
constexpr int kBins = 2048;                        // 11-bit digits
constexpr unsigned kFull = 0xffffffffu;

#ifdef TK_PHASE_TIMING
// Debug builds only: globaltimer stamps of block 0's second row.
__device__ unsigned long long g_rows_ns[16];
#define TR_STAMP(i)                                                                               \
  do {                                                                                            \
    if (blockIdx.x == 0 && threadIdx.x == 0 && row == gridDim.x) g_rows_ns[(i)] = globaltimer_ns(); \
  } while (0)
#define TR_VALUE(i, v)                                                                  \
  do {                                                                                  \
    if (blockIdx.x == 0 && threadIdx.x == 0 && row == gridDim.x) g_rows_ns[(i)] = (v); \
  } while (0)
#else
#define TR_STAMP(i) \
  do {              \
  } while (0)
#define TR_VALUE(i, v) \
  do {                 \
  } while (0)
#endif

struct RowsParams {
  const void* x;
  int64_t nsel, len;
  uint32_t flip;
  int vec;        // 16-byte loads are legal
  int64_t k;
  void* out_vals;
  int64_t* out_idx;
  int* status;
};

// Block-wide inclusive scan of one unsigned per thread; `tmp` has 32 words.
__device__ __forceinline__ unsigned scan_incl(unsigned v, unsigned* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const unsigned s = tmp[lane];
    unsigned si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(kFull, si, o);
      if (lane >= o) si += y;
    }
    tmp[lane] = si - s;
  }
  __syncthreads();
  return v + tmp[warp];  // (callers pass another barrier before tmp is written again)
}

// Number of keys in src[j0, j1) greater than v: rounds of eight independent,
// predicated loads (a slot past j1 reads as key 0, which is never greater).
__device__ __forceinline__ unsigned count_greater(const uint64_t* src, unsigned j0, unsigned j1, uint64_t v) {
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

// One radix-select pass over 32-bit keys, `n` per thread, key(i) giving the
// i-th (a flag bit of `valid` marks it present): digits of 11, 11 and 10 bits
// for passes 0, 1, 2.  Narrows prefix / pmask to the bin holding the rank-th
// largest (1-based, with multiplicity) and makes rank relative to that bin;
// *gt grows by the keys in bins above.  `hist` is all zero on entry and is
// left so.  All threads call it and get the same result.
template <int N, typename KeyAt>
__device__ void kth_pass(KeyAt key, uint32_t valid, int pass, uint32_t* prefix, uint32_t* pmask,
                         unsigned* rank, unsigned* gt, unsigned* hist, unsigned* tmp, unsigned* info) {
  const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
  const uint32_t dmask = pass == 2 ? 1023u : 2047u;
#pragma unroll
  for (int e = 0; e < N; ++e) {
    if ((valid >> e) & 1u) {
      const uint32_t k = key(e);
      if ((k & *pmask) == *prefix) atomicAdd(&hist[2047u - ((k >> shift) & dmask)], 1u);
    }
  }
  __syncthreads();
  // two bins per thread, descending key order; each thread clears its bins
  const unsigned c0 = hist[2 * threadIdx.x], c1 = hist[2 * threadIdx.x + 1];
  hist[2 * threadIdx.x] = 0u;
  hist[2 * threadIdx.x + 1] = 0u;
  const unsigned incl = scan_incl(c0 + c1, tmp);
  const unsigned ex = incl - c0 - c1;
  if (ex < *rank && *rank <= ex + c0) { info[0] = 2 * threadIdx.x; info[1] = ex; }
  else if (ex + c0 < *rank && *rank <= incl) { info[0] = 2 * threadIdx.x + 1; info[1] = ex + c0; }
  __syncthreads();
  *prefix |= (2047u - info[0]) << shift;
  *pmask |= dmask << shift;
  *rank -= info[1];
  *gt += info[1];
  __syncthreads();  // info is rewritten by the next pass
}

template <int DT>
__device__ __forceinline__ uint32_t raw_at(const void* x, int64_t i) {
  if (DT == kF32) return __ldg(static_cast<const uint32_t*>(x) + i);
  return __ldg(static_cast<const uint16_t*>(x) + i);
}

// The value is rebuilt from its key; only a zero or NaN key (whose key does
// not fix the sign or payload) reads the input again.
template <int DT>
__device__ __forceinline__ void write_winner(const RowsParams& a, int64_t row, int64_t place, uint64_t ck) {
  const uint32_t pos = 0xffffffffu - static_cast<uint32_t>(ck);
  const int64_t oi = row * a.k + place;
  a.out_idx[oi] = static_cast<int64_t>(pos);
  const uint32_t vk = static_cast<uint32_t>(ck >> 32) ^ a.flip;
  const uint32_t raw = (vk == Dt<DT>::kZeroKey || vk == Dt<DT>::kNanKey) ? raw_at<DT>(a.x, row * a.len + pos)
                                                                       : Dt<DT>::bits(vk);
  if (DT == kF32) static_cast<uint32_t*>(a.out_vals)[oi] = raw;
  else static_cast<uint16_t*>(a.out_vals)[oi] = static_cast<uint16_t>(raw);
}

template <int DT, bool LARGEST>
__global__ void __launch_bounds__(kRowBlock, 1) rows_kernel(RowsParams a) {
  using T = typename Dt<DT>::storage;
  constexpr int VEC = Dt<DT>::kVec;           // elements per 16-byte load
  constexpr int J = kRowElems / VEC;          // loads per thread
  constexpr int W = kRowElems * sizeof(T) / 4;  // 32-bit words of raw elements per thread
  __shared__ unsigned hist[kBins];
  __shared__ uint64_t cand[kRowCap];
  __shared__ unsigned tmp[32];
  __shared__ unsigned info[2];
  __shared__ unsigned s_cnt;
  __shared__ __align__(8) uint64_t row_bar;
  __shared__ int s_arrived;
  // the next row, fetched by the TMA engine while this one is worked on
  // (16-byte aligned rows only; others are read straight from global memory)
  extern __shared__ __align__(16) unsigned char next_row[];
  const int tid = threadIdx.x;
  const bool prefetch = a.vec != 0;
  const unsigned row_bytes = static_cast<unsigned>(a.len * sizeof(T));
  grid_dependency_wait();

  // one thread issues the whole row as bulk copies of at most 32 KB
  auto fetch = [&](int64_t r) {
    const unsigned char* src = static_cast<const unsigned char*>(a.x) + r * static_cast<int64_t>(row_bytes);
    mbar_expect_tx(&row_bar, row_bytes);
    for (unsigned off = 0; off < row_bytes; off += 32768u) {
      const unsigned n = row_bytes - off < 32768u ? row_bytes - off : 32768u;
      bulk_copy_g2s(next_row + off, src + off, n, &row_bar);
    }
  };
  for (int i = tid; i < kBins; i += kRowBlock) hist[i] = 0u;
  if (prefetch && tid == 0) {
    mbar_init(&row_bar, 1);
    if (static_cast<int64_t>(blockIdx.x) < a.nsel) fetch(blockIdx.x);
  }
  __syncthreads();
  unsigned parity = 0;

  for (int64_t row = blockIdx.x; row < a.nsel; row += gridDim.x) {
    // ---------------------------------------------------------------- load
    // element e of load j of thread t sits at position (j * 1024 + t) * VEC + e;
    // the raw elements stay packed in 32-bit words
    uint32_t w[W];
    uint32_t valid = 0;
    const int64_t base = row * a.len;
    TR_STAMP(0);
    if (prefetch) {
      // thread 0 waits (bounded) and tells the others
      if (tid == 0) s_arrived = mbar_wait(&row_bar, parity) ? 1 : 0;
      __syncthreads();
      if (!s_arrived) {
        // the copy did not land in time: report it, give it a last bounded
        // wait (it writes this block's shared memory) and stop
        if (tid == 0) {
          if (a.status) atomicCAS(a.status, kDevOk, kDevTimeout);
          mbar_wait(&row_bar, parity);
        }
        return;
      }
      parity ^= 1u;
    }
    TR_STAMP(1);
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int64_t p0 = (static_cast<int64_t>(j) * kRowBlock + tid) * VEC;
      if (a.vec && p0 + VEC <= a.len) {
        const uint4 q = prefetch ? *reinterpret_cast<const uint4*>(next_row + (p0 / VEC) * 16)
                                 : ld_stream_v4(static_cast<const T*>(a.x) + base + p0);
        w[4 * j] = q.x;
        w[4 * j + 1] = q.y;
        w[4 * j + 2] = q.z;
        w[4 * j + 3] = q.w;
        valid |= ((1u << VEC) - 1u) << (j * VEC);
      } else {
        uint32_t r[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const bool in = p0 + e < a.len;
          r[e] = in ? raw_at<DT>(a.x, base + p0 + e) : 0u;
          valid |= (in ? 1u : 0u) << (j * VEC + e);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[4 * j + q] = DT == kF32 ? r[q] : (r[2 * q] | (r[2 * q + 1] << 16));
      }
    }
    TR_STAMP(11);
    if (prefetch) {
      __syncthreads();  // every thread has its part of this row in registers
      TR_STAMP(12);
      if (tid == 0 && row + gridDim.x < a.nsel) {
        // the buffer was read through the generic proxy; order that before
        // the bulk copy overwrites it
        fence_proxy_async_smem();
        fetch(row + gridDim.x);
      }
    }
    TR_STAMP(2);
    auto raw = [&](int i) -> uint32_t {
      return DT == kF32 ? w[i] : ((w[i >> 1] >> ((i & 1) * 16)) & 0xffffu);
    };
    auto fval = [&](int i) -> float { return Dt<DT>::to_float(raw(i)); };
    auto key = [&](int i) -> uint32_t { return Dt<DT>::key(raw(i)) ^ a.flip; };
    auto pos_of = [&](int i) -> uint32_t {
      return static_cast<uint32_t>((static_cast<int64_t>(i / VEC) * kRowBlock + tid) * VEC + (i % VEC));
    };

    // ---------------------------------------------------------------- bound
    // L = a lower bound (in selection order) of the k-th best per-thread best
    // element: at least k elements rank at or above it.  The select over the
    // per-thread bests stops at the first digit whose bin's lower edge leaves
    // few enough candidates.  Elements are compared as floats against L's
    // value (NaN ranks first when largest, last when smallest; -0 == +0).
    float best = LARGEST ? -__int_as_float(0x7f800000) : __int_as_float(0x7f800000);
#pragma unroll
    for (int i = 0; i < kRowElems; ++i)
      if ((valid >> i) & 1u) {
        const float f = fval(i);
        if (LARGEST) asm("max.NaN.f32 %0, %0, %1;" : "+f"(best) : "f"(f));
        else best = fminf(best, f);
      }
    const uint32_t bkey = (Dt<DT>::key(DT == kF32 ? __float_as_uint(best) : (__float_as_uint(best) >> 16))) ^ a.flip;
    // (with fewer than k threads holding elements every element is a candidate)
    const int holders = __syncthreads_count(valid != 0u);
    TR_STAMP(3);
    uint32_t lp = 0, lm = 0;
    unsigned lrank = static_cast<unsigned>(a.k), lgt = 0;
    float fL = __int_as_float(0x7fffffff);  // NaN: every element passes
    unsigned C = 0;
    const int first = (a.len <= kRowCap || holders < a.k) ? 0 : 1;
#pragma unroll 1
    for (int pass = first; pass < 4; ++pass) {
      if (pass > 0) {
        if (holders < a.k) break;
        kth_pass<1>([&](int) { return bkey; }, valid ? 1u : 0u, pass - 1, &lp, &lm, &lrank, &lgt, hist, tmp,
                    info);
        // the bin's lower edge as a value (its key is lp)
        const uint32_t vb = Dt<DT>::bits(lp ^ a.flip);
        fL = Dt<DT>::to_float(vb);
      }
      // gather the candidates with one shared atomic per thread; the gather is
      // complete when their number fits
      if (tid == 0) s_cnt = 0u;
      __syncthreads();
      uint32_t cm = 0;
#pragma unroll
      for (int i = 0; i < kRowElems; ++i) {
        const float f = fval(i);
        const bool in = ((valid >> i) & 1u) && (LARGEST ? !(f < fL) : !(f > fL));
        cm |= (in ? 1u : 0u) << i;
      }
      const unsigned c = __popc(cm);
      unsigned slot = c ? atomicAdd(&s_cnt, c) : 0u;
      if (c && slot + c <= static_cast<unsigned>(kRowCap)) {
        // (position, raw bits) now; turned into composite keys once the
        // gather is known to be complete.  Static indices keep w[] in
        // registers.
#pragma unroll
        for (int i = 0; i < kRowElems; ++i)
          if ((cm >> i) & 1u) cand[slot++] = (static_cast<uint64_t>(pos_of(i)) << 32) | raw(i);
      }
      __syncthreads();
      C = s_cnt;
      TR_STAMP(4 + pass);
      if (C <= static_cast<unsigned>(kRowCap)) break;
      __syncthreads();  // s_cnt is reset next
    }

    if (C <= static_cast<unsigned>(kRowCap)) {
      // ------------------------------------------------------------ rank the candidates
      for (unsigned i = tid; i < C; i += kRowBlock) {
        const uint64_t e = cand[i];
        const uint32_t rk = (Dt<DT>::key(static_cast<uint32_t>(e)) ^ a.flip);
        cand[i] = (static_cast<uint64_t>(rk) << 32) | (0xffffffffu - static_cast<uint32_t>(e >> 32));
      }
      __syncthreads();
      TR_STAMP(8);
      for (unsigned i = tid; i < C; i += kRowBlock) {
        const uint64_t ck = cand[i];
        const unsigned r = count_greater(cand, 0u, C, ck);
        if (r < static_cast<unsigned>(a.k)) write_winner<DT>(a, row, r, ck);
      }
      __syncthreads();
      TR_STAMP(9);
      TR_VALUE(10, C);
      continue;
    }

    // -------------------------------------------------------------- many ties
    // exact k-th largest key over every element, then the tied elements in
    // position order.  (This rare path reads the row again from global memory,
    // where it is still in L2, which leaves the registers to the common path.)
    auto gkey = [&](int i) -> uint32_t { return Dt<DT>::key(raw_at<DT>(a.x, base + pos_of(i))) ^ a.flip; };
    auto gckey = [&](int i) -> uint64_t {
      return (static_cast<uint64_t>(gkey(i)) << 32) | (0xffffffffu - pos_of(i));
    };
    uint32_t vstar = 0, vm = 0;
    unsigned vrank = static_cast<unsigned>(a.k), above = 0;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass)
      kth_pass<kRowElems>(gkey, valid, pass, &vstar, &vm, &vrank, &above, hist, tmp, info);
    const unsigned need = static_cast<unsigned>(a.k) - above;  // tied elements taken
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    // winners above the value: any order
#pragma unroll
    for (int i = 0; i < kRowElems; ++i)
      if (((valid >> i) & 1u) && gkey(i) > vstar) cand[atomicAdd(&s_cnt, 1u)] = gckey(i);
    // tied ones: load by load, in position order (load j before j + 1; inside
    // a load, thread order, then element order)
    unsigned taken = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      unsigned tj = 0;
#pragma unroll
      for (int e = 0; e < VEC; ++e) tj += (((valid >> (j * VEC + e)) & 1u) && gkey(j * VEC + e) == vstar) ? 1u : 0u;
      const unsigned incl = scan_incl(tj, tmp);
      if (tid == kRowBlock - 1) info[0] = incl;
      __syncthreads();
      unsigned r = taken + incl - tj;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const int i = j * VEC + e;
        if (((valid >> i) & 1u) && gkey(i) == vstar) {
          if (r < need) cand[above + r] = gckey(i);
          ++r;
        }
      }
      taken += info[0];
      __syncthreads();
    }
    const unsigned K = static_cast<unsigned>(a.k);
    for (unsigned i = tid; i < K; i += kRowBlock) {
      const uint64_t ck = cand[i];
      write_winner<DT>(a, row, count_greater(cand, 0u, K, ck), ck);
    }
    __syncthreads();
  }
}

template <int DT, bool LARGEST>
cudaError_t launch_rows_t(const RowsParams& a, cudaStream_t st) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  const int64_t grid = a.nsel < sms ? a.nsel : sms;
  const size_t dyn = a.vec ? static_cast<size_t>(a.len) * sizeof(typename Dt<DT>::storage) : 0;
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(rows_kernel<DT, LARGEST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kRowMaxLen * sizeof(typename Dt<DT>::storage)));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  rows_kernel<DT, LARGEST><<<static_cast<unsigned>(grid), kRowBlock, dyn, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

#ifdef TK_PHASE_TIMING
int debug_rows_ns(unsigned long long* out) {
  return cudaMemcpyFromSymbol(out, g_rows_ns, sizeof(g_rows_ns)) == cudaSuccess ? 0 : -3;
}
#endif

bool rows_supported(const Problem& p, int64_t k) {
  return p.len <= kRowMaxLen && k <= kRowMaxK && k >= 1 && p.ib <= 32;
}

cudaError_t launch_rows(const Problem& p, int64_t k, void* out_vals, int64_t* out_idx, int* status,
                        cudaStream_t st) {
  if (!rows_supported(p, k)) return cudaErrorNotSupported;
  RowsParams a{p.x, p.nsel, p.len, p.flip, p.vec_ok ? 1 : 0, k, out_vals, out_idx, status};
  const bool largest = p.flip == 0;
  if (p.dtype == kF32) return largest ? launch_rows_t<kF32, true>(a, st) : launch_rows_t<kF32, false>(a, st);
  return largest ? launch_rows_t<kBF16, true>(a, st) : launch_rows_t<kBF16, false>(a, st);
}

}  // namespace tk
