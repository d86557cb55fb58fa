// Stage 1 of Prof-K (section 3, "Sampling"): S uniform positions per selection,
// drawn with Philox4x32-10, and the composite keys of the drawn elements.
//
// The draws are independent (with replacement); the parameter rule accounts
// for that exactly (see params.cpp).  Each thread makes one Philox call and
// turns its four 32-bit words into two 64-bit uniforms, i.e. two positions.
// The gathers are random 2- or 4-byte reads -- latency bound, so the grid is
// spread over every SM and each thread has both loads in flight at once.
// Optionally the keys are also counted by their leading 11 bits into a
// per-selection histogram, which is the threshold select's first digit.
//
// For one or a few selections the threshold (stage 2: the t-th largest
// sampled key) is computed by the same grid: a radix select whose digits are
// counted per block and merged in global histograms, one grid barrier per
// digit, the threads keeping their two keys in registers throughout.  Once
// the boundary bin holds few keys they are gathered, and the last block of
// the selection to finish ranks them ("Find the Cutoff Instead": count into
// buckets, recurse into the bucket holding the boundary).
#include "common.cuh"
#include "engine.h"
#include "rank.cuh"

namespace tk {

template <int DT>
__global__ void __launch_bounds__(256) sample_kernel(const void* __restrict__ x, int64_t len, int64_t S,
                                                     int ib, uint32_t flip, uint2 key, uint2 ctr_hi,
                                                     uint64_t* __restrict__ keys,
                                                     unsigned long long* __restrict__ counts,
                                                     DevHeader* __restrict__ hdr,
                                                     unsigned* __restrict__ hist_add,
                                                     unsigned* __restrict__ hist_zero) {
  using T = typename Dt<DT>::storage;
  constexpr unsigned DM = kSampleHistBins - 1;
  __shared__ unsigned sh[kSampleHistBins];
  TK_TL_BEGIN(0);
  grid_launch_dependents();  // the threshold select may start launching
  const uint32_t row = blockIdx.y;
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (pair == 0) {
    if (counts) counts[row] = 0ull;  // survivor counter of the filter that follows
    if (hdr && row == 0) {
      hdr->barrier[0] = 0u;  // arrival count of the fallback's grid barrier
      hdr->status = kDevOk;
      hdr->misses = 0ull;
      hdr->shortfalls = 0u;
    }
  }
  if (hist_add) {
    // (all of the other half: the next call may use other rows or levels)
    for (int i = threadIdx.x; i < kSampleHistBins; i += blockDim.x) sh[i] = 0u;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * gridDim.y * blockDim.x;
    for (int64_t i = (static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
         i < kSampleHistHalfWords; i += nthreads)
      hist_zero[i] = 0u;
    __syncthreads();
  }
  const bool one = 2 * pair < S, two = 2 * pair + 1 < S;
  uint64_t k0 = 0, k1 = 0;
  if (one) {
    uint64_t p0, p1;
    sample_pair(key, ctr_hi, row, static_cast<uint32_t>(pair), static_cast<uint64_t>(len), &p0, &p1);
    const T* xr = static_cast<const T*>(x) + static_cast<int64_t>(row) * len;
    const uint32_t v0 = __ldg(xr + p0);
    const uint32_t v1 = two ? static_cast<uint32_t>(__ldg(xr + p1)) : 0u;
    uint64_t* out = keys + static_cast<int64_t>(row) * S + 2 * pair;
    k0 = compose(Dt<DT>::key(v0) ^ flip, p0, ib);
    out[0] = k0;
    if (two) {
      k1 = compose(Dt<DT>::key(v1) ^ flip, p1, ib);
      out[1] = k1;
    }
  }
  if (hist_add) {
    // leading bits of the composite key = leading bits of the value key
    const int sh_bits = Dt<DT>::kKeyBits + ib - kSampleHistBits;
    if (one) atomicAdd(&sh[DM - static_cast<unsigned>((k0 >> sh_bits) & DM)], 1u);
    if (two) atomicAdd(&sh[DM - static_cast<unsigned>((k1 >> sh_bits) & DM)], 1u);
    __syncthreads();
    unsigned* h = hist_add + static_cast<int64_t>(row) * kSampleHistBins;
    for (int i = threadIdx.x; i < kSampleHistBins; i += blockDim.x)
      if (sh[i]) atomicAdd(h + i, sh[i]);
  }
  TK_TL_END(0);
}

namespace {

#ifdef TK_PHASE_TIMING
__device__ unsigned long long g_st_ns[2][16];  // debug: stamps of block 0 and of the ranking block
#define TK_ST(i)                                                                                 \
  do {                                                                                           \
    if (threadIdx.x == 0 && blockIdx.x == 0) g_st_ns[0][(i)] = globaltimer_ns();                 \
  } while (0)
#define TK_STL(i)                                                                                \
  do {                                                                                           \
    if (threadIdx.x == 0) g_st_ns[1][(i)] = globaltimer_ns();                                    \
  } while (0)
#else
#define TK_ST(i) \
  do {           \
  } while (0)
#define TK_STL(i) \
  do {            \
  } while (0)
#endif

struct SampleTauParams {
  const void* x;
  int64_t len;
  int64_t S;
  int ib;
  uint32_t flip;
  uint2 key, ctr;
  unsigned long long* counts;
  DevHeader* hdr;
  SampleTauScratch sc;
  uint64_t* tau_out;
  unsigned* refine_ctl;  // nullable: the grid refinement's control words; the largest sampled key goes there
  int64_t t;
  int q;      // blocks per selection
  int local;  // q * (t + 1) <= kTauGather: each block keeps its own top t (no grid barrier)
};

constexpr int kSampleBlock = 256;

// Barrier over a cooperative grid: arrivals in bar[0] (reset by the last
// block to arrive), generation in bar[1].  Gives up after kWaitLimitNs,
// records kDevTimeout and returns false.
__device__ bool tau_grid_barrier(unsigned* bar, int* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned gen = ld_acquire_u32(bar + 1);
    __threadfence();
    if (atomicAdd(bar, 1u) + 1u == gridDim.x) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u32(bar + 1) == gen) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicCAS(status, kDevOk, kDevTimeout);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

template <int DT>
__global__ void __launch_bounds__(kSampleBlock) sample_tau_kernel(SampleTauParams p) {
  using T = typename Dt<DT>::storage;
  constexpr int BLOCK = kSampleBlock;
  constexpr unsigned DM = kSampleHistBins - 1;
  __shared__ unsigned sh[kSampleHistBins];
  __shared__ uint64_t gk[kTauGather];
  __shared__ unsigned long long s_tmp[32];
  __shared__ unsigned long long s_info[3];
  __shared__ unsigned s_cnt;
  __shared__ int s_last;
  __shared__ uint64_t s_tau;
  __shared__ unsigned long long s_kmax;
  TK_TL_BEGIN(0);
  TK_ST(0);
  grid_launch_dependents();
  const int tid = threadIdx.x;
  const int row = static_cast<int>(blockIdx.x) / p.q;
  const int64_t pair = static_cast<int64_t>(static_cast<int>(blockIdx.x) % p.q) * BLOCK + tid;
  int* status = &p.hdr->status;
  if (pair == 0) {
    if (p.counts) p.counts[row] = 0ull;  // survivor counter of the filter that follows
    if (row == 0) {
      p.hdr->barrier[0] = 0u;  // arrival count of the fallback's grid barrier
      p.hdr->status = kDevOk;
      p.hdr->misses = 0ull;
      p.hdr->shortfalls = 0u;
    }
  }
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * BLOCK + tid; i < kSampleHistHalfWords;
       i += static_cast<int64_t>(gridDim.x) * BLOCK)
    p.sc.hist_zero[i] = 0u;  // the next call's histograms

  if (tid == 0) s_kmax = 0ull;
  if (p.refine_ctl) __syncthreads();

  // two sampled keys per thread, kept in registers
  const bool one = 2 * pair < p.S, two = 2 * pair + 1 < p.S;
  uint64_t k0 = 0, k1 = 0;
  if (one) {
    uint64_t p0, p1;
    sample_pair(p.key, p.ctr, static_cast<uint32_t>(row), static_cast<uint32_t>(pair), static_cast<uint64_t>(p.len),
                &p0, &p1);
    const T* xr = static_cast<const T*>(p.x) + static_cast<int64_t>(row) * p.len;
    const uint32_t v0 = __ldg(xr + p0);
    const uint32_t v1 = two ? static_cast<uint32_t>(__ldg(xr + p1)) : 0u;
    k0 = compose(Dt<DT>::key(v0) ^ p.flip, p0, p.ib);
    if (two) k1 = compose(Dt<DT>::key(v1) ^ p.flip, p1, p.ib);
  }
  if (p.refine_ctl) {
    // the largest sampled key: a warp maximum, a block maximum, one atomic per block
    unsigned long long m = k0 > k1 ? k0 : k1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(kFull, m, o);
      m = y > m ? y : m;
    }
    if ((tid & 31) == 0 && m) atomicMax(&s_kmax, m);
    __syncthreads();
    if (tid == 0 && s_kmax)
      atomicMax(reinterpret_cast<unsigned long long*>(p.refine_ctl + row * kRefineGridCtlWords + kRefineGridKmaxWord),
                s_kmax);
  }
  TK_ST(1);

  // Few candidates in all (q * (t + 1) <= kTauGather): the t largest sampled keys
  // are among the union of every block's own t largest, so each block ranks
  // its keys, keeps its top t, and the last block ranks the union -- no grid
  // barrier and no grid-wide histogram.
  uint64_t bound = 0ull;
  // small t: each block's t largest by warp rounds (no radix passes), appended
  // at once; the last block takes the t-th of their union the same way
  __shared__ uint64_t s_lists[(BLOCK / 32) * 32];
  __shared__ unsigned s_lcount[BLOCK / 32];
  __shared__ uint64_t s_top[kSmallTopT];
  __shared__ unsigned s_topn;
  const bool small_t = p.local && p.t <= kSmallTopT;
  if (small_t) {
    uint64_t v[2] = {k0, k1};
    const int nt = block_top_small<BLOCK, 2>(v, (one ? 1 : 0) + (two ? 1 : 0), static_cast<int>(p.t), s_lists,
                                             s_lcount, s_top, &s_topn);
    // this block's fixed slots [i t, i t + t) of the gather buffer (q t <=
    // kTauGather): no atomic to reserve them; a block with fewer than t keys
    // fills the rest with key 0, which ranks below every key or ties a key
    // of the same value, so the t-th largest of the union keeps its value
    uint64_t* gat0 = p.sc.gather + static_cast<int64_t>(row) * kTauGather;
    const int qi = static_cast<int>(blockIdx.x) % p.q;
    if (tid < static_cast<int>(p.t)) gat0[qi * p.t + tid] = tid < nt ? s_top[tid] : 0ull;
  } else if (p.local) {
    const int64_t first = 2 * (static_cast<int64_t>(static_cast<int>(blockIdx.x) % p.q) * BLOCK);
    const int64_t left = p.S - first;
    const unsigned nloc = static_cast<unsigned>(left < 2 * BLOCK ? left : 2 * BLOCK);
    if (one) gk[2 * tid] = k0;
    if (two) gk[2 * tid + 1] = k1;  // (the valid keys are gk[0 .. nloc))
    if (nloc > static_cast<unsigned>(p.t)) {
      bucket_kth<BLOCK>(gk, nloc, static_cast<unsigned long long>(p.t), sh, s_tmp, s_info, &s_cnt, &s_tau);
      __syncthreads();
      bound = s_tau;  // this block's t-th largest: keep the keys at or above it
    }
    __syncthreads();  // gk and s_tau are reused below
  }

  // radix select of the t-th largest key over the grid, one digit a level
  const int kb = Dt<DT>::kKeyBits + p.ib;
  uint64_t prefix = 0ull, pmask = (kb >= 64) ? 0ull : (~0ull << kb);
  int shift = kb - kSampleHistBits;
  unsigned long long rank = static_cast<unsigned long long>(p.t);
  for (int level = 0; !p.local; ++level) {
    for (int i = tid; i < kSampleHistBins; i += BLOCK) sh[i] = 0u;
    __syncthreads();
    if (one && (k0 & pmask) == prefix) atomicAdd(&sh[DM - static_cast<unsigned>((k0 >> shift) & DM)], 1u);
    if (two && (k1 & pmask) == prefix) atomicAdd(&sh[DM - static_cast<unsigned>((k1 >> shift) & DM)], 1u);
    __syncthreads();
    unsigned* h = p.sc.hist + (static_cast<int64_t>(level) * kSampleHistMaxRows + row) * kSampleHistBins;
    for (int i = tid; i < kSampleHistBins; i += BLOCK)
      if (sh[i]) atomicAdd(h + i, sh[i]);
    TK_ST(2 + 3 * (level < 3 ? level : 2));
    if (!tau_grid_barrier(p.sc.ctl, status)) return;
    TK_ST(3 + 3 * (level < 3 ? level : 2));
    // every block reads the same totals and finds the same boundary bin
    constexpr int kPer = kSampleHistBins / BLOCK;
    static_assert(kPer == 8, "two 16-byte loads per thread");
    unsigned c[kPer];
    unsigned long long sum = 0;
    {
      // 16-byte loads: each line of the totals is requested once per block
      const uint4 lo = ldcg_u4(h + tid * kPer), hi = ldcg_u4(h + tid * kPer + 4);
      c[0] = lo.x; c[1] = lo.y; c[2] = lo.z; c[3] = lo.w;
      c[4] = hi.x; c[5] = hi.y; c[6] = hi.z; c[7] = hi.w;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) sum += c[j];
    if (tid == 0) s_info[0] = ~0ull;
    const unsigned long long incl = block_scan_incl(sum, s_tmp);
    unsigned long long run = incl - sum;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (run < rank && rank <= run + c[j]) {
        s_info[0] = static_cast<unsigned long long>(tid * kPer + j);
        s_info[1] = run;
        s_info[2] = c[j];
      }
      run += c[j];
    }
    __syncthreads();
    const bool found = s_info[0] != ~0ull;
    if (found) {
      prefix |= static_cast<uint64_t>(DM - static_cast<unsigned>(s_info[0])) << shift;
      pmask |= static_cast<uint64_t>(DM) << shift;
      rank -= s_info[1];
    }
    const unsigned long long tot = s_info[2];
    __syncthreads();  // s_info is rewritten below
    TK_ST(4 + 3 * (level < 3 ? level : 2));
    // (the same totals in every block: every block leaves here together)
    if (!found || (tot > kTauGather && shift > 0 && level + 1 >= kSampleHistLevels)) {
      if (tid == 0) atomicCAS(status, kDevOk, kDevBadState);
      return;
    }
    if (tot <= kTauGather || shift == 0) break;
    shift = shift >= kSampleHistBits ? shift - kSampleHistBits : 0;
  }

  // gather the boundary bin (or each block's top t); the last block of the
  // selection ranks what was gathered
  unsigned* gctl = p.sc.ctl + 2 + 2 * row;  // gathered count, ticket
  uint64_t* gat = p.sc.gather + static_cast<int64_t>(row) * kTauGather;
  if (!small_t) {
    const bool w0 = one && (p.local ? k0 >= bound : (k0 & pmask) == prefix);
    const bool w1 = two && (p.local ? k1 >= bound : (k1 & pmask) == prefix);
    const unsigned s0 = warp_append_slot(gctl, w0);
    if (w0 && s0 < static_cast<unsigned>(kTauGather)) gat[s0] = k0;
    const unsigned s1 = warp_append_slot(gctl, w1);
    if (w1 && s1 < static_cast<unsigned>(kTauGather)) gat[s1] = k1;
  }
  __threadfence();
  __syncthreads();
  TK_ST(11);
  if (tid == 0) s_last = atomicAdd(gctl + 1, 1u) == static_cast<unsigned>(p.q - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  TK_STL(0);
  __threadfence();
  // every slot of the gather buffer and its count in one round of loads
  // (the slots past the count are dropped below)
  constexpr int kPerThread = kTauGather / BLOCK;
  uint64_t raw[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) raw[j] = __ldcg(gat + tid + j * BLOCK);
  const unsigned gn = small_t ? static_cast<unsigned>(p.q * p.t) : __ldcg(gctl);
  const unsigned n = gn < static_cast<unsigned>(kTauGather) ? gn : static_cast<unsigned>(kTauGather);
  if (small_t) {
    // the union (at most kTauGather keys: eight a thread), its t-th largest
    uint64_t v[kPerThread];
    int c = 0;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      const unsigned i = tid + j * BLOCK;
      v[j] = i < n ? raw[j] : 0ull;
      c += i < n ? 1 : 0;
    }
    if (tid == 0) {
      s_tau = 0ull;
      if (gn > static_cast<unsigned>(kTauGather)) atomicCAS(status, kDevOk, kDevBadState);
      gctl[0] = 0u;  // ready for the next call
      gctl[1] = 0u;
    }
    TK_STL(1);
    // (each thread's keys are a strided slice: the exchange network sorts them)
    const int nt = block_top_small<BLOCK, kPerThread>(v, c, static_cast<int>(p.t), s_lists, s_lcount, s_top, &s_topn);
    if (tid == 0) {
      if (nt == static_cast<int>(p.t)) s_tau = s_top[nt - 1];
      else atomicCAS(status, kDevOk, kDevBadState);
    }
    __syncthreads();
  } else {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j)
      if (tid + j * BLOCK < static_cast<int>(n)) gk[tid + j * BLOCK] = raw[j];
    if (tid == 0) {
      s_tau = 0ull;
      if (gn > static_cast<unsigned>(kTauGather)) atomicCAS(status, kDevOk, kDevBadState);
      gctl[0] = 0u;  // ready for the next call
      gctl[1] = 0u;
    }
    __syncthreads();
    TK_STL(1);
    bucket_kth<BLOCK>(gk, n, rank, sh, s_tmp, s_info, &s_cnt, &s_tau);
    __syncthreads();
  }
  TK_STL(2);
  if (tid == 0) p.tau_out[row] = s_tau;
#ifdef TK_PHASE_TIMING
  if (tid == 0) g_st_ns[1][3] = n;
#endif
  TK_TL_END(0);
}

template <int DT>
int sample_tau_capacity() {
  static int cap = -1;  // co-resident blocks of the fused grid on this device
  if (cap < 0) {
    int dev = 0, sms = 0, per = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, sample_tau_kernel<DT>, kSampleBlock, 0) != cudaSuccess)
      return 0;
    cap = sms * per;
  }
  return cap;
}

}  // namespace

bool sample_tau_supported(const Problem& p, int64_t S) {
  if (p.nsel > kSampleHistMaxRows || S < 1) return false;
  const int64_t q = ((S + 1) / 2 + kSampleBlock - 1) / kSampleBlock;
  const int cap = p.dtype == kF32 ? sample_tau_capacity<kF32>() : sample_tau_capacity<kBF16>();
  return q * p.nsel <= cap;
}

bool sample_tau_local(int64_t S, int64_t t) {
  const int64_t q = ((S + 1) / 2 + kSampleBlock - 1) / kSampleBlock;
  // (one key of slack per block: equal keys at a block's bound are all kept)
  return q * (t + 1) <= kTauGather;
}

cudaError_t launch_sample_tau(const Problem& p, int64_t S, int64_t t, uint64_t seed, uint64_t counter,
                              unsigned long long* counts_to_zero, DevHeader* hdr, const SampleTauScratch& sc,
                              uint64_t* tau_out, cudaStream_t st) {
  if (!sample_tau_supported(p, S) || t < 1 || t > S) return cudaErrorInvalidValue;
  SampleTauParams sp{};
  sp.x = p.x;
  sp.len = p.len;
  sp.S = S;
  sp.ib = p.ib;
  sp.flip = p.flip;
  sp.key = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  sp.ctr = make_uint2(static_cast<uint32_t>(counter), static_cast<uint32_t>(counter >> 32));
  sp.counts = counts_to_zero;
  sp.hdr = hdr;
  sp.sc = sc;
  sp.tau_out = tau_out;
  sp.refine_ctl = sc.refine_ctl;
  sp.t = t;
  sp.q = static_cast<int>(((S + 1) / 2 + kSampleBlock - 1) / kSampleBlock);
  sp.local = sample_tau_local(S, t) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sp.q * p.nsel), 1, 1);
  cfg.blockDim = dim3(kSampleBlock, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every block resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = sp.local ? 0 : 1;  // (no block waits on another in the local mode)
  if (p.dtype == kF32) return cudaLaunchKernelEx(&cfg, sample_tau_kernel<kF32>, sp);
  return cudaLaunchKernelEx(&cfg, sample_tau_kernel<kBF16>, sp);
}

cudaError_t launch_sample(const Problem& p, int64_t S, uint64_t seed, uint64_t counter,
                          uint64_t* keys, unsigned long long* counts_to_zero, DevHeader* hdr,
                          unsigned* hist_add, unsigned* hist_zero, cudaStream_t st) {
  if (hist_add && (!hist_zero || p.nsel > kSampleHistMaxRows)) return cudaErrorInvalidValue;
  const int64_t pairs = (S + 1) / 2;
  const dim3 block(256);
  const dim3 grid(static_cast<unsigned>((pairs + 255) / 256), static_cast<unsigned>(p.nsel));
  const uint2 key = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const uint2 ctr = make_uint2(static_cast<uint32_t>(counter), static_cast<uint32_t>(counter >> 32));
  if (p.dtype == kF32)
    sample_kernel<kF32><<<grid, block, 0, st>>>(p.x, p.len, S, p.ib, p.flip, key, ctr, keys,
                                                counts_to_zero, hdr, hist_add, hist_zero);
  else
    sample_kernel<kBF16><<<grid, block, 0, st>>>(p.x, p.len, S, p.ib, p.flip, key, ctr, keys,
                                                 counts_to_zero, hdr, hist_add, hist_zero);
  return cudaGetLastError();
}

#ifdef TK_PHASE_TIMING
TK_TIMELINE_ACCESSOR(debug_timeline_sample)
int debug_sample_tau_ns(unsigned long long* out) {
  return cudaMemcpyFromSymbol(out, g_st_ns, sizeof(g_st_ns)) == cudaSuccess ? 0 : -3;
}
#endif

}  // namespace tk
