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
// the source into per-warp shared-memory counters; the cluster's CTAs read one
// another's histograms through distributed shared memory, so every CTA finds
// the same boundary digit without touching global memory.  Once a CTA's
// elements at or above the current prefix fit in shared memory it caches them
// and stops re-reading the source.
//
// Sort (top-k only): the k winners (keys >= the k-th key; keys are distinct)
// are first spread evenly over the cluster, then sorted by a stable LSD radix
// sort, descending, one 8-bit digit per pass, skipping digits on which all
// winners agree.  Each pass ranks a CTA's items stably with __match_any_sync
// per warp, exchanges per-digit counts over DSMEM, and scatters every key
// straight into its destination CTA's shared memory.  The result is the order
// (value descending, index ascending), since the composite key encodes it.
#include <cooperative_groups.h>

#include "common.cuh"
#include "engine.h"

namespace cg = cooperative_groups;

namespace tk {

namespace {

constexpr unsigned kFull = 0xffffffffu;

struct SelParams {
  const uint64_t* keys;               // key source (SRC == 0)
  int64_t key_stride;
  const unsigned long long* counts;   // valid keys per selection (nullable)
  const void* x;                      // the input (SRC != 0, and for output values)
  int64_t len;                        // elements per selection of x
  int ib;
  uint32_t flip;
  int key_bits;                       // value-key bits (32 or 16)
  int64_t r;                          // rank sought (1-based)
  int want_topk;
  uint64_t* tau_out;
  void* out_vals;
  int64_t* out_idx;
  int* status;
};

template <int BLOCK, int P, int CB>
struct Layout {
  static constexpr int kWarps = BLOCK / 32;
  static constexpr int kItems = (P + BLOCK - 1) / BLOCK;
  static constexpr size_t kBufA = 0;
  static constexpr size_t kBufB = kBufA + sizeof(uint64_t) * P;
  static constexpr size_t kWhist = kBufB + sizeof(uint64_t) * CB;
  static constexpr size_t kHist = kWhist + sizeof(unsigned) * kWarps * 256;
  static constexpr size_t kGbase = kHist + sizeof(unsigned) * 256;
  static constexpr size_t kXch = kGbase + sizeof(unsigned) * 256;
  static constexpr size_t kBytes = kXch + sizeof(unsigned long long) * 4;
  static_assert(CB >= P, "cache buffer doubles as the second sort buffer");
  static_assert(BLOCK >= 256, "one thread per digit");
};

template <int SRC>
__device__ __forceinline__ uint64_t source_key(const SelParams& a, int64_t row, int64_t i) {
  if (SRC == 0) return __ldcg(a.keys + row * a.key_stride + i);
  if (SRC == 1) {
    const uint32_t u = __ldg(static_cast<const uint32_t*>(a.x) + row * a.len + i);
    return compose(order_key_f32(u) ^ a.flip, static_cast<uint64_t>(i), a.ib);
  }
  const uint32_t h = __ldg(static_cast<const uint16_t*>(a.x) + row * a.len + i);
  return compose(order_key_bf16(h) ^ a.flip, static_cast<uint64_t>(i), a.ib);
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

template <int BLOCK, int P, int CB, int SRC>
__global__ void __launch_bounds__(BLOCK, 1) select_kernel(SelParams a) {
  using L = Layout<BLOCK, P, CB>;
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* bufA = reinterpret_cast<uint64_t*>(smem + L::kBufA);
  uint64_t* bufB = reinterpret_cast<uint64_t*>(smem + L::kBufB);
  unsigned* whist = reinterpret_cast<unsigned*>(smem + L::kWhist);
  unsigned* hist = reinterpret_cast<unsigned*>(smem + L::kHist);
  unsigned* gbase = reinterpret_cast<unsigned*>(smem + L::kGbase);
  unsigned long long* xch = reinterpret_cast<unsigned long long*>(smem + L::kXch);
  __shared__ unsigned long long s_tmp[32];
  __shared__ unsigned long long s_info[4];
  __shared__ unsigned s_cnt;
  __shared__ int s_over;

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned G = cluster.num_blocks();
  const unsigned crank = cluster.block_rank();
  const int64_t row = blockIdx.x / G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int64_t valid = (SRC == 0) ? a.key_stride : a.len;
  if (SRC == 0 && a.counts) {
    const unsigned long long c = __ldcg(a.counts + row);
    if (c < static_cast<unsigned long long>(valid)) valid = static_cast<int64_t>(c);
  }
  const int64_t sb = valid * crank / G, se = valid * (crank + 1) / G;

  // ------------------------------------------------------------------ select
  const int kb = a.key_bits + a.ib;
  uint64_t prefix = 0, pmask = 0;
  unsigned long long rank = static_cast<unsigned long long>(a.r);
  bool cached = false;
  unsigned cache_n = 0;
  unsigned long long local_above = 0, local_bucket = static_cast<unsigned long long>(se - sb);
  bool failed = false;
  for (int shift = ((kb - 1) / 8) * 8; shift >= 0; shift -= 8) {
    const bool will_cache = !cached && (local_above + local_bucket) <= static_cast<unsigned long long>(CB);
    for (int i = tid; i < L::kWarps * 256; i += BLOCK) whist[i] = 0u;
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    unsigned* wh = whist + warp * 256;
    if (cached) {
      for (unsigned i = tid; i < cache_n; i += BLOCK) {
        const uint64_t k = bufB[i];
        if ((k & pmask) == prefix) atomicAdd(&wh[(k >> shift) & 255u], 1u);
      }
    } else {
      for (int64_t i = sb + tid; i < se; i += BLOCK) {
        const uint64_t k = source_key<SRC>(a, row, i);
        if ((k & pmask) == prefix) atomicAdd(&wh[(k >> shift) & 255u], 1u);
        if (will_cache && k >= prefix) bufB[atomicAdd(&s_cnt, 1u)] = k;
      }
    }
    __syncthreads();
    for (int d = tid; d < 256; d += BLOCK) {
      unsigned s = 0;
      for (int w = 0; w < L::kWarps; ++w) s += whist[w * 256 + d];
      hist[d] = s;
    }
    if (will_cache) {
      cache_n = s_cnt;
      cached = true;
    }
    if (tid == 0) s_info[0] = ~0ull;
    cluster.sync();
    // digit 255 - tid; inclusive scan from the top digit downwards
    unsigned long long tot = 0;
    const int d = 255 - tid;
    if (tid < 256)
      for (unsigned c = 0; c < G; ++c) tot += cluster.map_shared_rank(hist, c)[d];
    const unsigned long long incl = block_scan_incl(tot, s_tmp);
    if (tid < 256) {
      const unsigned long long excl = incl - tot;
      if (excl < rank && rank <= incl) {
        s_info[0] = static_cast<unsigned long long>(d);
        s_info[1] = excl;
        s_info[2] = hist[d];
        unsigned long long above = 0;
        for (int q = d + 1; q < 256; ++q) above += hist[q];
        s_info[3] = above;
      }
    }
    cluster.sync();
    if (s_info[0] == ~0ull) { failed = true; break; }
    prefix |= s_info[0] << shift;
    pmask |= 0xffull << shift;
    rank -= s_info[1];
    local_above += s_info[3];
    local_bucket = s_info[2];
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
  const int64_t k = a.r;
  const int64_t pe = (k + G - 1) / G;  // positions per CTA
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
        const uint64_t key = bufB[i];
        if (key >= tau) { ++cnt; orm |= key; andm &= key; }
      }
    } else {
      for (int64_t i = sb + tid; i < se; i += BLOCK) {
        const uint64_t key = source_key<SRC>(a, row, i);
        if (key >= tau) {
          ++cnt; orm |= key; andm &= key;
          const unsigned slot = atomicAdd(&s_cnt, 1u);
          if (slot < static_cast<unsigned>(CB)) bufB[slot] = key; else s_over = 1;
        }
      }
    }
    // count / or / and over the block; published in xch for the cluster
    const unsigned long long total = block_sum(cnt, s_tmp);
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
  // place the winners evenly: position base + local sequence -> CTA pos / pe
  {
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    if (cached || !s_over) {
      const unsigned n = cached ? cache_n : static_cast<unsigned>(xch[0]);
      for (unsigned i = tid; i < n; i += BLOCK) {
        const uint64_t key = bufB[i];
        if (cached && key < tau) continue;
        const unsigned long long pos = base + atomicAdd(&s_cnt, 1u);
        cluster.map_shared_rank(bufA, static_cast<unsigned>(pos / pe))[pos % pe] = key;
      }
    } else {
      for (int64_t i = sb + tid; i < se; i += BLOCK) {
        const uint64_t key = source_key<SRC>(a, row, i);
        if (key < tau) continue;
        const unsigned long long pos = base + atomicAdd(&s_cnt, 1u);
        cluster.map_shared_rank(bufA, static_cast<unsigned>(pos / pe))[pos % pe] = key;
      }
    }
  }
  cluster.sync();

  // ------------------------------------------------------------------ sort
  const int64_t my0 = static_cast<int64_t>(crank) * pe;
  const int n_c = static_cast<int>(my0 >= k ? 0 : (k - my0 < pe ? k - my0 : pe));
  const unsigned long long vary = all_or ^ all_and;
  uint64_t* src = bufA;
  uint64_t* dst = bufB;
  const int ipw = (n_c + L::kWarps - 1) / L::kWarps;  // items per warp segment
  const int seg0 = warp * ipw;
  const int seg1 = (seg0 + ipw < n_c) ? seg0 + ipw : n_c;
  const unsigned lt = lanemask_lt();
  for (int shift = 0; shift < 64; shift += 8) {
    if (((vary >> shift) & 0xffull) == 0) continue;  // cluster-uniform
    for (int i = tid; i < L::kWarps * 256; i += BLOCK) whist[i] = 0u;
    __syncthreads();
    unsigned* wh = whist + warp * 256;
    uint64_t key[L::kItems];
    unsigned dig[L::kItems], wr[L::kItems];
#pragma unroll
    for (int j = 0; j < L::kItems; ++j) {
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
    for (int d = tid; d < 256; d += BLOCK) {
      unsigned run = 0;
      for (int w = 0; w < L::kWarps; ++w) {
        const unsigned t = whist[w * 256 + d];
        whist[w * 256 + d] = run;
        run += t;
      }
      hist[d] = run;
    }
    cluster.sync();
    unsigned long long tot = 0, before_me = 0;
    if (tid < 256) {
      for (unsigned c = 0; c < G; ++c) {
        const unsigned h = cluster.map_shared_rank(hist, c)[tid];
        tot += h;
        if (c < crank) before_me += h;
      }
    }
    const unsigned long long incl = block_scan_incl(tot, s_tmp);
    if (tid < 256) gbase[tid] = static_cast<unsigned>(incl - tot + before_me);
    cluster.sync();
#pragma unroll
    for (int j = 0; j < L::kItems; ++j) {
      const int i = seg0 + j * 32 + lane;
      if (i < seg1) {
        const unsigned long long pos =
            static_cast<unsigned long long>(gbase[dig[j]]) + wh[dig[j]] + wr[j];
        cluster.map_shared_rank(dst, static_cast<unsigned>(pos / pe))[pos % pe] = key[j];
      }
    }
    cluster.sync();
    uint64_t* t = src; src = dst; dst = t;
  }

  // ------------------------------------------------------------------ output
  const int64_t obase = row * k + my0;
  for (int i = tid; i < n_c; i += BLOCK) {
    const uint64_t key = src[i];
    const uint64_t pos = position_of(key, a.ib);
    a.out_idx[obase + i] = static_cast<int64_t>(pos);
    const uint32_t vk = vkey_of(key, a.ib) ^ a.flip;
    if (a.key_bits == 32) {
      const uint32_t bits = (vk == Dt<kF32>::kZeroKey || vk == Dt<kF32>::kNanKey)
                                ? __ldg(static_cast<const uint32_t*>(a.x) + row * a.len + pos)
                                : value_bits_f32(vk);
      static_cast<uint32_t*>(a.out_vals)[obase + i] = bits;
    } else {
      const uint16_t bits = (vk == Dt<kBF16>::kZeroKey || vk == Dt<kBF16>::kNanKey)
                                ? __ldg(static_cast<const uint16_t*>(a.x) + row * a.len + pos)
                                : static_cast<uint16_t>(value_bits_bf16(vk));
      static_cast<uint16_t*>(a.out_vals)[obase + i] = bits;
    }
  }
}

// Kernel variants: (block, sort positions per CTA, cache/second buffer).
constexpr int kSmallBlock = 256, kSmallP = 512, kSmallCB = 2048;
constexpr int kBigBlock = 1024, kBigP = 11264, kBigCB = 11264;
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
  *used = G;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nsel * G), 1, 1);
  cfg.blockDim = dim3(BLOCK, 1, 1);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(G);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
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

cudaError_t launch_select(const Problem& p, const SelectJob& job, int64_t source_bound, int* cluster,
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
  a.r = job.r;
  a.want_topk = job.want_topk ? 1 : 0;
  a.tau_out = job.tau_out;
  a.out_vals = job.out_vals;
  a.out_idx = job.out_idx;
  a.status = job.status;
  const int src = job.keys ? 0 : (p.dtype == kF32 ? 1 : 2);
  const bool many = p.nsel >= sm_count();
  const int64_t sort_k = job.want_topk ? job.r : 1;
  const bool small = sort_k <= static_cast<int64_t>(kMaxCluster) * kSmallP;
  int G;
  if (small) {
    const int64_t g_min = (sort_k + kSmallP - 1) / kSmallP;
    const int64_t g_par = many ? 1 : (source_bound + kSmallBlock * 64 - 1) / (kSmallBlock * 64);
    G = pow2_at_least(g_min > g_par ? g_min : g_par);
  } else {
    const int64_t g_min = (sort_k + kBigP - 1) / kBigP;
    const int64_t g_par = many ? 1 : (source_bound + kBigBlock * 16 - 1) / (kBigBlock * 16);
    G = pow2_at_least(g_min > g_par ? g_min : g_par);
  }
  int used = G;
  const cudaError_t e = small ? launch_src<kSmallBlock, kSmallP, kSmallCB>(a, src, p.nsel, G, &used, st)
                              : launch_src<kBigBlock, kBigP, kBigCB>(a, src, p.nsel, G, &used, st);
  if (cluster) *cluster = used;
  return e;
}

}  // namespace tk
