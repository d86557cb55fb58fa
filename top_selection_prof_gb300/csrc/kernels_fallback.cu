// The exact fallback (Prof-K paper, section 3, stage 4, and Appendix D
// "Fallback as a Safety Mechanism") and the grid refinement for large k.
//
// fallback_kernel is a cooperative launch.  For every selection whose filter
// result missed k <= R <= M (or every selection when forced) it finds the
// k-th largest element exactly by radix select on the value key (8-bit digits,
// one grid-wide histogram per digit), resolves ties at that value by index --
// per-tile counts of the tied value, a scan and a lower bound over the running
// count ("Find It in log n"), then an ordered scan of one tile -- and re-runs
// the filter with that exact threshold, which keeps exactly k elements.
// Grid-wide steps use a bounded barrier that reports a timeout instead of
// hanging.  refine_grid_kernel runs the same miss check and fallback and then
// partitions the candidates of a few selections with many winners (below).
#include <cooperative_groups.h>

#include "binfo.cuh"
#include "filter_core.cuh"

namespace tk {

namespace {

// ---------------------------------------------------------------------------
// Fallback
// ---------------------------------------------------------------------------

struct FallbackParams {
  FilterParams fp;
  int64_t k;
  int force;
  FallbackScratch fs;
};

// Grid-wide barrier for a cooperative launch.  Gives up after fs.wait_ns and
// records kDevTimeout in the status word; returns false then (and when another
// block already reported an error).  Test knob: block fs.stall_block leaves
// without arriving (and returns false), so every other block's wait runs out.
__device__ bool grid_barrier(const FallbackScratch& fs) {
  __shared__ int s_ok;
  unsigned* bar = fs.barrier;
  int* status = fs.status;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    if (static_cast<int>(blockIdx.x) == fs.stall_block) {
      ok = 0;
    } else {
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
          if (*reinterpret_cast<volatile int*>(status) != kDevOk || globaltimer_ns() - t0 > fs.wait_ns) {
            atomicCAS(status, kDevOk, kDevTimeout);
            ok = 0;
            break;
          }
          __nanosleep(128);
        }
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
  __shared__ unsigned long long s_row_words[2];

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
    // (one thread loads the words the whole grid reads; the block shares them)
    __syncthreads();
    if (threadIdx.x == 0) {
      s_row_words[0] = __ldcg(fp.counts + row);
      s_row_words[1] = fs.relax_tau ? __ldcg(fs.relax_tau + row) : 0ull;
    }
    __syncthreads();
    const unsigned long long R = s_row_words[0];
    const unsigned long long kk = static_cast<unsigned long long>(a.k);
    // Relaxed recall: fewer than k survivors are the exact top-R and are
    // returned as they are.  Slots R..k-1 of the buffer get the sentinel keys
    // tau - 1 - j (below every survivor, distinct), written out as padding.
    // (Needs tau >= k for the sentinels; otherwise the row takes the exact
    // fallback like any other miss.)
    const uint64_t rtau = s_row_words[1];
    const bool shortfall = fs.relax_tau && !a.force && R < kk && rtau >= kk;
    const bool miss = a.force || (R < kk && !shortfall) || R > static_cast<unsigned long long>(fp.cap);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      fs.r_seen[row] = R;
      if (miss) atomicAdd(fs.misses, 1ull);
      if (shortfall) atomicAdd(fs.shortfalls, 1u);
      // the bound below which keys are padding (a missed row: its exact
      // k-th key, written below, which no key of the rebuilt buffer is under)
      if (fs.relax_tau && !miss) fs.tau_exact[row] = shortfall ? rtau : 0ull;
    }
    if (shortfall) {
      uint64_t* dst = fp.buf + row * fp.cap;
      for (int64_t j = static_cast<int64_t>(R) + gtid; j < a.k; j += nthreads)
        dst[j] = rtau - 1ull - static_cast<uint64_t>(j - static_cast<int64_t>(R));
      missed = 1;  // the buffer changed
      continue;
    }
    if (!miss) continue;
    missed = 1;
    const T* xr = static_cast<const T*>(fp.x) + row * fp.len;

    // -- zero the per-digit histograms
    TK_FB(0);
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) fs.ghist[i] = 0u;
    if (!grid_barrier(fs)) return -1;
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
      if (!grid_barrier(fs)) return -1;
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
    if (!grid_barrier(fs)) return -1;
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
    if (!grid_barrier(fs)) return -1;
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
  static_assert(kPartPer == 8, "two 16-byte loads per thread");
  unsigned c[kPartPer], sum = 0;
  {
    const uint4 lo = ldcg_u4(g + threadIdx.x * kPartPer), hi = ldcg_u4(g + threadIdx.x * kPartPer + 4);
    c[0] = lo.x; c[1] = lo.y; c[2] = lo.z; c[3] = lo.w;
    c[4] = hi.x; c[5] = hi.y; c[6] = hi.z; c[7] = hi.w;
  }
#pragma unroll
  for (int q = 0; q < kPartPer; ++q) sum += c[q];
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

// One winner to its output slot: the position, and the input's own bits (the
// key gives them back except for zeros and NaNs, whose bits are read from x).
__device__ __forceinline__ void write_winner(const FilterParams& fp, const RefineGridScratch& rg, int64_t row,
                                             int64_t k, int64_t slot, uint64_t key, uint64_t pad_below) {
  const int64_t oi = row * k + slot;
  if (key < pad_below) {  // a padding sentinel of relaxed recall
    rg.out_idx[oi] = -1;
    if (rg.unsorted == 1) static_cast<uint32_t*>(rg.out_vals)[oi] = fp.flip ? 0x7F800000u : 0xFF800000u;
    else static_cast<uint16_t*>(rg.out_vals)[oi] = static_cast<uint16_t>(fp.flip ? 0x7F80u : 0xFF80u);
    return;
  }
  const uint64_t pos = position_of(key, fp.ib);
  rg.out_idx[oi] = static_cast<int64_t>(pos);
  const uint32_t vk = vkey_of(key, fp.ib) ^ fp.flip;
  if (rg.unsorted == 1) {  // f32
    static_cast<uint32_t*>(rg.out_vals)[oi] =
        (vk == Dt<kF32>::kZeroKey || vk == Dt<kF32>::kNanKey)
            ? __ldg(static_cast<const uint32_t*>(fp.x) + row * fp.len + pos)
            : value_bits_f32(vk);
  } else {  // bf16
    static_cast<uint16_t*>(rg.out_vals)[oi] =
        (vk == Dt<kBF16>::kZeroKey || vk == Dt<kBF16>::kNanKey)
            ? __ldg(static_cast<const uint16_t*>(fp.x) + row * fp.len + pos)
            : static_cast<uint16_t>(value_bits_bf16(vk));
  }
}

__device__ bool partition_row(const RefineGridParams& a, int64_t row, uint64_t* cache, unsigned char* dsm,
                              bool hist_ok) {
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

  // ---- this block's slice of the buffer: bounds fixed by the capacity (the
  // host checks cap <= gridDim.x * kPartCache), so its loads are in flight
  // before R is known; keys at or beyond the valid count are dropped below
  // (when the filter also placed the survivors in bin regions they are
  // usually copied from there, and the slice is loaded only if not)
  const int64_t sb = fp.cap * blockIdx.x / gridDim.x, se = fp.cap * (blockIdx.x + 1) / gridDim.x;
  const uint64_t* src = fp.buf + row * fp.cap + sb;
  constexpr int kSliceLoads = kPartCache / kFilterBlock;
  uint64_t kv[kSliceLoads];
  auto load_slice = [&]() {
#pragma unroll
    for (int q = 0; q < kSliceLoads; ++q) {
      const int64_t i = tid + q * kFilterBlock;
      kv[q] = i < se - sb ? __ldcg(src + i) : 0ull;
    }
  };
  const bool regions = hist_ok && rg.region != nullptr;
  if (!regions) load_slice();

  // ---- the filter's histogram of the survivors' offsets above tau, when it
  // was kept and the buffer holds exactly the survivors it counted (no miss):
  // it gives every bin's total at once.  Usable when its top bin is empty
  // (every offset below 2047 << shift, so the bins are a plain digit of key -
  // tau) and the boundary bin fits the exchange buffer after the bins above.
  // The words every block reads are loaded by one thread each and shared: R,
  // the relaxed-recall tau, tau and the largest sampled key.
  __shared__ unsigned long long s_words[6];
  if (tid == 0) {
    s_words[0] = __ldcg(fp.counts + row);
    s_words[1] = fs.relax_tau ? __ldcg(fs.relax_tau + row) : 0ull;
    s_words[2] = hist_ok ? __ldcg(rg.tau + row) : 0ull;
    s_words[3] = hist_ok ? sampled_kmax(rg.ctl, row) : 0ull;
    s_words[4] = regions ? __ldcg(ctl + kRefineGridBinnedWord) : 1ull;  // 0: bin regions complete
    s_words[5] = regions ? __ldcg(ctl + kRefineGridFilterHist) : 1ull;  // the top (overflow) bin's count
  }
  if (regions && !rg.unsorted) {
    // Sorted output from complete bin regions: nothing to place here.  The
    // bin sort reads the filter's histogram and the regions itself; this
    // kernel only checked the miss (no miss: R is within [k, M] and the
    // histogram counts exactly the survivors) and publishes the digit.  The
    // bins below the top one are a plain digit of key - tau; the top bin
    // (keys beyond 2047 << shift) is not, so it may hold only a few keys,
    // none of them the k-th: a bin-sort block then never cuts it by digits
    // (it cuts only a bin larger than (kBinSortCap - its places) / 2 = 768).
    __syncthreads();
    if (s_words[4] == 0ull && s_words[5] <= kBinnedTopMax && s_words[5] < k) {
      if (blockIdx.x == 0 && tid == 0) {
        const uint64_t tau = s_words[2];
        const int hs = survivor_shift(tau, s_words[3]);
        const uint64_t pm = hs + kPartDigit >= 64 ? 0ull : (~0ull << (hs + kPartDigit));
        unsigned* bo = rg.binfo + row * binfo_words(static_cast<int64_t>(k));
        bo[kRefineGridBins] = 0u;
        bo[kRefineGridBins + 1] = 0u;
        bo[kRefineGridBins + 2] = static_cast<unsigned>(pm);
        bo[kRefineGridBins + 3] = static_cast<unsigned>(pm >> 32);
        bo[kRefineGridBins + 4] = static_cast<unsigned>(hs);
        bo[kRefineGridBins + 5] = 0u;  // (the bin sort finds the end of the boundary bin)
        bo[kRefineGridBins + 6] = static_cast<unsigned>(tau);
        bo[kRefineGridBins + 7] = static_cast<unsigned>(tau >> 32);
        bo[kRefineGridBins + 8] = 1u;  // the keys are in the bin regions
      }
      __syncthreads();  // (s_words is rewritten by the next selection)
      TK_RG(9);
      return true;
    }
  }
  bool fast = false, found = false;
  unsigned bb = 0, bb_start = 0, bb_tot = 0;
  if (hist_ok) {
    const unsigned* fh = ctl + kRefineGridFilterHist;
    if (find_rank_bin(fh, k, bst, s_ws, s_info)) {  // (synchronises the block)
      found = true;
      bb = s_info[0];
      bb_start = s_info[1];
      bb_tot = s_info[2];
      fast = bst[1] == 0u && static_cast<int64_t>(bb_start) + bb_tot <= rg.xstride;  // top bin empty
    }
  }
  __syncthreads();  // s_info is rewritten below; s_words are visible

  // ---- bin regions: the filter left every survivor in its bin's region,
  // so the winners' bins are copied out in place order -- no slice, no
  // histogram, no atomics here.  Sorted output: places [0, end of the
  // boundary bin) to the exchange buffer, as the partition below would have
  // placed them, for the bin sort.  Unsorted: the bins above the boundary
  // straight to the outputs, and block 0 ranks the boundary bin.
  if (regions && rg.unsorted && found && bb > 0u && s_words[4] == 0ull && bb_tot <= static_cast<unsigned>(kPartCache)) {
    // Unsorted output from complete bin regions: the bins above the
    // boundary (the top bin's keys too, whatever they are) go straight to
    // the outputs, split over every block but the last, which ranks the
    // boundary bin.
    TK_RG(3);
    const unsigned pend = bb_start;
    const unsigned ncopy = gridDim.x > 1 ? gridDim.x - 1 : 1u;
    const unsigned per = (pend + ncopy - 1) / ncopy;
    const unsigned p0 = blockIdx.x < ncopy && blockIdx.x * per < pend ? blockIdx.x * per : pend;
    const unsigned p1 = p0 + per < pend ? p0 + per : pend;
    // each place's bin by a binary search over the bin starts, four places
    // of a thread at once so that their searches and loads overlap (walking
    // the bins in order instead costs a step per bin, and the top bins are
    // mostly empty)
    constexpr int kCopyPer = 4;
    for (unsigned base = p0; base < p1; base += kCopyPer * kFilterBlock) {
      unsigned pl[kCopyPer], bl[kCopyPer];
      uint64_t key[kCopyPer];
#pragma unroll
      for (int j = 0; j < kCopyPer; ++j) {
        pl[j] = base + j * kFilterBlock + tid;
        bl[j] = 0u;
      }
      // (bst is non-decreasing and bst[0] = 0: the largest bin <= bb whose
      // start is <= the place, in a fixed number of steps)
#pragma unroll
      for (unsigned stp = kRefineGridBins / 2; stp > 0; stp >>= 1)
#pragma unroll
        for (int j = 0; j < kCopyPer; ++j)
          if (bl[j] + stp <= bb && bst[bl[j] + stp] <= pl[j]) bl[j] += stp;
#pragma unroll
      for (int j = 0; j < kCopyPer; ++j)
        key[j] = pl[j] < p1 ? __ldcg(rg.region + static_cast<int64_t>(bl[j]) * kBinRegionCap + (pl[j] - bst[bl[j]]))
                            : 0ull;
#pragma unroll
      for (int j = 0; j < kCopyPer; ++j)
        if (pl[j] < p1) write_winner(fp, rg, row, static_cast<int64_t>(k), pl[j], key[j], 0ull);
    }
    TK_RG(5);
    if (blockIdx.x == gridDim.x - 1) {
      // the top (k - bb_start) keys of the boundary bin (distinct keys:
      // exactly that many are >= the one of that rank)
      __shared__ unsigned long long s_tmp[32];
      __shared__ unsigned long long s_rinfo[3];
      __shared__ unsigned s_cnt;
      __shared__ uint64_t s_kappa;
      const unsigned r = static_cast<unsigned>(k) - bb_start;
      const uint64_t* rb = rg.region + static_cast<int64_t>(bb) * kBinRegionCap;
      for (unsigned i = tid; i < bb_tot; i += kFilterBlock) stg[i] = __ldcg(rb + i);
      __syncthreads();
      TK_RG(6);
      bucket_kth<kFilterBlock>(stg, bb_tot, r, mine, s_tmp, s_rinfo, &s_cnt, &s_kappa);
      __syncthreads();
      TK_RG(7);
      const uint64_t kap = s_kappa;
      if (tid == 0) s_cnt = 0u;
      __syncthreads();
      for (unsigned base = 0; base < bb_tot; base += kFilterBlock) {
        const unsigned i = base + tid;
        const uint64_t key = i < bb_tot ? stg[i] : 0ull;
        const bool w = i < bb_tot && key >= kap;
        const unsigned slot = warp_append_slot(&s_cnt, w);
        if (w && slot < r) write_winner(fp, rg, row, static_cast<int64_t>(k), bb_start + slot, key, 0ull);
      }
    }
    TK_RG(8);
    __syncthreads();  // the shared arrays are reused by the next selection
    TK_RG(9);
    return true;
  }

  // ---- the block's slice, cached; the base and the digit of the partition
  if (regions) load_slice();
  const unsigned long long R = s_words[0];
  int64_t n = R < static_cast<unsigned long long>(fp.cap) ? static_cast<int64_t>(R) : fp.cap;
  // relaxed recall: a row returned short holds sentinel keys up to slot k
  // (the fallback's decision, recomputed here from the same words)
  uint64_t pad_below = 0ull;
  if (fs.relax_tau && !a.fb.force && R < k) {
    const uint64_t rtau = s_words[1];
    if (rtau >= k) {
      n = static_cast<int64_t>(k);
      pad_below = rtau;
    }
  }
  // the valid keys of this slice: [sb, min(se, n))
  const int cn = static_cast<int>(n <= sb ? 0 : (n < se ? n - sb : se - sb));
  uint64_t kmin, pmask1;
  int shift1;
  const uint64_t prefix1 = 0ull;
  if (fast) {
    // digits of key - tau with the filter's shift; the cache holds key - tau
    kmin = s_words[2];
    shift1 = survivor_shift(kmin, s_words[3]);
    pmask1 = shift1 + kPartDigit >= 64 ? 0ull : (~0ull << (shift1 + kPartDigit));
#pragma unroll
    for (int q = 0; q < kSliceLoads; ++q) {
      const int i = tid + q * kFilterBlock;
      if (i < cn) cache[i] = kv[q] - kmin;
    }
    __syncthreads();
    TK_RG(3);
  } else {
    unsigned long long mn = ~0ull, mx = 0ull;
#pragma unroll
    for (int q = 0; q < kSliceLoads; ++q) {
      const int i = tid + q * kFilterBlock;
      if (i < cn) {
        cache[i] = kv[q];
        mn = kv[q] < mn ? kv[q] : mn;
        mx = kv[q] > mx ? kv[q] : mx;
      }
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
    if (!grid_barrier(fs)) return false;
    TK_RG(4);
    // Digits are taken of key - kmin: 2048 equal slices of the keys' range.
    // (Digits of the keys themselves below their top varying bit leave only a
    // few non-empty bins when the candidates' values cross a power of two.)
    // The cache holds key - kmin from here on; the order is the same.
    kmin = ~__ldcg(g_nmin);
    const uint64_t span = __ldcg(g_max) - kmin;
    const int hb = span ? 63 - __clzll(static_cast<long long>(span)) : 0;
    pmask1 = hb >= 63 ? 0ull : (~0ull << (hb + 1));
    shift1 = hb >= kPartDigit - 1 ? hb - (kPartDigit - 1) : 0;
    for (int i = tid; i < cn; i += kFilterBlock) cache[i] -= kmin;
    __syncthreads();
  }
  auto bin_of = [&](uint64_t key) { return kPartDM - static_cast<unsigned>((key >> shift1) & kPartDM); };

  // ---- first digit: this block's histogram, its range inside each bin
  for (int i = tid; i < kRefineGridBins; i += kFilterBlock) mine[i] = 0u;
  __syncthreads();
  for (int i = tid; i < cn; i += kFilterBlock) atomicAdd(&mine[bin_of(cache[i])], 1u);
  __syncthreads();
  {
    // every atomic of the thread in flight at once (each returns this
    // block's offset inside one bin)
    unsigned c[kPartPer], r[kPartPer];
#pragma unroll
    for (int q = 0; q < kPartPer; ++q) c[q] = mine[tid + q * kFilterBlock];
#pragma unroll
    for (int q = 0; q < kPartPer; ++q) r[q] = c[q] ? atomicAdd(g_lev + tid + q * kFilterBlock, c[q]) : 0u;
#pragma unroll
    for (int q = 0; q < kPartPer; ++q) cur[tid + q * kFilterBlock] = r[q];
  }
  TK_RG(5);
  if (!fast) {
    // the totals of every block's histogram
    if (!grid_barrier(fs)) return false;
    TK_RG(6);
    if (!find_rank_bin(g_lev, k, bst, s_ws, s_info)) {
      if (tid == 0) atomicCAS(fs.status, kDevOk, kDevBadState);
      return false;
    }
    bb = s_info[0];
    bb_start = s_info[1];
    bb_tot = s_info[2];
  } else {
    __syncthreads();  // cur is complete
  }
  TK_RG(7);
  // Unsorted output: only winners are written.  From the filter's histogram,
  // when the boundary bin is small, the bins above it are written straight
  // out and the boundary bin is placed whole in the exchange buffer; the
  // last block to finish ranks it (no grid barrier).  Otherwise further
  // digits find the exact k-th key first, one grid barrier each.
  const bool ufinish = rg.unsorted && fast && bb_tot <= static_cast<unsigned>(kPartCache);
  const bool whole = ufinish || (!rg.unsorted && (fast || static_cast<int64_t>(bb_start) + bb_tot <= rg.xstride));
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
      if (!grid_barrier(fs)) return false;
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
    if (pos >= xend) continue;
    if (rg.unsorted && !(ufinish && pos >= bb_start)) {
      write_winner(fp, rg, row, static_cast<int64_t>(k), pos, key + kmin, pad_below);
    } else {
      xb[pos] = key + kmin;
    }
  }
  if (ufinish) {
    // the last block to finish placing takes the top (k - bb_start) keys of
    // the boundary bin (distinct keys: exactly that many are >= the one of
    // that rank) to the places after the bins above it
    __shared__ int s_last;
    __shared__ unsigned long long s_tmp[32];
    __shared__ unsigned long long s_rinfo[3];
    __shared__ unsigned s_cnt;
    __shared__ uint64_t s_kappa;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(ctl + kRefineGridTicketWord, 1u) + 1u == gridDim.x ? 1 : 0;
    __syncthreads();
    if (s_last) {
      __threadfence();
      const unsigned r = static_cast<unsigned>(k) - bb_start;
      for (unsigned i = tid; i < bb_tot; i += kFilterBlock) stg[i] = __ldcg(xb + bb_start + i);
      __syncthreads();
      bucket_kth<kFilterBlock>(stg, bb_tot, r, mine, s_tmp, s_rinfo, &s_cnt, &s_kappa);
      __syncthreads();
      const uint64_t kap = s_kappa;
      if (tid == 0) s_cnt = 0u;
      __syncthreads();
      for (unsigned base = 0; base < bb_tot; base += kFilterBlock) {
        const unsigned i = base + tid;
        const uint64_t key = i < bb_tot ? stg[i] : 0ull;
        const bool w = i < bb_tot && key >= kap;
        const unsigned slot = warp_append_slot(&s_cnt, w);
        if (w && slot < r) write_winner(fp, rg, row, static_cast<int64_t>(k), bb_start + slot, key, 0ull);
      }
    }
  }
  if (!rg.unsorted) {
    // the bin sort's view of the partition, written by every block (each
    // holds the same bin starts): a slice of the starts and some chunks'
    // descriptors each, the digit description by block 0
    unsigned* bo = rg.binfo + row * binfo_words(static_cast<int64_t>(k));
    const int per = (kRefineGridBins + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    if (tid < per && static_cast<int>(blockIdx.x) * per + tid < kRefineGridBins)
      bo[blockIdx.x * per + tid] = bst[blockIdx.x * per + tid];
    publish_chunks(bst, xend, static_cast<int64_t>(k), bo + kRefineGridBins + kBinfoHeaderWords,
                   static_cast<int>(blockIdx.x) + tid * static_cast<int>(gridDim.x),
                   static_cast<int>(gridDim.x) * kFilterBlock);
  }
  if (blockIdx.x == 0 && !rg.unsorted) {
    unsigned* bo = rg.binfo + row * binfo_words(static_cast<int64_t>(k));
    if (tid == 0) {
      bo[kRefineGridBins] = static_cast<unsigned>(prefix1);
      bo[kRefineGridBins + 1] = static_cast<unsigned>(prefix1 >> 32);
      bo[kRefineGridBins + 2] = static_cast<unsigned>(pmask1);
      bo[kRefineGridBins + 3] = static_cast<unsigned>(pmask1 >> 32);
      bo[kRefineGridBins + 4] = static_cast<unsigned>(shift1);
      bo[kRefineGridBins + 5] = xend;
      bo[kRefineGridBins + 6] = static_cast<unsigned>(kmin);  // digits are of key - kmin
      bo[kRefineGridBins + 7] = static_cast<unsigned>(kmin >> 32);
      bo[kRefineGridBins + 8] = 0u;  // the keys are in the exchange buffer
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
  if (missed > 0 && !grid_barrier(a.fb.fs)) return;
  uint64_t* cache = &stage[0][0];
  const bool hist_ok = rg.tau != nullptr && missed == 0;
  for (int64_t row = 0; row < a.fb.fp.nsel; ++row)
    if (!partition_row(a, row, cache, part_smem, hist_ok)) return;
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
  cfg.numAttrs = pdl_edge(kPdlGridRefine) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, refine_grid_kernel<DT, LARGEST, VEC>, args);
}

template <int DT, bool LARGEST, int VEC>
int64_t refine_grid_capacity_t() {
  return static_cast<int64_t>(refine_grid_blocks<DT, LARGEST, VEC>()) * kPartCache;
}

}  // namespace

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
  RefineGridParams a{{{p.x, p.nsel, p.len, p.ib, p.flip, fs.tau_exact, cap, buf, counts, Divider{}}, k, force, fs},
                     rg};
  if (rg.unsorted && (!rg.out_vals || !rg.out_idx)) return cudaErrorInvalidValue;
  a.rg.unsorted = rg.unsorted ? (p.dtype == kF32 ? 1 : 2) : 0;  // the output's element type
  const bool largest = p.flip == 0;
  if (p.dtype == kF32) {
    if (p.vec_ok) return largest ? launch_refine_grid_t<kF32, true, 4>(a, st) : launch_refine_grid_t<kF32, false, 4>(a, st);
    return largest ? launch_refine_grid_t<kF32, true, 1>(a, st) : launch_refine_grid_t<kF32, false, 1>(a, st);
  }
  if (p.vec_ok) return largest ? launch_refine_grid_t<kBF16, true, 8>(a, st) : launch_refine_grid_t<kBF16, false, 8>(a, st);
  return largest ? launch_refine_grid_t<kBF16, true, 1>(a, st) : launch_refine_grid_t<kBF16, false, 1>(a, st);
}

#ifdef TK_PHASE_TIMING
TK_TIMELINE_ACCESSOR(debug_timeline_fallback)
int debug_refine_grid_ns(unsigned long long* out) {
  if (cudaMemcpyFromSymbol(out, g_rg_ns, sizeof(g_rg_ns)) != cudaSuccess) return -3;
  return cudaMemcpyFromSymbol(out + 16, g_fb_ns, sizeof(g_fb_ns)) == cudaSuccess ? 0 : -3;
}
#endif

}  // namespace tk
