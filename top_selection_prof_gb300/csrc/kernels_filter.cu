// Stage 3 of Prof-K (section 3, "Filtering").
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
// written.  The tile loop itself is in filter_core.cuh (the fallback re-runs it).
//
// A single selection with 16-byte aligned data (one long row, or BatchTopK
// over the flattened batch) takes filter_ring_kernel instead: there the TMA
// engine streams the block's tiles into a ring of shared-memory stages
// (cp.async.bulk completing on an mbarrier per stage) and the threads test
// them from shared memory.  The loads no longer wait on the threads' test
// work, and the first stages are requested before tau exists -- the input is
// the caller's, not the preceding grid's -- so they arrive while the sampling
// grid finishes.  A plain read of 1 GiB measured ~7.2-7.3 TB/s through such a
// ring against ~6.7-7.1 TB/s with 16-byte loads from registers.
#include "filter_core.cuh"

namespace tk {

namespace {

template <int DT, bool LARGEST, int VEC, bool HIST>
__global__ void __launch_bounds__(kFilterBlock) filter_kernel(FilterParams fp) {
  __shared__ uint64_t stage[kFilterBlock / 32][kWarpStage];
  __shared__ unsigned stage_n[kFilterBlock / 32];
  __shared__ unsigned sh_hist[HIST ? kRefineGridBins : 1];
  __shared__ uint4 queue_v[kFilterBlock / 32][kGroupQueue];
  __shared__ int64_t queue_pos[kFilterBlock / 32][kGroupQueue];
  TK_TL_BEGIN(2);
  if (HIST) {
    for (int i = threadIdx.x; i < kRefineGridBins; i += kFilterBlock) sh_hist[i] = 0u;
    __syncthreads();
  }
  grid_dependency_wait();  // tau and the zeroed counters come from the previous grid
  // the next grid may begin launching: its blocks take the SMs this grid's
  // blocks leave and wait there until this grid has finished
  grid_launch_dependents();
  if ((threadIdx.x & 31) == 0) stage_n[threadIdx.x >> 5] = 0u;
  __syncwarp();
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  const int64_t ntiles = fp.nsel * ((fp.len + kTile - 1) / kTile);
  const Stage st{stage[threadIdx.x >> 5], &stage_n[threadIdx.x >> 5]};
  const GroupQueue q{queue_v[threadIdx.x >> 5], queue_pos[threadIdx.x >> 5]};
  filter_tiles<DT, LARGEST, VEC, HIST>(fp, blockIdx.x, ntiles, gridDim.x, st, sh_hist, &q);
  TK_TL_END(2);
}

// Ring of tiles in shared memory: kRingStages stages of one tile each (16 KB),
// two blocks per SM (128 KB of stages per SM, ~100 KB of them in flight).
constexpr int kRingStages = 4;
constexpr unsigned kRingStageBytes = kFilterBlock * kFilterUnroll * 16;
constexpr int kRingBlocksPerSm = 2;
constexpr int kRingSmemBytes = kRingStages * static_cast<int>(kRingStageBytes);

template <int DT, bool LARGEST, bool HIST>
__global__ void __launch_bounds__(kFilterBlock, kRingBlocksPerSm) filter_ring_kernel(FilterParams fp) {
  using T = typename Dt<DT>::storage;
  constexpr int VEC = Dt<DT>::kVec;
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[kRingStages];
  __shared__ uint64_t stage[kFilterBlock / 32][kWarpStage];
  __shared__ unsigned stage_n[kFilterBlock / 32];
  __shared__ unsigned sh_hist[HIST ? kRefineGridBins : 1];
  __shared__ uint4 queue_v[kFilterBlock / 32][kGroupQueue];
  __shared__ int64_t queue_pos[kFilterBlock / 32][kGroupQueue];
  __shared__ uint64_t s_words[2];
  __shared__ int s_abort;
  TK_TL_BEGIN(2);
  const int tid = threadIdx.x;
  // the full tiles, dealt out by block index; the partial last one (if any)
  // goes to the block next in that order, after its full tiles
  const int64_t nfull = fp.len / kTile;
  const int64_t first = blockIdx.x, step = gridDim.x;
  const int64_t mine = first < nfull ? (nfull - 1 - first) / step + 1 : 0;
  const unsigned char* xb = static_cast<const unsigned char*>(fp.x);
  const uint64_t pol = l2_evict_first_policy();
  auto issue = [&](int64_t i) {  // this block's i-th tile into stage i % kRingStages
    const int s = static_cast<int>(i % kRingStages);
    mbar_expect_tx(&full[s], kRingStageBytes);
    bulk_copy_g2s(ring + s * kRingStageBytes, xb + (first + i * step) * kTile * static_cast<int64_t>(sizeof(T)),
                  kRingStageBytes, &full[s], pol);
  };
  if (tid == 0) {
    for (int s = 0; s < kRingStages; ++s) mbar_init(&full[s], 1u);
    s_abort = 0;
    s_filter_block_bad = 0;
    // the input does not come from the preceding grid: these copies may
    // start before it has finished (half the ring: the rest of the stream
    // would queue in front of that grid's last loads)
    for (int64_t i = 0; i < kRingStages / 2 && i < mine; ++i) issue(i);
    // where the preceding grid leaves HBM idle, the block's next tiles go to
    // L2 meanwhile, and their ring copies later hit there (at most half its
    // tiles: more crowds L2 and costs more than it saves)
    const int64_t ahead = fp.l2_ahead < mine / 2 ? fp.l2_ahead : mine / 2;
    for (int64_t i = kRingStages / 2; i < kRingStages / 2 + ahead && i < mine; ++i)
      bulk_prefetch_l2(xb + (first + i * step) * kTile * static_cast<int64_t>(sizeof(T)), kRingStageBytes);
  }
  if (HIST)
    for (int i = tid; i < kRefineGridBins; i += kFilterBlock) sh_hist[i] = 0u;
  if ((tid & 31) == 0) stage_n[tid >> 5] = 0u;
  if (fp.refine_ctl_next)  // the next call's control words (no kernel of this call uses them)
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kFilterBlock + tid; i < kRefineGridMaxSel * kRefineGridCtlWords;
         i += static_cast<int64_t>(gridDim.x) * kFilterBlock)
      fp.refine_ctl_next[i] = 0u;
  grid_dependency_wait();  // tau and the zeroed counters come from the previous grid
  grid_launch_dependents();
  if (tid == 0) {
    for (int64_t i = kRingStages / 2; i < kRingStages && i < mine; ++i) issue(i);
    s_words[0] = __ldcg(fp.tau);
    if (HIST) s_words[1] = sampled_kmax(fp.refine_ctl, 0);
  }
  __syncthreads();
  RowTau t = row_tau<DT>(s_words[0], fp.ib, fp.flip);
  t.hshift = HIST ? survivor_shift(t.key, s_words[1]) : 0;
  const Stage st{stage[tid >> 5], &stage_n[tid >> 5]};
  const GroupQueue q{queue_v[tid >> 5], queue_pos[tid >> 5]};
  unsigned qn = 0;
  int64_t i = 0;
  for (; i < mine; ++i) {
    const int s = static_cast<int>(i % kRingStages);
    if (!mbar_wait(&full[s], static_cast<unsigned>(i / kRingStages) & 1u)) s_abort = 1;
    const uint4* src = reinterpret_cast<const uint4*>(ring + s * kRingStageBytes);
    uint4 v[kFilterUnroll];
#pragma unroll
    for (int u = 0; u < kFilterUnroll; ++u) v[u] = src[u * kFilterBlock + tid];
    __syncthreads();  // the stage sits in registers everywhere: it may be refilled
    if (s_abort) break;
    if (tid == 0 && i + kRingStages < mine) {
      fence_proxy_async_smem();  // the generic reads above before the copy's writes
      issue(i + kRingStages);
    }
    single_tile_groups<DT, LARGEST, VEC, HIST>(v, (first + i * step) * kTile + tid * VEC, t, fp, st, sh_hist, q, qn);
  }
  if (s_abort) {
    // a copy did not land in time: report it, give the copies still in
    // flight (they write this block's shared memory) a last bounded wait and
    // stop
    if (tid == 0) {
      if (fp.status) atomicCAS(fp.status, kDevOk, kDevTimeout);
      for (int64_t j = i; j < i + kRingStages && j < mine; ++j)
        mbar_wait(&full[j % kRingStages], static_cast<unsigned>(j / kRingStages) & 1u);
    }
    __syncthreads();
    return;
  }
  if (qn) drain_groups<DT, LARGEST, VEC, HIST>(q, 0u, qn, t, fp, st, 0, sh_hist);
  const int64_t ntiles = (fp.len + kTile - 1) / kTile;
  if (ntiles > nfull && nfull % step == first) {
    // the partial last tile: whole 16-byte groups (the length is a multiple
    // of the group), each tested in place
    const T* x = static_cast<const T*>(fp.x);
#pragma unroll
    for (int u = 0; u < kFilterUnroll; ++u) {
      const int64_t pos = nfull * kTile + (static_cast<int64_t>(u) * kFilterBlock + tid) * VEC;
      if (pos < fp.len) test_group<DT, LARGEST, VEC, HIST>(load_group<DT, VEC>(x + pos, pol), pos, t, fp, st, 0, sh_hist);
    }
  }
  __syncthreads();  // every warp's stage, the block's counts and its flag are final
  if (HIST && fp.region && s_filter_block_bad) {
    // some survivors of this block left its stages: the regions are marked
    // incomplete, so only the histogram is added
    hist_flush(sh_hist, fp, 0);
  } else if (HIST && fp.region) {
    // Bin regions: one returning atomic per non-empty bin adds this block's
    // counts to the histogram and returns where its keys start in each
    // bin's region; then every survivor (all still in the warps' stages)
    // goes to its bin's region.  A bin that would overflow its region marks
    // the regions incomplete.
    unsigned* g = fp.refine_ctl + kRefineGridFilterHist;
    unsigned* cur = reinterpret_cast<unsigned*>(queue_v);  // (free now: 2048 counters)
    static_assert(sizeof(queue_v) >= sizeof(unsigned) * kRefineGridBins, "bin cursors");
    constexpr int kPer = kRefineGridBins / kFilterBlock;
    unsigned c[kPer], r[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) c[j] = sh_hist[tid + j * kFilterBlock];
#pragma unroll
    for (int j = 0; j < kPer; ++j) r[j] = c[j] ? atomicAdd(g + tid + j * kFilterBlock, c[j]) : 0u;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      sh_hist[tid + j * kFilterBlock] = r[j];
      cur[tid + j * kFilterBlock] = 0u;
    }
    __syncthreads();
    bool over = false;
    for (int idx = tid; idx < (kFilterBlock / 32) * kWarpStage; idx += kFilterBlock) {
      const int w = idx / kWarpStage, j = idx % kWarpStage;
      const unsigned nw = stage_n[w] < static_cast<unsigned>(kWarpStage) ? stage_n[w] : kWarpStage;
      if (static_cast<unsigned>(j) < nw) {
        const uint64_t key = stage[w][j];
        const unsigned b = survivor_bin(key, t.key, t.hshift);
        const unsigned slot = sh_hist[b] + atomicAdd(&cur[b], 1u);
        if (slot < static_cast<unsigned>(kBinRegionCap)) fp.region[static_cast<int64_t>(b) * kBinRegionCap + slot] = key;
        else over = true;
      }
    }
    if (over) *binned_bad_word(fp, 0) = 1u;
    __syncthreads();  // (stage_flush below clears the stage counts)
  }
  stage_flush(st, 0, fp.cap, fp.buf, fp.counts);
  if (HIST && !fp.region) hist_flush(sh_hist, fp, 0);
  TK_TL_END(2);
}

template <int DT, bool LARGEST, bool HIST>
cudaError_t launch_filter_ring(const FilterParams& fp, bool pdl, cudaStream_t st) {
  constexpr int VEC = Dt<DT>::kVec;
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  static int sms = 0, per_sm = 0;
  if (!sms) {
    int dev = 0, n = 0, b = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    const cudaError_t e = cudaFuncSetAttribute(filter_ring_kernel<DT, LARGEST, HIST>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemBytes);
    if (e != cudaSuccess) return e;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, filter_ring_kernel<DT, LARGEST, HIST>, kFilterBlock,
                                                  kRingSmemBytes);
    per_sm = b < 1 ? 1 : b;
    sms = n < 1 ? 1 : n;
  }
  const int64_t ntiles = (fp.len + kTile - 1) / kTile;
  FilterParams args = fp;
  args.tiles_per_row = make_divider(static_cast<uint64_t>(ntiles));
  int64_t grid = static_cast<int64_t>(sms) * per_sm;
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kFilterBlock, 1, 1);
  cfg.dynamicSmemBytes = kRingSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, filter_ring_kernel<DT, LARGEST, HIST>, args);
}

// One full wave: SMs x resident blocks per SM, less the SMs held by the
// preceding grid when this launch may overlap it (programmatic dependent
// launch): the tiles are dealt out by block index, so every block must start
// at once.
template <int DT, bool LARGEST, int VEC, bool HIST>
int filter_grid_size(int reserved_sms) {
  static int sms = 0, per_sm = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, filter_kernel<DT, LARGEST, VEC, HIST>, kFilterBlock, 0);
    if (per_sm < 1) per_sm = 1;
  }
  const int usable = sms - reserved_sms > sms / 2 ? sms - reserved_sms : sms / 2;
  return usable * per_sm;
}

template <int DT, bool LARGEST, int VEC, bool HIST>
cudaError_t launch_filter_t(const FilterParams& fp, int reserved_sms, cudaStream_t st) {
  constexpr int64_t kTile = static_cast<int64_t>(kFilterBlock) * kFilterUnroll * VEC;
  const int64_t ntiles = fp.nsel * ((fp.len + kTile - 1) / kTile);
  FilterParams args = fp;
  args.tiles_per_row = make_divider(static_cast<uint64_t>((fp.len + kTile - 1) / kTile));
  const bool pdl = reserved_sms >= 0 && pdl_edge(kPdlFilter);
  int64_t grid = filter_grid_size<DT, LARGEST, VEC, HIST>(pdl ? reserved_sms : 0);
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
  return cudaLaunchKernelEx(&cfg, filter_kernel<DT, LARGEST, VEC, HIST>, args);
}

template <int DT, bool LARGEST, int VEC>
cudaError_t launch_filter_h(const FilterParams& fp, int reserved_sms, cudaStream_t st) {
  return fp.refine_ctl ? launch_filter_t<DT, LARGEST, VEC, true>(fp, reserved_sms, st)
                 : launch_filter_t<DT, LARGEST, VEC, false>(fp, reserved_sms, st);
}

}  // namespace

cudaError_t launch_filter(const Problem& p, const uint64_t* tau, int64_t cap, uint64_t* buf,
                          unsigned long long* counts, int reserved_sms, cudaStream_t st, unsigned* refine_ctl,
                          int* status, uint64_t* region, unsigned* refine_ctl_next, int l2_ahead) {
  FilterParams fp{p.x, p.nsel, p.len, p.ib, p.flip, tau, cap, buf, counts, Divider{}};
  fp.l2_ahead = l2_ahead > 0 ? l2_ahead : 0;
  fp.refine_ctl = refine_ctl;
  fp.status = status;
  // (bin regions: the TMA-ring filter of one selection with the survivor histogram)
  fp.region = (p.nsel == 1 && p.vec_ok && refine_ctl) ? region : nullptr;
  fp.refine_ctl_next = fp.region ? refine_ctl_next : nullptr;
  const bool largest = p.flip == 0;
  if (p.nsel == 1 && p.vec_ok) {
    // (every block of the ring grid may start late: its tiles wait in the
    // ring, so the SMs a preceding grid holds need no reserving)
    const bool pdl = reserved_sms >= 0 && pdl_edge(kPdlFilter);
    const bool h = refine_ctl != nullptr;
    if (p.dtype == kF32)
      return largest ? (h ? launch_filter_ring<kF32, true, true>(fp, pdl, st)
                          : launch_filter_ring<kF32, true, false>(fp, pdl, st))
                     : (h ? launch_filter_ring<kF32, false, true>(fp, pdl, st)
                          : launch_filter_ring<kF32, false, false>(fp, pdl, st));
    return largest ? (h ? launch_filter_ring<kBF16, true, true>(fp, pdl, st)
                        : launch_filter_ring<kBF16, true, false>(fp, pdl, st))
                   : (h ? launch_filter_ring<kBF16, false, true>(fp, pdl, st)
                        : launch_filter_ring<kBF16, false, false>(fp, pdl, st));
  }
  if (p.dtype == kF32) {
    if (p.vec_ok) return largest ? launch_filter_h<kF32, true, 4>(fp, reserved_sms, st)
                                 : launch_filter_h<kF32, false, 4>(fp, reserved_sms, st);
    return largest ? launch_filter_h<kF32, true, 1>(fp, reserved_sms, st)
                   : launch_filter_h<kF32, false, 1>(fp, reserved_sms, st);
  }
  if (p.vec_ok) return largest ? launch_filter_h<kBF16, true, 8>(fp, reserved_sms, st)
                               : launch_filter_h<kBF16, false, 8>(fp, reserved_sms, st);
  return largest ? launch_filter_h<kBF16, true, 1>(fp, reserved_sms, st)
                 : launch_filter_h<kBF16, false, 1>(fp, reserved_sms, st);
}

#ifdef TK_PHASE_TIMING
TK_TIMELINE_ACCESSOR(debug_timeline_filter)
#endif

}  // namespace tk
