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
                          unsigned long long* counts, int reserved_sms, cudaStream_t st, unsigned* refine_ctl) {
  FilterParams fp{p.x, p.nsel, p.len, p.ib, p.flip, tau, cap, buf, counts, Divider{}};
  fp.refine_ctl = refine_ctl;
  const bool largest = p.flip == 0;
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
