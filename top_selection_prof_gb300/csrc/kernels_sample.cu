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
#include "common.cuh"
#include "engine.h"

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
    }
  }
  if (hist_add) {
    for (int i = threadIdx.x; i < kSampleHistBins; i += blockDim.x) sh[i] = 0u;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < kSampleHistBins;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
      hist_zero[static_cast<int64_t>(row) * kSampleHistBins + i] = 0u;
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
#endif

}  // namespace tk
