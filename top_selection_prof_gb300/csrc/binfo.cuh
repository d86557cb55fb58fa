// The bin information a partition publishes for the bin sort (kernels_select.cu),
// shared by its two producers: the refinement cluster (kernels_select.cu) and
// the grid refinement (kernels_fallback.cu).  Per selection, binfo_words(k)
// words: the kRefineGridBins bin starts (bins in descending key order),
// kBinfoHeaderWords words describing the first digit (prefix, mask, shift,
// the end of the placed keys, the base the digits are relative to; word 8:
// 1 when the keys stayed in the filter's bin regions, whose bins are these
// digits, and nothing else was published), then one descriptor of
// kChunkWords words per chunk of kBinSortChunk output places: the first and
// the last bin the chunk's places fall in, with the start and end of each,
// so that a bin-sort block reads its bins with one round of loads instead of
// every bin start.
#pragma once

#include "common.cuh"
#include "engine.h"

namespace tk {
namespace {

constexpr int kChunkWords = 6;

// Writes the descriptors of chunks c0, c0 + cstep, ... of the k output
// places to dst (kChunkWords each).  bst: the bin starts (shared memory,
// non-decreasing, bst[0] = 0); xend: the end of the placed keys (>= k).
__device__ void publish_chunks(const unsigned* bst, unsigned xend, int64_t k, unsigned* dst, int c0, int cstep) {
  constexpr unsigned NB = static_cast<unsigned>(kRefineGridBins);
  const int nch = static_cast<int>((k + kBinSortChunk - 1) / kBinSortChunk);
  auto bin_end = [&](unsigned b) {
    const unsigned e = b + 1 < NB ? bst[b + 1] : xend;
    return e < xend ? e : xend;
  };
  auto find = [&](unsigned p) {  // the last bin whose start is <= p: the bin holding place p
    unsigned lo = 0, hi = NB - 1;
    while (lo < hi) {
      const unsigned mid = (lo + hi + 1) / 2;
      if (bst[mid] <= p) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  for (int c = c0; c < nch; c += cstep) {
    const int64_t p0 = static_cast<int64_t>(c) * kBinSortChunk;
    const int64_t p1 = (p0 + kBinSortChunk < k ? p0 + kBinSortChunk : k) - 1;
    const unsigned bf = find(static_cast<unsigned>(p0)), bl = find(static_cast<unsigned>(p1));
    unsigned* d = dst + static_cast<int64_t>(c) * kChunkWords;
    d[0] = bf;
    d[1] = bl;
    d[2] = bst[bf];
    d[3] = bin_end(bf);
    d[4] = bst[bl];
    d[5] = bin_end(bl);
  }
}

}  // namespace
}  // namespace tk
