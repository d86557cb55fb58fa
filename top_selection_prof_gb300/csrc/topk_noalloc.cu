// topk_select_noalloc: the same selection as topk_select / topk_select_global,
// with every piece of scratch memory taken from one fixed device array that is
// part of the library image, so the call never allocates device memory.
//
// Who needs it: callers that must not allocate once they are running -- for
// example a serving loop whose device memory is entirely owned by another
// allocator (a framework's caching allocator that has reserved nearly all of
// HBM, where a hidden cudaMalloc can fail or fragment memory), or latency-
// critical code that cannot afford cudaMalloc's implicit device
// synchronisation and unpredictable cost.  They pass inputs and outputs as
// usual; the library's own workspace pool is not touched.
//
// The scratch array is a file-scope __device__ array of kNoAllocScratchBytes.
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; that first call should therefore come before any
// stream capture.  The selection itself is the pooled entry points' pipeline
// (select_with_fixed_scratch in topk_api.cu): the same kernels, the same
// choice of path, with the array as its workspace.  The array is zero when
// the module loads, and the pipeline keeps the regions that must start at
// zero clean between calls (alternating copies cleared by each call, and the
// header and counters reset by each call's first kernel).  All calls share
// the one array and it keeps the last call's contents; each device has its
// own copy, but on one device calls whose work overlaps on the GPU (for
// example calls issued to two streams with nothing ordering them) race on it
// and give wrong results: order such calls on one stream.
//
// The Prof-K method itself has no counterpart of this entry point; it is an
// engineering variant of the library's own pipeline.
#include <cstdint>
#include <map>
#include <mutex>

#include "../../include/topk.h"
#include "engine.h"

namespace tk {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct DeviceScratch {
  void* addr = nullptr;
  ScratchCounters counters;  // which alternating copies the next call uses
};
std::mutex g_addr_mu;
std::map<int, DeviceScratch> g_dev;  // device ordinal -> the array's address and counters

cudaError_t scratch_of_device(FixedScratch* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  DeviceScratch& d = g_dev[dev];
  if (!d.addr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    d.addr = p;
  }
  out->base = d.addr;
  out->bytes = kNoAllocScratchBytes;
  out->counters = &d.counters;  // (std::map nodes do not move)
  return cudaSuccess;
}

}  // namespace
}  // namespace tk

using namespace tk;

extern "C" int topk_select_noalloc(const void* x, int dtype, int64_t rows, int64_t n, int64_t k,
                                   int largest, double eps, void* out_vals, int64_t* out_idx,
                                   int global, void* stream) {
  // (arguments are checked by the pipeline before anything touches the device)
  if (dtype != TOPK_F32 && dtype != TOPK_BF16) return TOPK_EINVAL;
  if (rows < 0 || n < 1 || k < 1 || !(eps >= 0.0 && eps < 1.0)) return TOPK_EINVAL;
  if (rows == 0) return TOPK_OK;
  FixedScratch fs{};
  const cudaError_t e = scratch_of_device(&fs);
  if (e != cudaSuccess) return TOPK_ECUDA;
  return select_with_fixed_scratch(x, dtype, rows, n, k, largest, eps, out_vals, out_idx,
                                   static_cast<cudaStream_t>(stream), global != 0, fs);
}
