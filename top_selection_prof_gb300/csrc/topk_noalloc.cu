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
// stream capture.  All calls share the one array and it keeps the last call's
// contents: the kernels reset the counters they need (the sampler clears the
// survivor counts and the fallback's barrier and status words; the other paths
// clear them with cudaMemsetAsync).  Each device has its own copy of the
// array, but on one device calls whose work overlaps on the GPU (for example
// calls issued to two streams with nothing ordering them) race on it and give
// wrong results: order such calls on one stream.
//
// The Prof-K method itself has no counterpart of this entry point; it is an
// engineering variant of the library's own pipeline.
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>

#include "../../include/topk.h"
#include "common.cuh"
#include "engine.h"

namespace tk {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_addr_mu;
std::map<int, void*> g_addr;  // device ordinal -> device address of g_noalloc_scratch

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  auto it = g_addr.find(dev);
  if (it != g_addr.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  g_addr[dev] = p;
  *out = p;
  return cudaSuccess;
}

size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

int bits_for(int64_t len) {
  int b = 1;
  while (b < 63 && (int64_t(1) << b) < len) ++b;
  return b;
}

int to_status(cudaError_t e) {
  if (e == cudaSuccess) return TOPK_OK;
  if (e == cudaErrorMemoryAllocation) return TOPK_ENOMEM;
  return TOPK_ECUDA;
}

}  // namespace
}  // namespace tk

using namespace tk;

extern "C" int topk_select_noalloc(const void* x, int dtype, int64_t rows, int64_t n, int64_t k,
                                   int largest, double eps, void* out_vals, int64_t* out_idx,
                                   int global, void* stream) {
  if (dtype != TOPK_F32 && dtype != TOPK_BF16) return TOPK_EINVAL;
  if (rows < 0 || n < 1 || k < 1 || !(eps >= 0.0 && eps < 1.0)) return TOPK_EINVAL;
  if (rows == 0) return TOPK_OK;
  if (!x || !out_vals || !out_idx) return TOPK_EINVAL;
  if (global && rows > INT64_MAX / n) return TOPK_EUNSUPPORTED;
  const int64_t len = global ? rows * n : n;
  const int64_t nsel = global ? 1 : rows;
  if (k > len) return TOPK_EINVAL;
  if (!global && n >= (int64_t(1) << 31)) return TOPK_EUNSUPPORTED;
  if (len > (dtype == TOPK_F32 ? (int64_t(1) << 32) : (int64_t(1) << 48))) return TOPK_EUNSUPPORTED;
  if (k > select_max_k()) return TOPK_EUNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  Problem p;
  p.x = x;
  p.dtype = dtype;
  p.nsel = nsel;
  p.len = len;
  p.ib = bits_for(len);
  p.flip = largest ? 0u : (dtype == TOPK_F32 ? 0xffffffffu : 0xffffu);
  p.vec_ok = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (len % (dtype == TOPK_F32 ? 4 : 8) == 0);

  // path choice: as the pooled entry points
  int64_t S = 0, t = 0, M = 0;
  bool profk = false;
  if (eps > 0.0) {
    ParamRule pr;
    if (choose_params(len, k, eps, pr, &S, &t, &M))
      profk = t >= 1 && t <= S && 2 * S < len && 2 * M <= len && M >= k && nsel <= 65535;
  }
  int sms = 1, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int path = profk ? TOPK_PATH_PROFK
                         : ((len <= (int64_t(1) << 22) || nsel >= sms) ? TOPK_PATH_DIRECT : TOPK_PATH_EXACT);
  if (path != TOPK_PATH_PROFK) S = t = M = 0;
  const int64_t cap = path == TOPK_PATH_PROFK ? M : k;

  // scratch layout inside the static array
  size_t off = 0;
  const size_t o_hdr = off; off = up256(off + sizeof(DevHeader));
  const size_t o_counts = off; off = up256(off + sizeof(unsigned long long) * nsel);
  const size_t o_rseen = off; off = up256(off + sizeof(unsigned long long) * nsel);
  const size_t o_tau = off; off = up256(off + sizeof(uint64_t) * nsel);
  const size_t o_taux = off; off = up256(off + sizeof(uint64_t) * nsel);
  const size_t o_ghist = off; off = up256(off + sizeof(unsigned) * 8 * 256);
  const size_t o_tiles = off; off = up256(off + sizeof(unsigned) * ((len + kFallbackTile - 1) / kFallbackTile));
  const size_t o_samples = off; off = up256(off + sizeof(uint64_t) * nsel * S);
  const size_t o_buf = off; off = up256(off + sizeof(uint64_t) * nsel * cap);
  const size_t o_xbuf = off; off = up256(off + sizeof(uint64_t) * 2 * nsel * k);
  if (path == TOPK_PATH_DIRECT && rows_supported(p, k)) {
    // short rows: one block per row, the row in registers, no scratch at all
    const cudaError_t er = launch_rows(p, k, out_vals, out_idx, nullptr, st);
    return er == cudaSuccess ? TOPK_OK : to_status(er);
  }
  if (path == TOPK_PATH_DIRECT) {
    // the direct path needs only the header and the sort's exchange buffer
    if (up256(sizeof(DevHeader)) + sizeof(uint64_t) * 2 * nsel * k > kNoAllocScratchBytes)
      return TOPK_EUNSUPPORTED;
  } else if (off > kNoAllocScratchBytes) {
    return TOPK_EUNSUPPORTED;
  }

  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return to_status(e);
  char* base = static_cast<char*>(scratch);
  DevHeader* hdr = reinterpret_cast<DevHeader*>(base + o_hdr);

#define NA_TRY(expr)                       \
  do {                                     \
    const cudaError_t _e = (expr);         \
    if (_e != cudaSuccess) return to_status(_e); \
  } while (0)

  if (path == TOPK_PATH_DIRECT) {
    NA_TRY(cudaMemsetAsync(&hdr->status, 0, sizeof(int), st));
    SelectJob job{};
    job.r = k;
    job.want_topk = true;
    job.out_vals = out_vals;
    job.out_idx = out_idx;
    job.status = &hdr->status;
    job.xbuf = reinterpret_cast<uint64_t*>(base + up256(sizeof(DevHeader)));
    NA_TRY(launch_select(p, job, len, nullptr, st));
    return TOPK_OK;
  }

  auto* counts = reinterpret_cast<unsigned long long*>(base + o_counts);
  auto* tau = reinterpret_cast<uint64_t*>(base + o_tau);
  auto* buf = reinterpret_cast<uint64_t*>(base + o_buf);
  FallbackScratch fs{reinterpret_cast<unsigned*>(base + o_ghist), reinterpret_cast<unsigned*>(base + o_tiles),
                     hdr->barrier, &hdr->status, reinterpret_cast<unsigned long long*>(base + o_rseen),
                     &hdr->misses, reinterpret_cast<uint64_t*>(base + o_taux)};
  bool refine_checks = false;
  if (path == TOPK_PATH_PROFK) {
    static uint64_t calls = 0;  // Philox call counter of this entry point
    const uint64_t counter = __atomic_fetch_add(&calls, 1, __ATOMIC_RELAXED);
    auto* samples = reinterpret_cast<uint64_t*>(base + o_samples);
    NA_TRY(launch_sample(p, S, 0x243F6A8885A308D3ull, counter, samples, counts, hdr, nullptr, nullptr, st));
    SelectJob tj{};
    tj.keys = samples;
    tj.key_stride = S;
    tj.r = t;
    tj.tau_out = tau;
    tj.status = &hdr->status;
    int tau_cluster = 0;
    NA_TRY(launch_select(p, tj, S, &tau_cluster, st));
    NA_TRY(launch_filter(p, tau, cap, buf, counts, overlap_sms(tau_cluster, nsel), st));
    refine_checks = miss_in_refine(p, k, t, S, eps);
    if (!refine_checks) NA_TRY(launch_fallback(p, k, cap, buf, counts, fs, 0, st));
  } else {
    NA_TRY(cudaMemsetAsync(base, 0, o_tau, st));  // header, counts, r_seen
    NA_TRY(launch_fallback(p, k, cap, buf, counts, fs, 1, st));
  }
  SelectJob rj{};
  rj.keys = buf;
  rj.key_stride = cap;
  rj.counts = counts;
  rj.r = k;
  rj.want_topk = true;
  rj.out_vals = out_vals;
  rj.out_idx = out_idx;
  rj.status = &hdr->status;
  rj.xbuf = reinterpret_cast<uint64_t*>(base + o_xbuf);
  if (refine_checks) {  // the refinement checks for a miss itself
    rj.check_miss = true;
    rj.r_seen = reinterpret_cast<unsigned long long*>(base + o_rseen);
    rj.misses = &hdr->misses;
  }
  NA_TRY(launch_select(p, rj, cap, nullptr, st));
#undef NA_TRY
  return TOPK_OK;
}
