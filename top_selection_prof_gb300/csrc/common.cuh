// Device-side building blocks shared by the engine's kernels: the composite
// key, Philox4x32-10, PTX wrappers and the bounded device wait.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tk {

constexpr int kF32 = 0;
constexpr int kBF16 = 1;

// ---------------------------------------------------------------------------
// Order-preserving keys.  Unsigned order of the key == the selection order of
// the value: NaN above everything (all NaNs equal), -0 == +0.  The composite
// key appends the complemented position so that, among equal values, the lower
// position has the larger key -- the index tie-break of "Rank by Counting".
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint32_t order_key_f32(uint32_t u) {
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0xffffffffu;  // NaN
  if (u == 0x80000000u) u = 0u;                              // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__host__ __device__ __forceinline__ uint32_t order_key_bf16(uint32_t h) {
  if ((h & 0x7fffu) > 0x7f80u) return 0xffffu;
  if (h == 0x8000u) h = 0u;
  return (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
}

// Inverse of order_key_* for keys that are neither NaN nor zero (those two do
// not determine the input bits; the caller reads the input instead).
__host__ __device__ __forceinline__ uint32_t value_bits_f32(uint32_t key) {
  return (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
}
__host__ __device__ __forceinline__ uint32_t value_bits_bf16(uint32_t key) {
  return (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
}

template <int DT>
struct Dt;

template <>
struct Dt<kF32> {
  using storage = uint32_t;
  static constexpr int kKeyBits = 32;
  static constexpr uint32_t kKeyMask = 0xffffffffu;
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static uint32_t key(uint32_t u) { return order_key_f32(u); }
  __device__ __forceinline__ static uint32_t bits(uint32_t key) { return value_bits_f32(key); }
  __device__ __forceinline__ static float to_float(uint32_t u) { return __uint_as_float(u); }
  static constexpr uint32_t kZeroKey = 0x80000000u;
  static constexpr uint32_t kNanKey = 0xffffffffu;
};

template <>
struct Dt<kBF16> {
  using storage = uint16_t;
  static constexpr int kKeyBits = 16;
  static constexpr uint32_t kKeyMask = 0xffffu;
  static constexpr int kVec = 8;
  __device__ __forceinline__ static uint32_t key(uint32_t h) { return order_key_bf16(h); }
  __device__ __forceinline__ static uint32_t bits(uint32_t key) { return value_bits_bf16(key); }
  __device__ __forceinline__ static float to_float(uint32_t h) { return __uint_as_float(h << 16); }
  static constexpr uint32_t kZeroKey = 0x8000u;
  static constexpr uint32_t kNanKey = 0xffffu;
};

// Composite key: (value key << b) | (2^b - 1 - position).
__host__ __device__ __forceinline__ uint64_t compose(uint32_t vkey, uint64_t pos, int b) {
  const uint64_t mask = (b >= 64) ? ~0ull : ((1ull << b) - 1ull);
  return (static_cast<uint64_t>(vkey) << b) | (mask - pos);
}
__host__ __device__ __forceinline__ uint64_t position_of(uint64_t ck, int b) {
  const uint64_t mask = (1ull << b) - 1ull;
  return mask - (ck & mask);
}
__host__ __device__ __forceinline__ uint32_t vkey_of(uint64_t ck, int b) {
  return static_cast<uint32_t>(ck >> b);
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11): 10 rounds of two 32x32->64 multiplies,
// key bumped by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}

// Stage-1 draws j = 2*pair and 2*pair + 1 of selection `row`: counter
// (pair, row, call_lo, call_hi), key (seed_lo, seed_hi); the even draw takes
// the 64-bit word (w1 << 32 | w0), the odd one (w3 << 32 | w2); the position
// is floor(word * len / 2^64).
__device__ __forceinline__ void sample_pair(uint2 key, uint2 call, uint32_t row, uint32_t pair, uint64_t len,
                                            uint64_t* p0, uint64_t* p1) {
  const uint4 w = philox4x32_10(make_uint4(pair, row, call.x, call.y), key);
  *p0 = __umul64hi((static_cast<uint64_t>(w.y) << 32) | w.x, len);
  *p1 = __umul64hi((static_cast<uint64_t>(w.w) << 32) | w.z, len);
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
// Programmatic dependent launch: wait for the preceding grid (and its memory),
// and let the next grid start launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// L2 policy for data read once: its lines are evicted first, so a stream of
// it does not push out what later kernels reuse (their code, small buffers).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// Four consecutive 32-bit counters in one 16-byte load through L2 (p 16-byte
// aligned): a block reading a counter table then requests each line once.
__device__ __forceinline__ uint4 ldcg_u4(const unsigned* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

#ifdef TK_PHASE_TIMING
// Debug builds only: first-block start and last-block end of each kernel of
// a call (0 sample, 1 threshold, 2 filter, 3 refinement, 4 bin sort,
// 5 fallback), in globaltimer nanoseconds.
// (one copy per translation unit; each unit exports an accessor)
static __device__ unsigned long long g_timeline[8][2];
#define TK_TIMELINE_ACCESSOR(name)                                                      \
  int name(unsigned long long* out, int reset) {                                        \
    if (reset) {                                                                        \
      unsigned long long init[8][2];                                                    \
      for (int i = 0; i < 8; ++i) { init[i][0] = ~0ull; init[i][1] = 0ull; }            \
      return cudaMemcpyToSymbol(g_timeline, init, sizeof(init)) == cudaSuccess ? 0 : -3; \
    }                                                                                   \
    return cudaMemcpyFromSymbol(out, g_timeline, sizeof(g_timeline)) == cudaSuccess ? 0 : -3; \
  }
__device__ __forceinline__ void tl_begin(int id) {
  if (threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    atomicMin(&g_timeline[id][0], t);
  }
}
__device__ __forceinline__ void tl_end(int id) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    atomicMax(&g_timeline[id][1], t);
  }
}
#define TK_TL_BEGIN(id) tk::tl_begin(id)
#define TK_TL_END(id) tk::tl_end(id)
#else
#define TK_TL_BEGIN(id) \
  do {                  \
  } while (0)
#define TK_TL_END(id) \
  do {                \
  } while (0)
#endif

// Device status codes written to the workspace status word.
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 1;
constexpr int kDevBadState = 2;

// Upper bound of every device-side spin wait.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------------------
// Bulk copies (TMA engine, cp.async.bulk) into shared memory, completing on a
// shared-memory mbarrier.  Both addresses 16-byte aligned, the size a
// multiple of 16 bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}
// The same with an L2 cache policy for the source lines (e.g. evict-first).
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy) : "memory");
}
// Asks L2 to fetch [src, src + bytes) from global memory (no destination, no
// completion): src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Orders this thread's earlier generic-proxy accesses of shared memory before
// later bulk copies (async proxy) into it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// The same for every state space: what this thread has observed of global
// memory (e.g. counters other blocks added before a grid barrier) before
// its later bulk copies read it.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Waits for phase `parity` of the barrier to complete, for at most
// kWaitLimitNs; false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

}  // namespace tk
