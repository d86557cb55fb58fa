// Oracle: plain CPU top-k selection.  TEST INFRASTRUCTURE ONLY.
//
// This file is the reference answer the GPU engine is checked against.  It is
// deliberately slow and obvious and shares no code, header, table or helper
// with the CUDA path.  Only the test-suite, the smoke check and the bench's
// CPU-baseline leg may load it.
//
// What it computes (the plain definition of top-k):
//   "Given an input vector x in R^N and an integer k >= 1, return the k largest
//    entries of x together with their indices" -- Prof-K: Probabilistic
//    One-Pass Filtering for Efficient Top-k Selection, section 3 (Problem
//    Setup).  Batched inputs apply the same procedure to every row (same
//    section); the batch-global variant flattens the batch into one vector
//    (section 5, Application: BatchTopK Sparse Autoencoders).
//
// Order and tie-break:
//   Equal scores are ordered by index, the lower index first -- "Rank by
//   Counting" (top-k task 1), Goal and Requirements: an equal score outranks
//   you only when its index is lower.  The output lists the k winners from
//   rank 0 upward, i.e. sorted by (value descending, index ascending).
//   Readings where the pages are silent: NaN ranks above every number and all
//   NaNs are equal (they break ties by index); -0 equals +0; +-inf are ordinary
//   values.  With largest == 0 the value test is reversed (smallest first, NaN
//   last) and ties still go to the lower index.  bf16 inputs are widened to
//   float exactly before comparing.  Output values are the input's own bits.
//
// Steps: build (value, index) pairs, std::nth_element to put the k best in
// front, std::sort of those k.  No blocking, no keys, no bit tricks.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Item {
  float v;
  uint32_t bits;  // the input's own bit pattern (f32 bits, or bf16 bits)
  int64_t i;
};

// a comes before b in the largest-first order.
bool before_largest(const Item& a, const Item& b) {
  const bool an = std::isnan(a.v), bn = std::isnan(b.v);
  if (an != bn) return an;              // NaN ranks above every number
  if (!an && a.v != b.v) return a.v > b.v;
  return a.i < b.i;                     // equal values: lower index first
}

// a comes before b in the smallest-first order.
bool before_smallest(const Item& a, const Item& b) {
  const bool an = std::isnan(a.v), bn = std::isnan(b.v);
  if (an != bn) return bn;              // NaN ranks after every number
  if (!an && a.v != b.v) return a.v < b.v;
  return a.i < b.i;
}

float widen_bf16(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Selects the top k of items[0..n) in place; the first k entries end sorted.
void select_sorted(std::vector<Item>& items, int64_t k, int largest) {
  auto cmp = largest ? before_largest : before_smallest;
  const int64_t n = static_cast<int64_t>(items.size());
  if (k < n) std::nth_element(items.begin(), items.begin() + (k - 1), items.end(), cmp);
  std::sort(items.begin(), items.begin() + k, cmp);
}

}  // namespace

extern "C" {

// x: rows*n values, row-major; dtype 0 = f32, 1 = bf16 (raw uint16 bits).
// Per-row mode (global == 0): outputs are rows*k values / row-local indices.
// Global mode (global != 0): the rows*n values form one vector; outputs are k
// values / flat indices.  Returns 0 on success, -1 on bad arguments.
int oracle_topk(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                int global, void* out_vals, int64_t* out_idx) {
  if (rows < 0 || n < 0 || k < 1 || (dtype != 0 && dtype != 1)) return -1;
  if (rows == 0) return 0;
  const int64_t len = global ? rows * n : n;
  const int64_t nsel = global ? 1 : rows;
  if (k > len) return -1;
  std::vector<Item> items(static_cast<size_t>(len));
  for (int64_t r = 0; r < nsel; ++r) {
    for (int64_t i = 0; i < len; ++i) {
      Item& it = items[static_cast<size_t>(i)];
      it.i = i;
      if (dtype == 0) {
        const float* xf = static_cast<const float*>(x) + r * len;
        it.v = xf[i];
        std::memcpy(&it.bits, &xf[i], 4);
      } else {
        const uint16_t* xh = static_cast<const uint16_t*>(x) + r * len;
        it.v = widen_bf16(xh[i]);
        it.bits = xh[i];
      }
    }
    select_sorted(items, k, largest);
    for (int64_t j = 0; j < k; ++j) {
      const Item& it = items[static_cast<size_t>(j)];
      out_idx[r * k + j] = it.i;
      if (dtype == 0) {
        std::memcpy(static_cast<uint32_t*>(out_vals) + r * k + j, &it.bits, 4);
      } else {
        static_cast<uint16_t*>(out_vals)[r * k + j] = static_cast<uint16_t>(it.bits);
      }
    }
  }
  return 0;
}

// The same answer as oracle_topk from several host threads: each selection's
// elements are cut into `threads` contiguous chunks, each chunk keeps its own
// k best (nth_element) in parallel, and the union of those candidates -- which
// holds the k best of the whole selection -- is selected and sorted as
// above.  A CPU baseline over all host cores, not a reference answer: the
// tests check it against oracle_topk.
int oracle_topk_parallel(const void* x, int dtype, int64_t rows, int64_t n, int64_t k, int largest,
                         int global, int threads, void* out_vals, int64_t* out_idx) {
  if (rows < 0 || n < 0 || k < 1 || (dtype != 0 && dtype != 1) || threads < 1) return -1;
  if (rows == 0) return 0;
  const int64_t len = global ? rows * n : n;
  const int64_t nsel = global ? 1 : rows;
  if (k > len) return -1;
  auto cmp = largest ? before_largest : before_smallest;
  for (int64_t r = 0; r < nsel; ++r) {
    const int64_t nt = std::min<int64_t>(threads, std::max<int64_t>(1, len / std::max<int64_t>(k, 1)));
    std::vector<std::vector<Item>> kept(static_cast<size_t>(nt));
    std::vector<std::thread> pool;
    for (int64_t c = 0; c < nt; ++c) {
      pool.emplace_back([&, c]() {
        const int64_t b = len * c / nt, e = len * (c + 1) / nt;
        std::vector<Item>& v = kept[static_cast<size_t>(c)];
        v.resize(static_cast<size_t>(e - b));
        for (int64_t i = b; i < e; ++i) {
          Item& it = v[static_cast<size_t>(i - b)];
          it.i = i;
          if (dtype == 0) {
            const float* xf = static_cast<const float*>(x) + r * len;
            it.v = xf[i];
            std::memcpy(&it.bits, &xf[i], 4);
          } else {
            const uint16_t* xh = static_cast<const uint16_t*>(x) + r * len;
            it.v = widen_bf16(xh[i]);
            it.bits = xh[i];
          }
        }
        if (static_cast<int64_t>(v.size()) > k) {
          std::nth_element(v.begin(), v.begin() + (k - 1), v.end(), cmp);
          v.resize(static_cast<size_t>(k));
        }
      });
    }
    for (auto& t : pool) t.join();
    std::vector<Item> cand;
    for (auto& v : kept) cand.insert(cand.end(), v.begin(), v.end());
    select_sorted(cand, k, largest);
    for (int64_t j = 0; j < k; ++j) {
      const Item& it = cand[static_cast<size_t>(j)];
      out_idx[r * k + j] = it.i;
      if (dtype == 0) {
        std::memcpy(static_cast<uint32_t*>(out_vals) + r * k + j, &it.bits, 4);
      } else {
        static_cast<uint16_t*>(out_vals)[r * k + j] = static_cast<uint16_t>(it.bits);
      }
    }
  }
  return 0;
}

// Number of elements of one row that rank at or above element `pivot` in the
// chosen order (the pivot itself included).  This is R = |{i : x_i >= tau}|
// of the filtering stage (section 3, stage 3 and the design goal k <= R <= M)
// when tau is the element `pivot` and >= means "ranks at or above" in the
// (value, lower-index) total order.
int64_t oracle_count_at_or_above(const void* x, int dtype, int64_t len, int64_t pivot,
                                 int largest) {
  auto cmp = largest ? before_largest : before_smallest;
  Item p;
  p.i = pivot;
  p.v = dtype == 0 ? static_cast<const float*>(x)[pivot]
                   : widen_bf16(static_cast<const uint16_t*>(x)[pivot]);
  int64_t count = 0;
  for (int64_t i = 0; i < len; ++i) {
    Item it;
    it.i = i;
    it.v = dtype == 0 ? static_cast<const float*>(x)[i]
                      : widen_bf16(static_cast<const uint16_t*>(x)[i]);
    if (!cmp(p, it)) ++count;  // it does not come after the pivot
  }
  return count;
}

// The t-th best (1-based) of the sampled positions idx[0..s) of one row, with
// multiplicity (a position drawn twice occupies two places).  Returns its
// index.  This is tau = s_t of section 3, stage 2 (threshold estimation),
// expressed as the element it comes from.
int64_t oracle_sample_order_stat(const void* x, int dtype, const int64_t* idx, int64_t s,
                                 int64_t t, int largest) {
  std::vector<Item> items(static_cast<size_t>(s));
  for (int64_t j = 0; j < s; ++j) {
    Item& it = items[static_cast<size_t>(j)];
    it.i = idx[j];
    it.v = dtype == 0 ? static_cast<const float*>(x)[idx[j]]
                      : widen_bf16(static_cast<const uint16_t*>(x)[idx[j]]);
  }
  auto cmp = largest ? before_largest : before_smallest;
  std::sort(items.begin(), items.end(), cmp);
  return items[static_cast<size_t>(t - 1)].i;
}

}  // extern "C"
