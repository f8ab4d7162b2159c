// Row-wise top-k oracle: TEST INFRASTRUCTURE ONLY.
//
// This file is the plain, slow, obviously-correct CPU statement of what the
// selector computes.  Only the test suite, the smoke check and the benchmark's
// CPU-baseline leg may load it.  It shares no code, header, table or helper
// with the CUDA path, and the CUDA path never calls it.
//
// What is computed (definition, not algorithm).  For every row r, take the
// valid prefix  x_0 .. x_{L_r - 1}  of  scores[r * row_stride + i]  and order
// the pairs (x_i, i) so that a pair comes first when its value is larger, and
// among equal values the smaller in-row index comes first.  Emit the first
// min(k, L_r) pairs; fill the remaining k - min(k, L_r) slots with (-inf, -1).
//
//   * "Find the biggest 512 numbers in a list of a million", kept per query
//     row: The Secret GPU Kernel Behind DeepSeek V4.1 Flash (video transcript,
//     2:28-2:53); the selection size comes from the config line "index top k
//     512" (2:00-2:13).
//   * The selector returns the exact answer and "values come back bit-exact
//     and indices cannot duplicate": DeepSeek V4.1 Flash (kernelbench model
//     page, entry "Single-launch CUDA bitonic selection").
//
// Readings taken where the pages are silent:
//   * value order is the IEEE total order restricted to non-NaN values,
//     -inf < negatives < -0.0 < +0.0 < positives < +inf (the "monotonic key"
//     packing of the bitonic-selection entry orders floats this way);
//   * ties go to the smaller in-row index; output is value-descending;
//   * rows shorter than k return every valid position, then (-inf, -1) pads;
//   * NaN is not a value ("one bad value aborts the whole kernel", video
//     transcript 5:45-5:57): a NaN inside a valid prefix is reported through
//     the return code; that row's outputs are then all padding.
//
// Written with plain IEEE comparisons and an explicit signed-zero rule, not
// with any bit-packing trick, so that it stays independent of the GPU path.
//
// ORACLE_MUTANT (default 0) plants one deliberate mistake when set at compile
// time; the test suite uses it to show that the pins catch each mistake.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

namespace {

// a ranks strictly before b in the selection order.
bool ranks_before(float xa, int64_t ia, float xb, int64_t ib) {
#if ORACLE_MUTANT == 9
  // mistake: +inf clamped to the largest finite value
  if (std::isinf(xa) && xa > 0) xa = std::numeric_limits<float>::max();
  if (std::isinf(xb) && xb > 0) xb = std::numeric_limits<float>::max();
#endif
#if ORACLE_MUTANT == 3
  // mistake: ascending value order
  std::swap(xa, xb);
#endif
  if (xa > xb) return true;
  if (xa < xb) return false;
  // IEEE-equal: the same value, or +0.0 against -0.0.
  const bool neg_a = std::signbit(xa);
  const bool neg_b = std::signbit(xb);
#if ORACLE_MUTANT != 1  // mistake 1: signed zeros compared as equal
  if (neg_a != neg_b) return neg_b;  // +0.0 ranks before -0.0
#else
  (void)neg_a; (void)neg_b;
#endif
#if ORACLE_MUTANT == 2
  return ia > ib;  // mistake: ties go to the larger index
#else
  return ia < ib;  // ties go to the smaller in-row index
#endif
}

// One row.  Returns 0, or 5 when a NaN sits inside the valid prefix.
int select_row(const float* row, int64_t len, int32_t k, float* vals,
               int32_t* idx) {
  std::vector<int64_t> order;
  order.reserve(static_cast<size_t>(len));
  for (int64_t i = 0; i < len; ++i) {
    if (std::isnan(row[i])) {
      for (int32_t j = 0; j < k; ++j) {
        vals[j] = -std::numeric_limits<float>::infinity();
        idx[j] = -1;
      }
      return 5;
    }
#if ORACLE_MUTANT == 8
    if (std::isinf(row[i]) && row[i] < 0) continue;  // mistake: drops -inf
#endif
    order.push_back(i);
  }
  std::sort(order.begin(), order.end(), [row](int64_t a, int64_t b) {
    return ranks_before(row[a], a, row[b], b);
  });
  int64_t take = std::min<int64_t>(k, static_cast<int64_t>(order.size()));
#if ORACLE_MUTANT == 6
  if (take > 0 && take < k) take -= 1;  // mistake: off-by-one on short rows
#endif
  for (int64_t j = 0; j < take; ++j) {
    vals[j] = row[order[j]];
    idx[j] = static_cast<int32_t>(order[j]);
  }
  for (int64_t j = take; j < k; ++j) {
    vals[j] = -std::numeric_limits<float>::infinity();
#if ORACLE_MUTANT == 5
    idx[j] = 0;  // mistake: pads with index 0
#else
    idx[j] = -1;
#endif
  }
  return 0;
}

// a is a larger value than b in the same total order (+0.0 above -0.0).
bool value_greater(float a, float b) {
  if (a > b) return true;
  if (a < b) return false;
  return !std::signbit(a) && std::signbit(b);
}

// The block pool of one row.  Returns 0, or 5 when a NaN sits inside the
// valid prefix (the row's pool is then all -1).
int pool_row(const float* row, int64_t len, int32_t block, int32_t pool,
             int32_t pinned, int32_t* out) {
  for (int32_t j = 0; j < pool; ++j) out[j] = -1;
  for (int64_t i = 0; i < len; ++i)
    if (std::isnan(row[i])) return 5;
#if ORACLE_MUTANT == 13
  const int64_t nb = len / block;  // mistake: the short last block is dropped
#else
  const int64_t nb = (len + block - 1) / block;
#endif
  const int64_t pe = std::min<int64_t>(pinned, nb);
#if ORACLE_MUTANT == 14
  const int64_t ncand = nb;  // mistake: pinned blocks also compete
#else
  const int64_t ncand = nb - pe;
#endif
  // each candidate block's score: the largest value inside it
  std::vector<float> bmax(static_cast<size_t>(ncand));
  for (int64_t b = 0; b < ncand; ++b) {
    const int64_t lo = b * block, hi = std::min<int64_t>(len, lo + block);
    float m = row[lo];
#if ORACLE_MUTANT != 10  // mistake 10: the block's first score stands for it
    for (int64_t i = lo + 1; i < hi; ++i)
      if (value_greater(row[i], m)) m = row[i];
#else
    (void)hi;
#endif
    bmax[static_cast<size_t>(b)] = m;
  }
  std::vector<int64_t> order(static_cast<size_t>(ncand));
  for (int64_t b = 0; b < ncand; ++b) order[static_cast<size_t>(b)] = b;
  std::sort(order.begin(), order.end(), [&bmax](int64_t a, int64_t b) {
#if ORACLE_MUTANT == 12
    return ranks_before(bmax[a], -a, bmax[b], -b);  // mistake: ties to the larger block
#else
    return ranks_before(bmax[a], a, bmax[b], b);
#endif
  });
  std::vector<int64_t> kept;
  const int64_t take = std::min<int64_t>(pool - pe, ncand);
  for (int64_t j = 0; j < take; ++j) kept.push_back(order[static_cast<size_t>(j)]);
#if ORACLE_MUTANT == 11
  for (int64_t b = 0; b < pe; ++b) kept.push_back(b);  // mistake: oldest blocks pinned
#else
  for (int64_t b = nb - pe; b < nb; ++b) kept.push_back(b);
#endif
  std::sort(kept.begin(), kept.end());
  kept.erase(std::unique(kept.begin(), kept.end()), kept.end());
  for (size_t j = 0; j < kept.size() && j < static_cast<size_t>(pool); ++j)
    out[j] = static_cast<int32_t>(kept[j]);
  return 0;
}

}  // namespace

extern "C" {

// Shape checks mirror the library's documented contract so that the same
// arguments are accepted by both: rows >= 0, 1 <= n < 2^31, n <= row_stride,
// 1 <= k <= 2048, every length in [0, n].
//
// Returns 0 on success, 1 on a bad shape, 2 on a null pointer, 5 if any row
// held a NaN inside its valid prefix (that row's outputs are all padding),
// 6 if a length is outside [0, n].
int oracle_topk(const float* scores, int32_t rows, int64_t n,
                int64_t row_stride, const int32_t* lengths, int32_t k,
                float* out_vals, int32_t* out_idx, int32_t nthreads) {
  if (rows < 0 || n < 1 || n > INT32_MAX || row_stride < n || k < 1 ||
      k > 2048)
    return 1;
  if (rows == 0) return 0;
  if (!scores || !out_vals || !out_idx) return 2;
  if (lengths) {
    for (int32_t r = 0; r < rows; ++r)
      if (lengths[r] < 0 || lengths[r] > n) return 6;
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > rows) nthreads = rows;

  std::vector<int> row_status(static_cast<size_t>(rows), 0);
  auto run = [&](int32_t first, int32_t step) {
    for (int32_t r = first; r < rows; r += step) {
      int64_t len = lengths ? lengths[r] : n;
#if ORACLE_MUTANT == 4
      len = n;  // mistake: ignores the per-row lengths
#endif
#if ORACLE_MUTANT == 7
      const float* row = scores + static_cast<int64_t>(r) * n;  // mistake
#else
      const float* row = scores + static_cast<int64_t>(r) * row_stride;
#endif
      row_status[r] = select_row(row, len, k,
                                 out_vals + static_cast<int64_t>(r) * k,
                                 out_idx + static_cast<int64_t>(r) * k);
    }
  };
  if (nthreads == 1) {
    run(0, 1);
  } else {
    std::vector<std::thread> pool;
    for (int32_t t = 0; t < nthreads; ++t) pool.emplace_back(run, t, nthreads);
    for (auto& th : pool) th.join();
  }
  for (int s : row_status)
    if (s) return s;
  return 0;
}

// The layer-20 block pool (The Secret GPU Kernel Behind DeepSeek V4.1 Flash,
// video transcript 7:22-7:46): the sweep that scores every position also
// groups each row's valid prefix into blocks of `block` consecutive
// positions (the last block may be short), gives every block the largest
// score inside it, and keeps `pool` blocks: the `pinned` newest blocks (the
// highest block indices) always, and the best-scoring other blocks (value
// descending in the order above, ties to the smaller block index) until
// `pool` blocks are kept or none is left.  Output per row: the kept block
// indices in ascending order, padded with -1 to `pool` entries.
//
// Readings: the pages give blocks of eight and a pool of about 2,000
// blocks (16,000 positions) but not how many blocks are pinned, so that is
// a parameter; the pool is a set (upper indexers score inside it), emitted
// as ascending block indices.
//
// Returns 0, 1 on a bad shape (as oracle_topk, plus block < 1, pool < 1,
// pinned < 0, pinned > pool, pool - pinned > 2048), 2 on a null pointer,
// 5 if a row held a NaN (that row's pool is all -1), 6 on a bad length.
int oracle_block_pool(const float* scores, int32_t rows, int64_t n,
                      int64_t row_stride, const int32_t* lengths, int32_t block,
                      int32_t pool, int32_t pinned, int32_t* out,
                      int32_t nthreads) {
  if (rows < 0 || n < 1 || n > INT32_MAX || row_stride < n || block < 1 ||
      pool < 1 || pinned < 0 || pinned > pool || pool - pinned > 2048)
    return 1;
  if (rows == 0) return 0;
  if (!scores || !out) return 2;
  if (lengths) {
    for (int32_t r = 0; r < rows; ++r)
      if (lengths[r] < 0 || lengths[r] > n) return 6;
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > rows) nthreads = rows;
  std::vector<int> row_status(static_cast<size_t>(rows), 0);
  auto run = [&](int32_t first, int32_t step) {
    for (int32_t r = first; r < rows; r += step) {
      const int64_t len = lengths ? lengths[r] : n;
      row_status[r] = pool_row(scores + static_cast<int64_t>(r) * row_stride, len, block,
                               pool, pinned, out + static_cast<int64_t>(r) * pool);
    }
  };
  if (nthreads == 1) {
    run(0, 1);
  } else {
    std::vector<std::thread> th;
    for (int32_t t = 0; t < nthreads; ++t) th.emplace_back(run, t, nthreads);
    for (auto& t : th) t.join();
  }
  for (int s : row_status)
    if (s) return s;
  return 0;
}

// Number of hardware threads the host reports (for the baseline's core count).
int32_t oracle_hardware_threads(void) {
  unsigned c = std::thread::hardware_concurrency();
  return c ? static_cast<int32_t>(c) : 1;
}

}  // extern "C"
