// Row allocation for the static routing table (host only).
//
// "L³: Large Lookup Layers" (gist.science explainer), Technical Summary, "Information-
// Theoretic Embedding Allocation": a budget of v rows is spread over the vocabulary with
// 1 <= n_t <= k rows per token and more rows for frequent tokens. The corpus-driven
// Algorithm 1 is not on the pages; the library allocates by frequency instead:
// weights pow(freq, power) are water-filled into [n_min, n_max] so that they sum to v,
// and the real targets are rounded by largest remainder.
//
// The arithmetic is fixed step by step (sequential sums in id order, no fused
// multiply-add) so that the result is reproducible bit for bit.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <numeric>
#include <vector>

#include "l3.h"

namespace {

// sum_t clamp(c * w_t, lo, hi), left to right.
double filled(const std::vector<double>& w, double c, double lo, double hi) {
  double acc = 0.0;
  for (double wt : w) {
    double z = c * wt;
    z = z < lo ? lo : z;
    z = z > hi ? hi : z;
    acc += z;
  }
  return acc;
}

}  // namespace

extern "C" l3_status l3_alloc_offsets(const double* freq, int64_t vocab, int64_t v,
                                      int32_t n_min, int32_t n_max, double power,
                                      int32_t* offs_out) {
  if (!freq || !offs_out || vocab < 1 || n_min < 1 || n_max < n_min || !std::isfinite(power) ||
      v < 1 || v >= (int64_t(1) << 31))
    return L3_ERR_INVALID_ARG;
  for (int64_t t = 0; t < vocab; ++t)
    if (!(freq[t] > 0.0) || !std::isfinite(freq[t])) return L3_ERR_INVALID_ARG;
  if (vocab * int64_t(n_min) > v || v > vocab * int64_t(n_max)) return L3_ERR_INFEASIBLE;

  const size_t N = size_t(vocab);
  const double lo = double(n_min), hi = double(n_max);
  std::vector<double> w(N);
  double w_min = 0.0;
  for (size_t t = 0; t < N; ++t) {
    w[t] = std::pow(freq[t], power);
    if (!(w[t] > 0.0) || !std::isfinite(w[t])) return L3_ERR_INVALID_ARG;
    w_min = (t == 0 || w[t] < w_min) ? w[t] : w_min;
  }

  // Water level: F(c) = sum clamp(c w_t) is continuous and non-decreasing; bisect for
  // the smallest c with F(c) >= v, then read off the clamped sets there.
  double c_lo = 0.0, c_hi = 2.0 * hi / w_min;
  const double budget = double(v);
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (c_lo + c_hi);
    if (filled(w, mid, lo, hi) < budget)
      c_lo = mid;
    else
      c_hi = mid;
  }
  std::vector<double> r(N);
  std::vector<uint8_t> state(N);  // 0 free, 1 at the cap, 2 at the floor
  int64_t n_cap = 0, n_floor = 0;
  for (size_t t = 0; t < N; ++t) {
    double z = c_hi * w[t];
    if (z >= hi) {
      state[t] = 1;
      ++n_cap;
    } else if (z <= lo) {
      state[t] = 2;
      ++n_floor;
    } else {
      state[t] = 0;
    }
  }
  double w_free = 0.0;
  bool any_free = false;
  for (size_t t = 0; t < N; ++t)
    if (state[t] == 0) {
      w_free += w[t];
      any_free = true;
    }
  const double c_star =
      any_free ? (budget - hi * double(n_cap) - lo * double(n_floor)) / w_free : 0.0;
  for (size_t t = 0; t < N; ++t) {
    if (state[t] == 1) {
      r[t] = hi;
    } else if (state[t] == 2) {
      r[t] = lo;
    } else {
      double z = c_star * w[t];
      z = z < lo ? lo : z;
      z = z > hi ? hi : z;
      r[t] = z;
    }
  }

  // Largest remainder: floors first, then one more row to the D ids (below the cap)
  // with the largest fractional part; equal parts go to the lower id.
  std::vector<int64_t> n(N);
  int64_t floor_sum = 0;
  std::vector<int64_t> cand;
  cand.reserve(N);
  for (size_t t = 0; t < N; ++t) {
    n[t] = int64_t(std::floor(r[t]));
    floor_sum += n[t];
    if (n[t] < n_max) cand.push_back(int64_t(t));
  }
  const int64_t D = v - floor_sum;
  if (D < 0 || D > int64_t(cand.size())) return L3_ERR_INFEASIBLE;
  std::stable_sort(cand.begin(), cand.end(), [&](int64_t a, int64_t b) {
    double fa = r[size_t(a)] - double(n[size_t(a)]);
    double fb = r[size_t(b)] - double(n[size_t(b)]);
    return fa > fb;  // stable: equal fractional parts keep increasing id order
  });
  for (int64_t j = 0; j < D; ++j) n[size_t(cand[size_t(j)])] += 1;

  int64_t run = 0;
  offs_out[0] = 0;
  for (size_t t = 0; t < N; ++t) {
    if (n[t] < n_min || n[t] > n_max) return L3_ERR_INFEASIBLE;
    run += n[t];
    offs_out[t + 1] = int32_t(run);
  }
  return run == v ? L3_OK : L3_ERR_INFEASIBLE;
}

extern "C" l3_status l3_alloc_offsets_counts(const int64_t* counts, int64_t vocab, int64_t v,
                                             int32_t n_min, int32_t n_max, double power,
                                             double smoothing, int32_t* offs_out) {
  if (!counts || vocab < 1 || !(smoothing >= 0.0) || !std::isfinite(smoothing))
    return L3_ERR_INVALID_ARG;
  std::vector<double> freq(static_cast<size_t>(vocab));
  for (int64_t t = 0; t < vocab; ++t) {
    if (counts[t] < 0) return L3_ERR_INVALID_ARG;
    freq[size_t(t)] = double(counts[t]) + smoothing;  // l3_alloc_offsets rejects a zero
  }
  return l3_alloc_offsets(freq.data(), vocab, v, n_min, n_max, power, offs_out);
}
