// owners.cpp - one owner rank per matrix, balanced by predicted cost.
//
// "DMuon: Efficient Distributed Muon Training with Near-Adam Overhead"
// (gist.science summary, section 2.1): every matrix has exactly one owner,
// which keeps its optimizer state and runs its update; section 2.3: owners are
// chosen to minimise the predicted makespan (the largest per-rank load) over
// measured per-shape costs, with a greedy heuristic when the search space is
// large. Here: longest-processing-time-first greedy (largest cost to the
// least-loaded rank), then a local search that moves one matrix, or swaps
// two, between the most-loaded rank and another rank while that strictly
// lowers the makespan. Everything is deterministic, so every rank computes
// the same assignment from the same inputs without communicating.
#include <algorithm>
#include <cmath>
#include <numeric>
#include <vector>

#include "dmuon.h"
#include "internal.h"

namespace {

double ns_cost(int64_t rows, int64_t cols, int32_t ns_steps) {
  const double m = static_cast<double>(std::min(rows, cols)), n = static_cast<double>(std::max(rows, cols));
  return ns_steps * (m * (m + 1) * n + m * m * (m + 1) + 2 * m * m * n);
}

}  // namespace

extern "C" dmuon_status dmuon_assign_owners(const dmuon_shape* shapes, int32_t n_mats, int32_t ns_steps,
                                            const double* costs, int32_t n_ranks, int32_t* owner_out,
                                            double* load_out) {
  using dmuon::set_last_error;
  if (shapes == nullptr || owner_out == nullptr || n_mats <= 0)
    return set_last_error(DMUON_ERR_INVALID_ARG, "empty matrix list or NULL output");
  if (n_ranks < 1 || n_ranks > (1 << 20)) return set_last_error(DMUON_ERR_INVALID_ARG, "n_ranks must be >= 1");
  if (ns_steps < 0 || ns_steps > 16) return set_last_error(DMUON_ERR_INVALID_ARG, "ns_steps outside 0..16");
  std::vector<double> c(n_mats);
  for (int32_t i = 0; i < n_mats; ++i) {
    if (shapes[i].rows < 1 || shapes[i].cols < 1) return set_last_error(DMUON_ERR_INVALID_ARG, "bad shape");
    c[i] = costs ? costs[i] : ns_cost(shapes[i].rows, shapes[i].cols, std::max(ns_steps, 1));
    if (!(c[i] >= 0.0) || !std::isfinite(c[i]))
      return set_last_error(DMUON_ERR_INVALID_ARG, "costs must be finite and >= 0");
  }
  // greedy: largest cost first (ties: lower index), each to the least-loaded rank (ties: lower rank)
  std::vector<int32_t> order(n_mats);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return c[a] > c[b]; });
  std::vector<double> load(n_ranks, 0.0);
  std::vector<int32_t> own(n_mats, 0);
  for (int32_t i : order) {
    int32_t r = static_cast<int32_t>(std::min_element(load.begin(), load.end()) - load.begin());
    own[i] = r;
    load[r] += c[i];
  }
  // local search on the most-loaded rank: the best single move or swap; repeat while the makespan drops
  std::vector<std::vector<int32_t>> members(n_ranks);
  for (int iter = 0; iter < 4 * n_mats + 16; ++iter) {
    for (auto& m : members) m.clear();
    for (int32_t i = 0; i < n_mats; ++i) members[own[i]].push_back(i);
    const int32_t hi = static_cast<int32_t>(std::max_element(load.begin(), load.end()) - load.begin());
    const double span = load[hi];
    // the two largest loads among the other ranks, to get max over q not in {hi, r} in O(1)
    int32_t t1 = -1, t2 = -1;
    for (int32_t q = 0; q < n_ranks; ++q) {
      if (q == hi) continue;
      if (t1 < 0 || load[q] > load[t1]) {
        t2 = t1;
        t1 = q;
      } else if (t2 < 0 || load[q] > load[t2]) {
        t2 = q;
      }
    }
    double best = span;
    int32_t bi = -1, bj = -1, br = -1;
    for (int32_t r = 0; r < n_ranks; ++r) {
      if (r == hi) continue;
      const int32_t other = (r == t1) ? t2 : t1;
      const double rest = other >= 0 ? load[other] : 0.0;
      for (int32_t i : members[hi]) {
        const double mv = std::max(std::max(load[hi] - c[i], load[r] + c[i]), rest);
        if (mv < best - 1e-12 * span) {
          best = mv;
          bi = i;
          bj = -1;
          br = r;
        }
        for (int32_t j : members[r]) {
          if (c[j] >= c[i]) continue;
          const double sw = std::max(std::max(load[hi] - c[i] + c[j], load[r] + c[i] - c[j]), rest);
          if (sw < best - 1e-12 * span) {
            best = sw;
            bi = i;
            bj = j;
            br = r;
          }
        }
      }
    }
    if (bi < 0) break;
    load[hi] -= c[bi];
    load[br] += c[bi];
    own[bi] = br;
    if (bj >= 0) {
      load[br] -= c[bj];
      load[hi] += c[bj];
      own[bj] = hi;
    }
  }
  std::copy(own.begin(), own.end(), owner_out);
  if (load_out) std::copy(load.begin(), load.end(), load_out);
  return set_last_error(DMUON_OK, "");
}
