// muon_partition: which rank owns which matrix of a bank when the Muon step
// is spread over several processes (one per GPU).
//
// Each matrix's step (momentum, Newton-Schulz, update) depends on that
// matrix alone, so the bank splits into independent units.  The page
// "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术" (reposource.net),
// section "Muon优化器：动量正交化技术", has each rank orthogonalise its own
// slice of every size group of parameters and then gather the updates; here
// the assignment balances the Newton-Schulz work instead of slicing by
// position: matrices are taken from the heaviest down (identical shapes
// together) and each goes to the rank with the least work so far (greedy
// longest-processing-time rule), so no rank ends more than one matrix's work
// above the mean.  The result is a pure function of the shapes and the rank
// count, so every rank computes the same assignment with no communication.
// Host code only.
#include <algorithm>
#include <numeric>
#include <vector>

#include "../../include/muon.h"

namespace {

// Algorithmic Newton-Schulz FLOPs of one step of an R x C matrix
// (m = min, n = max): Gram m(m+1)n, polynomial m^2(m+1), update 2 m^2 n.
double ns_work(long long R, long long C) {
  const double m = static_cast<double>(std::min(R, C));
  const double n = static_cast<double>(std::max(R, C));
  return m * (m + 1.0) * n + m * m * (m + 1.0) + 2.0 * m * m * n;
}

}  // namespace

extern "C" muon_status_t muon_partition(const int64_t* rows, const int64_t* cols, int n_mats, int world,
                                        int* owner) {
  if (n_mats < 0 || world <= 0) return MUON_ERR_INVALID_ARG;
  if (n_mats == 0) return MUON_OK;
  if (!rows || !cols || !owner) return MUON_ERR_INVALID_ARG;
  for (int i = 0; i < n_mats; ++i)
    if (rows[i] <= 0 || cols[i] <= 0) return MUON_ERR_INVALID_ARG;
  std::vector<double> w(n_mats);
  for (int i = 0; i < n_mats; ++i) w[i] = ns_work(rows[i], cols[i]);
  std::vector<int> order(n_mats);
  std::iota(order.begin(), order.end(), 0);
  // heaviest first; equal work: identical shapes together (more rows first,
  // then more columns), so each shape group is dealt out evenly; then bank
  // order
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    if (w[a] != w[b]) return w[a] > w[b];
    if (rows[a] != rows[b]) return rows[a] > rows[b];
    return cols[a] > cols[b];
  });
  std::vector<double> load(world, 0.0);
  for (int i : order) {
    int best = 0;
    for (int r = 1; r < world; ++r)
      if (load[r] < load[best]) best = r;  // ties: lowest rank
    owner[i] = best;
    load[best] += w[i];
  }
  return MUON_OK;
}
