// Partition of the optimizer step over several ranks (host code).
//
// The OpenDM article (核心揭秘一 / 为 FSDP 分片量身定制的细节) runs Muon under
// FSDP: each rank holds a shard of every matrix, and MuonShardPlan all-gathers
// the shards so that Newton-Schulz sees whole matrices, then keeps its own
// slice of the result. Here the step itself is split instead:
//   - each Muon matrix is updated whole by one owner rank (Newton-Schulz needs
//     the whole matrix, so nothing is gathered before it); owners are chosen
//     longest-processing-time-first on the matrix's dense Newton-Schulz flops,
//     5 (4 s^2 l + 2 s^3), each to the rank with the least work so far (ties
//     to the lower rank);
//   - AdamW, which is elementwise, splits the concatenation of all AdamW
//     parameters (registration order) into `world` contiguous ranges of
//     nearly equal length; a cut that falls inside a parameter is moved down
//     to a multiple of 64 elements of that parameter, so every range starts
//     16-byte aligned wherever the parameter does;
//   - the global gradient norm is the square root of the sum over ranks of
//     each rank's sum of squares over the elements it owns (every element is
//     owned exactly once), so one all-reduce of one number per rank gives it.
// After the step, each rank's updated parameters are shared with the others
// (the caller's collectives: a broadcast per owned matrix, an all-gather of
// the AdamW ranges).
#include <algorithm>
#include <queue>
#include <utility>
#include <vector>

#include "internal.h"
#include "muon_adamw.h"

namespace ma {

void shard_partition(const std::vector<int>& group, const std::vector<int64_t>& numel,
                     const std::vector<int64_t>& rows, const std::vector<int64_t>& cols, int world,
                     std::vector<int>& owner, std::vector<int64_t>& begin, std::vector<int64_t>& end) {
  const size_t n = group.size();
  owner.assign(n, -1);
  begin.assign(n * (size_t)world, 0);
  end.assign(n * (size_t)world, 0);
  // Muon: whole matrices, longest first, each to the least-loaded rank
  std::vector<std::pair<double, size_t>> mats;
  for (size_t i = 0; i < n; ++i) {
    if (group[i] != MA_GROUP_MUON || numel[i] == 0) continue;
    const double s = (double)std::min(rows[i], cols[i]), l = (double)std::max(rows[i], cols[i]);
    mats.push_back({5.0 * (4.0 * s * s * l + 2.0 * s * s * s), i});
  }
  std::stable_sort(mats.begin(), mats.end(),
                   [](const std::pair<double, size_t>& a, const std::pair<double, size_t>& b) { return a.first > b.first; });
  using Load = std::pair<double, int>;  // (work so far, rank)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> least;
  for (int r = 0; r < world; ++r) least.push({0.0, r});
  for (const auto& m : mats) {
    const Load top = least.top();
    least.pop();
    owner[m.second] = top.second;
    begin[m.second * (size_t)world + (size_t)top.second] = 0;
    end[m.second * (size_t)world + (size_t)top.second] = numel[m.second];
    least.push({top.first + m.first, top.second});
  }
  // AdamW: contiguous ranges of the concatenation
  std::vector<size_t> adam;
  std::vector<int64_t> start;  // offset of each AdamW parameter in the concatenation
  int64_t total = 0;
  for (size_t i = 0; i < n; ++i) {
    if (group[i] != MA_GROUP_ADAMW || numel[i] == 0) continue;
    adam.push_back(i);
    start.push_back(total);
    total += numel[i];
  }
  if (adam.empty()) return;
  // cut r (r = 0..world) as a position in the concatenation, moved down to a
  // multiple of 64 elements of the parameter it falls in
  std::vector<int64_t> cut((size_t)world + 1);
  for (int r = 0; r <= world; ++r) {
    const int64_t c = total / world * r + total % world * r / world;  // floor(total r / world)
    if (c >= total) {
      cut[(size_t)r] = total;
      continue;
    }
    const size_t k = (size_t)(std::upper_bound(start.begin(), start.end(), c) - start.begin()) - 1;
    const int64_t local = c - start[k];
    cut[(size_t)r] = start[k] + local / 64 * 64;
  }
  for (int r = 0; r < world; ++r) {
    const int64_t lo = cut[(size_t)r], hi = cut[(size_t)r + 1];
    for (size_t k = 0; k < adam.size(); ++k) {
      const int64_t b = std::max(lo, start[k]) - start[k];
      const int64_t e = std::min(hi, start[k] + numel[adam[k]]) - start[k];
      if (e > b) {
        begin[adam[k] * (size_t)world + (size_t)r] = b;
        end[adam[k] * (size_t)world + (size_t)r] = e;
      }
    }
  }
}

}  // namespace ma
