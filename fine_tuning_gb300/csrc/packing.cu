// Best-Fit-Decreasing packing of variable-length sequences into bins of a
// fixed token capacity: the step that produces the packed batches (and
// their cu_seqlens) the QK-RoPE kernels consume.
//
// Chronicals (arXiv 2601.02609), abstract, optimisation (4): Best-Fit
// Decreasing sequence packing.  Host code (the data loader's side of the
// path); no device memory is touched.
//
// Longest sequence first (equal lengths: lower index first); each goes to
// the open bin with the least room that still holds it (equal room: lower
// bin index), else to a new bin.  Open bins are kept in an ordered set keyed
// by (room, bin), so the best fit is one lower_bound: O(n log n) time and
// O(n) memory in all.  The decreasing order is a counting sort (a table of
// capacity + 2 counts) only where that table is small beside the input,
// capacity <= 4 n + 1024; otherwise a stable comparison sort.
#include <algorithm>
#include <climits>
#include <new>
#include <set>
#include <utility>
#include <vector>

#include "ftk.h"

namespace {
// Counting sort only while its table (capacity + 2 counts) is O(n): at most
// 4 n + 1024 entries.
bool counting_sort_pays(int64_t n, int32_t capacity) {
  return (int64_t)capacity <= 4 * n + 1024;
}
}  // namespace

extern "C" FTK_API ftk_status ftk_bfd_pack(const int32_t *lengths, int64_t n, int32_t capacity,
                                           int32_t *bin_of, int64_t *order, int64_t *bin_start,
                                           int64_t *n_bins) {
  if (n < 0 || capacity < 1 || n >= INT32_MAX) return FTK_ERR_SHAPE;
  if (!n_bins || (n > 0 && (!lengths || !bin_of || !order || !bin_start)) || (!bin_start && n == 0))
    return FTK_ERR_NULL;
  for (int64_t i = 0; i < n; ++i)
    if (lengths[i] < 0 || lengths[i] > capacity) return FTK_ERR_SHAPE;
  try {
    // longest first, equal lengths in index order: a counting sort when the
    // capacity (the largest length) is small beside n, else a stable sort
    std::vector<int32_t> by_len(n);
    if (counting_sort_pays(n, capacity)) {
      std::vector<int64_t> at((size_t)capacity + 2, 0);
      for (int64_t i = 0; i < n; ++i) ++at[(size_t)(capacity - lengths[i]) + 1];
      for (size_t v = 1; v < at.size(); ++v) at[v] += at[v - 1];
      for (int64_t i = 0; i < n; ++i) by_len[at[(size_t)(capacity - lengths[i])]++] = (int32_t)i;
    } else {
      for (int64_t i = 0; i < n; ++i) by_len[i] = (int32_t)i;
      std::stable_sort(by_len.begin(), by_len.end(),
                       [&](int32_t a, int32_t b) { return lengths[a] > lengths[b]; });
    }
    std::set<std::pair<int32_t, int32_t>> open;  // (room left, bin)
    std::vector<int64_t> count;
    int32_t bins = 0;
    for (int32_t i : by_len) {
      const int32_t len = lengths[i];
      auto it = open.lower_bound({len, INT32_MIN});
      if (it == open.end()) {
        const int32_t b = bins++;
        open.insert({capacity - len, b});
        count.push_back(1);
        bin_of[i] = b;
      } else {
        // the bin's node is re-keyed in place (no allocation)
        auto node = open.extract(it);
        const int32_t b = node.value().second;
        node.value().first -= len;
        open.insert(std::move(node));
        ++count[b];
        bin_of[i] = b;
      }
    }
    // members of each bin, in the order they were placed
    bin_start[0] = 0;
    for (int32_t b = 0; b < bins; ++b) bin_start[b + 1] = bin_start[b] + count[b];
    std::vector<int64_t> fill(bin_start, bin_start + bins);
    for (int32_t i : by_len) order[fill[bin_of[i]]++] = i;
    *n_bins = bins;
  } catch (const std::bad_alloc &) {
    return FTK_ERR_WORKSPACE;
  }
  return FTK_OK;
}
