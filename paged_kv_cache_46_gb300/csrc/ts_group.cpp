// ts_group_prefixes: host-side greedy longest-shared-prefix grouping.
//
// Tokasaurus blog, "Dynamic prefix identification and exploration": before
// every forward pass a greedy depth-first search iteratively finds the longest
// possible shared prefixes, so that attention over each shared prefix can run
// once per group (Hydragen / cascade attention).
//
// Reading used here (the page fixes no tie-break or data format):
//   * a prefix is a run of whole pages shared by physical page id at the start
//     of the members' block-table rows; a member of length L may share at most
//     cap = (L - 1) / page_size pages, so it keeps at least one suffix token;
//   * the sequences form a trie keyed by page id; a depth-first walk handles
//     children (deeper prefixes) before their parent, and a node of depth >= 1
//     becomes a group of every still-ungrouped sequence below it once at least
//     min_group of them are left. Post-order over the trie is exactly "the
//     deepest prefix shared by >= min_group ungrouped sequences first";
//   * siblings are visited in increasing page id; members are listed in
//     increasing sequence index.
// Unary stretches of the trie (every member continues with the same page) are
// crossed in one scan, so the cost is about sum of shared pages plus a sort per
// branching node.
#include <algorithm>
#include <cstdint>
#include <utility>
#include <vector>

#include "ts_attn.h"

namespace ts {
ts_status fail(ts_status s, const char* fmt, ...);
}

namespace {

struct Grouper {
  const int32_t* bt;
  int64_t stride;
  const std::vector<int32_t>& cap;
  int min_group;
  std::vector<std::pair<int, std::vector<int32_t>>> groups;  // (depth, members)

  int32_t page(int32_t s, int d) const { return bt[s * stride + d]; }

  // Returns the members of the subtree rooted at (S, d) left ungrouped.
  std::vector<int32_t> visit(std::vector<int32_t> S, int d) {
    // cross the unary stretch: every member may go deeper and shares page d
    while (true) {
      bool extend = true;
      for (int32_t s : S)
        if (cap[s] <= d) {
          extend = false;
          break;
        }
      if (!extend) break;
      const int32_t p0 = page(S[0], d);
      for (int32_t s : S)
        if (page(s, d) != p0) {
          extend = false;
          break;
        }
      if (!extend) break;
      ++d;
    }
    std::vector<int32_t> left;
    std::vector<std::pair<int32_t, int32_t>> next;  // (page at depth d, sequence)
    for (int32_t s : S) {
      if (cap[s] <= d)
        left.push_back(s);
      else
        next.emplace_back(page(s, d), s);
    }
    std::sort(next.begin(), next.end());
    for (size_t i = 0; i < next.size();) {
      size_t j = i;
      while (j < next.size() && next[j].first == next[i].first) ++j;
      std::vector<int32_t> child;
      child.reserve(j - i);
      for (size_t t = i; t < j; ++t) child.push_back(next[t].second);
      if (static_cast<int>(child.size()) >= min_group) {
        std::vector<int32_t> rest = visit(std::move(child), d + 1);
        left.insert(left.end(), rest.begin(), rest.end());
      } else {
        left.insert(left.end(), child.begin(), child.end());
      }
      i = j;
    }
    if (d >= 1 && static_cast<int>(left.size()) >= min_group) {
      std::sort(left.begin(), left.end());
      groups.emplace_back(d, std::move(left));
      return {};
    }
    return left;
  }
};

}  // namespace

extern "C" ts_status ts_group_prefixes(const int32_t* block_table, int32_t bt_stride,
                                       const int32_t* seq_lens, int32_t B, int32_t page_size,
                                       int32_t min_group, ts_prefix_groups* out) {
  using ts::fail;
  if (!out) return fail(TS_ERR_INVALID_ARG, "ts_group_prefixes: null output");
  out->num_groups = 0;
  if (B < 0 || bt_stride <= 0 || page_size <= 0 || min_group < 2)
    return fail(TS_ERR_INVALID_ARG,
                "ts_group_prefixes: bad arguments (B=%d bt_stride=%d page_size=%d min_group=%d)", B,
                bt_stride, page_size, min_group);
  if (B > 0 && (!block_table || !seq_lens))
    return fail(TS_ERR_INVALID_ARG, "ts_group_prefixes: null block table or lengths");
  if (!out->prefix_indptr || !out->member_indptr || !out->prefix_len ||
      (B > 0 && (!out->member_ids || !out->group_of)) || out->capacity_groups < 0)
    return fail(TS_ERR_INVALID_ARG, "ts_group_prefixes: null output array");
  std::vector<int32_t> cap(static_cast<size_t>(B));
  std::vector<int32_t> roots;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t L = seq_lens[b];
    int64_t c = L > 0 ? (L - 1) / page_size : 0;
    if (c > bt_stride) c = bt_stride;
    cap[b] = static_cast<int32_t>(c);
    if (c >= 1) roots.push_back(b);
  }
  Grouper g{block_table, bt_stride, cap, min_group, {}};
  if (static_cast<int>(roots.size()) >= min_group) g.visit(std::move(roots), 0);

  const int32_t G = static_cast<int32_t>(g.groups.size());
  int64_t total_pages = 0, total_members = 0;
  for (const auto& gr : g.groups) {
    total_pages += gr.first;
    total_members += static_cast<int64_t>(gr.second.size());
  }
  if (G > out->capacity_groups || total_pages > out->capacity_prefix_pages ||
      total_members > out->capacity_members || (total_pages > 0 && !out->prefix_pages)) {
    out->num_groups = G;
    return fail(TS_ERR_CAPACITY,
                "ts_group_prefixes: need %d groups, %lld prefix pages, %lld members (capacities %d, "
                "%d, %d)",
                G, static_cast<long long>(total_pages), static_cast<long long>(total_members),
                out->capacity_groups, out->capacity_prefix_pages, out->capacity_members);
  }
  for (int32_t b = 0; b < B; ++b) out->group_of[b] = -1;
  int32_t pp = 0, mm = 0;
  out->prefix_indptr[0] = 0;
  out->member_indptr[0] = 0;
  for (int32_t gi = 0; gi < G; ++gi) {
    const int depth = g.groups[gi].first;
    const std::vector<int32_t>& members = g.groups[gi].second;
    for (int d = 0; d < depth; ++d)
      out->prefix_pages[pp++] = block_table[static_cast<int64_t>(members[0]) * bt_stride + d];
    out->prefix_indptr[gi + 1] = pp;
    out->prefix_len[gi] = depth * page_size;
    for (int32_t s : members) {
      out->member_ids[mm++] = s;
      out->group_of[s] = gi;
    }
    out->member_indptr[gi + 1] = mm;
  }
  out->num_groups = G;
  return TS_OK;
}
