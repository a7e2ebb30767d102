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
// crossed in one pass along each member's row (contiguous memory), so the cost
// is about the sum of shared pages plus a sort per branching node.
#include <algorithm>
#include <cstdint>
#include <cstring>
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
    // cross the unary stretch (every member may go deeper and shares the
    // page) in one pass along each member's row: it ends at the smallest cap
    // or at the first page where some row differs from the first member's
    {
      int32_t lim = cap[S[0]];
      for (int32_t s : S) lim = std::min(lim, cap[s]);
      if (lim > d) {
        const int32_t* r0 = bt + static_cast<int64_t>(S[0]) * stride;
        int32_t e = lim;
        for (size_t i = 1; i < S.size() && e > d; ++i) {
          const int32_t* rs = bt + static_cast<int64_t>(S[i]) * stride;
          if (std::memcmp(rs + d, r0 + d, static_cast<size_t>(e - d) * sizeof(int32_t)) == 0) continue;
          int32_t t = d;
          while (t < e && rs[t] == r0[t]) ++t;
          e = t;
        }
        d = e;
      }
    }
    // Branch on the page at depth d. Pages are counted in a hash table first,
    // so only pages held by at least min_group members become children
    // (visited in increasing page id); all others stay with this node.
    std::vector<int32_t> left;
    size_t cap2 = 16;
    while (cap2 < 2 * S.size()) cap2 <<= 1;
    std::vector<int32_t> key(cap2, 0), cnt(cap2, 0), child_of(cap2, -1);
    std::vector<uint8_t> used(cap2, 0);
    auto slot = [&](int32_t pg) {  // any int32 is a valid key (bad page ids included)
      size_t h = (static_cast<uint32_t>(pg) * 2654435761u) & (cap2 - 1);
      while (used[h] && key[h] != pg) h = (h + 1) & (cap2 - 1);
      return h;
    };
    for (int32_t s : S) {
      if (cap[s] <= d) continue;
      const size_t h = slot(page(s, d));
      used[h] = 1;
      key[h] = page(s, d);
      ++cnt[h];
    }
    std::vector<std::pair<int32_t, size_t>> kids;  // (page, table slot) of children
    for (size_t h = 0; h < cap2; ++h)
      if (used[h] && cnt[h] >= min_group) kids.emplace_back(key[h], h);
    std::sort(kids.begin(), kids.end());
    std::vector<std::vector<int32_t>> members(kids.size());
    for (size_t c = 0; c < kids.size(); ++c) {
      child_of[kids[c].second] = static_cast<int32_t>(c);
      members[c].reserve(cnt[kids[c].second]);
    }
    for (int32_t s : S) {  // S is in increasing sequence order, and so are the children
      if (cap[s] <= d) {
        left.push_back(s);
        continue;
      }
      const int32_t c = child_of[slot(page(s, d))];
      if (c >= 0)
        members[c].push_back(s);
      else
        left.push_back(s);
    }
    for (size_t c = 0; c < kids.size(); ++c) {
      std::vector<int32_t> rest = visit(std::move(members[c]), d + 1);
      left.insert(left.end(), rest.begin(), rest.end());
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
