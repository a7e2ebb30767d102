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

// ---------------------------------------------------------------------------
// ts_group_prefixes_nested: the same greedy search kept as a tree.
//
// Tokasaurus blog, "Dynamic prefix identification and exploration": the
// search iteratively finds the longest shared prefixes. Kept as a tree, a
// prefix shared by a large set and a longer one shared by a subset are both
// used: the short one once for the whole set, the extension once for the
// subset. Reading used here:
//   * a node is a maximal stretch of whole pages [d0, d1) shared by physical
//     page id by a set of at least min_group sequences that all share the
//     path above it and may all share d1 pages (cap, as above); its members
//     are all of them;
//   * at the node's end the members that can go deeper branch on the next
//     page; branches of at least min_group sequences become child nodes, the
//     others (and the members whose cap is reached) end at this node;
//   * a sequence's node is the deepest one it belongs to, so its shared depth
//     is the largest d for which at least min_group sequences (itself
//     included) share its first d pages within their caps;
//   * nodes are listed level by level (roots first), each level in visiting
//     order (increasing page ids), members in increasing sequence index.
// ---------------------------------------------------------------------------
namespace {

struct NestedGrouper {
  const int32_t* bt;
  int64_t stride;
  const std::vector<int32_t>& cap;
  int min_group;
  struct Node {
    int parent, level, d0, d1;
    std::vector<int32_t> members;
  };
  std::vector<Node> nodes;
  std::vector<int32_t> deepest;  // per sequence

  int32_t page(int32_t s, int d) const { return bt[s * stride + d]; }

  // end of the stretch that all of M share from depth d (>= d + 1: they share page d)
  int stretch_end(const std::vector<int32_t>& M, int d) const {
    int32_t lim = cap[M[0]];
    for (int32_t s : M) lim = std::min(lim, cap[s]);
    const int32_t* r0 = bt + static_cast<int64_t>(M[0]) * stride;
    int32_t e = lim;
    for (size_t i = 1; i < M.size() && e > d + 1; ++i) {
      const int32_t* rs = bt + static_cast<int64_t>(M[i]) * stride;
      if (std::memcmp(rs + d, r0 + d, static_cast<size_t>(e - d) * sizeof(int32_t)) == 0) continue;
      int32_t t = d;
      while (t < e && rs[t] == r0[t]) ++t;
      e = t;
    }
    return e;
  }

  // S: sequences sharing pages [0, d) under `parent`; branch on page d.
  void branch(const std::vector<int32_t>& S, int d, int parent, int level) {
    std::vector<std::pair<int32_t, int32_t>> keyed;  // (page at d, sequence)
    keyed.reserve(S.size());
    for (int32_t s : S)
      if (cap[s] > d) keyed.emplace_back(page(s, d), s);
    std::sort(keyed.begin(), keyed.end());
    for (size_t i = 0; i < keyed.size();) {
      size_t j = i;
      while (j < keyed.size() && keyed[j].first == keyed[i].first) ++j;
      if (static_cast<int>(j - i) >= min_group) {
        std::vector<int32_t> M;
        M.reserve(j - i);
        for (size_t t = i; t < j; ++t) M.push_back(keyed[t].second);  // increasing index
        const int e = stretch_end(M, d);
        const int id = static_cast<int>(nodes.size());
        nodes.push_back(Node{parent, level, d, e, M});
        for (int32_t s : M) deepest[s] = id;
        branch(M, e, id, level + 1);
      }
      i = j;
    }
  }
};

}  // namespace

extern "C" ts_status ts_group_prefixes_nested(const int32_t* block_table, int32_t bt_stride,
                                              const int32_t* seq_lens, int32_t B, int32_t page_size,
                                              int32_t min_group, ts_prefix_forest* out) {
  using ts::fail;
  const char* who = "ts_group_prefixes_nested";
  if (!out) return fail(TS_ERR_INVALID_ARG, "%s: null output", who);
  out->num_nodes = 0;
  out->num_levels = 0;
  if (B < 0 || bt_stride <= 0 || page_size <= 0 || min_group < 2)
    return fail(TS_ERR_INVALID_ARG, "%s: bad arguments (B=%d bt_stride=%d page_size=%d min_group=%d)", who, B,
                bt_stride, page_size, min_group);
  if (B > 0 && (!block_table || !seq_lens)) return fail(TS_ERR_INVALID_ARG, "%s: null block table or lengths", who);
  if (!out->prefix_indptr || !out->member_indptr || !out->prefix_len || !out->level_indptr || !out->parent ||
      (B > 0 && (!out->member_ids || !out->group_of)) || out->capacity_nodes < 0)
    return fail(TS_ERR_INVALID_ARG, "%s: null output array", who);
  std::vector<int32_t> cap(static_cast<size_t>(B));
  std::vector<int32_t> all;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t L = seq_lens[b];
    int64_t c = L > 0 ? (L - 1) / page_size : 0;
    if (c > bt_stride) c = bt_stride;
    cap[b] = static_cast<int32_t>(c);
    all.push_back(b);
  }
  NestedGrouper g{block_table, bt_stride, cap, min_group, {}, std::vector<int32_t>(static_cast<size_t>(B), -1)};
  g.branch(all, 0, -1, 0);

  // level order: stable by level keeps each level's visiting order
  const int32_t N = static_cast<int32_t>(g.nodes.size());
  std::vector<int32_t> order(static_cast<size_t>(N));
  for (int32_t i = 0; i < N; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return g.nodes[a].level < g.nodes[b].level; });
  std::vector<int32_t> rank(static_cast<size_t>(N));
  for (int32_t i = 0; i < N; ++i) rank[order[i]] = i;
  int32_t levels = 0;
  int64_t total_pages = 0, total_members = 0;
  for (const auto& nd : g.nodes) {
    levels = std::max(levels, nd.level + 1);
    total_pages += nd.d1 - nd.d0;
    total_members += static_cast<int64_t>(nd.members.size());
  }
  if (N > out->capacity_nodes || levels > out->capacity_levels || total_pages > out->capacity_prefix_pages ||
      total_members > out->capacity_members || (total_pages > 0 && !out->prefix_pages)) {
    out->num_nodes = N;
    out->num_levels = levels;
    return fail(TS_ERR_CAPACITY,
                "%s: need %d nodes, %d levels, %lld prefix pages, %lld members (capacities %d, %d, %d, %d)", who,
                N, levels, static_cast<long long>(total_pages), static_cast<long long>(total_members),
                out->capacity_nodes, out->capacity_levels, out->capacity_prefix_pages, out->capacity_members);
  }
  int32_t pp = 0, mm = 0;
  out->prefix_indptr[0] = 0;
  out->member_indptr[0] = 0;
  for (int32_t l = 0; l <= levels; ++l) out->level_indptr[l] = 0;
  for (int32_t i = 0; i < N; ++i) {
    const auto& nd = g.nodes[order[i]];
    out->level_indptr[nd.level + 1] = i + 1;
    for (int d = nd.d0; d < nd.d1; ++d)
      out->prefix_pages[pp++] = block_table[static_cast<int64_t>(nd.members[0]) * bt_stride + d];
    out->prefix_indptr[i + 1] = pp;
    out->prefix_len[i] = nd.d1 * page_size;  // tokens shared from the root through this node
    out->parent[i] = nd.parent >= 0 ? rank[nd.parent] : -1;
    for (int32_t s : nd.members) out->member_ids[mm++] = s;
    out->member_indptr[i + 1] = mm;
  }
  for (int32_t b = 0; b < B; ++b) out->group_of[b] = g.deepest[b] >= 0 ? rank[g.deepest[b]] : -1;
  out->num_nodes = N;
  out->num_levels = levels;
  return TS_OK;
}
