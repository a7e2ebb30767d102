"""Invariant checker for shared-prefix groups. TEST INFRASTRUCTURE ONLY.

Tokasaurus blog (Stanford), "Dynamic prefix identification and exploration":
before every forward pass a greedy depth-first search iteratively finds the
longest possible shared prefixes, so that attention over each shared prefix
can be computed once for the whole group (Hydragen / cascade attention).

The pages fix no tie-break, depth or data format, so several groupings can be
valid. This module therefore does not re-implement the search; it checks the
properties any output of the reading below must have (several correct results:
compare what is unique, check the rest is valid):

* prefixes are whole pages, shared *by physical page id* in the block table;
* every member keeps at least one suffix token (``n_pages * page_size <= L - 1``);
* each sequence is in at most one group, and every group has at least
  ``min_group`` members;
* a group's prefix is maximal: its members do not all share the next page too;
* greedy longest-first: a sequence that starts with a group's whole prefix
  (and may share that many pages) is in that group or in a deeper one;
* deepest first, at every depth d: no ``min_group`` sequences placed
  shallower than d (ungrouped = depth 0) share their first d pages within
  their caps, since the search would have grouped them at depth d first;
* nothing is missed: among ungrouped sequences that could share a page, no
  ``min_group`` of them start with the same page id.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List

import numpy as np


@dataclass
class PrefixGroups:
    """Single-level prefix groups in CSR form (host copy).

    prefix_indptr[G+1] / prefix_pages: each group's shared physical page ids.
    prefix_len[G]: shared tokens (= pages * page_size).
    member_indptr[G+1] / member_ids: the sequences of each group.
    """

    prefix_indptr: np.ndarray
    prefix_pages: np.ndarray
    prefix_len: np.ndarray
    member_indptr: np.ndarray
    member_ids: np.ndarray
    num_groups: int = field(default=0)

    def groups(self):
        for gi in range(self.num_groups):
            pages = self.prefix_pages[self.prefix_indptr[gi]:self.prefix_indptr[gi + 1]]
            members = self.member_ids[self.member_indptr[gi]:self.member_indptr[gi + 1]]
            yield gi, pages, int(self.prefix_len[gi]), members


def shareable_pages(seq_len: int, page_size: int) -> int:
    """Whole pages a sequence may share while keeping >= 1 suffix token."""
    return max(0, (int(seq_len) - 1) // page_size)


def check_prefix_groups(block_table, seq_lens, page_size: int, min_group: int,
                        groups: PrefixGroups) -> List[str]:
    """Return a list of violated invariants (empty when ``groups`` is valid)."""
    bt = np.asarray(block_table)
    lens = np.asarray(seq_lens)
    B = len(lens)
    errors: List[str] = []
    owner = np.full(B, -1, dtype=np.int64)
    for gi, pages, plen, members in groups.groups():
        n = len(pages)
        if n < 1:
            errors.append(f"group {gi}: empty prefix")
            continue
        if plen != n * page_size:
            errors.append(f"group {gi}: prefix_len {plen} != {n} pages * {page_size}")
        if len(members) < min_group:
            errors.append(f"group {gi}: {len(members)} members < min_group {min_group}")
        for b in members:
            b = int(b)
            if not 0 <= b < B:
                errors.append(f"group {gi}: member {b} out of range")
                continue
            if owner[b] >= 0:
                errors.append(f"sequence {b} in groups {owner[b]} and {gi}")
            owner[b] = gi
            if n > shareable_pages(lens[b], page_size):
                errors.append(f"group {gi}: member {b} (L={lens[b]}) keeps no suffix token")
                continue
            if not np.array_equal(bt[b, :n], pages):
                errors.append(f"group {gi}: member {b} does not start with the group prefix")
        # maximality: not every member shares page n as well
        valid = [int(b) for b in members if 0 <= int(b) < B]
        if valid and all(shareable_pages(lens[b], page_size) > n for b in valid):
            nxt = {int(bt[b, n]) for b in valid}
            if len(nxt) == 1:
                errors.append(f"group {gi}: prefix not maximal (all members share page {n})")
    # greedy longest-first: whoever starts with a group's whole prefix belongs
    # to it or to a deeper group
    depth = np.zeros(B, dtype=np.int64)
    for gi, pages, plen, members in groups.groups():
        for b in members:
            if 0 <= int(b) < B:
                depth[int(b)] = len(pages)
    caps = np.maximum(0, (lens.astype(np.int64) - 1) // page_size)
    for gi, pages, plen, members in groups.groups():
        n = len(pages)
        if n < 1 or n > bt.shape[1]:
            continue
        starts = np.all(bt[:, :n] == np.asarray(pages)[None, :], axis=1) & (caps >= n)
        bad = np.nonzero(starts & (owner != gi) & (depth <= n))[0]
        for b in bad[:5]:
            errors.append(f"sequence {b} starts with group {gi}'s prefix but is not in it or deeper")
    # completeness: ungrouped sequences with a shareable first page
    first_counts = {}
    for b in range(B):
        if owner[b] < 0 and shareable_pages(lens[b], page_size) >= 1:
            first_counts.setdefault(int(bt[b, 0]), []).append(b)
    for page, seqs in first_counts.items():
        if len(seqs) >= min_group:
            errors.append(f"{len(seqs)} ungrouped sequences share first page {page}")
    errors.extend(_deepest_first_violations(bt, caps, depth, min_group))
    return errors


def _deepest_first_violations(bt, caps, depth, min_group: int) -> List[str]:
    """Greedy deepest shared prefix first, checked at every depth d: among the
    sequences placed shallower than d (ungrouped counts as depth 0) that may
    share d pages, no ``min_group`` share the same first d page ids. If they
    did, the greedy search would have formed their depth-d group before
    settling any of them higher up.

    Exhaustive over d; the first d pages of each row are identified by
    interning (id of the first d-1 pages, page d-1) pairs, so every depth
    costs one pass over the rows."""
    B = bt.shape[0]
    errors: List[str] = []
    max_d = int(min(caps.max(initial=0), bt.shape[1]))
    prefix_id = np.zeros(B, dtype=np.int64)
    for d in range(1, max_d + 1):
        pairs = np.stack([prefix_id, bt[:, d - 1].astype(np.int64)], axis=1)
        _, prefix_id = np.unique(pairs, axis=0, return_inverse=True)
        prefix_id = prefix_id.reshape(-1)
        open_rows = np.nonzero((caps >= d) & (depth < d))[0]
        if len(open_rows) < min_group:
            continue
        ids, counts = np.unique(prefix_id[open_rows], return_counts=True)
        for pid in ids[counts >= min_group][:5]:
            seqs = open_rows[prefix_id[open_rows] == pid]
            errors.append(f"sequences {seqs[:8].tolist()} share their first {d} pages but are placed "
                          f"shallower (not deepest-first)")
    return errors


def shared_depth_brute_force(block_table, seq_lens, page_size: int, min_group: int) -> np.ndarray:
    """Per sequence: the largest d such that at least ``min_group`` sequences
    (itself included) share its first d pages by id, each within its cap
    ((L - 1) // page_size pages). Plain O(B^2 * depth) search for small inputs."""
    bt = np.asarray(block_table)
    B = len(seq_lens)
    cap = [shareable_pages(seq_lens[b], page_size) for b in range(B)]
    out = np.zeros(B, dtype=np.int64)
    for b in range(B):
        for d in range(cap[b], 0, -1):
            n = sum(1 for t in range(B) if cap[t] >= d and np.array_equal(bt[t, :d], bt[b, :d]))
            if n >= min_group:
                out[b] = d
                break
    return out


def check_prefix_forest(block_table, seq_lens, page_size: int, min_group: int, forest: dict):
    """Invariants of a nested (tree) grouping, raising AssertionError on the first violation.

    Tokasaurus blog, "Dynamic prefix identification and exploration" (greedy
    search for the longest shared prefixes), kept as a tree: nodes level by
    level, each node a stretch of whole pages shared by id by all its members
    below its parent's path, members within their caps, at least
    ``min_group`` members, children's members inside their parent's, and
    every sequence's shared depth the largest possible (brute force).
    """
    bt = np.asarray(block_table)
    B = len(seq_lens)
    N = int(forest["num_nodes"])
    lvl = forest["level_indptr"]
    ptr, pages, plen = forest["prefix_indptr"], forest["prefix_pages"], forest["prefix_len"]
    mptr, mids, parent, group_of = forest["member_indptr"], forest["member_ids"], forest["parent"], forest["group_of"]
    level_of = np.full(N, -1)
    for l in range(int(forest["num_levels"])):
        level_of[lvl[l]:lvl[l + 1]] = l
    assert N == 0 or (lvl[0] == 0 and lvl[-1] == N and np.all(level_of >= 0)), "level ranges"
    members = [set(mids[mptr[i]:mptr[i + 1]].tolist()) for i in range(N)]
    depth_end = plen // page_size
    for i in range(N):
        par = int(parent[i])
        assert (par == -1) == (level_of[i] == 0), f"node {i}: roots are exactly level 0"
        d0 = 0 if par < 0 else int(depth_end[par])
        if par >= 0:
            assert level_of[par] == level_of[i] - 1 and members[i] <= members[par], f"node {i}: parent"
        d1 = int(depth_end[i])
        own = pages[ptr[i]:ptr[i + 1]]
        assert plen[i] % page_size == 0 and d1 - d0 == len(own) >= 1, f"node {i}: stretch"
        assert len(members[i]) >= min_group, f"node {i}: {len(members[i])} members"
        m_sorted = mids[mptr[i]:mptr[i + 1]]
        assert np.all(np.diff(m_sorted) > 0), f"node {i}: members not increasing"
        for m in members[i]:
            assert shareable_pages(seq_lens[m], page_size) >= d1, f"node {i}: member {m} over its cap"
            assert np.array_equal(bt[m, d0:d1], own), f"node {i}: member {m} does not share the pages"
        # maximal stretch: the members do not all continue with one more shared page
        ext = [m for m in members[i] if shareable_pages(seq_lens[m], page_size) > d1]
        assert not (len(ext) == len(members[i]) and len({int(bt[m, d1]) for m in ext}) == 1), \
            f"node {i}: stretch could go on"
    # each sequence's node is the deepest holding it, on one chain, at the largest shared depth
    want = shared_depth_brute_force(bt, seq_lens, page_size, min_group)
    for b in range(B):
        holding = [i for i in range(N) if b in members[i]]
        g = int(group_of[b])
        if not holding:
            assert g == -1 and want[b] == 0, f"sequence {b}: ungrouped but depth {want[b]} is shared"
            continue
        assert g == max(holding, key=lambda i: depth_end[i]), f"sequence {b}: not its deepest node"
        chain, i = set(), g
        while i >= 0:
            chain.add(i)
            i = int(parent[i])
        assert chain == set(holding), f"sequence {b}: nodes off its chain"
        assert depth_end[g] == want[b], f"sequence {b}: shared depth {depth_end[g]} != {want[b]}"
