"""The host grouping pass ts_group_prefixes (C++, through the C ABI), checked by
the oracle's invariant checker (CPU only)."""

import time

import numpy as np
import pytest

import paged_kv_cache_46_gb300 as ts
import workloads
import oracle
from oracle import PrefixGroups, check_prefix_groups
from paged_kv_cache_46_gb300 import build as ts_build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ts_build.build()


def _as_oracle(g):
    return PrefixGroups(g["prefix_indptr"], g["prefix_pages"], g["prefix_len"], g["member_indptr"],
                        g["member_ids"], num_groups=g["num_groups"])


def _check(bt, lens, ps, min_group=2):
    g = ts.ts_group_prefixes(bt, lens, ps, min_group)
    errs = check_prefix_groups(bt, lens, ps, min_group, _as_oracle(g))
    assert errs == [], errs[:5]
    for gi in range(g["num_groups"]):
        members = g["member_ids"][g["member_indptr"][gi]:g["member_indptr"][gi + 1]]
        assert np.all(g["group_of"][members] == gi)
    assert np.sum(g["group_of"] >= 0) == len(g["member_ids"])
    return g


def test_hand_example():
    bt = np.array([[10, 11, 12, 13, 0], [10, 11, 12, 14, 0], [10, 11, 15, 0, 0], [10, 11, 16, 0, 0],
                   [20, 21, 0, 0, 0], [20, 22, 0, 0, 0], [30, 31, 32, 33, 0], [10, 0, 0, 0, 0]], dtype=np.int32)
    lens = np.array([14, 16, 10, 9, 6, 8, 13, 4], dtype=np.int32)
    g = _check(bt, lens, 4)
    got = {(tuple(g["prefix_pages"][g["prefix_indptr"][i]:g["prefix_indptr"][i + 1]]),
            tuple(g["member_ids"][g["member_indptr"][i]:g["member_indptr"][i + 1]])) for i in range(g["num_groups"])}
    assert got == {((10, 11, 12), (0, 1)), ((10, 11), (2, 3)), ((20,), (4, 5))}
    # min_group 3: only 0-3 (shared [10, 11]) qualify
    g = ts.ts_group_prefixes(bt, lens, 4, 3)
    assert g["num_groups"] == 1 and list(g["member_ids"]) == [0, 1, 2, 3] and list(g["prefix_pages"]) == [10, 11]


def test_cascade_workload_recovers_constructed_groups():
    """Shared-prefix cascade workload (16 groups x 1024, 2048-token prefixes):
    the pass recovers exactly the constructed groups."""
    case = workloads.shared_prefix_cascade(values=False)
    t = time.perf_counter()
    g = _check(case.block_table, case.seq_lens, 16)
    elapsed = time.perf_counter() - t
    assert g["num_groups"] == 16
    assert np.all(g["prefix_len"] == 2048)
    truth = {tuple(np.sort(m)) for m in case.groups_truth}
    got = {tuple(g["member_ids"][g["member_indptr"][i]:g["member_indptr"][i + 1]]) for i in range(16)}
    assert got == truth
    assert elapsed < 5.0


def test_cascade_with_ungrouped_and_short_members():
    case = workloads.shared_prefix_cascade(groups=5, members=7, prefix_tokens=64, suffix_lo=1, suffix_hi=40,
                                           ungrouped=9, values=False)
    g = _check(case.block_table, case.seq_lens, 16)
    assert g["num_groups"] == 5


def _random_tree_case(seed):
    rng = np.random.default_rng(seed)
    ps = int(rng.choice([4, 16]))
    B = int(rng.integers(2, 120))
    max_pages = 24
    bt = np.zeros((B, max_pages), dtype=np.int32)
    next_page = 0
    for b in range(B):
        if b > 0 and rng.random() < 0.7:
            src = int(rng.integers(0, b))
            k = int(rng.integers(1, max_pages))
            bt[b, :k] = bt[src, :k]
        else:
            k = 0
        for j in range(k, max_pages):
            bt[b, j] = next_page
            next_page += 1
    lens = rng.integers(0, max_pages * ps + 1, size=B).astype(np.int32)
    return bt, lens, ps


@pytest.mark.parametrize("seed", range(6))
def test_random_nested_prefix_trees(seed):
    """Random nested sharing: sequences copy a random-length prefix of another
    sequence's block-table row (a random tree of shared prefixes)."""
    bt, lens, ps = _random_tree_case(seed)
    for min_group in (2, 3):
        _check(bt, lens, ps, min_group)


def _one_level_grouper(bt, lens, ps, min_group):
    """A planted mistake: each run of sequences sharing a first page becomes one
    group at the run's longest common prefix (within every member's cap), and
    the search never goes deeper into sub-runs."""
    caps = [(int(L) - 1) // ps if L > 0 else 0 for L in lens]
    runs = {}
    for b in range(len(lens)):
        if caps[b] >= 1:
            runs.setdefault(int(bt[b, 0]), []).append(b)
    groups = []
    for _, members in sorted(runs.items()):
        if len(members) < min_group:
            continue
        n = 0
        while n < min(caps[m] for m in members) and len({int(bt[m, n]) for m in members}) == 1:
            n += 1
        groups.append((bt[members[0], :n].tolist(), members))
    pi, pp, pl, mi, mm = [0], [], [], [0], []
    for pages, members in groups:
        pp += pages
        pi.append(len(pp))
        pl.append(len(pages) * ps)
        mm += members
        mi.append(len(mm))
    return PrefixGroups(np.array(pi), np.array(pp, np.int64), np.array(pl), np.array(mi),
                        np.array(mm, np.int64), num_groups=len(groups))


def test_one_level_grouper_fails_on_random_trees():
    """The checker is not satisfied by a grouper that stops at the first level:
    wherever its output differs from the greedy pass's, it is reported."""
    differing = 0
    for seed in range(6):
        bt, lens, ps = _random_tree_case(seed)
        for min_group in (2, 3):
            good = _as_oracle(ts.ts_group_prefixes(bt, lens, ps, min_group))
            shallow = _one_level_grouper(bt, lens, ps, min_group)
            as_sets = lambda g: {(tuple(p.tolist()), tuple(sorted(m.tolist()))) for _, p, _, m in g.groups()}
            if as_sets(good) == as_sets(shallow):
                assert check_prefix_groups(bt, lens, ps, min_group, shallow) == []
                continue
            differing += 1
            errs = check_prefix_groups(bt, lens, ps, min_group, shallow)
            assert any("not deepest-first" in e for e in errs), (seed, min_group, errs[:3])
    assert differing >= 6


def test_capacity_and_argument_errors():
    bt = np.array([[1, 2], [1, 3]], dtype=np.int32)
    lens = np.array([20, 20], dtype=np.int32)
    with pytest.raises(ts.TSError) as e:
        ts.ts_group_prefixes(bt, lens, 16, 1)
    assert e.value.status == ts.TS_ERR_INVALID_ARG
    g = ts.ts_group_prefixes(bt, lens, 16, 2)
    assert g["num_groups"] == 1 and list(g["prefix_pages"]) == [1]
    g = ts.ts_group_prefixes(np.zeros((0, 4), np.int32), np.zeros(0, np.int32), 16, 2)
    assert g["num_groups"] == 0


# ---------------------------------------------------------------------------
# Nested (tree) grouping: ts_group_prefixes_nested against the invariant
# checker, whose maximality pin is a brute-force search.
# ---------------------------------------------------------------------------

def _check_forest(bt, lens, ps, min_group=2):
    f = ts.ts_group_prefixes_nested(bt, lens, ps, min_group)
    oracle.check_prefix_forest(bt, lens, ps, min_group, f)
    return f


def test_forest_hand_example():
    # pages: 0-3 = system prompt (4 pages); seqs 0-3 share it; 0,1 share 2 more pages; 4 is alone
    ps = 4
    bt = np.array([[0, 1, 2, 3, 10, 11, 20, 21],
                   [0, 1, 2, 3, 10, 11, 22, 23],
                   [0, 1, 2, 3, 12, 13, 24, 25],
                   [0, 1, 2, 3, 14, 15, 26, 27],
                   [30, 31, 32, 33, 34, 35, 36, 37]], np.int32)
    lens = np.array([29, 32, 20, 30, 32], np.int32)
    f = _check_forest(bt, lens, ps)
    assert f["num_nodes"] == 2 and f["num_levels"] == 2
    assert f["prefix_len"].tolist() == [16, 24]
    assert f["prefix_pages"].tolist() == [0, 1, 2, 3, 10, 11]
    assert f["member_ids"].tolist() == [0, 1, 2, 3, 0, 1]
    assert f["group_of"].tolist() == [1, 1, 0, 0, -1] and f["parent"].tolist() == [-1, 0]


def test_forest_cap_splits_a_stretch():
    # all three share 6 pages, but sequence 2 may share only 3 (length 13, page 4)
    ps = 4
    bt = np.array([[5, 6, 7, 8, 9, 1, 40], [5, 6, 7, 8, 9, 1, 41], [5, 6, 7, 8, 9, 1, 42]], np.int32)
    lens = np.array([28, 25, 13], np.int32)
    f = _check_forest(bt, lens, ps)
    assert f["prefix_len"].tolist() == [12, 24] and f["group_of"].tolist() == [1, 1, 0]


@pytest.mark.parametrize("seed", range(6))
def test_forest_random_prefix_trees(seed):
    rng = np.random.default_rng(100 + seed)
    B, ps, depth = 40, 4, 12
    # random tree: each sequence walks down a small random trie of shared pages
    bt = np.zeros((B, depth), np.int32)
    nxt = [1000]
    children = {}
    for b in range(B):
        node = ()
        for d in range(depth):
            kids = children.setdefault(node, [])
            if kids and rng.random() < 0.7:
                pg = kids[rng.integers(len(kids))]
            else:
                pg = nxt[0]
                nxt[0] += 1
                kids.append(pg)
            bt[b, d] = pg
            node = node + (pg,)
    lens = rng.integers(1, depth * ps + 1, size=B).astype(np.int32)
    for mg in (2, 3, 5):
        _check_forest(bt, lens, ps, mg)


def test_forest_on_the_cascade_workload_structure():
    case = workloads.shared_prefix_cascade(groups=2, members=64, values=False)
    f = _check_forest(case.block_table, case.attn_lens, case.page_size)
    assert f["num_levels"] >= 1 and set(f["group_of"].tolist()) != {-1}


def test_forest_arguments():
    bt = np.zeros((2, 2), np.int32)
    lens = np.array([9, 9], np.int32)
    with pytest.raises(ts.TSError):
        ts.ts_group_prefixes_nested(bt, lens, 4, 1)  # min_group < 2
    f = ts.ts_group_prefixes_nested(np.zeros((0, 1), np.int32), np.zeros(0, np.int32), 4)
    assert f["num_nodes"] == 0


def _hand_forest_case():
    ps = 4
    bt = np.array([[0, 1, 2, 3, 10, 11, 20, 21],
                   [0, 1, 2, 3, 10, 11, 22, 23],
                   [0, 1, 2, 3, 12, 13, 24, 25],
                   [0, 1, 2, 3, 14, 15, 26, 27],
                   [30, 31, 32, 33, 34, 35, 36, 37]], np.int32)
    lens = np.array([29, 32, 20, 30, 32], np.int32)
    return bt, lens, ps


def test_shared_depth_brute_force_hand_values():
    """The brute-force shared depth on the hand example: sequences 0 and 1
    share 6 pages, 2 and 3 only the 4-page system prompt, 4 nothing; with
    min_group 3 the pair's deeper stretch no longer counts."""
    bt, lens, ps = _hand_forest_case()
    assert oracle.shared_depth_brute_force(bt, lens, ps, 2).tolist() == [6, 6, 4, 4, 0]
    assert oracle.shared_depth_brute_force(bt, lens, ps, 3).tolist() == [4, 4, 4, 4, 0]
    assert oracle.shared_depth_brute_force(bt, lens, ps, 5).tolist() == [0, 0, 0, 0, 0]


def _copy_forest(f):
    return {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in f.items()}


def test_forest_checker_rejects_planted_mistakes():
    """Mistakes planted in a valid forest are caught: a member dropped from
    the deeper node (its sequence's shared depth is no longer the largest), a
    node's stretch cut short, a sequence pointed at a shallower node, and a
    member that does not share the node's pages."""
    bt, lens, ps = _hand_forest_case()
    good = ts.ts_group_prefixes_nested(bt, lens, ps, 2)
    oracle.check_prefix_forest(bt, lens, ps, 2, good)

    bad = _copy_forest(good)   # node 1 loses member 1
    bad["member_ids"] = np.array([0, 1, 2, 3, 0], np.int32)
    bad["member_indptr"] = np.array([0, 4, 5], np.int32)
    bad["group_of"] = np.array([1, 0, 0, 0, -1], np.int32)
    with pytest.raises(AssertionError):
        oracle.check_prefix_forest(bt, lens, ps, 2, bad)

    bad = _copy_forest(good)   # node 1's stretch cut to one page
    bad["prefix_pages"] = np.array([0, 1, 2, 3, 10], np.int32)
    bad["prefix_indptr"] = np.array([0, 4, 5], np.int32)
    bad["prefix_len"] = np.array([16, 20], np.int32)
    with pytest.raises(AssertionError):
        oracle.check_prefix_forest(bt, lens, ps, 2, bad)

    bad = _copy_forest(good)   # sequence 0 pointed at the root instead of its deepest node
    bad["group_of"] = np.array([0, 1, 0, 0, -1], np.int32)
    with pytest.raises(AssertionError):
        oracle.check_prefix_forest(bt, lens, ps, 2, bad)

    bad = _copy_forest(good)   # sequence 4 planted into the root it does not share
    bad["member_ids"] = np.array([0, 1, 2, 3, 4, 0, 1], np.int32)
    bad["member_indptr"] = np.array([0, 5, 7], np.int32)
    bad["group_of"] = np.array([1, 1, 0, 0, 0], np.int32)
    with pytest.raises(AssertionError):
        oracle.check_prefix_forest(bt, lens, ps, 2, bad)
