"""Pins for the shared-prefix group checker (CPU only).

The checker is pinned by hand-built groupings whose validity is known, by the
ground truth of the cascade workload's own construction, and by planted
mistakes (one per invariant) that it must report.
"""

import numpy as np

import workloads
from oracle import PrefixGroups, check_prefix_groups


def _csr(groups, page_size):
    """groups: list of (prefix_pages, members)."""
    pi, pp, pl, mi, mm = [0], [], [], [0], []
    for pages, members in groups:
        pp.extend(pages)
        pi.append(len(pp))
        pl.append(len(pages) * page_size)
        mm.extend(members)
        mi.append(len(mm))
    return PrefixGroups(np.array(pi), np.array(pp, dtype=np.int64), np.array(pl),
                        np.array(mi), np.array(mm, dtype=np.int64), num_groups=len(groups))


# Hand example, page size 4. Sequences 0-3 share pages [10, 11]; 0 and 1 also
# share page 12; 4 and 5 share [20]; 6 owns its pages; 7 shares page 10 but is
# only 4 tokens long, so it may share nothing (it must keep one suffix token).
BT = np.array([
    [10, 11, 12, 13, 0],
    [10, 11, 12, 14, 0],
    [10, 11, 15, 0, 0],
    [10, 11, 16, 0, 0],
    [20, 21, 0, 0, 0],
    [20, 22, 0, 0, 0],
    [30, 31, 32, 33, 0],
    [10, 0, 0, 0, 0],
])
LENS = np.array([14, 16, 10, 9, 6, 8, 13, 4])
GOOD = [([10, 11, 12], [0, 1]), ([10, 11], [2, 3]), ([20], [4, 5])]


def test_valid_hand_grouping_passes():
    assert check_prefix_groups(BT, LENS, 4, 2, _csr(GOOD, 4)) == []


def test_shallow_grouping_is_rejected_as_not_greedy():
    # One group at depth 2 for 0-3 covers every sequence and is maximal (0-3 do
    # not all share page 12), but it is not deepest-first: 0 and 1 share three
    # pages and sit at depth 2.
    shallow = [([10, 11], [0, 1, 2, 3]), ([20], [4, 5])]
    errs = check_prefix_groups(BT, LENS, 4, 2, _csr(shallow, 4))
    assert any("[0, 1] share their first 3 pages" in e for e in errs), errs
    assert not any("maximal" in e for e in errs)
    # 0 and 1 left out entirely is caught as well
    only_deep_missing = [([10, 11], [2, 3]), ([20], [4, 5])]
    errs = check_prefix_groups(BT, LENS, 4, 2, _csr(only_deep_missing, 4))
    assert any("not in it or deeper" in e for e in errs)
    assert any("[0, 1] share their first 3 pages" in e for e in errs)


def test_deepest_first_keeps_a_leftover_ungrouped():
    # 0 and 1 share [10, 11, 12]; 2 shares only [10, 11]. Deepest-first groups
    # 0 and 1 at depth 3 and leaves 2 alone (fewer than min_group = 2), which is
    # valid; pulling all three into [10, 11] is not.
    bt = np.array([[10, 11, 12, 13], [10, 11, 12, 14], [10, 11, 15, 0]])
    lens = np.array([16, 16, 12])
    assert check_prefix_groups(bt, lens, 4, 2, _csr([([10, 11, 12], [0, 1])], 4)) == []
    errs = check_prefix_groups(bt, lens, 4, 2, _csr([([10, 11], [0, 1, 2])], 4))
    assert any("share their first 3 pages" in e for e in errs), errs
    # with min_group 3 the pair does not qualify, so [10, 11] for all three is right
    assert check_prefix_groups(bt, lens, 4, 3, _csr([([10, 11], [0, 1, 2])], 4)) == []
    # the cap counts: if 1 may share only 2 pages, 0 alone is left at depth 3
    lens_capped = np.array([16, 12, 12])
    assert check_prefix_groups(bt, lens_capped, 4, 2, _csr([([10, 11], [0, 1, 2])], 4)) == []


def test_planted_mistakes_are_reported():
    cases = {
        "not start with": [([10, 11, 12], [0, 1, 6]), ([10, 11], [2, 3]), ([20], [4, 5])],
        "keeps no suffix": [([10, 11, 12], [0, 1]), ([10, 11], [2, 3]), ([20, 21], [4, 5])],
        "min_group": [([10, 11, 12], [0]), ([10, 11], [1, 2, 3]), ([20], [4, 5])],
        "in groups": [([10, 11, 12], [0, 1]), ([10, 11], [1, 2, 3]), ([20], [4, 5])],
        "not maximal": [([10, 11], [0, 1]), ([10, 11], [2, 3]), ([20], [4, 5])],
        "share first page 20": [([10, 11, 12], [0, 1]), ([10, 11], [2, 3])],
        "prefix_len": None,
    }
    for needle, groups in cases.items():
        if groups is None:
            bad = _csr(GOOD, 4)
            bad.prefix_len = bad.prefix_len + 1
        else:
            bad = _csr(groups, 4)
        errs = check_prefix_groups(BT, LENS, 4, 2, bad)
        assert any(needle in e for e in errs), (needle, errs)


def test_cascade_construction_truth_passes():
    case = workloads.shared_prefix_cascade(groups=3, members=5, prefix_tokens=32,
                                           suffix_lo=1, suffix_hi=40, ungrouped=4)
    truth = [(case.block_table[m[0], :case.prefix_pages_truth].tolist(), m.tolist())
             for m in case.groups_truth]
    assert check_prefix_groups(case.block_table, case.seq_lens, 16, 2, _csr(truth, 16)) == []
    # dropping one member is caught
    truth[0] = (truth[0][0], truth[0][1][1:])
    assert check_prefix_groups(case.block_table, case.seq_lens, 16, 2, _csr(truth, 16)) != []
