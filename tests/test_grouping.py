"""The host grouping pass ts_group_prefixes (C++, through the C ABI), checked by
the oracle's invariant checker (CPU only)."""

import time

import numpy as np
import pytest

import paged_kv_cache_46_gb300 as ts
import workloads
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


@pytest.mark.parametrize("seed", range(6))
def test_random_nested_prefix_trees(seed):
    """Random nested sharing: sequences copy a random-length prefix of another
    sequence's block-table row (a random tree of shared prefixes)."""
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
    for min_group in (2, 3):
        _check(bt, lens, ps, min_group)


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
