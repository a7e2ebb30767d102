"""GPU parity of the shared-prefix (cascade) path: ts_group_prefixes on the host,
ts_cascade_decode_attn on the GPU (tensor-core prefix kernel + paged suffix +
LSE merge), against the oracle's FLAT attention over prefix ++ suffix (the
oracle never splits or merges)."""

import numpy as np
import pytest
import torch

import paged_kv_cache_46_gb300 as ts
import workloads
from gpu_helpers import compare, device_metadata, oracle_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_46_gb300 import build
    build.build()


def _run_cascade(case, min_group=2):
    groups = ts.ts_group_prefixes(case.block_table, case.seq_lens, case.page_size, min_group)
    gdev = ts.groups_to_device(groups, DEV)
    bt, lens, _ = device_metadata(case)
    ws = ts.new_workspace(ts.ts_cascade_decode_workspace_size(case.B, case.H_q, case.D), DEV)
    out, lse = ts.ts_cascade_decode_attn(case.q, case.k_pool, case.v_pool, gdev, bt, lens, case.scale,
                                         workspace=ws, return_lse=True)
    torch.cuda.synchronize()
    assert ts.ts_read_device_error(ws) == 0
    return out, lse, groups


@pytest.mark.parametrize("groups,members,prefix_tokens,ungrouped", [
    (3, 40, 256, 5),     # two full key tiles, a partial member tile, ungrouped sequences
    (2, 33, 48, 0),      # a prefix of 3 pages: one partial key tile
    (1, 128, 2048, 3),   # a 16-tile prefix, 4 member tiles
    (4, 2, 16, 2),       # one-page prefixes, two members each
])
def test_cascade_matches_flat_attention(groups, members, prefix_tokens, ungrouped):
    case = workloads.shared_prefix_cascade(device=DEV, seed=40 + groups, groups=groups, members=members,
                                           prefix_tokens=prefix_tokens, suffix_lo=1, suffix_hi=100,
                                           ungrouped=ungrouped)
    out, lse, g = _run_cascade(case)
    assert g["num_groups"] == groups
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"cascade {groups}x{members} prefix {prefix_tokens}")


def test_cascade_with_split_suffixes():
    """Long suffixes are cut across CTAs: the split merge also folds in the prefix."""
    case = workloads.shared_prefix_cascade(device=DEV, seed=47, groups=2, members=20, prefix_tokens=512,
                                           suffix_lo=2000, suffix_hi=6000, ungrouped=2)
    out, lse, _ = _run_cascade(case)
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, "cascade split suffixes")


def test_cascade_full_workload_sampled_and_cross_checked():
    """Shared-prefix cascade at full size (16 groups x 1024 members, 2048-token
    prefixes, suffixes U[64,512]): a seeded sample of 256 sequences (with the
    shortest and longest) against the oracle, and every output against the
    flat paged path."""
    case = workloads.shared_prefix_cascade(device=DEV)
    out, lse, g = _run_cascade(case)
    assert g["num_groups"] == 16
    idx = workloads.sample_sequences(case, 256)
    o_ref, l_ref = oracle_decode(case, seq_idx=idx)
    dev_idx = torch.from_numpy(idx).to(DEV)
    compare(out[dev_idx], o_ref, "bf16", lse[dev_idx], l_ref, "cascade 16x1024 sample")
    bt, lens, _ = device_metadata(case)
    flat, flat_lse = ts.ts_paged_decode_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale,
                                             return_lse=True)
    torch.cuda.synchronize()
    diff = (out.float() - flat.float()).abs().max().item()
    assert diff <= 2e-2, diff
    assert (lse - flat_lse).abs().max().item() <= 1e-3


def test_cascade_without_groups_is_the_paged_path():
    case = workloads.build_case("nogroups", 49, B=6, H_q=32, H_kv=8, D=64, page_size=16,
                                seq_lens=[5, 100, 17, 300, 1, 64], dtype="bf16", scale=0.125, device=DEV)
    out, lse, g = _run_cascade(case)
    assert g["num_groups"] == 0
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, "cascade no groups")


# ---------------------------------------------------------------------------
# Nested (tree) prefixes: ts_group_prefixes_nested + ts_cascade_nested_decode_attn
# against the oracle's flat attention.
# ---------------------------------------------------------------------------

def _run_nested(case, min_group=2):
    forest = ts.ts_group_prefixes_nested(case.block_table, case.seq_lens, case.page_size, min_group)
    fdev = ts.forest_to_device(forest, DEV)
    bt, lens, _ = device_metadata(case)
    ws = ts.new_workspace(ts.ts_cascade_decode_workspace_size(case.B, case.H_q, case.D), DEV)
    out, lse = ts.ts_cascade_nested_decode_attn(case.q, case.k_pool, case.v_pool, fdev, bt, lens, case.scale,
                                                workspace=ws, return_lse=True)
    torch.cuda.synchronize()
    assert ts.ts_read_device_error(ws) == 0
    return out, lse, forest


@pytest.mark.parametrize("roots,subs,members,root_tokens,sub_tokens", [
    (2, 3, 40, 256, 256),   # two levels, partial member tiles
    (1, 2, 130, 48, 2048),  # a 3-page root, 16-tile second level, 2 member tiles per node
    (3, 1, 9, 16, 16),      # one-page stretches
])
def test_nested_cascade_matches_flat_attention(roots, subs, members, root_tokens, sub_tokens):
    case = workloads.nested_prefix_cascade(device=DEV, seed=60 + roots, roots=roots, subs=subs, members=members,
                                           root_tokens=root_tokens, sub_tokens=sub_tokens, suffix_lo=1,
                                           suffix_hi=300)
    out, lse, f = _run_nested(case)
    assert f["num_levels"] == (2 if subs > 1 else 1)
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"nested {roots}x{subs}x{members}")


def test_nested_cascade_random_trees_and_deep_levels():
    """Sequences walking a random trie of shared pages: several levels, nodes of
    different depths, ungrouped sequences; every output against the oracle."""
    rng = np.random.default_rng(71)
    B, ps, depth = 96, 16, 10
    paths, nxt, children = np.zeros((B, depth), np.int64), [0], {}
    for b in range(B):
        node = ()
        for d in range(depth):
            kids = children.setdefault(node, [])
            if kids and rng.random() < 0.75:
                pg = kids[rng.integers(len(kids))]
            else:
                pg = nxt[0]
                nxt[0] += 1
                kids.append(pg)
            paths[b, d] = pg
            node = node + (pg,)
    lens = rng.integers(1, depth * ps + 1, size=B)
    # map the trie's page labels onto a shuffled pool; pages past a sequence's
    # length are its own (so that two sequences never write one page)
    n_pages = nxt[0] + B * depth
    perm = rng.permutation(n_pages).astype(np.int32)
    bt = perm[paths].astype(np.int32)
    for b in range(B):
        used = (int(lens[b]) + ps - 1) // ps
        # a sequence's last (partial) page and beyond must be its own
        bt[b, max(0, used - 1):] = perm[nxt[0] + b * depth + np.arange(max(0, used - 1), depth)]
    case = workloads.build_case("nested_random", 72, B=B, H_q=32, H_kv=8, D=64, page_size=ps, seq_lens=lens,
                                dtype="bf16", scale=0.125, device=DEV, layout=(bt, n_pages))
    out, lse, f = _run_nested(case)
    assert f["num_levels"] >= 2
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, "nested random trie")


def test_nested_cascade_full_workload_sampled():
    """4 root prefixes x 4 second-level prefixes x 256 members (1024 + 1024
    shared tokens, suffixes U[64,512]): a seeded sample of 256 sequences against
    the oracle, every output against the single-level cascade."""
    case = workloads.nested_prefix_cascade(device=DEV)
    out, lse, f = _run_nested(case)
    assert f["num_nodes"] == 20 and f["num_levels"] == 2
    idx = workloads.sample_sequences(case, 256)
    o_ref, l_ref = oracle_decode(case, seq_idx=idx)
    dev_idx = torch.from_numpy(idx).to(DEV)
    compare(out[dev_idx], o_ref, "bf16", lse[dev_idx], l_ref, "nested 4x4x256 sample")
    flat, flat_lse, _ = _run_cascade(case)
    assert (out.float() - flat.float()).abs().max().item() <= 2e-2
    assert (lse - flat_lse).abs().max().item() <= 1e-3
