"""GPU parity of tree verification (ts_paged_decode_tree_attn: each draft
token attends the context and its own path in the draft tree, on the
tensor-core multi-query kernel) against the fp64 oracle."""

import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_46_gb300 as ts
import workloads
from gpu_helpers import compare, device_metadata

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_46_gb300 import build
    build.build()


def _case(seed, lens, n, H_q=32, H_kv=8, D=128, shape="random"):
    rng = np.random.default_rng(seed + 500)
    case = workloads.build_case(f"tree_{seed}", seed, B=len(lens), H_q=H_q, H_kv=H_kv, D=D, page_size=16,
                                seq_lens=lens, dtype="bf16", scale=D ** -0.5, device=DEV, q_len=n)
    return case, workloads.draft_trees(len(lens), n, rng, shape)


def _run(case, parents, head_group=None):
    bt, lens, _ = device_metadata(case)
    par = torch.from_numpy(parents).to(DEV)
    if head_group is not None:
        os.environ["TS_MULTI_QUERY_HEAD_GROUP"] = str(head_group)
    try:
        ws = ts.new_workspace(256, DEV)
        out, lse = ts.ts_paged_decode_tree_attn(case.q, case.k_pool, case.v_pool, bt, lens, par, case.scale,
                                                workspace=ws, return_lse=True)
        torch.cuda.synchronize()
        err = ts.ts_read_device_error(ws)
    finally:
        os.environ.pop("TS_MULTI_QUERY_HEAD_GROUP", None)
    return out, lse, err


def _oracle(case, parents, seq_idx=None):
    v = workloads.oracle_view(case, seq_idx)
    par = parents if seq_idx is None else parents[seq_idx]
    return oracle.tree_verify_decode_attention(v["q"], v["k_pool"], v["v_pool"], v["block_table"], v["seq_lens"],
                                               par, case.scale)


@pytest.mark.parametrize("shape", ["random", "beam", "star", "chain"])
@pytest.mark.parametrize("n,H_q,H_kv,D", [(8, 32, 8, 128), (6, 8, 2, 64), (32, 32, 8, 128), (64, 16, 8, 64)])
def test_tree_shapes(shape, n, H_q, H_kv, D):
    """Ragged lengths: the draft tokens are the whole context (L = n), draft
    keys straddling a page and a key tile, exact pages, long contexts."""
    lens = [n, n + 15, n + 17, 128, 16 * 9 + 3, 1000, 3001, 130]
    case, parents = _case(80 + n, lens, n, H_q, H_kv, D, shape)
    out, lse, err = _run(case, parents)
    assert err == 0, f"device error word {err:#x}"
    o_ref, l_ref = _oracle(case, parents)
    compare(out, o_ref, "bf16", lse, l_ref, f"tree {shape} n={n} {H_q}/{H_kv} D={D}", margin=0.8)


@pytest.mark.parametrize("hg", [1, 2, 4])
def test_head_groups(hg):
    case, parents = _case(90, [9, 700, 2049, 33], 8)
    out, lse, err = _run(case, parents, hg)
    assert err == 0
    o_ref, l_ref = _oracle(case, parents)
    compare(out, o_ref, "bf16", lse, l_ref, f"tree hg={hg}", margin=0.8)


def test_chain_tree_is_causal_multi_query_bit_for_bit():
    case, parents = _case(91, [8, 40, 700, 2049, 129], 8, shape="chain")
    out, lse, err = _run(case, parents)
    assert err == 0
    bt, lens, _ = device_metadata(case)
    os.environ["TS_MULTI_QUERY_PATH"] = "tensor"
    try:
        out2, lse2 = ts.ts_paged_decode_multi_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale,
                                                   return_lse=True)
        torch.cuda.synchronize()
    finally:
        os.environ.pop("TS_MULTI_QUERY_PATH", None)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_bad_parent_is_flagged_without_fault():
    case, parents = _case(92, [50, 60], 6)
    parents = parents.copy()
    parents[1, 3] = 3            # its own parent: not an earlier node
    out, lse, err = _run(case, parents)
    assert err & ts.TS_DEVERR_TREE
    assert torch.isfinite(out).all()
    o_ref, l_ref = _oracle(case, parents[:1], seq_idx=np.array([0]))
    compare(out[:1], o_ref, "bf16", lse[:1], l_ref, "tree neighbour of a bad parent")


def test_unsupported_shapes_are_rejected():
    case, parents = _case(93, [70, 80], 65, H_q=8, H_kv=8, D=64)   # n > 64
    bt, lens, _ = device_metadata(case)
    with pytest.raises(ts.TSError) as e:
        ts.ts_paged_decode_tree_attn(case.q, case.k_pool, case.v_pool, bt, lens,
                                     torch.from_numpy(parents).to(DEV), case.scale)
    assert e.value.status == ts.TS_ERR_UNSUPPORTED


def test_speculative_tree_workload_sampled():
    """The Llama-3-8B layer shape verifying 16-token random draft trees (B = 64,
    lens U[512, 4096]) in the benchmark's launch configuration: a seeded
    sample of sequences (shortest and longest included) against the oracle."""
    case, parents = workloads.speculative_tree(device=DEV)
    out, lse, err = _run(case, parents)
    assert err == 0
    idx = workloads.sample_sequences(case, 12, seed=4)
    o_ref, l_ref = _oracle(case, parents, idx)
    sel = torch.from_numpy(idx).to(DEV)
    compare(out[sel], o_ref, "bf16", lse[sel], l_ref, "speculative tree sample", margin=0.8)
