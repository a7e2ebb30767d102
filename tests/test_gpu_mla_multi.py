"""GPU parity of multi-query absorbed-MLA decode (ts_mla_paged_decode_multi:
q_len tokens per sequence folded into the 128 rows of a tile by
fold_sq_factor, causal among the new tokens) against the fp64 oracle."""

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


def _case(seed, lens, H, q_len):
    return workloads.build_case(f"mla_mq_{seed}", seed, B=len(lens), H_q=H, H_kv=1, D=576, Dv=512, page_size=64,
                                seq_lens=lens, dtype="bf16", scale=192 ** -0.5, mla=True, device=DEV,
                                q_len=q_len)


def _run(case, clusters=None):
    bt, lens, _ = device_metadata(case)
    if clusters is not None:
        os.environ["TS_MLA_CLUSTERS"] = str(clusters)
    try:
        ws = ts.new_workspace(ts.ts_mla_multi_workspace_size(case.B, case.q_len, case.H_q, 512), DEV)
        q = case.q if case.q.dim() == 4 else case.q.unsqueeze(1)   # [B, q_len, H, 576]
        out, lse = ts.ts_mla_paged_decode_multi(q, case.k_pool, bt, lens, case.scale, workspace=ws,
                                                return_lse=True)
        torch.cuda.synchronize()
        err = ts.ts_read_device_error(ws)
    finally:
        os.environ.pop("TS_MLA_CLUSTERS", None)
    assert err == 0, f"device error word {err:#x}"
    return out, lse


def _oracle(case, seq_idx=None):
    v = workloads.oracle_view(case, seq_idx)
    return oracle.mla_multi_query_decode_attention(v["q"], v["k_pool"], v["block_table"], v["seq_lens"],
                                                   case.scale, case.Dv)


def test_fold_factor_of_the_worked_example():
    # 64 heads, 4 query tokens: F = 2, two 128-row tiles per sequence
    assert ts.ts_fold_sq_factor(64, 4, 128) == 2
    B = 3
    one_step = ts.ts_mla_workspace_size(B * 2, 128, 512)
    assert ts.ts_mla_multi_workspace_size(B, 4, 64, 512) == one_step


@pytest.mark.parametrize("clusters", [None, 1, 3])
def test_worked_example_64_heads_4_tokens(clusters):
    """The page's example shape: 64 heads x 4 tokens, ragged lengths: the
    whole context is the new tokens (4), masked keys straddling a page
    boundary (65, 66), exact pages (64, 128), a long sequence cut across
    clusters."""
    case = _case(71, [4, 65, 66, 700, 64, 128, 5000, 131], H=64, q_len=4)
    out, lse = _run(case, clusters)
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"mla 64x4 clusters={clusters}", margin=0.8)


@pytest.mark.parametrize("H,q_len", [(128, 2), (128, 3), (32, 4), (16, 8), (64, 2)])
def test_other_folds(H, q_len):
    case = _case(72 + q_len, [q_len, 63 + q_len, 900, 2049], H=H, q_len=q_len)
    out, lse = _run(case)
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"mla H={H} q_len={q_len}", margin=0.8)


def test_one_token_is_plain_mla_bit_for_bit():
    case = _case(73, [1, 65, 700, 64, 130], H=128, q_len=1)
    out, lse = _run(case)
    bt, lens, _ = device_metadata(case)
    out1, lse1 = ts.ts_mla_paged_decode(case.q, case.k_pool, bt, lens, case.scale, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], out1) and torch.equal(lse[:, 0], lse1)


def test_rows_that_see_no_key():
    """A context shorter than the new tokens: tokens 0 and 1 of a 2-token
    context with q_len 4 see no key (O = 0, LSE = -inf); tokens 2 and 3 see
    keys 0 and 0..1."""
    case = _case(74, [2, 300], H=64, q_len=4)
    out, lse = _run(case)
    assert torch.all(out[0, :2] == 0) and torch.all(torch.isneginf(lse[0, :2]))
    v = workloads.oracle_view(case)
    for j in (2, 3):
        o_ref, l_ref = oracle.mla_decode_attention(v["q"][:, j], v["k_pool"], v["block_table"],
                                                   v["seq_lens"] - 4 + 1 + j, case.scale, 512)
        compare(out[:, j], o_ref, "bf16", lse[:, j], l_ref, f"token {j}", margin=0.8)


def test_unsupported_folds_are_rejected():
    case = _case(75, [10, 20], H=64, q_len=3)    # F = 1: 64-row tiles
    bt, lens, _ = device_metadata(case)
    with pytest.raises(ts.TSError) as e:
        ts.ts_mla_paged_decode_multi(case.q, case.k_pool, bt, lens, case.scale)
    assert e.value.status == ts.TS_ERR_UNSUPPORTED


def test_speculative_mla_workload_sampled():
    """64 heads x 4 draft tokens over the absorbed-MLA workload's lengths
    (B = 64, U[8192, 50000]) in the benchmark's launch configuration: a
    seeded sample of sequences (shortest and longest included) against the
    oracle, all outputs finite."""
    case = workloads.absorbed_mla_multi(device=DEV)
    out, lse = _run(case)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    idx = workloads.sample_sequences(case, 8, seed=3)
    o_ref, l_ref = _oracle(case, idx)
    sel = torch.from_numpy(idx).to(DEV)
    compare(out[sel], o_ref, "bf16", lse[sel], l_ref, "mla speculative sample", margin=0.8)
