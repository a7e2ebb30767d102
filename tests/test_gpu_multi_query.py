"""GPU parity: ts_paged_decode_multi_attn (q_len query tokens per sequence,
causal among the new tokens) against the fp64 oracle, through the C ABI."""

import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_46_gb300 as ts
import workloads
from gpu_helpers import as_f64, compare

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_46_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _case(name, seed, lens, q_len, H_q=32, H_kv=8, D=128, ps=16, dtype="bf16"):
    return workloads.build_case(name, seed, B=len(lens), H_q=H_q, H_kv=H_kv, D=D, page_size=ps,
                                seq_lens=lens, dtype=dtype, scale=D ** -0.5, device=DEV, q_len=q_len)


def _run(case, q_len, ctas=None, path=None, hg=None):
    """path: None = the library's choice, "tensor" = the tcgen05 kernel where the
    shape allows it, "cuda" = the CUDA-core split-KV kernel; hg: kv heads per
    CTA of the tcgen05 kernel (None = the library's choice)."""
    bt = torch.from_numpy(case.block_table).to(DEV)
    lens = torch.from_numpy(case.seq_lens).to(DEV)
    if ctas is not None:
        os.environ["TS_PAGED_DECODE_CTAS"] = str(ctas)
    if path is not None:
        os.environ["TS_MULTI_QUERY_PATH"] = path
    if hg is not None:
        os.environ["TS_MULTI_QUERY_HEAD_GROUP"] = str(hg)
    try:
        ws = ts.new_workspace(ts.ts_paged_decode_multi_workspace_size(case.B, q_len, case.H_q, case.D))
        out, lse = ts.ts_paged_decode_multi_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale,
                                                 workspace=ws, return_lse=True)
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
    finally:
        os.environ.pop("TS_PAGED_DECODE_CTAS", None)
        os.environ.pop("TS_MULTI_QUERY_PATH", None)
        os.environ.pop("TS_MULTI_QUERY_HEAD_GROUP", None)
    return out, lse


def _oracle(case):
    v = workloads.oracle_view(case)
    return oracle.multi_query_decode_attention(v["q"], v["k_pool"], v["v_pool"], v["block_table"],
                                               v["seq_lens"], case.scale)


@pytest.mark.parametrize("q_len,H_q,H_kv,D,dtype", [
    (2, 32, 8, 128, "bf16"),   # g=4: both tokens folded into 8 rows, one pass
    (4, 32, 8, 128, "bf16"),   # g=4: fold 2, two passes
    (3, 32, 8, 64, "bf16"),    # g=4: 3 is odd, three passes
    (8, 8, 8, 64, "bf16"),     # g=1: all 8 tokens folded
    (3, 16, 8, 64, "bf16"),    # g=2: fold 1 (2*3 rows is not a compiled row count)
    (2, 64, 8, 128, "bf16"),   # g=8: fold 1, two passes
    (2, 8, 2, 64, "f32"),
    (4, 4, 4, 128, "f32"),     # g=1, fold 4
])
def test_multi_query_matches_oracle(q_len, H_q, H_kv, D, dtype):
    rng = np.random.default_rng(q_len * 100 + H_q + D)
    lens = rng.integers(q_len, 700, size=7)
    lens[0] = q_len            # the context is only the new tokens
    lens[1] = 16 + q_len - 1   # new tokens straddle a page boundary
    lens[2] = 33
    case = _case(f"mq_{q_len}_{H_q}_{H_kv}_{D}_{dtype}", 61 + q_len, lens, q_len, H_q, H_kv, D, dtype=dtype)
    o_ref, l_ref = _oracle(case)
    for ctas, path in ((None, "tensor"), (None, "cuda"), (5, "cuda")):
        out, lse = _run(case, q_len, ctas, path)
        compare(out, o_ref, dtype, lse, l_ref, f"q_len={q_len} {H_q}/{H_kv} D={D} {dtype} ctas={ctas} path={path}", margin=0.8 if dtype == "bf16" else 1.0)


@pytest.mark.parametrize("ctas", [1, 7, None, 1000])
def test_multi_query_independent_of_split_pattern(ctas):
    lens = [4, 5, 19, 64, 700, 2049, 31, 300]
    case = _case("mq_split", 71, lens, 4)
    out, lse = _run(case, 4, ctas, "cuda")
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"ctas={ctas}", margin=0.8)


def test_q_len_one_equals_single_query_decode():
    lens = [1, 17, 300, 2000, 45]
    case = _case("mq_one", 73, lens, 1)
    bt = torch.from_numpy(case.block_table).to(DEV)
    dl = torch.from_numpy(case.seq_lens).to(DEV)
    q4 = case.q.view(case.B, 1, case.H_q, case.D)
    o1, l1 = ts.ts_paged_decode_multi_attn(q4, case.k_pool, case.v_pool, bt, dl, case.scale, return_lse=True)
    o0, l0 = ts.ts_paged_decode_attn(case.q, case.k_pool, case.v_pool, bt, dl, case.scale, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o1.view_as(o0), o0) and torch.equal(l1.view_as(l0), l0)


def test_full_llama_shape_with_two_draft_tokens():
    """Llama-3-8B layer shape (B=64, 32/8 heads, D=128) verifying 2 tokens
    per sequence; every output row checked against the oracle."""
    rng = np.random.default_rng(2)
    lens = rng.integers(512, 4097, size=64)
    case = _case("mq_llama", 2, lens, 2)
    o_ref, l_ref = _oracle(case)
    for path in ("tensor", "cuda"):
        out, lse = _run(case, 2, path=path)
        compare(out, o_ref, "bf16", lse, l_ref, f"llama shape q_len=2 path={path}", margin=0.8)


@pytest.mark.parametrize("q_len,H_q,H_kv,D,hg", [
    (4, 32, 8, 128, 1), (4, 32, 8, 128, 2), (4, 32, 8, 128, 4),   # 16 rows: 1, 2 or 4 kv heads per CTA
    (2, 32, 8, 64, 4), (8, 64, 8, 128, 1), (8, 64, 8, 128, 2),    # 8 and 64 rows
    (16, 32, 4, 64, 1), (3, 8, 1, 64, 1)])                         # 128 rows; one kv head
def test_tensor_core_path_shapes(q_len, H_q, H_kv, D, hg):
    """Rows q_len * g from 8 to 128 on the tensor-core path, with 1, 2 or 4 kv
    heads per CTA, including sequences shorter than a key tile, a context of
    only the new tokens, and one past a tile boundary."""
    rng = np.random.default_rng(q_len * 7 + D)
    lens = rng.integers(q_len, 3000, size=6)
    lens[0], lens[1], lens[2] = q_len, 127 + q_len, 128
    lens[3] = 16 * (8 // hg) + 1        # one key past a tile of 8 / hg pages
    case = _case(f"mq_tc_{q_len}_{H_q}_{H_kv}_{D}", 91 + q_len, lens, q_len, H_q, H_kv, D)
    out, lse = _run(case, q_len, path="tensor", hg=hg)
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"tc q_len={q_len} {H_q}/{H_kv} D={D} hg={hg}", margin=0.8)


@pytest.mark.parametrize("B,hg", [(40, 1), (40, 4), (129, 2), (300, 2)])
def test_tensor_core_path_work_order(B, hg):
    """Up to 128 sequences the CTAs take them longest first, above that in index
    order: both against the oracle, with runs of equal lengths (ties in the
    ranking) and lengths of zero, one and a tile boundary mixed in."""
    rng = np.random.default_rng(B)
    lens = rng.integers(4, 700, size=B)
    lens[: B // 4] = 257                   # a block of ties
    lens[B // 4] = 4
    lens[B // 4 + 1] = 128
    rng.shuffle(lens)
    case = _case(f"mq_tc_order_{B}", 300 + B, lens, 4)
    out, lse = _run(case, 4, path="tensor", hg=hg)
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"tc work order B={B} hg={hg}", margin=0.8)


def test_full_speculative_verify_four_tokens_sampled():
    """The benchmark's 4-draft-token workload at full size (B=64, 32/8 heads,
    D=128) through the library's choice (the tensor-core kernel, 2 kv heads
    per CTA, longest first): a seeded sample of 12 sequences against the
    oracle."""
    case = workloads.speculative_verify(device=DEV, q_len=4)
    out, lse = _run(case, 4)
    idx = workloads.sample_sequences(case, 12)
    v = workloads.oracle_view(case, idx)
    o_ref, l_ref = oracle.multi_query_decode_attention(v["q"], v["k_pool"], v["v_pool"], v["block_table"],
                                                       v["seq_lens"], case.scale)
    dev_idx = torch.from_numpy(idx).to(DEV)
    compare(out[dev_idx], o_ref, "bf16", lse[dev_idx], l_ref, "speculative verify q4 full sample", margin=0.8)
