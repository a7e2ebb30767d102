"""GPU parity of absorbed-MLA decode on the fp8 input path
(ts_mla_paged_decode_fp8: e4m3 query and latent codes with per-row scales,
kind::f8f6f4 products) against the fp64 oracle over the reconstructed rows."""

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


def _case(seed, lens, H=128, q_len=1):
    return workloads.build_mla_fp8_case(f"mla_fp8_{seed}", seed, B=len(lens), H=H, seq_lens=lens,
                                        scale=192 ** -0.5, q_len=q_len, device=DEV)


def _run(case, clusters=None):
    bt, lens, _ = device_metadata(case)
    if clusters is not None:
        os.environ["TS_MLA_CLUSTERS"] = str(clusters)
    try:
        ws = ts.new_workspace(ts.ts_mla_multi_workspace_size(case.B, case.q_len, case.H_q, 512), DEV)
        out, lse = ts.ts_mla_paged_decode_fp8(case.q, case.meta["q_scale"], case.k_pool, case.k_scale, bt, lens,
                                              case.scale, workspace=ws, return_lse=True)
        torch.cuda.synchronize()
        err = ts.ts_read_device_error(ws)
    finally:
        os.environ.pop("TS_MLA_CLUSTERS", None)
    assert err == 0, f"device error word {err:#x}"
    return out, lse


def _oracle(case, seq_idx=None):
    v = workloads.oracle_view(case, seq_idx)
    if case.q_len == 1:
        return oracle.mla_decode_attention_fp8(v["q"], v["q_scale"], v["k_pool"], v["k_scale"], v["block_table"],
                                               v["seq_lens"], case.scale, 512)
    qd = oracle.dequantize(v["q"], v["q_scale"]).astype(np.float64)
    cd = oracle.dequantize(v["k_pool"], v["k_scale"]).astype(np.float64)
    return oracle.mla_multi_query_decode_attention(qd, cd, v["block_table"], v["seq_lens"], case.scale, 512)


@pytest.mark.parametrize("clusters", [None, 1, 3])
def test_fp8_mla_small_ragged(clusters):
    case = _case(81, [1, 65, 700, 64, 0, 130, 2])
    out, lse = _run(case, clusters)
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"fp8 mla clusters={clusters}")


def test_fp8_mla_long_sequence_split_over_many_clusters():
    case = _case(82, [20000, 3, 900])
    out, lse = _run(case)
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, "fp8 mla long split")


def test_fp8_mla_token_scales_spanning_many_powers_of_two():
    """Latent-row scales spread over nine powers of two (2^-9 .. 1 times the
    drawn scale): the gain G on P changes from tile to tile and must rescale
    the accumulator exactly, while the outputs stay of order one."""
    case = _case(83, [3000, 129, 64, 500])
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    spread = torch.exp2(torch.rand(case.k_scale.shape, generator=g, device=DEV) * -9)
    case.k_scale = torch.where(torch.isnan(case.k_scale), case.k_scale, case.k_scale * spread)
    out, lse = _run(case)
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, "fp8 mla spread scales")


@pytest.mark.parametrize("H,q_len", [(64, 4), (128, 2)])
def test_fp8_mla_multi_query(H, q_len):
    case = _case(84 + q_len, [q_len, 66, 700, 2049], H=H, q_len=q_len)
    out, lse = _run(case)
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"fp8 mla H={H} q_len={q_len}")


def test_fp8_mla_workload_sampled():
    """The absorbed-MLA workload on the fp8 path (B = 64, 128 heads, lens
    U[8192, 50000]) in the benchmark's launch configuration: a seeded sample of
    sequences (shortest and longest included) against the oracle."""
    case = workloads.absorbed_mla_fp8(device=DEV)
    out, lse = _run(case)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    idx = workloads.sample_sequences(case, 12, seed=5)
    o_ref, l_ref = _oracle(case, idx)
    sel = torch.from_numpy(idx).to(DEV)
    compare(out[sel], o_ref, "bf16", lse[sel], l_ref, "fp8 mla workload sample")
