"""GPU parity of absorbed-MLA decode (ts_mla_paged_decode: a two-CTA cluster per
page range, tcgen05 with Q and P in TMEM, partial scores swapped through
distributed shared memory) against the fp64 oracle."""

import os

import numpy as np
import pytest
import torch

import paged_kv_cache_46_gb300 as ts
import workloads
from gpu_helpers import compare, device_metadata, oracle_mla

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_46_gb300 import build
    build.build()


def _mla_case(seed, lens):
    return workloads.build_case(f"mla_{seed}", seed, B=len(lens), H_q=128, H_kv=1, D=576, Dv=512, page_size=64,
                                seq_lens=lens, dtype="bf16", scale=192 ** -0.5, mla=True, device=DEV)


def _run_mla(case, clusters=None):
    bt, lens, _ = device_metadata(case)
    if clusters is not None:
        os.environ["TS_MLA_CLUSTERS"] = str(clusters)
    try:
        ws = ts.new_workspace(ts.ts_mla_workspace_size(case.B, 128, 512), DEV)
        out, lse = ts.ts_mla_paged_decode(case.q, case.k_pool, bt, lens, case.scale, workspace=ws, return_lse=True)
        torch.cuda.synchronize()
        err = ts.ts_read_device_error(ws)
    finally:
        os.environ.pop("TS_MLA_CLUSTERS", None)
    assert err == 0, f"device error word {err:#x}"
    return out, lse


@pytest.mark.parametrize("clusters", [None, 1, 3])
def test_mla_small_ragged(clusters):
    case = _mla_case(61, [1, 65, 700, 64, 0, 130])
    out, lse = _run_mla(case, clusters)
    o_ref, l_ref = oracle_mla(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"mla small clusters={clusters}")


def test_mla_long_sequence_split_over_many_clusters():
    case = _mla_case(62, [20000, 3, 900])
    out, lse = _run_mla(case)
    o_ref, l_ref = oracle_mla(case)
    compare(out, o_ref, "bf16", lse, l_ref, "mla long split")


def test_mla_full_workload():
    """Absorbed-MLA decode at full size (B=64, 128 heads, latent 576, page 64,
    lens U[8192, 50000]), in the launch configuration the benchmark times:
    every sequence, head and dim against the oracle."""
    case = workloads.absorbed_mla(device=DEV)
    out, lse = _run_mla(case)
    o_ref, l_ref = oracle_mla(case)
    compare(out, o_ref, "bf16", lse, l_ref, "mla full workload")
