"""The allocation-free decode entry point, checked against the workspace one.

ts_paged_decode_attn_noalloc serves callers that cannot allocate device
memory (a plugin given only its inputs and outputs by a host runtime, or an
engine whose KV-cache pool already holds all free HBM): its split-KV scratch
is a fixed array inside the library. This file sorts last so that a run
stopping at its first failure has already run every other test. It must pass
alone in a fresh process and after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_46_gb300 as ts
import workloads
from gpu_helpers import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_46_gb300 import build
    build.build()
    return ts.lib()


def _case(seed, lens, D=128, H_q=32, H_kv=8):
    return workloads.build_case(f"noalloc_{seed}", seed, B=len(lens), H_q=H_q, H_kv=H_kv, D=D, page_size=16,
                                seq_lens=lens, dtype="bf16", scale=D ** -0.5, device=DEV)


def _noalloc_call(lib, case, bt, lens, out, lse):
    """Direct C-ABI call (no Python-side allocation)."""
    return lib.ts_paged_decode_attn_noalloc(
        ctypes.c_void_p(case.q.data_ptr()), ctypes.c_void_p(case.k_pool.data_ptr()),
        ctypes.c_void_p(case.v_pool.data_ptr()), ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
        ctypes.c_void_p(lens.data_ptr()), case.B, case.H_q, case.H_kv, case.D, case.page_size,
        case.num_pages, ctypes.c_float(case.scale), ts.TS_BF16, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice(lib):
    rng = np.random.default_rng(5)
    cases = [_case(61, [0, 1, 17, 4096, 300, 2500, 16, 999]),
             _case(62, rng.integers(1, 3000, size=40).tolist(), D=64)]
    for case in cases:  # two calls in a row; the second reuses the scratch the first left
        bt = torch.from_numpy(case.block_table).to(DEV)
        lens = torch.from_numpy(case.attn_lens).to(DEV)
        ref_out, ref_lse = ts.ts_paged_decode_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale,
                                                   return_lse=True)
        out = torch.full_like(case.q, float("nan"))
        lse = torch.full((case.B, case.H_q), float("nan"), device=DEV)
        st = _noalloc_call(lib, case, bt, lens, out, lse)
        assert st == ts.TS_OK, lib.ts_last_error_detail()
        torch.cuda.synchronize()
        ref_o = ref_out.double().cpu().numpy()
        compare(out, ref_o, "bf16", lse, ref_lse.double().cpu().numpy(), f"noalloc {case.name}")


def test_noalloc_rejects_sizes_beyond_the_static_scratch(lib):
    case = _case(63, [5, 9], D=128, H_q=256, H_kv=8)   # 2 x SMs x 256 x 128 fp32 partials > 16 MiB
    bt = torch.from_numpy(case.block_table).to(DEV)
    lens = torch.from_numpy(case.attn_lens).to(DEV)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.B, case.H_q, device=DEV)
    st = _noalloc_call(lib, case, bt, lens, out, lse)
    assert st == ts.TS_ERR_WORKSPACE
    assert b"static scratch" in lib.ts_last_error_detail()
