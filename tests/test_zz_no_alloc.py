"""The allocation-free decode entry point, checked against the oracle and,
bit for bit, against the workspace entry point.

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
from gpu_helpers import compare, oracle_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_46_gb300 import build
    build.build()
    return ts.lib()


def _case(seed, lens, D=128, H_q=32, H_kv=8, dtype="bf16"):
    return workloads.build_case(f"noalloc_{seed}", seed, B=len(lens), H_q=H_q, H_kv=H_kv, D=D, page_size=16,
                                seq_lens=lens, dtype=dtype, scale=D ** -0.5, device=DEV)


def _noalloc_call(lib, case, bt, lens, out, lse, B=None, dtype=ts.TS_BF16):
    """Direct C-ABI call (no Python-side allocation)."""
    return lib.ts_paged_decode_attn_noalloc(
        ctypes.c_void_p(case.q.data_ptr()), ctypes.c_void_p(case.k_pool.data_ptr()),
        ctypes.c_void_p(case.v_pool.data_ptr()), ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
        ctypes.c_void_p(lens.data_ptr()), case.B if B is None else B, case.H_q, case.H_kv, case.D,
        case.page_size, case.num_pages, ctypes.c_float(case.scale), dtype, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _meta(case):
    return torch.from_numpy(case.block_table).to(DEV), torch.from_numpy(case.attn_lens).to(DEV)


def test_noalloc_matches_oracle_and_workspace_entry_point_twice(lib):
    rng = np.random.default_rng(5)
    cases = [_case(61, [0, 1, 17, 4096, 300, 2500, 16, 999]),
             _case(62, rng.integers(1, 3000, size=40).tolist(), D=64)]
    for case in cases:  # two calls in a row; the second reuses the scratch the first left
        bt, lens = _meta(case)
        ref_out, ref_lse = ts.ts_paged_decode_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale,
                                                   return_lse=True)
        out = torch.full_like(case.q, float("nan"))
        lse = torch.full((case.B, case.H_q), float("nan"), device=DEV)
        st = _noalloc_call(lib, case, bt, lens, out, lse)
        assert st == ts.TS_OK, lib.ts_last_error_detail()
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(None) == 0
        # same kernels, same cut: identical bits
        assert torch.equal(out, ref_out), f"{case.name}: O differs from the workspace entry point"
        assert torch.equal(lse, ref_lse), f"{case.name}: LSE differs from the workspace entry point"
        o_ref, l_ref = oracle_decode(case)
        compare(out, o_ref, "bf16", lse, l_ref, f"noalloc {case.name}")


def test_noalloc_reports_and_then_clears_device_errors(lib):
    """A bad page id is flagged in the static scratch's error word (read with
    a NULL workspace); the next clean call starts from a cleared word."""
    case = _case(64, [40, 20, 33, 9], D=64, H_q=8, H_kv=2, dtype="f32")
    bt, lens = _meta(case)
    bad_bt = bt.clone()
    bad_bt[1, 0] = case.num_pages + 5        # out of range: the kernel's bounds check flags it
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((case.B, case.H_q), float("nan"), device=DEV)
    assert _noalloc_call(lib, case, bad_bt, lens, out, lse, dtype=ts.TS_F32) == ts.TS_OK
    torch.cuda.synchronize()
    assert ts.ts_read_device_error(None) & ts.TS_DEVERR_PAGE_RANGE
    good = np.array([0, 2, 3])
    o_ref, l_ref = oracle_decode(case, seq_idx=good)
    idx = torch.from_numpy(good).to(DEV)
    compare(out[idx], o_ref, "f32", lse[idx], l_ref, "noalloc bad page neighbours")
    assert _noalloc_call(lib, case, bt, lens, out, lse, dtype=ts.TS_F32) == ts.TS_OK
    torch.cuda.synchronize()
    assert ts.ts_read_device_error(None) == 0
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "f32", lse, l_ref, "noalloc after a flagged call")


def test_noalloc_steady_state_allocates_nothing(lib):
    case = _case(65, [700, 33, 2048, 5])
    bt, lens = _meta(case)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.B, case.H_q, device=DEV)
    assert _noalloc_call(lib, case, bt, lens, out, lse) == ts.TS_OK
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc_call(lib, case, bt, lens, out, lse) == ts.TS_OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before


def test_noalloc_rejects_sizes_beyond_the_static_scratch(lib):
    """A supported shape (64 query heads over 8 kv heads, D 128) with a batch
    large enough that its split records overflow the static scratch."""
    H_q, H_kv, D = 64, 8, 128
    B = 1 << 16
    while ts.ts_paged_decode_workspace_size(B, H_q, D) <= ts.TS_NOALLOC_SCRATCH_BYTES:
        B *= 2
    assert B <= 1 << 21
    q = torch.zeros(B, H_q, D, dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(q)
    lse = torch.empty(B, H_q, device=DEV)
    pool = torch.zeros(1, 16, H_kv, D, dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros(B, 1, dtype=torch.int32, device=DEV)
    lens = torch.ones(B, dtype=torch.int32, device=DEV)
    st = lib.ts_paged_decode_attn_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(pool.data_ptr()), ctypes.c_void_p(pool.data_ptr()),
        ctypes.c_void_p(bt.data_ptr()), 1, ctypes.c_void_p(lens.data_ptr()), B, H_q, H_kv, D, 16, 1,
        ctypes.c_float(D ** -0.5), ts.TS_BF16, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ts.TS_ERR_WORKSPACE
    assert b"static scratch" in lib.ts_last_error_detail()
    del q, out


def test_noalloc_reports_unsupported_shapes_as_such(lib):
    case = _case(63, [5, 9], D=128, H_q=256, H_kv=8)   # group size 32: not a supported shape
    bt, lens = _meta(case)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.B, case.H_q, device=DEV)
    assert _noalloc_call(lib, case, bt, lens, out, lse) == ts.TS_ERR_UNSUPPORTED
