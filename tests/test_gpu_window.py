"""GPU parity of decode over a sliding-window KV group (ts_paged_decode_window_attn)
against the oracle's decode_attention_window. The block-table slots wholly in
front of each window point at an all-NaN placeholder page, and the rows of the
window's first page in front of the window are overwritten with NaN, so any
read outside the window shows in the output."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_46_gb300 as ts
import workloads
from gpu_helpers import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_46_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _windowed_case(name, seed, lens, window, H_q=32, H_kv=8, D=128, ps=16, dtype="bf16"):
    case = workloads.build_case(name, seed, B=len(lens), H_q=H_q, H_kv=H_kv, D=D, page_size=ps,
                                seq_lens=np.asarray(lens), dtype=dtype, scale=D ** -0.5, device=DEV)
    bt = case.block_table.copy()
    nan = float("nan")
    for b, L in enumerate(case.seq_lens):
        start = max(0, int(L) - window)
        bt[b, :start // ps] = case.sentinel_page  # placeholders: an all-NaN page
        if start % ps:
            first = int(bt[b, start // ps])
            case.k_pool[first, :start % ps] = nan
            case.v_pool[first, :start % ps] = nan
    case.block_table = bt
    return case


def _run(case, window):
    bt = torch.from_numpy(case.block_table).to(DEV)
    lens = torch.from_numpy(case.seq_lens).to(DEV)
    ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D), DEV)
    out, lse = ts.ts_paged_decode_window_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale, window,
                                              workspace=ws, return_lse=True)
    torch.cuda.synchronize()
    assert ts.ts_read_device_error(ws) == 0
    return out, lse


def _oracle(case, window):
    v = workloads.oracle_view(case)
    return oracle.decode_attention_window(v["q"], v["k_pool"], v["v_pool"], v["block_table"], v["seq_lens"],
                                          case.scale, window)


@pytest.mark.parametrize("window,H_q,H_kv,D,dtype", [
    (1024, 32, 8, 128, "bf16"),   # whole pages
    (1000, 32, 8, 128, "bf16"),   # the window starts mid-page
    (37, 32, 8, 64, "bf16"),      # shorter than most contexts, D = 64
    (1, 8, 8, 64, "bf16"),        # one token: O = V[L-1]
    (300, 16, 2, 64, "f32"),      # fp32, g = 8
])
def test_window_matches_oracle(window, H_q, H_kv, D, dtype):
    rng = np.random.default_rng(window + D)
    lens = rng.integers(1, 3000, size=12)
    lens[:5] = [window, window + 1, max(1, window - 1), 1, window + 16]
    case = _windowed_case(f"win_{window}", 500 + window, lens, window, H_q, H_kv, D, dtype=dtype)
    out, lse = _run(case, window)
    o_ref, l_ref = _oracle(case, window)
    compare(out, o_ref, dtype, lse, l_ref, f"window {window} {H_q}/{H_kv} D={D} {dtype}")


def test_long_windows_cut_across_ctas():
    """Windows of 8000 tokens inside contexts of up to 40000: each window's
    pages are split over several CTAs and merged."""
    lens = np.array([40000, 8001, 12345, 39999, 7999, 33], dtype=np.int64)
    case = _windowed_case("win_long", 77, lens, 8000, D=64)
    out, lse = _run(case, 8000)
    o_ref, l_ref = _oracle(case, 8000)
    compare(out, o_ref, "bf16", lse, l_ref, "long windows")


def test_window_covering_the_context_is_plain_decode():
    lens = np.array([5, 100, 17, 300, 1, 64, 2048, 999])
    case = workloads.build_case("win_full", 78, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                seq_lens=lens, dtype="bf16", scale=128 ** -0.5, device=DEV)
    out, lse = _run(case, 4096)
    bt = torch.from_numpy(case.block_table).to(DEV)
    lens_d = torch.from_numpy(case.seq_lens).to(DEV)
    ref, ref_lse = ts.ts_paged_decode_attn(case.q, case.k_pool, case.v_pool, bt, lens_d, case.scale,
                                           return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_window_below_one_is_an_argument_error():
    case = workloads.build_case("win_bad", 79, B=2, H_q=8, H_kv=2, D=64, page_size=16, seq_lens=[5, 9],
                                dtype="bf16", scale=0.125, device=DEV)
    bt = torch.from_numpy(case.block_table).to(DEV)
    lens = torch.from_numpy(case.seq_lens).to(DEV)
    with pytest.raises(ts.TSError):
        ts.ts_paged_decode_window_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale, 0)


def test_window_full_workload_sampled():
    """The benchmark's sliding-window workload at full size (B=64, contexts
    U[4096, 32768], W=4096, placeholder slots in front of every window), in
    the launch configuration bench.py times: a seeded sample of 8 sequences
    (with the shortest and longest) against the oracle."""
    case = workloads.sliding_window(device=DEV)
    bt = torch.from_numpy(case.block_table).to(DEV)
    lens = torch.from_numpy(case.seq_lens).to(DEV)
    ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D), DEV)
    out, lse = ts.ts_paged_decode_window_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale, case.window,
                                              workspace=ws, return_lse=True)
    torch.cuda.synchronize()
    assert ts.ts_read_device_error(ws) == 0
    idx = workloads.sample_sequences(case, 8)
    v = workloads.oracle_view(case, idx)
    o_ref, l_ref = oracle.decode_attention_window(v["q"], v["k_pool"], v["v_pool"], v["block_table"],
                                                  v["seq_lens"], case.scale, case.window)
    dev_idx = torch.from_numpy(idx).to(DEV)
    compare(out[dev_idx], o_ref, "bf16", lse[dev_idx], l_ref, "sliding window full workload sample")
