"""GPU parity: ts_kv_append (bit-exact) and ts_paged_decode_attn / ts_merge_states
against the fp64 oracle, through the C ABI. Needs a GB300 and the built library."""

import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_46_gb300 as ts
import workloads
from gpu_helpers import as_f64, compare, device_metadata, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_46_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _run_decode(case, ctas=None, check_error_word=True):
    bt, lens, pos = device_metadata(case)
    if ctas is not None:
        os.environ["TS_PAGED_DECODE_CTAS"] = str(ctas)
    try:
        ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D))
        out, lse = ts.ts_paged_decode_attn(case.q, case.k_pool, case.v_pool, bt, lens, case.scale,
                                           workspace=ws, return_lse=True)
        torch.cuda.synchronize()
        err = ts.ts_read_device_error(ws)
    finally:
        os.environ.pop("TS_PAGED_DECODE_CTAS", None)
    if check_error_word:
        assert err == 0, f"device error word {err:#x}"
    return out, lse, err


def _append(case):
    bt, lens, pos = device_metadata(case)
    ts.ts_kv_append(case.k_new, case.v_new, case.k_pool, case.v_pool, bt, pos)


def test_tiny_gqa_append_fp32():
    """Tiny paged GQA decode with one appended token (fp32, 8/2 heads, D=64,
    page 16, lens {17,40,64,100}, 64-page pool)."""
    case = workloads.tiny_gqa_append(device=DEV)
    k0, v0 = case.k_pool.clone(), case.v_pool.clone()
    _append(case)
    torch.cuda.synchronize()
    # bit-exact pools (NaN sentinels included) against the oracle's append
    ok, ov = oracle.kv_append(k0.cpu().numpy().view(np.uint32), v0.cpu().numpy().view(np.uint32),
                              case.k_new.cpu().numpy().view(np.uint32), case.v_new.cpu().numpy().view(np.uint32),
                              case.block_table, case.positions, case.page_size)
    assert np.array_equal(case.k_pool.cpu().numpy().view(np.uint32), ok)
    assert np.array_equal(case.v_pool.cpu().numpy().view(np.uint32), ov)
    out, lse, _ = _run_decode(case)
    o_ref, l_ref = oracle_decode(case, k_pool=k0, v_pool=v0)
    compare(out, o_ref, "f32", lse, l_ref, "tiny fp32")


def test_kv_append_bf16_bit_exact_and_untouched_rows():
    case = workloads.llama3_8b_layer(device=DEV, B=16, lo=1, hi=300)
    k0, v0 = case.k_pool.clone(), case.v_pool.clone()
    _append(case)
    torch.cuda.synchronize()
    ok, ov = oracle.kv_append(k0.cpu().view(torch.int16).numpy(), v0.cpu().view(torch.int16).numpy(),
                              case.k_new.cpu().view(torch.int16).numpy(), case.v_new.cpu().view(torch.int16).numpy(),
                              case.block_table, case.positions, case.page_size)
    assert np.array_equal(case.k_pool.cpu().view(torch.int16).numpy(), ok)
    assert np.array_equal(case.v_pool.cpu().view(torch.int16).numpy(), ov)


def test_llama3_8b_layer_full_batch():
    """Llama-3-8B-shaped decode layer at full size (B=64, 32/8 heads, D=128,
    bf16, lens U[512,4096], shuffled 1.25x pool, one appended token): every
    output compared with the oracle."""
    case = workloads.llama3_8b_layer(device=DEV)
    k0, v0 = case.k_pool.clone(), case.v_pool.clone()
    _append(case)
    out, lse, _ = _run_decode(case)
    o_ref, l_ref = oracle_decode(case, k_pool=k0, v_pool=v0)
    compare(out, o_ref, "bf16", lse, l_ref, "llama3 layer B=64")


def test_mixed_lengths_full_batch():
    """Mixed-length batch at full size (lens {20..1000} x 32, B=256, D=64)."""
    case = workloads.mixed_lengths(device=DEV)
    out, lse, _ = _run_decode(case)
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, "mixed lengths")


@pytest.mark.parametrize("ctas", [1, 2, 7, 64, None, 1000])
def test_result_independent_of_split_pattern(ctas):
    """The CTA count decides where sequences are cut; every cut must give the
    oracle's result (1 CTA: no split at all; 1000: many empty ranges)."""
    lens = [0, 1, 15, 16, 17, 33, 700, 2049, 5, 64, 0, 300]
    case = workloads.build_case("split_sweep", 21, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                seq_lens=lens, dtype="bf16", scale=0.0884, device=DEV)
    out, lse, _ = _run_decode(case, ctas=ctas)
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"ctas={ctas}")
    assert np.all(as_f64(out[0]) == 0) and np.all(np.isneginf(as_f64(lse[0])))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_many_sequences_few_ctas(dtype):
    """500 sequences (more than a CTA's 384 threads) over 7 and 3 CTAs: the
    prologue gathers the lengths through shared memory, and the merge takes
    its per-CTA grid (each CTA records the one cut sequence it starts); every
    cut sequence is merged once."""
    rng = np.random.default_rng(61)
    lens = rng.integers(0, 300, size=500)
    lens[::17] = 0
    case = workloads.build_case(f"many_few_{dtype}", 62, B=len(lens), H_q=32, H_kv=8, D=64, page_size=16,
                                seq_lens=lens, dtype=dtype, scale=0.125, device=DEV)
    for ctas in (7, 3):
        out, lse, _ = _run_decode(case, ctas=ctas)
        o_ref, l_ref = oracle_decode(case)
        compare(out, o_ref, dtype, lse, l_ref, f"{dtype} 500 sequences over {ctas} CTAs")


@pytest.mark.parametrize("ctas", [7, None])
def test_one_workspace_serves_calls_with_different_cuts(ctas):
    """The per-CTA records of cut sequences are rewritten by every call, so a
    workspace reused across calls whose lengths cut the batch differently
    (and leave some CTAs without a cut sequence) gives each call's result."""
    lens_sets = [[700, 2049, 5, 64, 300, 17], [16, 33, 2049, 1, 800, 0], [4000, 3, 3, 3, 90, 512],
                 [1, 1, 1, 1, 1, 1]]
    ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(6, 32, 64))
    for i, lens in enumerate(lens_sets):
        case = workloads.build_case(f"reuse_{i}", 51 + i, B=6, H_q=32, H_kv=8, D=64, page_size=16,
                                    seq_lens=lens, dtype="bf16", scale=0.125, device=DEV)
        bt, dlens, _ = device_metadata(case)
        if ctas is not None:
            os.environ["TS_PAGED_DECODE_CTAS"] = str(ctas)
        try:
            out, lse = ts.ts_paged_decode_attn(case.q, case.k_pool, case.v_pool, bt, dlens, case.scale,
                                               workspace=ws, return_lse=True)
            torch.cuda.synchronize()
        finally:
            os.environ.pop("TS_PAGED_DECODE_CTAS", None)
        assert ts.ts_read_device_error(ws) == 0
        o_ref, l_ref = oracle_decode(case)
        compare(out, o_ref, "bf16", lse, l_ref, f"reuse call {i} ctas={ctas}")


@pytest.mark.parametrize("dtype,D,H_q,H_kv,ps", [
    ("f32", 64, 8, 2, 16), ("f32", 128, 8, 8, 16), ("bf16", 64, 8, 8, 16), ("bf16", 64, 16, 2, 32),
    ("bf16", 128, 64, 8, 16), ("bf16", 128, 8, 1, 8), ("bf16", 64, 4, 4, 16), ("f32", 64, 16, 8, 32),
    # head dim 64, four query rows per kv head, with 2, 1 and 4 kv heads
    ("bf16", 64, 8, 2, 16), ("bf16", 64, 4, 1, 8), ("bf16", 64, 16, 4, 32),
])
def test_shapes(dtype, D, H_q, H_kv, ps):
    rng = np.random.default_rng(D + H_q + H_kv + ps)
    lens = rng.integers(1, 400, size=9)
    lens[2] = ps
    case = workloads.build_case(f"shape_{dtype}_{D}_{H_q}_{H_kv}_{ps}", 31, B=9, H_q=H_q, H_kv=H_kv, D=D,
                                page_size=ps, seq_lens=lens, dtype=dtype, scale=D ** -0.5, device=DEV)
    for ctas in (None, 5):
        out, lse, _ = _run_decode(case, ctas=ctas)
        o_ref, l_ref = oracle_decode(case)
        compare(out, o_ref, dtype, lse, l_ref, f"{dtype} D={D} {H_q}/{H_kv} ps={ps} ctas={ctas}")


def test_edge_cases():
    # single one-token sequence: O = V exactly up to the bf16 output rounding
    case = workloads.build_case("one_token", 41, B=1, H_q=32, H_kv=8, D=128, page_size=16, seq_lens=[1],
                                dtype="bf16", scale=0.1, device=DEV)
    out, lse, _ = _run_decode(case)
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, "one token")
    # all sequences empty
    for dt in ("f32", "bf16"):
        case = workloads.build_case("all_empty", 42, B=5, H_q=8, H_kv=2, D=64, page_size=16, seq_lens=[0] * 5,
                                    dtype=dt, scale=0.1, device=DEV)
        out, lse, _ = _run_decode(case)
        assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    # one long sequence among short ones: cut across most CTAs
    lens = [3] * 20 + [60000] + [7] * 20
    case = workloads.build_case("long_among_short", 43, B=len(lens), H_q=32, H_kv=8, D=64, page_size=16,
                                seq_lens=lens, dtype="bf16", scale=0.125, device=DEV)
    out, lse, _ = _run_decode(case)
    o_ref, l_ref = oracle_decode(case)
    compare(out, o_ref, "bf16", lse, l_ref, "long among short")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_out_of_range_page_is_flagged_not_dereferenced(dtype):
    """A bad page id is caught by the kernel's bounds check: the error word gets
    TS_DEVERR_PAGE_RANGE, nothing faults, other sequences stay correct."""
    case = workloads.build_case("bad_page", 51, B=4, H_q=8, H_kv=2, D=64, page_size=16,
                                seq_lens=[40, 20, 33, 9], dtype=dtype, scale=0.125, device=DEV)
    case.block_table = case.block_table.copy()
    case.block_table[1, 0] = case.num_pages + 5
    out, lse, err = _run_decode(case, check_error_word=False)
    assert err & ts.TS_DEVERR_PAGE_RANGE
    good = np.array([0, 2, 3])
    o_ref, l_ref = oracle_decode(case, seq_idx=good)
    compare(out[torch.from_numpy(good).to(DEV)], o_ref, dtype, lse[torch.from_numpy(good).to(DEV)], l_ref,
            "bad page neighbours")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_merge_states(dtype):
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    rows, D = 1000, 128
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    # attention outputs are convex combinations of value rows: O(1) magnitudes
    o_a = (0.5 * torch.randn(rows, D, generator=g, device=DEV)).to(tdt)
    o_b = (0.5 * torch.randn(rows, D, generator=g, device=DEV)).to(tdt)
    l_a = torch.randn(rows, generator=g, device=DEV) * 4
    l_b = torch.randn(rows, generator=g, device=DEV) * 4
    l_a[::7] = -float("inf")
    l_b[::11] = -float("inf")
    o, l = ts.ts_merge_states(o_a, l_a, o_b, l_b)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.merge_states(as_f64(o_a), as_f64(l_a), as_f64(o_b), as_f64(l_b))
    if dtype == "f32":
        compare(o, o_ref, "f32", l, l_ref, "merge f32")
    else:
        compare(o, o_ref, "bf16", l, l_ref, "merge bf16")


def test_launch_trace_records_each_kernel_of_a_call():
    """With the launch trace on, one append + one decode call record the
    append kernel, the split-KV kernel and the merge kernel, in launch order,
    each with a positive device time; results stay correct."""
    case = workloads.tiny_gqa_append(device=DEV)
    k0, v0 = case.k_pool.clone(), case.v_pool.clone()
    ts.ts_trace_collect()
    ts.ts_trace_enable(True)
    try:
        _append(case)
        out, lse, _ = _run_decode(case)
    finally:
        ts.ts_trace_enable(False)
    recs = ts.ts_trace_collect()
    assert [r[0] for r in recs] == ["kv_append_kernel", "paged_decode_kernel", "split_merge_kernel"]
    assert all(ms > 0 for _, ms in recs)
    o_ref, l_ref = oracle_decode(case, k_pool=k0, v_pool=v0)
    compare(out, o_ref, "f32", lse, l_ref, "traced tiny append")
    assert ts.ts_trace_collect() == []


def test_decode_step_replays_from_a_cuda_graph():
    """One decode step (append + split-KV attention + merge) captured once in a
    CUDA graph and replayed with new inputs written in place: new queries and
    new K/V rows, then shorter lengths. The split plan is computed on the
    device from seq_lens at every launch, so the replays need no host work."""
    case = workloads.llama3_8b_layer(device=DEV, B=8, lo=100, hi=900)
    k0, v0 = case.k_pool.clone(), case.v_pool.clone()
    bt, lens, pos = device_metadata(case)
    q, kn, vn = case.q.clone(), case.k_new.clone(), case.v_new.clone()
    out = torch.empty_like(q)
    lse = torch.empty(case.B, case.H_q, dtype=torch.float32, device=DEV)
    ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D))
    stream = torch.cuda.Stream()

    def step():
        ts.ts_kv_append(kn, vn, case.k_pool, case.v_pool, bt, pos, stream=stream)
        ts.ts_paged_decode_attn(q, case.k_pool, case.v_pool, bt, lens, case.scale, out=out, lse=lse,
                                workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        step()  # warm-up outside the capture (function attributes, tensor maps)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    gen = torch.Generator(device=DEV).manual_seed(123)
    for attempt, shorten in ((0, False), (1, False), (2, True)):
        q.copy_(torch.randn(q.shape, generator=gen, device=DEV).to(q.dtype))
        kn.copy_(torch.randn(kn.shape, generator=gen, device=DEV).to(kn.dtype))
        vn.copy_(torch.randn(vn.shape, generator=gen, device=DEV).to(vn.dtype))
        new_lens = case.attn_lens.copy()
        if shorten:
            new_lens = np.maximum(new_lens // 3, 1).astype(np.int32)
        lens.copy_(torch.from_numpy(new_lens))
        graph.replay()
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
        view = workloads.oracle_view(case, k_pool=k0, v_pool=v0)
        view["q"] = as_f64(q)
        view["k_new"], view["v_new"] = as_f64(kn), as_f64(vn)
        kp, vp = oracle.kv_append(view["k_pool"], view["v_pool"], view["k_new"], view["v_new"],
                                  view["block_table"], view["positions"], case.page_size)
        o_ref, l_ref = oracle.decode_attention(view["q"], kp, vp, view["block_table"],
                                               new_lens.astype(np.int64), case.scale)
        compare(out, o_ref, "bf16", lse, l_ref, f"graph replay {attempt}")
