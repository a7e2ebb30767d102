"""GPU parity for the fp8 (e4m3fn) cache through the C ABI: the quantizing
append is bit-exact with the oracle's token-group quantizer, and decode over
the codes matches the fp64 oracle on the float32 reconstruction."""

import os

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


def _meta(case):
    return (torch.from_numpy(case.block_table).to(DEV), torch.from_numpy(case.attn_lens).to(DEV),
            torch.from_numpy(case.positions).to(DEV))


def _decode(case, ctas=None, path=None, hg=None, expect_kernel=None):
    """path: None = the library's choice, "tensor" = the tcgen05 kernel where the
    shape allows it, "cuda" = the CUDA-core split-KV kernel; hg: kv heads per
    CTA of the tcgen05 kernel; expect_kernel: the decode kernel the launch
    trace must show."""
    bt, lens, _ = _meta(case)
    env = {"TS_PAGED_DECODE_CTAS": ctas, "TS_FP8_DECODE_PATH": path, "TS_FP8_HEAD_GROUP": hg}
    for k, v in env.items():
        if v is not None:
            os.environ[k] = str(v)
    ts.ts_trace_collect()
    ts.ts_trace_enable(expect_kernel is not None)
    try:
        ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D))
        out, lse = ts.ts_paged_decode_fp8_attn(case.q, case.k_pool, case.v_pool, case.k_scale, case.v_scale,
                                               bt, lens, case.scale, workspace=ws, return_lse=True)
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
    finally:
        ts.ts_trace_enable(False)
        for k in env:
            os.environ.pop(k, None)
    recs = ts.ts_trace_collect()
    if expect_kernel is not None:
        assert recs and recs[0][0] == expect_kernel, recs
    return out, lse


def _oracle(case, view=None):
    v = view or workloads.oracle_view(case)
    return oracle.decode_attention_fp8(v["q"], v["k_pool"], v["v_pool"], v["k_scale"], v["v_scale"],
                                       v["block_table"], v["seq_lens"], case.scale)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_append_fp8_bit_exact(dtype):
    lens = [0, 15, 16, 31, 100, 1]
    case = workloads.build_fp8_case("fp8_append", 81, B=len(lens), H_q=16, H_kv=4, D=128, page_size=16,
                                    seq_lens=lens, scale=0.09, append=True, device=DEV)
    kn, vn = case.k_new, case.v_new
    if dtype == "f32":  # f32 rows that are not bf16 values
        g = torch.Generator(device=DEV).manual_seed(5)
        kn = torch.randn(kn.shape, generator=g, device=DEV) * 3
        vn = torch.randn(vn.shape, generator=g, device=DEV) * 0.01
        vn[0, 0] = 0.0  # an all-zero group takes the 1e-10 scale floor
    before = [t.clone() for t in (case.k_pool, case.v_pool, case.k_scale, case.v_scale)]
    bt, _, pos = _meta(case)
    ts.ts_kv_append_fp8(kn, vn, case.k_pool, case.v_pool, case.k_scale, case.v_scale, bt, pos)
    torch.cuda.synchronize()
    ref = oracle.kv_append_fp8(*(t.cpu().numpy() for t in before), kn.float().cpu().numpy(),
                               vn.float().cpu().numpy(), case.block_table, case.positions, case.page_size)
    got = [t.cpu().numpy() for t in (case.k_pool, case.v_pool, case.k_scale, case.v_scale)]
    for r, gt, what in zip(ref, got, ("k codes", "v codes", "k scales", "v scales")):
        if r.dtype == np.float32:  # NaN sentinels stay NaN: compare bit patterns
            np.testing.assert_array_equal(r.view(np.uint32), gt.view(np.uint32), err_msg=what)
        else:
            np.testing.assert_array_equal(r, gt, err_msg=what)


@pytest.mark.parametrize("D,H_q,H_kv,ps", [(128, 32, 8, 16), (64, 32, 8, 16), (128, 8, 8, 8), (64, 16, 8, 32),
                                           (128, 4, 1, 16), (64, 8, 4, 16)])
def test_decode_fp8_matches_oracle(D, H_q, H_kv, ps):
    rng = np.random.default_rng(D + H_q + ps)
    lens = rng.integers(1, 900, size=9)
    lens[0], lens[1] = 1, ps
    case = workloads.build_fp8_case(f"fp8_{D}_{H_q}_{H_kv}_{ps}", 83, B=9, H_q=H_q, H_kv=H_kv, D=D,
                                    page_size=ps, seq_lens=lens, scale=D ** -0.5, device=DEV)
    o_ref, l_ref = _oracle(case)
    for ctas in (None, 5):
        out, lse = _decode(case, ctas, path="cuda")
        compare(out, o_ref, "bf16", lse, l_ref, f"fp8 D={D} {H_q}/{H_kv} ps={ps} ctas={ctas}")


@pytest.mark.parametrize("ctas", [1, 7, 1000])
def test_decode_fp8_independent_of_split_pattern(ctas):
    lens = [0, 1, 15, 16, 17, 700, 2049, 64]
    case = workloads.build_fp8_case("fp8_split", 85, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                    seq_lens=lens, scale=0.0884, device=DEV)
    out, lse = _decode(case, ctas, path="cuda")
    o_ref, l_ref = _oracle(case)
    compare(out, o_ref, "bf16", lse, l_ref, f"ctas={ctas}")


def test_llama_fp8_step_append_then_decode():
    """The Llama-3-8B layer shape over an fp8 cache, one append then decode,
    every output row against the oracle (which quantizes the new rows itself)."""
    case = workloads.llama3_8b_layer_fp8(device=DEV)
    view = workloads.oracle_view(case)
    bt, lens, pos = _meta(case)
    ts.ts_kv_append_fp8(case.k_new, case.v_new, case.k_pool, case.v_pool, case.k_scale, case.v_scale, bt, pos)
    out, lse = _decode(case, expect_kernel="paged_decode_kernel")  # the library's choice: the CUDA-core kernel
    kp, vp, ks, vs = oracle.kv_append_fp8(view["k_pool"], view["v_pool"], view["k_scale"], view["v_scale"],
                                          view["k_new"], view["v_new"], view["block_table"], view["positions"],
                                          case.page_size)
    o_ref, l_ref = oracle.decode_attention_fp8(view["q"], kp, vp, ks, vs, view["block_table"], view["seq_lens"],
                                               case.scale)
    compare(out, o_ref, "bf16", lse, l_ref, "llama fp8 step")


@pytest.mark.parametrize("D,H_q,H_kv,hg", [(128, 32, 8, 2), (128, 32, 8, 4), (64, 32, 8, 2), (64, 16, 4, 4),
                                           (128, 16, 2, 2), (128, 64, 4, 2)])
def test_decode_fp8_tensor_core_path(D, H_q, H_kv, hg):
    """The tcgen05 kernel (2 or 4 kv heads per CTA, codes widened to f16 by
    converter warps, scales on the scores and probabilities) against the
    oracle: a one-token context, exact page and tile multiples, one key past
    a tile, longer contexts; the launch trace shows the kernel ran."""
    rng = np.random.default_rng(D * 7 + H_q + hg)
    lens = rng.integers(1, 2500, size=10)
    tile = 16 * (8 // hg)
    lens[:5] = [1, 16, tile, tile + 1, 2 * tile - 1]
    case = workloads.build_fp8_case(f"fp8_tc_{D}_{H_q}_{H_kv}_{hg}", 87, B=len(lens), H_q=H_q, H_kv=H_kv, D=D,
                                    page_size=16, seq_lens=lens, scale=D ** -0.5, device=DEV)
    o_ref, l_ref = _oracle(case)
    out, lse = _decode(case, path="tensor", hg=hg, expect_kernel="fp8_tc_kernel")
    compare(out, o_ref, "bf16", lse, l_ref, f"fp8 tensor core D={D} {H_q}/{H_kv} hg={hg}")


def test_decode_fp8_paths_agree_on_the_llama_shape():
    """The Llama-3-8B layer shape over an fp8 cache: the tensor-core and the
    CUDA-core kernels against each other (every output) and the oracle on a
    sample of 16 sequences."""
    case = workloads.llama3_8b_layer_fp8(device=DEV, append=False)
    o_tc, l_tc = _decode(case, path="tensor", expect_kernel="fp8_tc_kernel")
    o_cc, l_cc = _decode(case, path="cuda")
    assert (o_tc.float() - o_cc.float()).abs().max().item() <= 2e-2
    assert (l_tc - l_cc).abs().max().item() <= 1e-3
    idx = workloads.sample_sequences(case, 16)
    view = workloads.oracle_view(case, idx)
    o_ref, l_ref = _oracle(case, view)
    dev_idx = torch.from_numpy(idx).to(DEV)
    compare(o_tc[dev_idx], o_ref, "bf16", l_tc[dev_idx], l_ref, "llama fp8 tensor core sample")


@pytest.mark.parametrize("ctas", [None, 1, 3, 7, 64, 1000])
def test_decode_fp8_code_mma_kernel(ctas):
    """The kernel that multiplies the codes on the tensor cores
    (TS_FP8_DECODE_PATH=mma; 32/8 heads, head dim 128, page 16) against the oracle: empty
    sequences, one key, a page minus one, one page, a page plus one, long
    contexts. The CTA count sweeps the cut: one CTA holds every page,
    sequences cut across several CTAs (merged by the last to arrive), more
    CTAs than pages. The launch trace shows the kernel ran."""
    lens = [0, 1, 15, 16, 17, 700, 2049, 64, 5000, 0, 333]
    case = workloads.build_fp8_case("fp8_mma", 89, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                    seq_lens=lens, scale=128 ** -0.5, device=DEV)
    o_ref, l_ref = _oracle(case)
    out, lse = _decode(case, ctas, path="mma", expect_kernel="fp8_mma_kernel")
    compare(out, o_ref, "bf16", lse, l_ref, f"fp8 code products ctas={ctas}")


def test_decode_fp8_code_mma_bad_page_is_flagged_without_fault():
    """A page id past the pool: the error word reports it, the page reads as
    zeros (no out-of-range access), every output stays finite and the other
    sequences are unaffected."""
    lens = [40, 300, 33, 900]
    case = workloads.build_fp8_case("fp8_mma_bad", 90, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                    seq_lens=lens, scale=128 ** -0.5, device=DEV)
    case.block_table = case.block_table.copy()
    case.block_table[1, 3] = case.num_pages + 5
    bt, dlens, _ = _meta(case)
    ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D))
    os.environ["TS_FP8_DECODE_PATH"] = "mma"
    try:
        out, lse = ts.ts_paged_decode_fp8_attn(case.q, case.k_pool, case.v_pool, case.k_scale, case.v_scale, bt,
                                               dlens, case.scale, workspace=ws, return_lse=True)
        torch.cuda.synchronize()
    finally:
        os.environ.pop("TS_FP8_DECODE_PATH", None)
    assert ts.ts_read_device_error(ws) & ts.TS_DEVERR_PAGE_RANGE
    assert torch.isfinite(out.float()).all()
    good = np.array([0, 2, 3])
    view = workloads.oracle_view(case, good)
    o_ref, l_ref = _oracle(case, view)
    sel = torch.from_numpy(good).to(DEV)
    compare(out[sel], o_ref, "bf16", lse[sel], l_ref, "fp8 code products, bad page neighbours")


def test_decode_fp8_code_mma_repeats_bit_for_bit_and_replays_from_a_graph():
    """Launches on one workspace without clearing it, and replays of a captured
    CUDA graph (the same launch epoch every time: the counters of the cut
    sequences must return to zero), all give the same bits, and those match
    the oracle. 40 CTAs cut most sequences."""
    rng = np.random.default_rng(91)
    lens = rng.integers(1, 3000, size=24)
    case = workloads.build_fp8_case("fp8_mma_rep", 91, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                    seq_lens=lens, scale=128 ** -0.5, device=DEV)
    bt, dlens, _ = _meta(case)
    os.environ["TS_PAGED_DECODE_CTAS"] = "40"
    os.environ["TS_FP8_DECODE_PATH"] = "mma"
    try:
        ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D))
        out = torch.empty_like(case.q)
        lse = torch.empty(case.B, case.H_q, dtype=torch.float32, device=DEV)
        stream = torch.cuda.Stream()

        def call():
            ts.ts_paged_decode_fp8_attn(case.q, case.k_pool, case.v_pool, case.k_scale, case.v_scale, bt, dlens,
                                        case.scale, out=out, lse=lse, workspace=ws, stream=stream)

        with torch.cuda.stream(stream):
            call()
        torch.cuda.synchronize()
        first = (out.clone(), lse.clone())
        for _ in range(2):
            with torch.cuda.stream(stream):
                call()
            torch.cuda.synchronize()
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1])
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            call()
        for _ in range(3):
            out.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1])
        assert ts.ts_read_device_error(ws) == 0
    finally:
        os.environ.pop("TS_PAGED_DECODE_CTAS", None)
        os.environ.pop("TS_FP8_DECODE_PATH", None)
    o_ref, l_ref = _oracle(case)
    compare(first[0], o_ref, "bf16", first[1], l_ref, "fp8 code products, repeated")


def test_decode_fp8_code_mma_on_the_llama_shape():
    """The Llama-3-8B layer workload over an fp8 cache (B = 64, lengths
    U[512, 4096]) in the benchmark's launch configuration: the code-multiplying
    kernel against the CUDA-core kernel on every output, and against the
    oracle on a sample of 16 sequences."""
    case = workloads.llama3_8b_layer_fp8(device=DEV, append=False)
    o_mm, l_mm = _decode(case, path="mma", expect_kernel="fp8_mma_kernel")
    o_cc, l_cc = _decode(case, path="cuda", expect_kernel="paged_decode_kernel")
    assert (o_mm.float() - o_cc.float()).abs().max().item() <= 2e-2
    assert (l_mm - l_cc).abs().max().item() <= 2e-4
    idx = workloads.sample_sequences(case, 16)
    view = workloads.oracle_view(case, idx)
    o_ref, l_ref = _oracle(case, view)
    dev_idx = torch.from_numpy(idx).to(DEV)
    compare(o_mm[dev_idx], o_ref, "bf16", l_mm[dev_idx], l_ref, "llama fp8 code products sample")
