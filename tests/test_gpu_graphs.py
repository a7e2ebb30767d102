"""CUDA-graph capture of the tensor-core multi-query path and of the
sliding-window path: captured once, replayed with new queries and new
lengths written in place, every replay against the oracle. Both plan their
work on the device (the multi-query kernel ranks the sequences itself, the
window kernel cuts its pages from seq_lens), so replays need no host work."""


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


def _capture(step, stream):
    with torch.cuda.stream(stream):
        step()  # warm-up outside the capture (function attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    return graph


def test_tensor_core_multi_query_replays_from_a_cuda_graph(monkeypatch):
    monkeypatch.setenv("TS_MULTI_QUERY_PATH", "tensor")
    rng = np.random.default_rng(9)
    lens = rng.integers(200, 1500, size=12).astype(np.int32)
    case = workloads.build_case("graph_mq", 90, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16, seq_lens=lens,
                                dtype="bf16", scale=128 ** -0.5, device=DEV, q_len=4)
    bt = torch.from_numpy(case.block_table).to(DEV)
    dlens = torch.from_numpy(case.seq_lens).to(DEV)
    q = case.q.clone()
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    ws = ts.new_workspace(ts.ts_paged_decode_multi_workspace_size(case.B, 4, case.H_q, case.D))
    stream = torch.cuda.Stream()

    def step():
        ts.ts_paged_decode_multi_attn(q, case.k_pool, case.v_pool, bt, dlens, case.scale, out=out, lse=lse,
                                      workspace=ws, stream=stream)
    ts.ts_trace_collect()
    ts.ts_trace_enable(True)  # an eager call: the tensor-core kernel is the one that runs
    try:
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
    finally:
        ts.ts_trace_enable(False)
    assert [r[0] for r in ts.ts_trace_collect()] == ["mq_tc_kernel"]
    graph = _capture(step, stream)
    gen = torch.Generator(device=DEV).manual_seed(7)
    for attempt, shorten in ((0, False), (1, True)):
        q.copy_(torch.randn(q.shape, generator=gen, device=DEV).to(q.dtype))
        new_lens = case.seq_lens.copy()
        if shorten:
            new_lens = np.maximum(new_lens // 3, 4).astype(np.int32)
        dlens.copy_(torch.from_numpy(new_lens))
        graph.replay()
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
        view = workloads.oracle_view(case)
        o_ref, l_ref = oracle.multi_query_decode_attention(as_f64(q), view["k_pool"], view["v_pool"],
                                                           view["block_table"], new_lens.astype(np.int64),
                                                           case.scale)
        compare(out, o_ref, "bf16", lse, l_ref, f"multi-query graph replay {attempt}")


def test_window_decode_replays_from_a_cuda_graph():
    lens = np.array([3000, 10, 1024, 1025, 700, 2048, 33, 1500], dtype=np.int32)
    window = 1000
    case = workloads.build_case("graph_win", 91, B=len(lens), H_q=32, H_kv=8, D=64, page_size=16, seq_lens=lens,
                                dtype="bf16", scale=0.125, device=DEV)
    bt = torch.from_numpy(case.block_table).to(DEV)
    dlens = torch.from_numpy(case.seq_lens).to(DEV)
    q = case.q.clone()
    out = torch.empty_like(q)
    lse = torch.empty(case.B, case.H_q, dtype=torch.float32, device=DEV)
    ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D))
    stream = torch.cuda.Stream()
    graph = _capture(lambda: ts.ts_paged_decode_window_attn(q, case.k_pool, case.v_pool, bt, dlens, case.scale,
                                                            window, out=out, lse=lse, workspace=ws, stream=stream),
                     stream)
    gen = torch.Generator(device=DEV).manual_seed(8)
    for attempt, shorten in ((0, False), (1, True)):
        q.copy_(torch.randn(q.shape, generator=gen, device=DEV).to(q.dtype))
        new_lens = case.seq_lens.copy()
        if shorten:
            new_lens = np.maximum(new_lens // 2, 1).astype(np.int32)
        dlens.copy_(torch.from_numpy(new_lens))
        graph.replay()
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
        view = workloads.oracle_view(case)
        o_ref, l_ref = oracle.decode_attention_window(as_f64(q), view["k_pool"], view["v_pool"],
                                                      view["block_table"], new_lens.astype(np.int64), case.scale,
                                                      window)
        compare(out, o_ref, "bf16", lse, l_ref, f"window graph replay {attempt}")
