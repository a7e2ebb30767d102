"""Pools past 4 GiB: byte offsets into a K/V (or latent) pool no longer fit 32
bits. Every path runs once on a small pool and once on a pool of more than
5 GiB that holds the same pages at high page ids (the block table remapped,
the pages spread every other id up to the top of the pool). Page ids only
select rows, so the two runs must agree bit for bit; the small-pool results
are themselves held to the oracle by the other parity tests."""

import numpy as np
import pytest
import torch

import paged_kv_cache_46_gb300 as ts
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
BIG_BYTES = 5 << 30  # per pool


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_46_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    yield
    torch.cuda.empty_cache()


def _relocate(tensors, bt):
    """Copy pools (and per-page scale arrays) [P, ...] into pools of more than
    BIG_BYTES bytes: page p moves to id big - 1 - 2p. Returns the new tensors,
    the remapped block table and the new page count."""
    P = tensors[0].shape[0]
    page_bytes = tensors[0][0].numel() * tensors[0].element_size()
    big = max(2 * P, BIG_BYTES // page_bytes + 1)
    new_id = big - 1 - 2 * np.arange(P, dtype=np.int64)
    ids = torch.from_numpy(new_id).to(DEV)
    out = []
    for t in tensors:
        b = torch.empty((big,) + tuple(t.shape[1:]), dtype=t.dtype, device=DEV)
        b.index_copy_(0, ids, t)
        out.append(b)
    assert out[0].numel() * out[0].element_size() > (4 << 30)
    bt_new = np.where((bt >= 0) & (bt < P), new_id[np.clip(bt, 0, P - 1)], bt).astype(np.int32)
    return out, bt_new, big, ids


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _same(a, b, what):
    """Bitwise equality (pool rows holding no token are NaN)."""
    if a.dtype in (torch.bfloat16, torch.float16):
        a, b = a.view(torch.int16), b.view(torch.int16)
    elif a.dtype == torch.float32:
        a, b = a.view(torch.int32), b.view(torch.int32)
    assert torch.equal(a, b), f"{what}: large-pool result differs"


def test_append_and_decode_on_a_pool_past_4_gib():
    lens = np.array([700, 1, 4000, 33, 2048, 15, 1500, 999], dtype=np.int32)
    case = workloads.build_case("big_pool", 81, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                seq_lens=lens, dtype="bf16", scale=128 ** -0.5, device=DEV, append=True)
    (kb, vb), bt_big, big, ids = _relocate([case.k_pool, case.v_pool], case.block_table)
    pos = _dev(case.positions)
    lens_dev = _dev(case.attn_lens)
    results = []
    for kp, vp, bt in ((case.k_pool.clone(), case.v_pool.clone(), case.block_table), (kb, vb, bt_big)):
        btd = _dev(bt)
        ts.ts_kv_append(case.k_new, case.v_new, kp, vp, btd, pos)
        ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D), DEV)
        out, lse = ts.ts_paged_decode_attn(case.q, kp, vp, btd, lens_dev, case.scale, workspace=ws,
                                           return_lse=True)
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
        results.append((kp, vp, out, lse))
    (k0, v0, o0, l0), (k1, v1, o1, l1) = results
    _same(k1.index_select(0, ids), k0, "appended K rows")
    _same(v1.index_select(0, ids), v0, "appended V rows")
    _same(o1, o0, "decode output")
    _same(l1, l0, "decode LSE")


@pytest.mark.parametrize("hg", [1, 2])
def test_tensor_core_multi_query_on_a_pool_past_4_gib(hg, monkeypatch):
    lens = np.array([4, 3000, 129, 2500, 640, 77, 4096, 1200], dtype=np.int32)
    case = workloads.build_case("big_pool_mq", 82, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                seq_lens=lens, dtype="bf16", scale=128 ** -0.5, device=DEV, q_len=4)
    (kb, vb), bt_big, big, _ = _relocate([case.k_pool, case.v_pool], case.block_table)
    monkeypatch.setenv("TS_MULTI_QUERY_PATH", "tensor")
    monkeypatch.setenv("TS_MULTI_QUERY_HEAD_GROUP", str(hg))
    lens_dev = _dev(case.seq_lens)
    res = []
    for kp, vp, bt in ((case.k_pool, case.v_pool, case.block_table), (kb, vb, bt_big)):
        ws = ts.new_workspace(ts.ts_paged_decode_multi_workspace_size(case.B, 4, case.H_q, case.D), DEV)
        out, lse = ts.ts_paged_decode_multi_attn(case.q, kp, vp, _dev(bt), lens_dev, case.scale, workspace=ws,
                                                 return_lse=True)
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
        res.append((out, lse))
    _same(res[1][0], res[0][0], f"multi-query output hg={hg}")
    _same(res[1][1], res[0][1], f"multi-query LSE hg={hg}")


def test_fp8_append_and_decode_on_a_pool_past_4_gib():
    lens = np.array([500, 2, 3000, 17, 1024, 4095, 60, 800], dtype=np.int32)
    case = workloads.build_fp8_case("big_pool_fp8", 83, B=len(lens), H_q=32, H_kv=8, D=128, page_size=16,
                                    seq_lens=lens, scale=128 ** -0.5, device=DEV, append=True)
    (kb, vb, ksb, vsb), bt_big, big, ids = _relocate([case.k_pool, case.v_pool, case.k_scale, case.v_scale],
                                                     case.block_table)
    pos = _dev(case.positions)
    lens_dev = _dev(case.attn_lens)
    res = []
    small = (case.k_pool.clone(), case.v_pool.clone(), case.k_scale.clone(), case.v_scale.clone(), case.block_table)
    for kp, vp, ks, vs, bt in (small, (kb, vb, ksb, vsb, bt_big)):
        btd = _dev(bt)
        ts.ts_kv_append_fp8(case.k_new, case.v_new, kp, vp, ks, vs, btd, pos)
        ws = ts.new_workspace(ts.ts_paged_decode_workspace_size(case.B, case.H_q, case.D), DEV)
        out, lse = ts.ts_paged_decode_fp8_attn(case.q, kp, vp, ks, vs, btd, lens_dev, case.scale, workspace=ws,
                                               return_lse=True)
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
        res.append((kp, ks, out, lse))
    (k0, s0, o0, l0), (k1, s1, o1, l1) = res
    _same(k1.index_select(0, ids), k0, "appended fp8 K codes")
    _same(s1.index_select(0, ids), s0, "appended K scales")
    _same(o1, o0, "fp8 decode output")
    _same(l1, l0, "fp8 decode LSE")


def test_cascade_on_a_pool_past_4_gib():
    case = workloads.shared_prefix_cascade(device=DEV, seed=84, groups=2, members=40, prefix_tokens=512,
                                           suffix_lo=1, suffix_hi=300, ungrouped=3)
    (kb, vb), bt_big, big, _ = _relocate([case.k_pool, case.v_pool], case.block_table)
    lens_dev = _dev(case.attn_lens)
    res = []
    for kp, vp, bt in ((case.k_pool, case.v_pool, case.block_table), (kb, vb, bt_big)):
        groups = ts.ts_group_prefixes(bt, case.seq_lens, case.page_size, 2)
        assert groups["num_groups"] == 2
        gdev = ts.groups_to_device(groups, DEV)
        ws = ts.new_workspace(ts.ts_cascade_decode_workspace_size(case.B, case.H_q, case.D), DEV)
        out, lse = ts.ts_cascade_decode_attn(case.q, kp, vp, gdev, _dev(bt), lens_dev, case.scale, workspace=ws,
                                             return_lse=True)
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
        res.append((out, lse))
    _same(res[1][0], res[0][0], "cascade output")
    _same(res[1][1], res[0][1], "cascade LSE")


def test_mla_on_a_pool_past_4_gib():
    case = workloads.absorbed_mla(device=DEV, seed=85, B=4, lo=900, hi=3000)
    (pb,), bt_big, big, _ = _relocate([case.k_pool], case.block_table)
    lens_dev = _dev(case.attn_lens)
    res = []
    for pool, bt in ((case.k_pool, case.block_table), (pb, bt_big)):
        ws = ts.new_workspace(ts.ts_mla_workspace_size(case.B, case.H_q, case.Dv), DEV)
        out, lse = ts.ts_mla_paged_decode(case.q, pool, _dev(bt), lens_dev, case.scale, d_v=case.Dv, workspace=ws,
                                          return_lse=True)
        torch.cuda.synchronize()
        assert ts.ts_read_device_error(ws) == 0
        res.append((out, lse))
    _same(res[1][0], res[0][0], "MLA output")
    _same(res[1][1], res[0][1], "MLA LSE")
