"""Pins for the oracle's tree verification, multi-query MLA and fp8 MLA
functions (CPU only).

Each check ties a function to something other than itself: torch's fp64
scaled_dot_product_attention with a mask built here, the single-query oracle
functions on inputs rearranged here, torch's float8_e4m3fn conversion, hand
values, and planted mistakes that a pin must catch.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
import oracle.fp8 as of8


def _paged(rng, rows, lens, page_size, spare=3):
    """Scatter contiguous per-sequence rows [B, Lmax, ...] into a shuffled pool
    whose unowned rows are NaN; returns (pool, block_table)."""
    B = rows.shape[0]
    n_pages = [(int(L) + page_size - 1) // page_size for L in lens]
    P = sum(n_pages) + spare
    perm = rng.permutation(P)
    pool = np.full((P, page_size) + rows.shape[2:], np.nan)
    bt = np.full((B, max(n_pages) + 1), perm[-1], dtype=np.int64)
    c = 0
    for b in range(B):
        for j in range(n_pages[b]):
            bt[b, j] = perm[c]
            c += 1
        for t in range(int(lens[b])):
            pool[bt[b, t // page_size], t % page_size] = rows[b, t]
    return pool, bt


# ---------------------------------------------------------------------------
# Tree verification
# ---------------------------------------------------------------------------

def test_tree_ancestors_hand_values():
    #        ctx
    #       /   \
    #      0     1
    #     / \     \
    #    2   3     4
    #        |
    #        5
    assert oracle.tree_ancestors([-1, -1, 0, 0, 1, 3]) == [[0], [1], [0, 2], [0, 3], [1, 4], [0, 3, 5]]
    assert oracle.tree_ancestors([-1, 0, 1, 2]) == [[0], [0, 1], [0, 1, 2], [0, 1, 2, 3]]
    with pytest.raises(ValueError):
        oracle.tree_ancestors([-1, 2, 0])      # parent after the child


TREES = {
    "branchy": [-1, -1, 0, 0, 1, 3],
    "chain": [-1, 0, 1, 2, 3, 4],
    "star": [-1, -1, -1, -1, -1, -1],
    "two_level": [-1, 0, 0, 0, 1, 2],
}


def _tree_problem(seed, n=6, B=4, H_q=8, H_kv=2, D=16, page_size=4, Lmax=31, trees=None):
    rng = np.random.default_rng(seed)
    lens = rng.integers(n, Lmax + 1, size=B)
    lens[0] = Lmax
    lens[1] = n                      # the draft tokens are the whole context
    K = rng.standard_normal((B, Lmax, H_kv, D))
    V = rng.standard_normal((B, Lmax, H_kv, D))
    q = rng.standard_normal((B, n, H_q, D))
    kp, bt = _paged(rng, K, lens, page_size)
    vp = np.full_like(kp, np.nan)
    for b in range(B):
        for t in range(int(lens[b])):
            vp[bt[b, t // page_size], t % page_size] = V[b, t]
    names = trees or list(TREES)
    parents = np.array([TREES[names[b % len(names)]] for b in range(B)])
    return q, K, V, lens, kp, vp, bt, parents


def _tree_sdpa_reference(q, K, V, lens, parents, scale, g):
    """torch fp64 SDPA with an explicit mask: node j sees the context and the
    draft positions of the nodes on its path, walked up here from the parents."""
    B, n, H_q, D = q.shape
    out = np.zeros((B, n, H_q, V.shape[3]))
    for b in range(B):
        L = int(lens[b])
        ctx = L - n
        mask = torch.zeros(n, L, dtype=torch.bool)
        mask[:, :ctx] = True
        for j in range(n):
            a = j
            while a >= 0:
                mask[j, ctx + a] = True
                a = int(parents[b, a])
        k = torch.from_numpy(K[b, :L]).permute(1, 0, 2).repeat_interleave(g, dim=0)
        v = torch.from_numpy(V[b, :L]).permute(1, 0, 2).repeat_interleave(g, dim=0)
        qq = torch.from_numpy(q[b]).permute(1, 0, 2)
        o = F.scaled_dot_product_attention(qq[None], k[None], v[None], attn_mask=mask, scale=scale)
        out[b] = o[0].permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_verify_matches_masked_torch_sdpa(seed):
    q, K, V, lens, kp, vp, bt, parents = _tree_problem(60 + seed)
    o, lse = oracle.tree_verify_decode_attention(q, kp, vp, bt, lens, parents, 0.33)
    ref = _tree_sdpa_reference(q, K, V, lens, parents, 0.33, 4)
    np.testing.assert_allclose(o, ref, atol=1e-12, rtol=0)
    # LSE of node 5 of the branchy tree (path 0, 3, 5): scipy over its keys
    b, j, n = 0, 5, q.shape[1]
    ctx = int(lens[b]) - n
    keys = list(range(ctx)) + [ctx + 0, ctx + 3, ctx + 5]
    for h in range(q.shape[2]):
        s = 0.33 * K[b, keys, h // 4] @ q[b, j, h]
        assert abs(lse[b, j, h] - logsumexp(s)) < 1e-12


def test_chain_tree_is_causal_multi_query():
    q, K, V, lens, kp, vp, bt, parents = _tree_problem(70, trees=["chain"])
    o, lse = oracle.tree_verify_decode_attention(q, kp, vp, bt, lens, parents, 0.27)
    o2, l2 = oracle.multi_query_decode_attention(q, kp, vp, bt, lens, 0.27)
    np.testing.assert_allclose(o, o2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse, l2, atol=1e-13, rtol=0)


def test_tree_rows_are_single_queries_over_context_plus_path():
    """Each node equals plain decode over a cache holding only the context
    followed by its path's rows, re-paged into fresh pages (test-side copy)."""
    q, K, V, lens, kp, vp, bt, parents = _tree_problem(71)
    o, lse = oracle.tree_verify_decode_attention(q, kp, vp, bt, lens, parents, 0.31)
    B, n = q.shape[:2]
    rng = np.random.default_rng(5)
    for b in range(B):
        ctx = int(lens[b]) - n
        for j in range(n):
            path = [j]
            while parents[b, path[-1]] >= 0:
                path.append(int(parents[b, path[-1]]))
            keys = list(range(ctx)) + [ctx + a for a in reversed(path)]
            Lb = len(keys)
            kp1, bt1 = _paged(rng, K[b:b + 1, keys], [Lb], 4)
            vp1 = np.full_like(kp1, np.nan)    # V at the same pages as K
            for t in range(Lb):
                vp1[bt1[0, t // 4], t % 4] = V[b, keys[t]]
            o1, l1 = oracle.decode_attention(q[b:b + 1, j], kp1, vp1, bt1, [Lb], 0.31)
            np.testing.assert_allclose(o[b, j], o1[0], atol=1e-13, rtol=0)
            np.testing.assert_allclose(lse[b, j], l1[0], atol=1e-13, rtol=0)


def test_tree_rows_ignore_rows_off_their_path():
    q, K, V, lens, kp, vp, bt, parents = _tree_problem(72, trees=["branchy"])
    o, _ = oracle.tree_verify_decode_attention(q, kp, vp, bt, lens, parents, 0.3)
    b, n = 0, q.shape[1]
    pos = int(lens[b]) - n + 4        # node 4 (child of 1): on the paths of 4 only
    page, row = bt[b, pos // 4], pos % 4
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[page, row] += 4.0
    vp2[page, row] -= 2.0
    o2, _ = oracle.tree_verify_decode_attention(q, kp2, vp2, bt, lens, parents, 0.3)
    for j in (0, 1, 2, 3, 5):
        np.testing.assert_array_equal(o2[b, j], o[b, j])
    assert not np.allclose(o2[b, 4], o[b, 4])


def test_mutation_sibling_visible_mask_is_caught(monkeypatch):
    """A causal mask in place of the ancestor mask (every earlier draft token
    visible) fails the masked-SDPA pin on a branching tree."""
    def causal(q, k_pool, v_pool, block_table, seq_lens, parents, scale):
        return oracle.multi_query_decode_attention(q, k_pool, v_pool, block_table, seq_lens, scale)
    monkeypatch.setattr(oracle, "tree_verify_decode_attention", causal)
    with pytest.raises(AssertionError):
        test_tree_verify_matches_masked_torch_sdpa(0)


# ---------------------------------------------------------------------------
# Multi-query absorbed MLA
# ---------------------------------------------------------------------------

def _mla_problem(seed, q_len, B=3, H=6, Dqk=24, Dv=16, ps=8, Lmax=45):
    rng = np.random.default_rng(seed)
    lens = rng.integers(q_len, Lmax + 1, size=B)
    lens[0] = Lmax
    lens[1] = q_len
    C = rng.standard_normal((B, Lmax, Dqk))
    q = rng.standard_normal((B, q_len, H, Dqk))
    pool, bt = _paged(rng, C, lens, ps)
    return q, C, lens, pool, bt, Dv


@pytest.mark.parametrize("q_len", [1, 2, 4])
def test_mla_multi_query_matches_causal_torch_sdpa(q_len):
    q, C, lens, pool, bt, Dv = _mla_problem(80 + q_len, q_len)
    o, lse = oracle.mla_multi_query_decode_attention(q, pool, bt, lens, 0.21, Dv)
    B, _, H, Dqk = q.shape
    for b in range(B):
        L = int(lens[b])
        k = torch.from_numpy(C[b, :L])[None, None].expand(1, H, L, Dqk)
        v = torch.from_numpy(C[b, :L, :Dv])[None, None].expand(1, H, L, Dv)
        qq = torch.from_numpy(q[b]).permute(1, 0, 2)[None]      # [1, H, q_len, Dqk]
        mask = torch.arange(L)[None, :] <= (L - q_len + torch.arange(q_len))[:, None]
        ref = F.scaled_dot_product_attention(qq, k, v, attn_mask=mask, scale=0.21)
        np.testing.assert_allclose(o[b], ref[0].permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)
        for j in range(q_len):
            Lj = L - q_len + 1 + j
            s = 0.21 * (q[b, j] @ C[b, :Lj].T)
            np.testing.assert_allclose(lse[b, j], logsumexp(s, axis=-1), atol=1e-12)


def test_mla_multi_query_of_one_token_is_mla_decode():
    q, C, lens, pool, bt, Dv = _mla_problem(90, 1)
    o, lse = oracle.mla_multi_query_decode_attention(q, pool, bt, lens, 0.3, Dv)
    o1, l1 = oracle.mla_decode_attention(q[:, 0], pool, bt, lens, 0.3, Dv)
    np.testing.assert_array_equal(o[:, 0], o1)
    np.testing.assert_array_equal(lse[:, 0], l1)


def test_mla_multi_query_rows_are_single_queries_over_shortened_contexts():
    q_len = 4
    q, C, lens, pool, bt, Dv = _mla_problem(91, q_len)
    o, lse = oracle.mla_multi_query_decode_attention(q, pool, bt, lens, 0.3, Dv)
    for j in range(q_len):
        o1, l1 = oracle.mla_decode_attention(q[:, j], pool, bt, lens - q_len + 1 + j, 0.3, Dv)
        np.testing.assert_array_equal(o[:, j], o1)
        np.testing.assert_array_equal(lse[:, j], l1)


def test_mutation_mla_multi_query_without_mask_is_caught(monkeypatch):
    def unmasked(q, kv_pool, block_table, seq_lens, scale, d_v):
        outs = [oracle.mla_decode_attention(q[:, j], kv_pool, block_table, seq_lens, scale, d_v)
                for j in range(q.shape[1])]
        return np.stack([x[0] for x in outs], 1), np.stack([x[1] for x in outs], 1)
    monkeypatch.setattr(oracle, "mla_multi_query_decode_attention", unmasked)
    with pytest.raises(AssertionError):
        test_mla_multi_query_matches_causal_torch_sdpa(4)


# ---------------------------------------------------------------------------
# fp8 MLA input path
# ---------------------------------------------------------------------------

def _torch_dequant(codes, scale):
    """Test-side reconstruction through torch's float8_e4m3fn conversion."""
    v = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float32)
    return (v * torch.from_numpy(np.asarray(scale, np.float32))[..., None]).numpy().astype(np.float64)


def _fp8_mla_problem(seed, B=3, H=4, Dqk=32, Dv=16, ps=8, Lmax=40, P=12):
    rng = np.random.default_rng(seed)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    q_codes = rng.choice(finite, size=(B, H, Dqk)).astype(np.uint8)
    q_scale = rng.uniform(0.002, 0.01, size=(B, H)).astype(np.float32)
    kv_codes = rng.choice(finite, size=(P, ps, Dqk)).astype(np.uint8)
    kv_scale = rng.uniform(0.002, 0.01, size=(P, ps)).astype(np.float32)
    lens = np.array([Lmax, 1, 17])[:B]
    bt = np.stack([rng.permutation(P) for _ in range(B)])
    return q_codes, q_scale, kv_codes, kv_scale, bt, lens, Dv


def test_fp8_mla_equals_mla_on_torch_dequantized_inputs():
    q_codes, q_scale, kv_codes, kv_scale, bt, lens, Dv = _fp8_mla_problem(100)
    o, lse = oracle.mla_decode_attention_fp8(q_codes, q_scale, kv_codes, kv_scale, bt, lens, 0.07, Dv)
    qd = _torch_dequant(q_codes, q_scale)
    cd = _torch_dequant(kv_codes, kv_scale)
    o2, l2 = oracle.mla_decode_attention(qd, cd, bt, lens, 0.07, Dv)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, l2)
    # one-token context: O is that latent row's reconstructed first Dv columns
    page = bt[1, 0]
    np.testing.assert_allclose(o[1], np.broadcast_to(cd[page, 0, :Dv], o[1].shape), atol=1e-15)


def test_mutation_fp8_mla_scale_left_out_is_caught(monkeypatch):
    real = of8.dequantize
    monkeypatch.setattr(of8, "dequantize", lambda codes, scale: real(codes, np.ones_like(scale)))
    with pytest.raises(AssertionError):
        test_fp8_mla_equals_mla_on_torch_dequantized_inputs()
