"""Pins for the fp64 attention oracle (CPU only).

Each check ties the oracle to something other than itself: a library routine
(torch's fp64 scaled_dot_product_attention, scipy's logsumexp), a closed form,
an invariant, or an independent scatter written here. The mutation tests at the
bottom plant plausible mistakes in the oracle and show a pin catches each.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
import oracle.attention as oa
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _paged_from_contiguous(rng, K, V, lens, page_size, spare_pages=3):
    """Scatter contiguous per-sequence K/V into a shuffled page pool (test-side code).

    K, V: [B, Lmax, H_kv, D]. Returns pools [P, ps, H_kv, D] and block tables.
    Unowned rows are NaN so any stray read poisons the result.
    """
    B, Lmax, H_kv, D = K.shape
    n_pages = [(int(L) + page_size - 1) // page_size for L in lens]
    P = sum(n_pages) + spare_pages
    perm = rng.permutation(P)
    kp = np.full((P, page_size, H_kv, D), np.nan)
    vp = np.full((P, page_size, H_kv, V.shape[3]), np.nan)
    bt = np.full((B, max(n_pages) + 2), perm[-1], dtype=np.int64)
    c = 0
    for b in range(B):
        for j in range(n_pages[b]):
            bt[b, j] = perm[c]
            c += 1
        for t in range(int(lens[b])):
            kp[bt[b, t // page_size], t % page_size] = K[b, t]
            vp[bt[b, t // page_size], t % page_size] = V[b, t]
    return kp, vp, bt


def _sdpa_reference(q, K, V, lens, scale, g):
    """torch fp64 SDPA per sequence on the unpaged K/V; GQA by repeating kv heads."""
    B, H_q, D = q.shape
    out = np.zeros((B, H_q, V.shape[3]))
    for b in range(B):
        L = int(lens[b])
        k = torch.from_numpy(K[b, :L]).permute(1, 0, 2).repeat_interleave(g, dim=0)  # [H_q, L, D]
        v = torch.from_numpy(V[b, :L]).permute(1, 0, 2).repeat_interleave(g, dim=0)
        qq = torch.from_numpy(q[b])[:, None, :]  # [H_q, 1, D]
        o = F.scaled_dot_product_attention(qq[None], k[None], v[None], scale=scale)
        out[b] = o[0, :, 0].numpy()
    return out


def _random_problem(seed, B=5, H_q=8, H_kv=2, D=16, page_size=4, Lmax=37, Dv=None):
    rng = np.random.default_rng(seed)
    Dv = Dv or D
    lens = rng.integers(1, Lmax + 1, size=B)
    lens[0] = Lmax           # a full-length row
    lens[-1] = page_size     # exactly one full page
    q = rng.standard_normal((B, H_q, D))
    K = rng.standard_normal((B, Lmax, H_kv, D))
    V = rng.standard_normal((B, Lmax, H_kv, Dv))
    return rng, q, K, V, lens


@pytest.mark.parametrize("seed,H_q,H_kv,page_size", [(0, 8, 2, 4), (1, 4, 4, 3), (2, 6, 1, 5), (3, 8, 8, 16)])
def test_decode_matches_torch_sdpa_unpaged(seed, H_q, H_kv, page_size):
    rng, q, K, V, lens = _random_problem(seed, H_q=H_q, H_kv=H_kv, page_size=page_size)
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, page_size)
    scale = 0.37
    o, _ = oracle.decode_attention(q, kp, vp, bt, lens, scale)
    ref = _sdpa_reference(q, K, V, lens, scale, H_q // H_kv)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_lse_matches_scipy_logsumexp():
    rng, q, K, V, lens = _random_problem(4)
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, 4)
    scale = 0.5
    _, lse = oracle.decode_attention(q, kp, vp, bt, lens, scale)
    g = q.shape[1] // K.shape[2]
    for b in range(len(lens)):
        L = int(lens[b])
        for h in range(q.shape[1]):
            scores = torch.from_numpy(K[b, :L, h // g]) @ torch.from_numpy(q[b, h]) * scale
            assert abs(lse[b, h] - logsumexp(scores.numpy())) < 1e-12


def test_page_permutation_invariance():
    rng, q, K, V, lens = _random_problem(5, B=6, page_size=4)
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, 4)
    o1, l1 = oracle.decode_attention(q, kp, vp, bt, lens, 0.3)
    perm = rng.permutation(kp.shape[0])          # new physical slot of page p is perm[p]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    o2, l2 = oracle.decode_attention(q, kp2, vp2, perm[bt], lens, 0.3)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(6)
    B, H_q, H_kv, D, ps, L = 2, 4, 2, 8, 4, 11
    K = np.broadcast_to(rng.standard_normal((1, 1, H_kv, D)), (B, L, H_kv, D)).copy()
    V = rng.standard_normal((B, L, H_kv, D))
    q = rng.standard_normal((B, H_q, D))
    lens = np.array([L, 7])
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, ps)
    o, lse = oracle.decode_attention(q, kp, vp, bt, lens, 0.9)
    for b in range(B):
        for h in range(H_q):
            np.testing.assert_allclose(o[b, h], V[b, :lens[b], h // 2].mean(axis=0), atol=1e-13)
            s = 0.9 * q[b, h] @ K[0, 0, h // 2]
            assert abs(lse[b, h] - (s + math.log(lens[b]))) < 1e-12


def test_one_token_context_returns_v_exactly():
    rng = np.random.default_rng(7)
    B, H_q, H_kv, D, ps = 3, 4, 2, 8, 16
    K = rng.standard_normal((B, 1, H_kv, D))
    V = rng.standard_normal((B, 1, H_kv, D))
    q = rng.standard_normal((B, H_q, D))
    lens = np.ones(B, dtype=np.int64)
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, ps)
    o, lse = oracle.decode_attention(q, kp, vp, bt, lens, 0.25)
    for b in range(B):
        for h in range(H_q):
            assert np.array_equal(o[b, h], V[b, 0, h // 2])
            assert abs(lse[b, h] - 0.25 * float(q[b, h] @ K[b, 0, h // 2])) < 1e-14


def test_two_token_sigmoid_closed_form():
    # q = (1, 0); k1 = (2, 0), k2 = (0, 0): s1 = 2, s2 = 0 at scale 1.
    q = np.array([[[1.0, 0.0]]])
    K = np.array([[[[2.0, 0.0]], [[0.0, 0.0]]]])
    V = np.array([[[[1.0, -3.0]], [[5.0, 7.0]]]])
    kp, vp, bt = _paged_from_contiguous(np.random.default_rng(0), K, V, [2], 1)
    o, lse = oracle.decode_attention(q, kp, vp, bt, np.array([2]), 1.0)
    p1 = 1.0 / (1.0 + math.exp(-2.0))
    np.testing.assert_allclose(o[0, 0], p1 * V[0, 0, 0] + (1 - p1) * V[0, 1, 0], atol=1e-15)
    assert abs(lse[0, 0] - math.log(math.exp(2.0) + 1.0)) < 1e-15


def test_empty_context_gives_zero_and_neg_inf():
    rng, q, K, V, lens = _random_problem(8, B=3)
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, 4)
    lens = lens.copy()
    lens[1] = 0
    o, lse = oracle.decode_attention(q, kp, vp, bt, lens, 0.5)
    assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(o[0])) and np.all(np.isfinite(lse[2]))


def test_cascade_prefix_suffix_merge_equals_flat():
    rng = np.random.default_rng(9)
    B, H_q, H_kv, D, ps = 4, 8, 2, 16, 4
    prefix_pages = 3
    lens = np.array([17, 13, 30, 21])
    Lmax = int(lens.max())
    K = rng.standard_normal((B, Lmax, H_kv, D))
    V = rng.standard_normal((B, Lmax, H_kv, D))
    K[:, :prefix_pages * ps] = K[0, :prefix_pages * ps]   # shared prefix content
    V[:, :prefix_pages * ps] = V[0, :prefix_pages * ps]
    q = rng.standard_normal((B, H_q, D))
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, ps)
    bt[:, :prefix_pages] = bt[0, :prefix_pages]          # share the prefix pages by id
    flat_o, flat_l = oracle.decode_attention(q, kp, vp, bt, lens, 0.4)
    pre_o, pre_l = oracle.decode_attention(q, kp, vp, bt, np.full(B, prefix_pages * ps), 0.4)
    suf_o, suf_l = oracle.decode_attention(q, kp, vp, bt[:, prefix_pages:], lens - prefix_pages * ps, 0.4)
    o, l = oracle.merge_states(pre_o, pre_l, suf_o, suf_l)
    np.testing.assert_allclose(o, flat_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, flat_l, rtol=0, atol=1e-12)


def test_n_way_split_merge_equals_flat():
    rng = np.random.default_rng(10)
    B, H_q, H_kv, D, ps = 3, 4, 1, 8, 2
    lens = np.array([40, 23, 9])
    K = rng.standard_normal((B, 40, H_kv, D))
    V = rng.standard_normal((B, 40, H_kv, D))
    q = rng.standard_normal((B, H_q, D))
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, ps)
    flat_o, flat_l = oracle.decode_attention(q, kp, vp, bt, lens, 0.7)
    for b in range(B):
        n_pages = (lens[b] + ps - 1) // ps
        cuts = np.sort(rng.choice(np.arange(1, n_pages), size=min(3, n_pages - 1), replace=False))
        bounds = [0] + [int(c) for c in cuts] + [int(n_pages)]
        os_, ls_ = [], []
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            seg_len = min(int(lens[b]), hi * ps) - lo * ps
            o, l = oracle.decode_attention(q[b:b + 1], kp, vp, bt[b:b + 1, lo:], [seg_len], 0.7)
            os_.append(o)
            ls_.append(l)
        o, l = oracle.merge_states_many(os_, ls_)
        np.testing.assert_allclose(o[0], flat_o[b], atol=1e-12)
        np.testing.assert_allclose(l[0], flat_l[b], atol=1e-12)


def test_merge_with_empty_state():
    rng = np.random.default_rng(11)
    o = rng.standard_normal((3, 5))
    l = rng.standard_normal(3)
    empty_o = np.full((3, 5), 123.0)   # contents of an empty state must not matter
    empty_l = np.full(3, -np.inf)
    mo, ml = oracle.merge_states(o, l, empty_o, empty_l)
    np.testing.assert_allclose(mo, o, atol=1e-15)
    np.testing.assert_allclose(ml, l, atol=1e-15)
    mo, ml = oracle.merge_states(empty_o, empty_l, empty_o, empty_l)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))


def test_mla_matches_torch_sdpa():
    rng = np.random.default_rng(12)
    B, H, Dqk, Dv, ps, Lmax = 3, 6, 24, 16, 8, 50
    lens = np.array([50, 1, 33])
    C = rng.standard_normal((B, Lmax, 1, Dqk))
    q = rng.standard_normal((B, H, Dqk))
    pool, _, bt = _paged_from_contiguous(rng, C, C, lens, ps)
    o, lse = oracle.mla_decode_attention(q, pool[:, :, 0, :], bt, lens, 0.2, Dv)
    for b in range(B):
        L = int(lens[b])
        k = torch.from_numpy(C[b, :L, 0])[None, None].expand(1, H, L, Dqk)
        v = torch.from_numpy(C[b, :L, 0, :Dv])[None, None].expand(1, H, L, Dv)
        ref = F.scaled_dot_product_attention(torch.from_numpy(q[b])[None, :, None], k, v, scale=0.2)
        np.testing.assert_allclose(o[b], ref[0, :, 0].numpy(), atol=1e-12)
        scores = (torch.from_numpy(q[b]) @ torch.from_numpy(C[b, :L, 0]).T * 0.2).numpy()
        np.testing.assert_allclose(lse[b], logsumexp(scores, axis=-1), atol=1e-12)
    # one-token context: O is the latent row's first Dv columns exactly
    assert np.array_equal(o[1], np.broadcast_to(C[1, 0, 0, :Dv], (H, Dv)))


def _expected_append_loop(kp, vp, kn, vn, bt, pos, ps):
    """Element-by-element expected pools after the append (test-side code)."""
    ek, ev = kp.copy(), vp.copy()
    for b in range(len(pos)):
        page = bt[b][pos[b] // ps]
        row = pos[b] % ps
        for h in range(kn.shape[1]):
            for d in range(kn.shape[2]):
                ek[page, row, h, d] = kn[b, h, d]
                ev[page, row, h, d] = vn[b, h, d]
    return ek, ev


def test_kv_append_exact_and_only_target_rows_change():
    case = workloads.tiny_gqa_append()                    # lens {17, 40, 64, 100}
    kp = case.k_pool.numpy().view(np.uint32)              # exact bit patterns, NaNs included
    vp = case.v_pool.numpy().view(np.uint32)
    kn = case.k_new.numpy().view(np.uint32)
    vn = case.v_new.numpy().view(np.uint32)
    pos = case.positions
    ok, ov = oracle.kv_append(kp, vp, kn, vn, case.block_table, pos, case.page_size)
    ek, ev = _expected_append_loop(kp, vp, kn, vn, case.block_table, pos, case.page_size)
    assert np.array_equal(ok, ek) and np.array_equal(ov, ev)
    changed = np.argwhere(np.any(ok != kp, axis=(2, 3)))
    expect = {(int(case.block_table[b][pos[b] // 16]), int(pos[b] % 16)) for b in range(4)}
    assert {tuple(x) for x in changed} == expect
    # position 64 opens the fifth page (page index 4) of sequence 2
    assert (int(case.block_table[2][4]), 0) in expect
    # inputs untouched
    assert np.array_equal(kp, case.k_pool.numpy().view(np.uint32))


def test_kv_bytes_model_matches_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes_example.json")))
    per_layer = workloads.kv_cache_bytes(g["tokens"], g["kv_heads"], g["head_dim"], g["head_dim"],
                                         g["bytes_per_element"])
    assert per_layer * g["layers"] == g["kv_bytes"]
    assert g["kv_bytes"] == g["per_request_mib"] * 2 ** 20


def test_fold_sq_factor_matches_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "fold_sq_factor_example.json")))
    f = oracle.fold_sq_factor(g["num_heads"], g["q_seqlen"], g["tile_rows"])
    assert f == g["F"]
    assert g["num_heads"] * f == g["H_eff"] and g["q_seqlen"] // f == g["q_seqlen_eff"]


@pytest.mark.parametrize("H,q_len,tile,F_expected", [
    (128, 4, 128, 1),   # the head count alone fills the tile
    (32, 4, 128, 4),    # all four tokens fit
    (64, 3, 128, 1),    # 3 is prime and 64 * 3 > 128
    (16, 6, 128, 6),    # a non-power-of-two factor
    (48, 4, 128, 2),    # 48 * 4 > 128 >= 48 * 2
    (200, 2, 128, 1),   # more heads than tile rows
    (4, 8, 8, 2),       # an 8-row tile
    (1, 7, 8, 7),
])
def test_fold_sq_factor_hand_values(H, q_len, tile, F_expected):
    assert oracle.fold_sq_factor(H, q_len, tile) == F_expected


def _causal_sdpa_reference(q, K, V, lens, scale, g):
    """torch fp64 SDPA with an explicit boolean mask: query j of sequence b
    sees keys 0 .. L_b - q_len + j (test-side code)."""
    B, q_len, H_q, D = q.shape
    out = np.zeros((B, q_len, H_q, V.shape[3]))
    for b in range(B):
        L = int(lens[b])
        k = torch.from_numpy(K[b, :L]).permute(1, 0, 2).repeat_interleave(g, dim=0)  # [H_q, L, D]
        v = torch.from_numpy(V[b, :L]).permute(1, 0, 2).repeat_interleave(g, dim=0)
        qq = torch.from_numpy(q[b]).permute(1, 0, 2)  # [H_q, q_len, D]
        pos = torch.arange(L)[None, :]
        last = (L - q_len + torch.arange(q_len))[:, None]
        mask = pos <= last  # [q_len, L]
        o = F.scaled_dot_product_attention(qq[None], k[None], v[None], attn_mask=mask, scale=scale)
        out[b] = o[0].permute(1, 0, 2).numpy()
    return out


def _multi_query_problem(seed, q_len, B=4, H_q=8, H_kv=2, D=16, page_size=4, Lmax=29):
    rng, q1, K, V, lens = _random_problem(seed, B=B, H_q=H_q, H_kv=H_kv, D=D, page_size=page_size, Lmax=Lmax)
    lens = np.maximum(lens, q_len)
    lens[1] = q_len  # the new tokens are the whole context
    q = rng.standard_normal((B, q_len, H_q, D))
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, page_size)
    return q, K, V, lens, kp, vp, bt


@pytest.mark.parametrize("q_len", [1, 2, 3, 4])
def test_multi_query_matches_causal_torch_sdpa(q_len):
    q, K, V, lens, kp, vp, bt = _multi_query_problem(40 + q_len, q_len)
    o, lse = oracle.multi_query_decode_attention(q, kp, vp, bt, lens, 0.41)
    ref = _causal_sdpa_reference(q, K, V, lens, 0.41, 4)
    np.testing.assert_allclose(o, ref, atol=1e-12, rtol=0)
    # LSE of row j: scipy over the scores of its visible keys
    for b in range(len(lens)):
        for j in range(q_len):
            Lj = int(lens[b]) - q_len + 1 + j
            for h in range(q.shape[2]):
                s = 0.41 * K[b, :Lj, h // 4] @ q[b, j, h]
                assert abs(lse[b, j, h] - logsumexp(s)) < 1e-12


def test_multi_query_rows_are_single_queries_over_shortened_contexts():
    q_len = 3
    q, K, V, lens, kp, vp, bt = _multi_query_problem(47, q_len)
    o, lse = oracle.multi_query_decode_attention(q, kp, vp, bt, lens, 0.29)
    for j in range(q_len):
        o1, l1 = oracle.decode_attention(q[:, j], kp, vp, bt, lens - q_len + 1 + j, 0.29)
        np.testing.assert_array_equal(o[:, j], o1)
        np.testing.assert_array_equal(lse[:, j], l1)


def test_multi_query_rows_ignore_later_keys():
    q_len = 4
    q, K, V, lens, kp, vp, bt = _multi_query_problem(48, q_len)
    o, _ = oracle.multi_query_decode_attention(q, kp, vp, bt, lens, 0.3)
    b, L = 0, int(lens[0])
    last_pos = L - 1
    page, row = bt[b, last_pos // 4], last_pos % 4
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[page, row] += 5.0
    vp2[page, row] -= 3.0
    o2, _ = oracle.multi_query_decode_attention(q, kp2, vp2, bt, lens, 0.3)
    np.testing.assert_array_equal(o2[b, :q_len - 1], o[b, :q_len - 1])  # earlier tokens cannot see it
    assert not np.allclose(o2[b, q_len - 1], o[b, q_len - 1])


# ---------------------------------------------------------------------------
# Mutation checks: a plausible mistake planted in the oracle must fail a pin.
# ---------------------------------------------------------------------------

def _sdpa_pin_holds():
    rng, q, K, V, lens = _random_problem(13, H_q=8, H_kv=2, page_size=4)
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, 4)
    o, _ = oracle.decode_attention(q, kp, vp, bt, lens, 0.37)
    ref = _sdpa_reference(q, K, V, lens, 0.37, 4)
    return bool(np.all(np.isfinite(o)) and np.allclose(o, ref, atol=1e-10))


def test_mutation_wrong_row_index_is_caught(monkeypatch):
    real = oa.gather_sequence

    def off_by_one(pool, row, length, page_size):
        return real(pool, row, length + 1, page_size)[1:]   # shifted by one token
    monkeypatch.setattr(oa, "gather_sequence", off_by_one)
    assert not _sdpa_pin_holds()


def test_mutation_wrong_gqa_mapping_is_caught(monkeypatch):
    real = oa.decode_attention

    def interleaved(q, k_pool, v_pool, block_table, seq_lens, scale):
        # head h reads kv head h % H_kv instead of h // g
        H_q, H_kv = q.shape[1], k_pool.shape[2]
        g = H_q // H_kv
        slot = np.array([(h % H_kv) * g + h // H_kv for h in range(H_q)])
        q_perm = np.empty_like(q)
        q_perm[:, slot] = q
        o, l = real(q_perm, k_pool, v_pool, block_table, seq_lens, scale)
        return o[:, slot], l[:, slot]
    monkeypatch.setattr(oracle, "decode_attention", interleaved)
    assert not _sdpa_pin_holds()


def test_mutation_missing_scale_is_caught(monkeypatch):
    real = oa._softmax_attend
    monkeypatch.setattr(oa, "_softmax_attend", lambda s, v: real(s / 0.37, v))
    assert not _sdpa_pin_holds()


def test_mutation_merge_sign_error_is_caught(monkeypatch):
    real = oa.merge_states

    def wrong(o_a, l_a, o_b, l_b):
        return real(o_a, l_a, o_b, -np.asarray(l_b))
    monkeypatch.setattr(oracle, "merge_states", wrong)
    with pytest.raises(AssertionError):
        test_cascade_prefix_suffix_merge_equals_flat()


def test_mutation_causal_off_by_one_is_caught(monkeypatch):
    real = oa.multi_query_decode_attention

    def shifted(q, k_pool, v_pool, block_table, seq_lens, scale):
        # every query token also sees the next token (limit one too far)
        q_len = q.shape[1]
        o = np.zeros(q.shape[:3] + (v_pool.shape[3],))
        l = np.zeros(q.shape[:3])
        for j in range(q_len):
            lens_j = np.minimum(np.asarray(seq_lens) - q_len + 2 + j, np.asarray(seq_lens))
            oj, lj = oracle.decode_attention(q[:, j], k_pool, v_pool, block_table, lens_j, scale)
            o[:, j], l[:, j] = oj, lj
        return o, l
    monkeypatch.setattr(oracle, "multi_query_decode_attention", shifted)
    with pytest.raises(AssertionError):
        test_multi_query_matches_causal_torch_sdpa(3)


# ---------------------------------------------------------------------------
# Sliding-window KV groups (decode_attention_window)
# ---------------------------------------------------------------------------

def _window_problem(seed, window, page_size=4, Lmax=37):
    rng, q, K, V, lens = _random_problem(seed, page_size=page_size, Lmax=Lmax)
    lens[1] = min(window, Lmax)       # exactly the window
    lens[2] = min(window + 1, Lmax)   # one token past it
    lens[3] = 1
    kp, vp, bt = _paged_from_contiguous(rng, K, V, lens, page_size)
    return rng, q, K, V, lens, kp, vp, bt


@pytest.mark.parametrize("seed,window", [(20, 5), (21, 8), (22, 13), (23, 1)])
def test_window_equals_full_decode_on_a_cache_holding_only_the_window(seed, window):
    """Each sequence's last min(L, W) tokens re-paged from row 0 of fresh pages:
    plain decode over that cache is the windowed decode over the original."""
    rng, q, K, V, lens, kp, vp, bt = _window_problem(seed, window)
    B, Lmax = K.shape[0], K.shape[1]
    Kw, Vw = np.zeros_like(K), np.zeros_like(V)
    wl = np.minimum(lens, window)
    for b in range(B):
        L = int(lens[b])
        Kw[b, :wl[b]] = K[b, L - wl[b]:L]
        Vw[b, :wl[b]] = V[b, L - wl[b]:L]
    kp2, vp2, bt2 = _paged_from_contiguous(rng, Kw, Vw, wl, 4)
    o_ref, l_ref = oracle.decode_attention(q, kp2, vp2, bt2, wl, 0.37)
    o, l = oracle.decode_attention_window(q, kp, vp, bt, lens, 0.37, window)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, rtol=0, atol=1e-12)


def test_window_at_least_the_length_is_full_decode():
    rng, q, K, V, lens, kp, vp, bt = _window_problem(24, 37)
    o_ref, l_ref = oracle.decode_attention(q, kp, vp, bt, lens, 0.25)
    o, l = oracle.decode_attention_window(q, kp, vp, bt, lens, 0.25, 37)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(l, l_ref)
    o2, l2 = oracle.decode_attention_window(q, kp, vp, bt, lens, 0.25, 10 ** 6)
    np.testing.assert_array_equal(o2, o_ref)


def test_one_token_window_returns_the_last_value_exactly():
    rng, q, K, V, lens, kp, vp, bt = _window_problem(25, 1)
    g = q.shape[1] // K.shape[2]
    o, l = oracle.decode_attention_window(q, kp, vp, bt, lens, 0.5, 1)
    for b in range(q.shape[0]):
        L = int(lens[b])
        for h in range(q.shape[1]):
            np.testing.assert_array_equal(o[b, h], V[b, L - 1, h // g])
            assert l[b, h] == pytest.approx(0.5 * float(q[b, h] @ K[b, L - 1, h // g]), abs=1e-12)


def test_placeholders_in_front_of_the_window_are_never_read():
    """Slots wholly before the window point at a NaN placeholder page and the
    window's first page holds NaN before the window: the result stays finite
    and equal to the windowed decode over the intact cache."""
    window, ps = 6, 4
    rng, q, K, V, lens, kp, vp, bt = _window_problem(26, window, page_size=ps)
    o_ref, l_ref = oracle.decode_attention_window(q, kp, vp, bt, lens, 0.3, window)
    P = kp.shape[0]
    kp2 = np.concatenate([kp, np.full((1,) + kp.shape[1:], np.nan)])
    vp2 = np.concatenate([vp, np.full((1,) + vp.shape[1:], np.nan)])
    bt2 = bt.copy()
    for b in range(q.shape[0]):
        start = max(0, int(lens[b]) - window)
        bt2[b, :start // ps] = P  # the placeholder
        first = bt2[b, start // ps]
        kp2[first, :start % ps] = np.nan
        vp2[first, :start % ps] = np.nan
    o, l = oracle.decode_attention_window(q, kp2, vp2, bt2, lens, 0.3, window)
    assert np.all(np.isfinite(o))
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(l, l_ref)


def test_mutation_window_off_by_one_is_caught(monkeypatch):
    real = oracle.decode_attention_window

    def wider(q, k_pool, v_pool, block_table, seq_lens, scale, window):
        return real(q, k_pool, v_pool, block_table, seq_lens, scale, window + 1)
    monkeypatch.setattr(oracle, "decode_attention_window", wider)
    with pytest.raises(AssertionError):
        test_window_equals_full_decode_on_a_cache_holding_only_the_window(21, 8)
