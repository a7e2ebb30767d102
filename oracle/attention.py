"""fp64 oracle: paged gather, decode attention (GQA and absorbed MLA), LSE merge,
and the KV append. TEST INFRASTRUCTURE ONLY (see the package docstring).

Conventions (readings of points the pages leave open; each is also listed in
the design notes):

* Pool layout is ``[num_pages, page_size, H_kv, D]`` ("NHD"): row ``r`` of
  physical page ``p`` holds token ``page_slot * page_size + r`` of whatever
  sequence owns the page. The MLA latent pool is ``[num_pages, page_size, 576]``.
* Query head ``h`` reads kv head ``h // g`` with ``g = H_q // H_kv``.
* ``LSE`` is the natural-log log-sum-exp of the scaled scores.
* An empty context (length 0) gives ``O = 0`` and ``LSE = -inf``.

No blocking, fusion or reordering beyond the definition: gather the rows,
score them, softmax, weight the values.
"""

from __future__ import annotations

import numpy as np


def gather_sequence(pool: np.ndarray, block_table_row: np.ndarray, length: int,
                    page_size: int) -> np.ndarray:
    """Rows ``0 .. length-1`` of one sequence, gathered through its block table.

    SwiftLLM page, section 3.1: a request's cache is a list of non-contiguous
    fixed-size blocks found through its block table; token ``t`` lives in block
    ``block_table[t // page_size]`` at row ``t % page_size``.

    Pinned by: brute-force unpaged attention (the test scatters contiguous K/V
    into shuffled pages itself) and page-permutation invariance.
    """
    length = int(length)
    if length == 0:
        return np.zeros((0,) + pool.shape[2:], dtype=pool.dtype)
    n_pages = (length + page_size - 1) // page_size
    pages = np.asarray(block_table_row[:n_pages], dtype=np.int64)
    rows = pool[pages]  # [n_pages, page_size, ...]
    rows = rows.reshape((n_pages * page_size,) + pool.shape[2:])
    return rows[:length]


def _softmax_attend(scores: np.ndarray, values: np.ndarray):
    """softmax over the last axis of ``scores`` [n, L], then weight ``values`` [L, Dv].

    Returns (O [n, Dv], LSE [n]) in float64.
    """
    m = scores.max(axis=-1, keepdims=True)
    e = np.exp(scores - m)
    s = e.sum(axis=-1, keepdims=True)
    out = (e @ values) / s
    lse = (m + np.log(s))[:, 0]
    return out, lse


def decode_attention(q, k_pool, v_pool, block_table, seq_lens, scale):
    """One decode step of GQA attention over a paged KV cache, in float64.

    For every sequence ``b`` and query head ``h`` (kv head ``kh = h // g``):
    ``s_t = scale * <q[b,h], K_b[t,kh]>`` for ``t < L_b``, ``p = softmax(s)``,
    ``O[b,h] = sum_t p_t V_b[t,kh]`` and ``LSE[b,h] = log sum_t exp(s_t)``.

    SwiftLLM page, sections 3.1 and 5.1 (query, block tables and context
    lengths are the attention inputs); the GQA sharing of one kv head by
    ``g`` consecutive query heads is the reading stated in the module docstring.

    Args:
        q: [B, H_q, D] float array.
        k_pool, v_pool: [P, page_size, H_kv, D] float arrays.
        block_table: [B, >= max pages] integer array of physical page ids.
        seq_lens: [B] context lengths (tokens attended).
        scale: softmax scale.

    Returns:
        (O [B, H_q, D] float64, LSE [B, H_q] float64).

    Pinned by: torch's fp64 scaled_dot_product_attention on the unpaged K/V,
    scipy's logsumexp, page-permutation invariance, identical keys (O = mean V),
    one-token context (O = V exactly) and the two-token sigmoid closed form.
    """
    q = np.asarray(q, dtype=np.float64)
    B, H_q, D = q.shape
    page_size, H_kv = k_pool.shape[1], k_pool.shape[2]
    if H_q % H_kv != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    g = H_q // H_kv
    Dv = v_pool.shape[3]
    out = np.zeros((B, H_q, Dv), dtype=np.float64)
    lse = np.full((B, H_q), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        K = gather_sequence(k_pool, block_table[b], L, page_size).astype(np.float64)
        V = gather_sequence(v_pool, block_table[b], L, page_size).astype(np.float64)
        for kh in range(H_kv):
            heads = slice(kh * g, (kh + 1) * g)
            scores = scale * (q[b, heads] @ K[:, kh, :].T)  # [g, L]
            o, l = _softmax_attend(scores, V[:, kh, :])
            out[b, heads] = o
            lse[b, heads] = l
    return out, lse


def decode_attention_window(q, k_pool, v_pool, block_table, seq_lens, scale, window):
    """Decode attention over a sliding-window KV group, in float64.

    TokenSpeed deep dive (wth2jhl.online), section 4.1: a ``sliding_window``
    KV group declares ``sliding_window_tokens``; tokenspeed 딥다이브
    (fiv.co.kr), section 6-3: such a group's block table keeps the real
    blocks at the back of the window and a placeholder (block 0) in the
    slots in front of it. Reading (listed in the design notes): the query of
    a sequence with ``L`` tokens attends its last ``min(L, window)`` tokens,
    positions ``L - window .. L - 1``; token ``t`` still lives in slot
    ``t // page_size`` at row ``t % page_size``, so slots wholly before the
    window (placeholders) and rows of the window's first page before it are
    never read. Otherwise as :func:`decode_attention`.

    Args: as :func:`decode_attention`, plus ``window`` >= 1 (tokens).

    Pinned by: window >= L equal to :func:`decode_attention`, a one-token
    window giving O = V[L-1] exactly, equality with :func:`decode_attention`
    on a cache re-paged to hold only each window (from row 0 of fresh pages),
    NaN placeholder pages that leave the result finite, and a planted
    off-by-one window caught.
    """
    if int(window) < 1:
        raise ValueError("window must be >= 1 token")
    q = np.asarray(q, dtype=np.float64)
    B, H_q, D = q.shape
    page_size, H_kv = k_pool.shape[1], k_pool.shape[2]
    if H_q % H_kv != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    g = H_q // H_kv
    Dv = v_pool.shape[3]
    out = np.zeros((B, H_q, Dv), dtype=np.float64)
    lse = np.full((B, H_q), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        pos = np.arange(max(0, L - int(window)), L)
        pages = np.asarray(block_table[b])[pos // page_size]
        K = k_pool[pages, pos % page_size].astype(np.float64)  # [n, H_kv, D]
        V = v_pool[pages, pos % page_size].astype(np.float64)
        for kh in range(H_kv):
            heads = slice(kh * g, (kh + 1) * g)
            scores = scale * (q[b, heads] @ K[:, kh, :].T)
            o, l = _softmax_attend(scores, V[:, kh, :])
            out[b, heads] = o
            lse[b, heads] = l
    return out, lse


def fold_sq_factor(num_heads: int, q_len: int, tile_rows: int = 128) -> int:
    """Number of query tokens folded into the head (row) dimension of a tile.

    TokenSpeed deep dive, section 7.2: ``F`` is the largest factor with
    ``q_len % F == 0`` and ``num_heads * F <= tile_rows``; the kernel then sees
    ``H_eff = num_heads * F`` rows per query step and ``q_len / F`` steps. A
    head count that alone exceeds the tile folds nothing (``F = 1``).

    Pinned by: the page's worked example (64 heads, 4 query tokens, 128-row
    tile: F = 2, H_eff = 128, 2 steps; ``tests/golden/fold_sq_factor_example.json``)
    and hand-checked values for prime, non-power-of-two and oversized cases.
    """
    if num_heads <= 0 or q_len <= 0 or tile_rows <= 0:
        raise ValueError("num_heads, q_len and tile_rows must be positive")
    best = 1
    for f in range(1, q_len + 1):
        if q_len % f == 0 and num_heads * f <= tile_rows:
            best = f
    return best


def multi_query_decode_attention(q, k_pool, v_pool, block_table, seq_lens, scale):
    """Decode with several new query tokens per sequence (speculative verify).

    ``q`` holds ``q_len`` consecutive query tokens per sequence whose K/V rows
    are already in the cache: ``seq_lens[b]`` counts them. Query token ``j``
    sits at position ``L_b - q_len + j`` and attends tokens ``0 .. L_b - q_len + j``
    (causal among the new tokens); each (token, head) row is otherwise the
    single-query GQA decode of :func:`decode_attention`.

    TokenSpeed deep dive, section 7 fig. 3 and 7.2 (decode over ``q_seqlen``
    query tokens per sequence, the workspace sized by ``H * q_len`` rows);
    the causal placement of the new tokens at the end of the context is the
    reading listed in the design notes.

    Args:
        q: [B, q_len, H_q, D]; pools and block table as :func:`decode_attention`;
        seq_lens: [B] context lengths including the q_len new tokens (>= q_len).

    Returns:
        (O [B, q_len, H_q, D] float64, LSE [B, q_len, H_q] float64).

    Pinned by: q_len = 1 equals :func:`decode_attention`; every row equals
    :func:`decode_attention` of that one query over the shortened context;
    torch's fp64 scaled_dot_product_attention with an explicit causal mask on
    the unpaged K/V; rows unaffected by K/V rows after their position.
    """
    q = np.asarray(q, dtype=np.float64)
    B, q_len, H_q, D = q.shape
    page_size, H_kv = k_pool.shape[1], k_pool.shape[2]
    if H_q % H_kv != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    g = H_q // H_kv
    Dv = v_pool.shape[3]
    out = np.zeros((B, q_len, H_q, Dv), dtype=np.float64)
    lse = np.full((B, q_len, H_q), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L < q_len:
            raise ValueError("seq_lens must count the q_len new tokens")
        K = gather_sequence(k_pool, block_table[b], L, page_size).astype(np.float64)
        V = gather_sequence(v_pool, block_table[b], L, page_size).astype(np.float64)
        for j in range(q_len):
            Lj = L - q_len + 1 + j
            for kh in range(H_kv):
                heads = slice(kh * g, (kh + 1) * g)
                scores = scale * (q[b, j, heads] @ K[:Lj, kh, :].T)  # [g, Lj]
                o, l = _softmax_attend(scores, V[:Lj, kh, :])
                out[b, j, heads] = o
                lse[b, j, heads] = l
    return out, lse


def tree_ancestors(parents) -> list:
    """Ancestor-or-self sets of the nodes of a draft tree.

    ``parents[j]`` is node ``j``'s parent among the draft tokens (``< j``), or
    -1 for a node that hangs directly off the committed context. Returns, per
    node, the sorted list of node indices on its path from the context down to
    itself.
    """
    out = []
    for j, par in enumerate(int(x) for x in parents):
        if par >= j or par < -1:
            raise ValueError(f"parents[{j}] = {par}: must be -1 or an earlier node")
        out.append((out[par] if par >= 0 else []) + [j])
    return out


def tree_verify_decode_attention(q, k_pool, v_pool, block_table, seq_lens, parents, scale):
    """Verify a tree of draft tokens in one decode step (tree speculation).

    Each sequence carries ``n`` draft tokens that form a tree: node ``j`` has
    parent ``parents[b, j]`` (an earlier node, or -1 for a child of the last
    committed token). Their K/V rows are already in the cache at positions
    ``L_b - n + j`` (``seq_lens[b]`` counts them), in node order. Node ``j``'s
    query attends the committed context, positions ``0 .. L_b - n - 1``, and
    the rows of the nodes on its own path (its ancestors and itself), and no
    other draft token: a sibling branch is another candidate continuation.

    TokenSpeed deep dive (wth2jhl.online), section 0 (the tree-speculation
    design document) and the closing section (tree speculation as a serving
    workload). The pages fix no mask; the ancestor mask above is the reading
    listed in the design notes. A chain (``parents[j] = j - 1``) is causal
    multi-token verification.

    Args:
        q: [B, n, H_q, D]; pools, block table as :func:`decode_attention`;
        seq_lens: [B] context lengths including the n draft tokens (>= n);
        parents: [B, n] integer array.

    Returns:
        (O [B, n, H_q, D] float64, LSE [B, n, H_q] float64).

    Pinned by: the chain tree equal to :func:`multi_query_decode_attention`;
    every node's row equal to :func:`decode_attention` over the context
    followed by its path's rows, re-paged into fresh pages; torch's fp64
    scaled_dot_product_attention with the explicit ancestor mask; rows
    unchanged when rows off their path are overwritten; a planted causal
    (sibling-visible) mask caught on a branching tree.
    """
    q = np.asarray(q, dtype=np.float64)
    B, n, H_q, D = q.shape
    page_size, H_kv = k_pool.shape[1], k_pool.shape[2]
    if H_q % H_kv != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    g = H_q // H_kv
    Dv = v_pool.shape[3]
    out = np.zeros((B, n, H_q, Dv), dtype=np.float64)
    lse = np.full((B, n, H_q), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L < n:
            raise ValueError("seq_lens must count the n draft tokens")
        K = gather_sequence(k_pool, block_table[b], L, page_size).astype(np.float64)
        V = gather_sequence(v_pool, block_table[b], L, page_size).astype(np.float64)
        ctx = L - n
        for j, path in enumerate(tree_ancestors(parents[b])):
            keys = np.concatenate([np.arange(ctx), ctx + np.asarray(path, dtype=np.int64)])
            for kh in range(H_kv):
                heads = slice(kh * g, (kh + 1) * g)
                scores = scale * (q[b, j, heads] @ K[keys, kh, :].T)
                o, l = _softmax_attend(scores, V[keys, kh, :])
                out[b, j, heads] = o
                lse[b, j, heads] = l
    return out, lse


def mla_decode_attention(q, kv_pool, block_table, seq_lens, scale, d_v):
    """Absorbed-MLA decode: every query head attends one shared latent head.

    ``s[h,t] = scale * <q[b,h,0:Dqk], C_b[t,0:Dqk]>``, softmax over ``t``,
    ``O[b,h] = sum_t p[h,t] C_b[t,0:d_v]`` (the values are the first ``d_v``
    columns of the same latent rows).

    TokenSpeed deep dive (wth2jhl.online), section 7, fig. 3: MLA decode with a
    512-wide output per head row; the 576 = 512 latent + 64 rope row width and
    ``V = C[:, :512]`` are the workload's statement of the absorbed form.

    Args:
        q: [B, H, Dqk]; kv_pool: [P, page_size, Dqk]; d_v <= Dqk.

    Returns:
        (O [B, H, d_v] float64, LSE [B, H] float64).

    Pinned by: torch's fp64 scaled_dot_product_attention with one kv head and a
    value width different from the key width, and the one-token closed form.
    """
    q = np.asarray(q, dtype=np.float64)
    B, H, Dqk = q.shape
    page_size = kv_pool.shape[1]
    out = np.zeros((B, H, d_v), dtype=np.float64)
    lse = np.full((B, H), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        C = gather_sequence(kv_pool, block_table[b], L, page_size).astype(np.float64)
        scores = scale * (q[b] @ C.T)  # [H, L]
        o, l = _softmax_attend(scores, C[:, :d_v])
        out[b] = o
        lse[b] = l
    return out, lse


def mla_multi_query_decode_attention(q, kv_pool, block_table, seq_lens, scale, d_v):
    """Absorbed-MLA decode with ``q_len`` new query tokens per sequence.

    Query token ``j`` of sequence ``b`` sits at position ``L_b - q_len + j``
    (its latent row is already cached: ``seq_lens[b]`` counts the new tokens)
    and, for every head, attends latent rows ``0 .. L_b - q_len + j``; each
    (token, head) row is otherwise :func:`mla_decode_attention`.

    TokenSpeed deep dive (wth2jhl.online), section 7, fig. 3 and 7.2: MLA
    decode over ``q_seqlen`` query tokens, whose tokens are folded into the
    head rows of a tile (``fold_sq_factor``); causal placement at the end of
    the context is the same reading as :func:`multi_query_decode_attention`.

    Args:
        q: [B, q_len, H, Dqk]; kv_pool: [P, page_size, Dqk]; seq_lens >= q_len.

    Returns:
        (O [B, q_len, H, d_v] float64, LSE [B, q_len, H] float64).

    Pinned by: q_len = 1 equal to :func:`mla_decode_attention`; every row
    equal to :func:`mla_decode_attention` of that query over the shortened
    context; torch's fp64 scaled_dot_product_attention with one kv head, a
    value width of d_v and an explicit causal mask.
    """
    q = np.asarray(q, dtype=np.float64)
    B, q_len, H, Dqk = q.shape
    page_size = kv_pool.shape[1]
    out = np.zeros((B, q_len, H, d_v), dtype=np.float64)
    lse = np.full((B, q_len, H), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L < q_len:
            raise ValueError("seq_lens must count the q_len new tokens")
        C = gather_sequence(kv_pool, block_table[b], L, page_size).astype(np.float64)
        for j in range(q_len):
            Lj = L - q_len + 1 + j
            scores = scale * (q[b, j] @ C[:Lj].T)  # [H, Lj]
            o, l = _softmax_attend(scores, C[:Lj, :d_v])
            out[b, j] = o
            lse[b, j] = l
    return out, lse


def merge_states(o_a, lse_a, o_b, lse_b):
    """Merge two attention states over disjoint key sets by their log-sum-exp.

    With ``m = max(lse_a, lse_b)``, ``w_a = exp(lse_a - m)``, ``w_b = exp(lse_b - m)``:
    ``O = (w_a O_a + w_b O_b) / (w_a + w_b)`` and ``LSE = m + log(w_a + w_b)``.
    A state with ``LSE = -inf`` (no keys) has weight 0; two empty states merge
    to ``O = 0``, ``LSE = -inf``.

    TokenSpeed deep dive, section 7 fig. 3 (stage 3 reduces the split partials
    by their LSE) and section 7.1; Tokasaurus blog, "Dynamic prefix
    identification and exploration" (shared-prefix attention is combined with
    the per-sequence part).

    Args: o_* [..., D]; lse_* [...] (natural log).
    Returns: (O [..., D] float64, LSE [...] float64).

    Pinned by: prefix-state merged with suffix-state equals flat attention over
    prefix ++ suffix (an independent oracle call), and N-way associativity.
    """
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    m = np.maximum(lse_a, lse_b)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    w_a = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - m_safe))
    w_b = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - m_safe))
    w = w_a + w_b
    w_div = np.where(empty, 1.0, w)
    o = (w_a[..., None] * o_a + w_b[..., None] * o_b) / w_div[..., None]
    o = np.where(empty[..., None], 0.0, o)
    lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, w)))
    return o, lse


def merge_states_many(os, lses):
    """Left fold of :func:`merge_states` over a list of states (split-KV reduce)."""
    o, lse = os[0], lses[0]
    for o_n, lse_n in zip(os[1:], lses[1:]):
        o, lse = merge_states(o, lse, o_n, lse_n)
    return np.asarray(o, dtype=np.float64), np.asarray(lse, dtype=np.float64)


def kv_append(k_pool, v_pool, k_new, v_new, block_table, positions, page_size):
    """Write one new token's K/V per sequence into its page; return new pools.

    SwiftLLM page, section 3.1: blocks are handed to a request on demand, so the
    token at position ``pos`` goes to page ``block_table[b][pos // page_size]``,
    row ``pos % page_size``. Works on raw element arrays of any dtype (bf16 is
    carried as uint16 bit patterns), so the copy is exact; the inputs are not
    modified.

    Args:
        k_pool, v_pool: [P, page_size, H_kv, D]; k_new, v_new: [B, H_kv, D];
        positions: [B] token index to write (= context length before append).

    Pinned by: an element-wise loop in the tests that writes the expected pool
    cell by cell, and the check that every other byte is unchanged.
    """
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    for b in range(len(positions)):
        pos = int(positions[b])
        page = int(block_table[b][pos // page_size])
        row = pos % page_size
        k_out[page, row] = k_new[b]
        v_out[page, row] = v_new[b]
    return k_out, v_out
