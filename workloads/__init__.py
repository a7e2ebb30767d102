"""Seeded synthetic inputs for decode attention over a paged KV cache.

This module is shared by the tests, the benchmark and the smoke check. It holds
none of the attention arithmetic: only shapes, lengths, page placement and
random values. Both the CUDA library and the CPU oracle read the inputs it
builds; neither reads the other's outputs.

Recipe (all seeded):
* structure (lengths, page permutation, block tables) comes from
  ``numpy.random.default_rng(seed)`` on the host;
* values (q, K, V, new-token K/V) are N(0, 1) drawn by a ``torch.Generator``
  seeded with ``seed`` on the device the case lives on; bf16 values are the
  float32 draws rounded to nearest-even by torch;
* every pool row no sequence owns is a NaN sentinel: unused pages, the rows
  past each sequence's length in its last page, and the row a pending append
  will fill. Block-table entries past a sequence's pages point at an unused
  (all-NaN) page, so a masked-read bug shows as NaN instead of a stray access.

Layouts: pools are ``[P, page_size, H_kv, D]`` (MLA: ``[P, page_size, Dqk]``),
block tables ``int32 [B, bt_stride]`` row-major, lengths ``int32 [B]``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class PagedCase:
    """One decode-step workload over a paged cache (GQA or MLA)."""

    name: str
    seed: int
    B: int
    H_q: int
    H_kv: int           # 1 for MLA
    D: int              # key width (Dqk for MLA)
    Dv: int             # value width (= D for GQA, 512 for MLA)
    page_size: int
    num_pages: int
    dtype: str          # "f32" | "bf16"
    scale: float
    mla: bool
    append: bool
    seq_lens: np.ndarray        # int32 [B]: cached tokens before this step's append
    block_table: np.ndarray     # int32 [B, bt_stride]
    sentinel_page: int          # an all-NaN page (or 0 if the pool has none spare)
    q: torch.Tensor = None
    k_pool: torch.Tensor = None  # MLA: the latent pool
    v_pool: Optional[torch.Tensor] = None
    k_new: Optional[torch.Tensor] = None
    v_new: Optional[torch.Tensor] = None
    groups_truth: Optional[List[np.ndarray]] = None  # cascade: members per constructed group
    q_len: int = 1              # query tokens per sequence (q [B, q_len, H_q, D] when > 1)
    # fp8 (e4m3fn) cache: k_pool / v_pool hold uint8 codes, with float32
    # scales [num_pages, page_size, H_kv] per (page, row, kv head)
    kv_fp8: bool = False
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    prefix_pages_truth: int = 0
    window: int = 0             # sliding-window KV group: tokens a query attends (0: all of them)
    meta: Dict = field(default_factory=dict)

    @property
    def attn_lens(self) -> np.ndarray:
        """Tokens attended by the step (one more than cached when appending)."""
        return (self.seq_lens + (1 if self.append else 0)).astype(np.int32)

    @property
    def attended_lens(self) -> np.ndarray:
        """Tokens each query reads: the attended length, capped by the window."""
        L = self.attn_lens
        return np.minimum(L, self.window).astype(np.int32) if self.window > 0 else L

    @property
    def bt_stride(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def positions(self) -> np.ndarray:
        """Append positions (= cached length before the append)."""
        return self.seq_lens.astype(np.int32)

    def kv_bytes_read(self) -> int:
        """Algorithmic K/V (or latent) bytes one attention pass must read."""
        esize = 4 if self.dtype == "f32" else 2
        tokens = int(self.attended_lens.astype(np.int64).sum())
        if self.mla:  # fp8: one-byte codes plus a float32 scale per latent row
            return tokens * (self.D + 4) if self.kv_fp8 else tokens * self.D * esize
        if self.kv_fp8:  # one-byte codes plus a float32 scale per row and kv head, K and V
            return kv_cache_bytes(tokens, self.H_kv, self.D, self.Dv, 1) + tokens * self.H_kv * 2 * 4
        return kv_cache_bytes(tokens, self.H_kv, self.D, self.Dv, esize)


def kv_cache_bytes(tokens: int, H_kv: int, D: int, Dv: int, elem_bytes: int) -> int:
    """Bytes of uncompressed K plus V rows for ``tokens`` tokens of one layer.

    Same count as the approximate KV-size formula of the tokenspeed deep dive
    (fiv.co.kr), section 7-2 (there multiplied by the layer count).
    """
    return int(tokens) * int(H_kv) * (int(D) + int(Dv)) * int(elem_bytes)


def _pages_for(n_tokens: np.ndarray, page_size: int) -> np.ndarray:
    return (n_tokens.astype(np.int64) + page_size - 1) // page_size


def _randn(shape, generator, device, dtype: str, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """N(0,1) draws in float32 rounded to ``dtype``, generated in chunks."""
    numel = int(np.prod(shape))
    out = torch.empty(numel, dtype=_TORCH_DTYPE[dtype], device=device)
    for start in range(0, numel, chunk_elems):
        n = min(chunk_elems, numel - start)
        out[start:start + n] = torch.randn(n, generator=generator, device=device,
                                           dtype=torch.float32).to(out.dtype)
    return out.view(*shape)


def build_case(name: str, seed: int, *, B: int, H_q: int, H_kv: int, D: int,
               page_size: int, seq_lens: Sequence[int], dtype: str, scale: float,
               append: bool = False, mla: bool = False, Dv: Optional[int] = None,
               pool_factor: float = 1.25, shared_groups: Optional[List[np.ndarray]] = None,
               shared_pages: int = 0, device="cpu", rng: Optional[np.random.Generator] = None,
               extra_pages: int = 1, num_pages: Optional[int] = None, values: bool = True,
               q_len: int = 1, layout: Optional[tuple] = None) -> PagedCase:
    """Build a case: lengths -> page need -> shuffled pool -> block tables -> values.

    ``q_len`` > 1 draws ``q_len`` query tokens per sequence (q [B, q_len, H_q, D]);
    ``seq_lens`` then already count them. ``layout`` = (block_table, num_pages)
    replaces the page assignment (a caller-built sharing structure).

    ``shared_groups``: lists of sequence ids; each list shares its first
    ``shared_pages`` pages by physical id (the cascade workload).
    """
    rng = rng if rng is not None else np.random.default_rng(seed)
    lens = np.asarray(seq_lens, dtype=np.int32)
    assert len(lens) == B
    attn = lens + (1 if append else 0)
    if layout is not None:
        bt, num_pages = np.asarray(layout[0], dtype=np.int32), int(layout[1])
        return _finish_case(name, seed, B, H_q, H_kv, D, page_size, lens, dtype, scale, append, mla, Dv,
                            num_pages, bt, 0, None, 0, values, device, q_len)
    n_alloc = _pages_for(attn, page_size)                  # pages each sequence needs
    own = n_alloc.copy()
    if shared_groups:
        for members in shared_groups:
            own[members] -= shared_pages
    need = int(own.sum()) + (len(shared_groups) * shared_pages if shared_groups else 0)
    if num_pages is None:
        num_pages = max(int(math.ceil(pool_factor * need)), need + extra_pages)
    assert num_pages >= need
    perm = rng.permutation(num_pages).astype(np.int32)
    sentinel = int(perm[need]) if num_pages > need else 0
    bt_stride = max(1, int(n_alloc.max()) if B else 1)
    bt = np.full((B, bt_stride), sentinel, dtype=np.int32)
    cursor = 0
    grouped = np.zeros(B, dtype=bool)
    if shared_groups:
        for members in shared_groups:
            pages = perm[cursor:cursor + shared_pages]
            cursor += shared_pages
            bt[np.asarray(members), :shared_pages] = pages
            grouped[np.asarray(members)] = True
    for b in range(B):
        start = shared_pages if grouped[b] else 0
        n_own = int(n_alloc[b]) - start
        bt[b, start:start + n_own] = perm[cursor:cursor + n_own]
        cursor += n_own
    assert cursor == need

    return _finish_case(name, seed, B, H_q, H_kv, D, page_size, lens, dtype, scale, append, mla, Dv, num_pages,
                        bt, sentinel, shared_groups, shared_pages, values, device, q_len)


def _finish_case(name, seed, B, H_q, H_kv, D, page_size, lens, dtype, scale, append, mla, Dv, num_pages, bt,
                 sentinel, shared_groups, shared_pages, values, device, q_len) -> PagedCase:
    """Values of a case whose page layout is fixed: NaN sentinels on rows holding
    no cached token, seeded N(0,1) pools, queries and appended rows."""
    # NaN sentinel mask over [num_pages, page_size]: everything not holding a
    # cached token of some sequence (the pending append row included).
    sentinel_rows = np.ones((num_pages, page_size), dtype=bool)
    for b in range(B):
        L = int(lens[b])
        full, rem = divmod(L, page_size)
        if full:
            sentinel_rows[bt[b, :full]] = False
        if rem:
            sentinel_rows[bt[b, full], :rem] = False

    Dv = Dv if Dv is not None else D
    if not values:  # structure only (block tables and lengths), no tensors
        return PagedCase(name=name, seed=seed, B=B, H_q=H_q, H_kv=H_kv, D=D, Dv=Dv, page_size=page_size,
                         num_pages=num_pages, dtype=dtype, scale=scale, mla=mla, append=append,
                         seq_lens=lens, block_table=bt, sentinel_page=sentinel,
                         groups_truth=[np.asarray(m) for m in shared_groups] if shared_groups else None,
                         prefix_pages_truth=shared_pages if shared_groups else 0)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if mla:
        k_pool = _randn((num_pages, page_size, D), g, device, dtype)
        v_pool = None
    else:
        k_pool = _randn((num_pages, page_size, H_kv, D), g, device, dtype)
        v_pool = _randn((num_pages, page_size, H_kv, Dv), g, device, dtype)
    q = _randn((B, H_q, D) if q_len == 1 else (B, q_len, H_q, D), g, device, dtype)
    k_new = v_new = None
    if append:
        k_new = _randn((B, H_kv, D), g, device, dtype)
        v_new = _randn((B, H_kv, Dv), g, device, dtype)
    mask = torch.from_numpy(sentinel_rows).to(device)
    nan = float("nan")
    k_pool.view(num_pages, page_size, -1).masked_fill_(mask[:, :, None], nan)
    if v_pool is not None:
        v_pool.view(num_pages, page_size, -1).masked_fill_(mask[:, :, None], nan)
    return PagedCase(name=name, seed=seed, B=B, H_q=H_q, H_kv=H_kv, D=D, Dv=Dv,
                     page_size=page_size, num_pages=num_pages, dtype=dtype, scale=scale,
                     mla=mla, append=append, seq_lens=lens, block_table=bt,
                     sentinel_page=sentinel, q=q, k_pool=k_pool, v_pool=v_pool,
                     k_new=k_new, v_new=v_new, q_len=q_len,
                     groups_truth=[np.asarray(m) for m in shared_groups] if shared_groups else None,
                     prefix_pages_truth=shared_pages if shared_groups else 0)


# --------------------------------------------------------------------------
# The five workloads (sizes as stated by the workload list) and small variants
# --------------------------------------------------------------------------

def build_fp8_case(name: str, seed: int, *, B: int, H_q: int, H_kv: int, D: int, page_size: int,
                   seq_lens: Sequence[int], scale: float, append: bool = False, device="cpu",
                   rng: Optional[np.random.Generator] = None) -> PagedCase:
    """A case over an fp8 (e4m3fn) cache: the same page placement as
    :func:`build_case`, with uniformly drawn non-NaN e4m3 codes and per-row
    scales U[2.5, 3.5] / 448 (a row of N(0,1) values has its maximum there).
    Rows holding no cached token carry the NaN code 0x7F and NaN scales.
    Queries (and appended rows) are bf16 N(0,1)."""
    base = build_case(name, seed, B=B, H_q=H_q, H_kv=H_kv, D=D, page_size=page_size, seq_lens=seq_lens,
                      dtype="bf16", scale=scale, append=append, device=device, rng=rng, values=False)
    P = base.num_pages
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    def codes():
        c = torch.randint(0, 256, (P, page_size, H_kv, D), generator=g, device=device, dtype=torch.int32)
        c = torch.where((c & 0x7F) == 0x7F, c - 1, c)  # no NaN codes among cached rows
        return c.to(torch.uint8)
    def scales():
        return (torch.rand((P, page_size, H_kv), generator=g, device=device) + 2.5) / 448.0
    k_pool, v_pool = codes(), codes()
    k_scale, v_scale = scales(), scales()
    q = _randn((B, H_q, D), g, device, "bf16")
    k_new = v_new = None
    if append:
        k_new = _randn((B, H_kv, D), g, device, "bf16")
        v_new = _randn((B, H_kv, D), g, device, "bf16")
    lens = base.seq_lens
    sentinel_rows = np.ones((P, page_size), dtype=bool)
    for b in range(B):
        full, rem = divmod(int(lens[b]), page_size)
        if full:
            sentinel_rows[base.block_table[b, :full]] = False
        if rem:
            sentinel_rows[base.block_table[b, full], :rem] = False
    mask = torch.from_numpy(sentinel_rows).to(device)
    for pool in (k_pool, v_pool):
        pool.view(P, page_size, -1).masked_fill_(mask[:, :, None], 0x7F)
    for sc in (k_scale, v_scale):
        sc.masked_fill_(mask[:, :, None], float("nan"))
    base.q, base.k_pool, base.v_pool, base.k_new, base.v_new = q, k_pool, v_pool, k_new, v_new
    base.kv_fp8, base.k_scale, base.v_scale = True, k_scale, v_scale
    return base


def build_mla_fp8_case(name: str, seed: int, *, B: int, H: int, seq_lens: Sequence[int], scale: float,
                       q_len: int = 1, page_size: int = 64, device="cpu",
                       rng: Optional[np.random.Generator] = None) -> PagedCase:
    """An absorbed-MLA case on the fp8 input path: the page placement of
    :func:`build_case`; uniformly drawn non-NaN e4m3 codes for the latent rows
    [P, ps, 576] and the query rows [B, (q_len,) H, 576], with one scale per
    row drawn U[2.5, 3.5] / 448 (``k_scale`` [P, ps]; the query scales in
    ``meta["q_scale"]``). Rows holding no cached token carry the NaN code 0x7F
    and NaN scales."""
    base = build_case(name, seed, B=B, H_q=H, H_kv=1, D=576, Dv=512, page_size=page_size, seq_lens=seq_lens,
                      dtype="bf16", scale=scale, mla=True, device=device, rng=rng, values=False, q_len=q_len)
    P = base.num_pages
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    def codes(shape):
        c = torch.randint(0, 256, shape, generator=g, device=device, dtype=torch.int32)
        return torch.where((c & 0x7F) == 0x7F, c - 1, c).to(torch.uint8)  # no NaN codes
    def scales(shape):
        return (torch.rand(shape, generator=g, device=device) + 2.5) / 448.0
    kv = codes((P, page_size, 576))
    kv_scale = scales((P, page_size))
    qshape = (B, H) if q_len == 1 else (B, q_len, H)
    q = codes(qshape + (576,))
    q_scale = scales(qshape)
    lens = base.seq_lens
    sentinel_rows = np.ones((P, page_size), dtype=bool)
    for b in range(B):
        full, rem = divmod(int(lens[b]), page_size)
        if full:
            sentinel_rows[base.block_table[b, :full]] = False
        if rem:
            sentinel_rows[base.block_table[b, full], :rem] = False
    mask = torch.from_numpy(sentinel_rows).to(device)
    kv.masked_fill_(mask[:, :, None], 0x7F)
    kv_scale.masked_fill_(mask, float("nan"))
    base.q, base.k_pool, base.k_scale, base.q_len = q, kv, kv_scale, q_len
    base.kv_fp8 = True
    base.meta["q_scale"] = q_scale
    return base


def absorbed_mla_fp8(device="cpu", seed: int = 11, B: int = 64, lo: int = 8192, hi: int = 50000) -> PagedCase:
    """The absorbed-MLA workload (B=64, 128 heads, latent 576, page 64, lens
    U[lo, hi], scale 1/sqrt(192)) on the fp8 input path."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    return build_mla_fp8_case(f"absorbed_mla_fp8_B{B}", seed, B=B, H=128, seq_lens=lens,
                              scale=1.0 / math.sqrt(192), device=device, rng=rng)


def nested_prefix_cascade(device="cpu", seed: int = 8, roots: int = 4, subs: int = 4, members: int = 256,
                          root_tokens: int = 1024, sub_tokens: int = 1024, suffix_lo: int = 64,
                          suffix_hi: int = 512, values: bool = True) -> PagedCase:
    """Two-level shared prefixes: ``roots`` root prefixes (``root_tokens``
    each, e.g. a system prompt) each followed by ``subs`` second-level
    prefixes (``sub_tokens``, e.g. a problem statement) each shared by
    ``members`` sequences with their own suffix U[suffix_lo, suffix_hi];
    32/8 heads, D=64, bf16, page 16; pages shuffled over a 1.25x pool."""
    ps = 16
    rng = np.random.default_rng(seed)
    B = roots * subs * members
    rp, sp = root_tokens // ps, sub_tokens // ps
    suffix = rng.integers(suffix_lo, suffix_hi + 1, size=B).astype(np.int32)
    lens = (rp + sp) * ps + suffix
    own = _pages_for(lens, ps) - rp - sp
    need = roots * rp + roots * subs * sp + int(own.sum())
    num_pages = int(math.ceil(1.25 * need))
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((B, int((rp + sp + own).max())), perm[need], dtype=np.int32)
    cur = 0
    for r in range(roots):
        root = perm[cur:cur + rp]
        cur += rp
        for k in range(subs):
            sub = perm[cur:cur + sp]
            cur += sp
            for m in range(members):
                b = (r * subs + k) * members + m
                bt[b, :rp], bt[b, rp:rp + sp] = root, sub
    for b in range(B):
        bt[b, rp + sp:rp + sp + own[b]] = perm[cur:cur + own[b]]
        cur += int(own[b])
    assert cur == need
    case = build_case(f"nested_cascade_{roots}x{subs}x{members}", seed, B=B, H_q=32, H_kv=8, D=64, page_size=ps,
                      seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(64), device=device, rng=rng,
                      values=values, layout=(bt, num_pages))
    case.meta.update(roots=roots, subs=subs, members=members, root_pages=rp, sub_pages=sp)
    return case


def llama3_8b_layer_fp8(device="cpu", seed: int = 7, B: int = 64, lo: int = 512, hi: int = 4096,
                        append: bool = True) -> PagedCase:
    """The Llama-3-8B-shaped layer over an fp8 cache (same lengths and shapes)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    return build_fp8_case(f"llama3_8b_layer_fp8_B{B}", seed, B=B, H_q=32, H_kv=8, D=128, page_size=16,
                          seq_lens=lens, scale=1.0 / math.sqrt(128), append=append, device=device, rng=rng)


def tiny_gqa_append(device="cpu", seed: int = 1) -> PagedCase:
    """Tiny paged GQA decode: B=4, 8/2 heads, D=64, page 16, fp32, lens
    {17, 40, 64, 100}, 64-page pool, scale 1/8, one appended token."""
    return build_case("tiny_gqa_append_fp32", seed, B=4, H_q=8, H_kv=2, D=64, page_size=16,
                      seq_lens=[17, 40, 64, 100], dtype="f32", scale=1.0 / math.sqrt(64),
                      append=True, num_pages=64, device=device)


def llama3_8b_layer(device="cpu", seed: int = 2, B: int = 64, lo: int = 512, hi: int = 4096,
                    append: bool = True) -> PagedCase:
    """Llama-3-8B-shaped decode layer: 32/8 heads, D=128, bf16, page 16,
    lens ~ U[lo, hi], pool 1.25x the need."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    return build_case(f"llama3_8b_layer_B{B}", seed, B=B, H_q=32, H_kv=8, D=128, page_size=16,
                      seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(128),
                      append=append, device=device, rng=rng)


def speculative_verify(device="cpu", seed: int = 6, B: int = 64, q_len: int = 4, lo: int = 512,
                       hi: int = 4096) -> PagedCase:
    """Llama-3-8B-shaped layer verifying q_len draft tokens per sequence:
    32/8 heads, D=128, bf16, page 16, lens ~ U[lo, hi] counting the draft
    tokens (their K/V already in the cache), pool 1.25x the need."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    return build_case(f"speculative_verify_B{B}_q{q_len}", seed, B=B, H_q=32, H_kv=8, D=128,
                      page_size=16, seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(128),
                      device=device, rng=rng, q_len=q_len)


def draft_trees(B: int, n: int, rng: np.random.Generator, shape: str = "random") -> np.ndarray:
    """Parents [B, n] (int32) of B draft-token trees: node j's parent is an
    earlier node or -1 (a child of the last committed token).

    "random": each node hangs under a uniformly drawn earlier node or the
    context; "chain": a single causal chain; "star": every node under the
    context; "beam": levels of up to 4 children per node, breadth first."""
    par = np.empty((B, n), dtype=np.int32)
    for b in range(B):
        if shape == "chain":
            par[b] = np.arange(-1, n - 1)
        elif shape == "star":
            par[b] = -1
        elif shape == "beam":
            par[b, 0] = -1
            for j in range(1, n):
                par[b, j] = (j - 1) // 4
        else:
            par[b] = [int(rng.integers(-1, j)) if j > 0 else -1 for j in range(n)]
    return par


def speculative_tree(device="cpu", seed: int = 10, B: int = 64, n: int = 16, lo: int = 512,
                     hi: int = 4096, shape: str = "random"):
    """Llama-3-8B-shaped layer verifying a tree of n draft tokens per
    sequence (32/8 heads, D=128, bf16, page 16, lens ~ U[lo, hi] counting
    the draft tokens). Returns (case, parents int32 [B, n])."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    case = build_case(f"speculative_tree_B{B}_n{n}", seed, B=B, H_q=32, H_kv=8, D=128, page_size=16,
                      seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(128), device=device, rng=rng, q_len=n)
    return case, draft_trees(B, n, rng, shape)


def sliding_window(device="cpu", seed: int = 8, B: int = 64, lo: int = 4096, hi: int = 32768,
                   window: int = 4096) -> PagedCase:
    """Llama-3-8B-shaped layer over a sliding-window KV group: 32/8 heads,
    D=128, bf16, page 16, lens ~ U[lo, hi], each query attending its last
    ``window`` tokens. As in such a group's block table (tokenspeed 딥다이브,
    section 6-3), the slots wholly in front of the window hold a placeholder
    page; only the window's pages are real (pool 1.25x of them)."""
    rng = np.random.default_rng(seed)
    ps = 16
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    slots = _pages_for(lens, ps)
    first = np.maximum(0, lens.astype(np.int64) - window) // ps
    need = slots - first
    num_pages = int(np.ceil(need.sum() * 1.25)) + 1
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((B, int(slots.max())), perm[-1], dtype=np.int32)  # perm[-1]: the placeholder
    c = 0
    for b in range(B):
        bt[b, first[b]:slots[b]] = perm[c:c + need[b]]
        c += int(need[b])
    case = build_case(f"sliding_window_B{B}_W{window}", seed, B=B, H_q=32, H_kv=8, D=128, page_size=ps,
                      seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(128), device=device, rng=rng,
                      layout=(bt, num_pages))
    case.window = int(window)
    return case


def mixed_lengths(device="cpu", seed: int = 3, repeat: int = 32) -> PagedCase:
    """Mixed-length batch: lens {20,30,50,80,120,200,500,1000} x repeat, shuffled;
    32/8 heads, D=64, bf16, page 16, random page placement."""
    rng = np.random.default_rng(seed)
    base = np.array([20, 30, 50, 80, 120, 200, 500, 1000], dtype=np.int32)
    lens = rng.permutation(np.tile(base, repeat)).astype(np.int32)
    return build_case(f"mixed_lengths_B{len(lens)}", seed, B=len(lens), H_q=32, H_kv=8, D=64,
                      page_size=16, seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(64),
                      device=device, rng=rng)


def shared_prefix_cascade(device="cpu", seed: int = 4, groups: int = 16, members: int = 1024,
                          prefix_tokens: int = 2048, suffix_lo: int = 64,
                          suffix_hi: int = 512, ungrouped: int = 0, values: bool = True) -> PagedCase:
    """Shared-prefix cascade: ``groups`` x ``members`` sequences, each group one
    shared prefix of ``prefix_tokens`` tokens (whole pages, shared by id) plus
    per-sequence suffix ~ U[suffix_lo, suffix_hi]; 32/8 heads, D=64, bf16,
    page 16. Sequence order is shuffled; ``ungrouped`` extra sequences own
    all their pages."""
    ps = 16
    assert prefix_tokens % ps == 0
    rng = np.random.default_rng(seed)
    B = groups * members + ungrouped
    order = rng.permutation(B)
    group_lists = [np.sort(order[gi * members:(gi + 1) * members]) for gi in range(groups)]
    suffix = rng.integers(suffix_lo, suffix_hi + 1, size=B).astype(np.int32)
    lens = (prefix_tokens + suffix).astype(np.int32)
    return build_case(f"cascade_{groups}x{members}", seed, B=B, H_q=32, H_kv=8, D=64,
                      page_size=ps, seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(64),
                      shared_groups=group_lists, shared_pages=prefix_tokens // ps,
                      device=device, rng=rng, values=values)


def absorbed_mla(device="cpu", seed: int = 5, B: int = 64, lo: int = 8192,
                 hi: int = 50000) -> PagedCase:
    """Absorbed-MLA paged decode: 128 heads, one latent head of 576 (V = first
    512), bf16, page 64, lens ~ U[lo, hi], scale 1/sqrt(192)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    return build_case(f"absorbed_mla_B{B}", seed, B=B, H_q=128, H_kv=1, D=576, Dv=512,
                      page_size=64, seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(192),
                      mla=True, device=device, rng=rng)


def absorbed_mla_multi(device="cpu", seed: int = 9, B: int = 64, H: int = 64, q_len: int = 4,
                       lo: int = 8192, hi: int = 50000) -> PagedCase:
    """Absorbed-MLA decode verifying q_len draft tokens per sequence with H
    heads (the fold example's 64 heads x 4 tokens by default): latent 576
    (V = first 512), bf16, page 64, lens ~ U[lo, hi] counting the draft
    tokens, scale 1/sqrt(192)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    return build_case(f"absorbed_mla_B{B}_H{H}_q{q_len}", seed, B=B, H_q=H, H_kv=1, D=576, Dv=512,
                      page_size=64, seq_lens=lens, dtype="bf16", scale=1.0 / math.sqrt(192),
                      mla=True, device=device, rng=rng, q_len=q_len)


# --------------------------------------------------------------------------
# Moving inputs to the oracle (data movement only)
# --------------------------------------------------------------------------

def _to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def oracle_view(case: PagedCase, seq_idx: Optional[Sequence[int]] = None,
                k_pool: Optional[torch.Tensor] = None,
                v_pool: Optional[torch.Tensor] = None) -> Dict[str, np.ndarray]:
    """The inputs of sequences ``seq_idx`` as float64 numpy arrays.

    Only the pages those sequences own are copied; their block-table rows are
    renumbered to the compacted pool. ``k_pool``/``v_pool`` default to the
    case's pools (pass a snapshot taken before an append to get pre-append data).
    """
    B = case.B
    idx = np.arange(B) if seq_idx is None else np.asarray(seq_idx, dtype=np.int64)
    lens = case.attn_lens[idx]
    n_alloc = _pages_for(lens, case.page_size)
    rows = case.block_table[idx]
    used = np.unique(np.concatenate([rows[i, :n_alloc[i]] for i in range(len(idx))] + [np.zeros(0, np.int32)]))
    remap = {int(p): i for i, p in enumerate(used)}
    bt = np.zeros((len(idx), max(1, rows.shape[1])), dtype=np.int64)
    for i in range(len(idx)):
        for j in range(int(n_alloc[i])):
            bt[i, j] = remap[int(rows[i, j])]
    kp = case.k_pool if k_pool is None else k_pool
    vp = case.v_pool if v_pool is None else v_pool
    dev_pages = torch.from_numpy(used.astype(np.int64)).to(kp.device)
    # fp8 caches travel as their raw codes (uint8) and float32 scales
    conv = (lambda t: t.cpu().numpy()) if case.kv_fp8 else _to_f64
    dev_idx = torch.from_numpy(idx).to(case.q.device)
    fp8_q = case.mla and case.kv_fp8   # MLA fp8 path: the queries are codes too
    out = {
        "q": case.q[dev_idx].cpu().numpy() if fp8_q else _to_f64(case.q[dev_idx]),
        "k_pool": conv(kp.index_select(0, dev_pages)) if len(used) else None,
        "v_pool": conv(vp.index_select(0, dev_pages)) if (vp is not None and len(used)) else None,
        "block_table": bt,
        "seq_lens": lens.astype(np.int64),
        "positions": case.seq_lens[idx].astype(np.int64),
        "page_of_remapped": used,
    }
    if case.kv_fp8:
        out["k_scale"] = case.k_scale.index_select(0, dev_pages).cpu().numpy() if len(used) else None
        if case.v_scale is not None:
            out["v_scale"] = case.v_scale.index_select(0, dev_pages).cpu().numpy() if len(used) else None
    if fp8_q:
        out["q_scale"] = case.meta["q_scale"][dev_idx].cpu().numpy()
    if "parents" in case.meta:
        out["parents"] = np.asarray(case.meta["parents"])[idx]
    if case.append:
        dev_idx = torch.from_numpy(idx).to(case.q.device)
        out["k_new"] = _to_f64(case.k_new[dev_idx])
        out["v_new"] = _to_f64(case.v_new[dev_idx])
    return out


def sample_sequences(case: PagedCase, n: int, seed: int = 0) -> np.ndarray:
    """A seeded sample of sequence ids that always includes the shortest and
    the longest sequence (ragged extremes)."""
    rng = np.random.default_rng(seed + 1000 * case.seed)
    n = min(n, case.B)
    pick = set(rng.choice(case.B, size=n, replace=False).tolist())
    pick.add(int(np.argmin(case.attn_lens)))
    pick.add(int(np.argmax(case.attn_lens)))
    return np.array(sorted(pick), dtype=np.int64)
