"""Seeded synthetic workloads for cascade verify and prefix-hit prefill.

This module only *makes inputs*: random bf16 tensors, page tables and
sequence lengths.  It holds none of the attention arithmetic, so both the
fp64 oracle (``oracle/``) and the CUDA path (``cascade_paged_attention_gb300``)
can consume the same bits without sharing any of the method's code.

Layout conventions written here (the reader side lives separately in the
oracle's C code and in the CUDA kernels):

* K/V page pool: ``[num_pages, page_size, H_kv, head_dim]`` bf16 (stored as
  uint16 bit patterns).  Logical position ``pos`` of a sequence lives in page
  ``table[pos // page_size]`` at slot ``pos % page_size`` (the block-table rule
  of the KV-cache tutorial, "PagedAttention" section, ``append_token``).
* Queries ``q``: ``[T, H_q, head_dim]``; for verify, token
  ``t = (b * topk + k) * S + s`` is draft token ``s`` of branch ``k`` of
  request ``b``.
* Page tables are int32, padded with -1 past each row's used pages.

Values are N(0, 1) fp32 rounded to bf16 (round-to-nearest-even).  Slots of a
page that lie past a sequence's end are filled with ``pad_fill`` ("random" or
"nan") so that a reader which touches them shows up in the results.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = [
    "build_pool",
    "table_matrix",
    "VerifyWorkload",
    "PrefillWorkload",
    "make_verify",
    "make_prefill",
    "TreeWorkload",
    "make_tree_verify",
    "random_bfs_tree",
    "chain_forest",
    "TREE_CONFIGS",
    "Fp8VerifyWorkload",
    "make_verify_fp8",
    "e4m3_codes",
    "SharedWorkload",
    "make_shared_verify",
    "SHARED_CONFIGS",
    "VERIFY_CONFIGS",
    "PREFILL_CONFIG",
    "bf16_bits_from_f32",
    "f32_from_bf16_bits",
]


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_NAN_BF16 = np.uint16(0x7FC0)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    chunk = 1 << 24
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = bf16_bits_from_f32(rng.standard_normal(hi - lo, dtype=np.float32))
    return out.reshape(shape)


@dataclasses.dataclass
class VerifyWorkload:
    """Inputs of one verify step (one layer): B requests, topk chain branches of S drafts."""

    B: int
    topk: int
    S: int
    H_q: int
    H_kv: int
    head_dim: int
    page_size: int
    prefix_lens: np.ndarray          # int32 [B]
    q: np.ndarray                    # uint16 [B*topk*S, H_q, d]
    k_pages: np.ndarray              # uint16 [num_pages, P, H_kv, d]
    v_pages: np.ndarray              # uint16 [num_pages, P, H_kv, d]
    prefix_page_table: np.ndarray    # int32 [B, max_prefix_pages]
    draft_page_table: np.ndarray     # int32 [B*topk, max_draft_pages]
    max_prefix_len: int
    # Logical (de-paged) K/V, only when requested: lists indexed by request /
    # virtual request, each uint16 [len, H_kv, d].
    prefix_k: Optional[list] = None
    prefix_v: Optional[list] = None
    draft_k: Optional[list] = None
    draft_v: Optional[list] = None

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def n_tokens(self) -> int:
        return self.B * self.topk * self.S

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def unique_kv_tokens(self) -> int:
        """Prefix tokens once per request plus every branch's own drafts."""
        return int(self.prefix_lens.astype(np.int64).sum()) + self.B * self.topk * self.S

    def naive_kv_tokens(self) -> int:
        """Every virtual request (b, k) re-reads its request's prefix plus its drafts."""
        return int(self.topk * (self.prefix_lens.astype(np.int64) + self.S).sum())

    def kv_bytes_per_token(self) -> int:
        return 2 * self.H_kv * self.head_dim * 2


@dataclasses.dataclass
class PrefillWorkload:
    """Inputs of a prefill after a prefix-cache hit of H tokens (same N for every request)."""

    B: int
    N: int
    H: int
    H_q: int
    H_kv: int
    head_dim: int
    page_size: int
    q: np.ndarray           # uint16 [B*M, H_q, d] suffix queries, M = N - H
    k_pages: np.ndarray     # uint16 [num_pages, P, H_kv, d]
    v_pages: np.ndarray
    page_table: np.ndarray  # int32 [B, ceil(N/P)]
    seq_k: Optional[list] = None  # logical K per request [N, H_kv, d] (optional)
    seq_v: Optional[list] = None

    @property
    def M(self) -> int:
        return self.N - self.H

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def visible_pairs(self) -> int:
        """Query-key pairs the suffix must still compute, per request and q head."""
        N, H = self.N, self.H
        return (N * (N + 1) - H * (H + 1)) // 2


def build_pool(k_seqs, v_seqs, page_size: int, perm_rng: np.random.Generator,
               pad_fill: str = "random", spare_pages: int = 0):
    """Page a list of logical sequences into one K pool and one V pool.

    ``k_seqs[i]`` / ``v_seqs[i]`` are uint16 ``[len_i, H_kv, d]``.  Each
    sequence gets ``ceil(len_i / page_size)`` physical pages drawn from one
    random permutation of the pool; token ``pos`` goes to page
    ``table_i[pos // page_size]``, slot ``pos % page_size``.  Returns
    ``(k_pages, v_pages, tables)`` with ``tables[i]`` an int32 array.
    """
    assert len(k_seqs) == len(v_seqs)
    P = page_size
    if k_seqs:
        H_kv, d = k_seqs[0].shape[1], k_seqs[0].shape[2]
    else:
        H_kv, d = 1, 1
    counts = [(int(x.shape[0]) + P - 1) // P for x in k_seqs]
    total = int(sum(counts)) + spare_pages
    perm = perm_rng.permutation(total).astype(np.int32)
    shape = (total, P, H_kv, d)
    if pad_fill == "nan":
        k_pages = np.full(shape, _NAN_BF16, dtype=np.uint16)
        v_pages = np.full(shape, _NAN_BF16, dtype=np.uint16)
    elif pad_fill == "random":
        k_pages = _normal_bf16(perm_rng, shape)
        v_pages = _normal_bf16(perm_rng, shape)
    elif pad_fill == "zero":
        k_pages = np.zeros(shape, dtype=np.uint16)
        v_pages = np.zeros(shape, dtype=np.uint16)
    else:
        raise ValueError(pad_fill)
    tables = []
    cur = 0
    for ks, vs, n in zip(k_seqs, v_seqs, counts):
        tab = perm[cur:cur + n].copy()
        cur += n
        pos = np.arange(ks.shape[0])
        if pos.size:
            k_pages[tab[pos // P], pos % P] = ks
            v_pages[tab[pos // P], pos % P] = vs
        tables.append(tab)
    return k_pages, v_pages, tables


def table_matrix(tables, width: int) -> np.ndarray:
    """Stack per-sequence page lists into an int32 matrix padded with -1."""
    out = np.full((len(tables), max(1, width)), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        out[i, :len(t)] = t
    return out


def make_verify(B: int, topk: int, S: int, H_q: int, H_kv: int, head_dim: int = 128,
                page_size: int = 16, L: Optional[int] = None,
                L_range: Optional[tuple[int, int]] = None, prefix_lens=None,
                seed: int = 0, perm_seed: Optional[int] = None, pad_fill: str = "random",
                spare_pages: int = 0, keep_logical: bool = False) -> VerifyWorkload:
    """Build one verify workload.

    The logical contents (q, every sequence's K/V) depend only on ``seed``;
    the physical placement of pages depends only on ``perm_seed``, so two
    workloads that differ in ``perm_seed`` hold the same logical data.
    """
    rng = np.random.default_rng(seed)
    if prefix_lens is not None:
        lens = np.asarray(prefix_lens, dtype=np.int32).copy()
        assert lens.shape == (B,)
    elif L_range is not None:
        lens = rng.integers(L_range[0], L_range[1] + 1, size=B).astype(np.int32)
    else:
        assert L is not None
        lens = np.full(B, L, dtype=np.int32)
    P = page_size
    d = head_dim
    T = B * topk * S
    q = _normal_bf16(rng, (T, H_q, d))
    pk = [_normal_bf16(rng, (int(lens[b]), H_kv, d)) for b in range(B)]
    pv = [_normal_bf16(rng, (int(lens[b]), H_kv, d)) for b in range(B)]
    dk = [_normal_bf16(rng, (S, H_kv, d)) for _ in range(B * topk)]
    dv = [_normal_bf16(rng, (S, H_kv, d)) for _ in range(B * topk)]

    perm_rng = np.random.default_rng(seed * 7919 + 17 if perm_seed is None else perm_seed)
    k_pages, v_pages, tables = build_pool(pk + dk, pv + dv, P, perm_rng, pad_fill, spare_pages)
    max_prefix_len = int(lens.max()) if B > 0 else 0
    prefix_pt = table_matrix(tables[:B], (max_prefix_len + P - 1) // P)
    draft_pt = table_matrix(tables[B:], (S + P - 1) // P)

    wl = VerifyWorkload(B=B, topk=topk, S=S, H_q=H_q, H_kv=H_kv, head_dim=d, page_size=P,
                        prefix_lens=lens, q=q, k_pages=k_pages, v_pages=v_pages,
                        prefix_page_table=prefix_pt, draft_page_table=draft_pt,
                        max_prefix_len=max_prefix_len)
    if keep_logical:
        wl.prefix_k, wl.prefix_v, wl.draft_k, wl.draft_v = pk, pv, dk, dv
    return wl


def make_prefill(B: int, N: int, H: int, H_q: int, H_kv: int, head_dim: int = 128,
                 page_size: int = 16, seed: int = 0, perm_seed: Optional[int] = None,
                 pad_fill: str = "random", keep_logical: bool = False) -> PrefillWorkload:
    """Build one prefix-hit prefill workload: every request has N tokens, the first H cached."""
    assert 0 <= H <= N
    rng = np.random.default_rng(seed)
    P = page_size
    d = head_dim
    M = N - H
    q = _normal_bf16(rng, (B * M, H_q, d))
    sk = [_normal_bf16(rng, (N, H_kv, d)) for _ in range(B)]
    sv = [_normal_bf16(rng, (N, H_kv, d)) for _ in range(B)]
    perm_rng = np.random.default_rng(seed * 7919 + 17 if perm_seed is None else perm_seed)
    k_pages, v_pages, tables = build_pool(sk, sv, P, perm_rng, pad_fill)
    pt = table_matrix(tables, (N + P - 1) // P)
    wl = PrefillWorkload(B=B, N=N, H=H, H_q=H_q, H_kv=H_kv, head_dim=d, page_size=P, q=q,
                         k_pages=k_pages, v_pages=v_pages, page_table=pt)
    if keep_logical:
        wl.seq_k, wl.seq_v = sk, sv
    return wl


def random_bfs_tree(rng: np.random.Generator, N: int, n_roots: int = 1,
                    max_children: int = 4) -> np.ndarray:
    """A random draft tree of N nodes, returned as a BFS-ordered parent array.

    Nodes are produced level by level: the first ``n_roots`` nodes are roots
    (parent -1); each later node picks its parent uniformly among the nodes of
    the previous level that still have fewer than ``max_children`` children,
    and a new level starts once a level's nodes are used up.  Because nodes
    are numbered in creation order and parents are picked in ascending order,
    the numbering is a BFS order (every parent precedes its children and the
    children of an earlier node precede those of a later one).
    """
    assert 1 <= n_roots <= N
    parents = [-1] * n_roots
    level = list(range(n_roots))
    while len(parents) < N:
        n_next = int(rng.integers(1, max_children * len(level) + 1))
        n_next = min(n_next, N - len(parents))
        picks = sorted(int(x) for x in rng.choice(
            np.repeat(np.array(level), max_children), size=n_next, replace=False))
        start = len(parents)
        parents.extend(picks)
        level = list(range(start, len(parents)))
    return np.asarray(parents, dtype=np.int32)


def chain_forest(topk: int, S: int) -> np.ndarray:
    """Parent array of topk independent chains of S drafts, in BFS order.

    Level s holds draft s of every branch, so draft s of branch k is node
    ``s*topk + k`` and its parent is node ``(s-1)*topk + k``.
    """
    par = np.full(topk * S, -1, dtype=np.int32)
    for s in range(1, S):
        for k in range(topk):
            par[s * topk + k] = (s - 1) * topk + k
    return par


@dataclasses.dataclass
class TreeWorkload:
    """Inputs of one tree-verify step: B requests, each with a BFS-flattened draft tree of N nodes."""

    B: int
    N: int
    H_q: int
    H_kv: int
    head_dim: int
    page_size: int
    prefix_lens: np.ndarray          # int32 [B]
    parents: np.ndarray              # int32 [B, N], -1 for roots
    q: np.ndarray                    # uint16 [B*N, H_q, d], token b*N + i
    k_pages: np.ndarray
    v_pages: np.ndarray
    prefix_page_table: np.ndarray    # int32 [B, max_prefix_pages]
    tree_page_table: np.ndarray      # int32 [B, ceil(N/P)]
    max_prefix_len: int
    prefix_k: Optional[list] = None  # logical K/V per request (optional)
    prefix_v: Optional[list] = None
    tree_k: Optional[list] = None
    tree_v: Optional[list] = None

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def n_tokens(self) -> int:
        return self.B * self.N

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def unique_kv_tokens(self) -> int:
        return int(self.prefix_lens.astype(np.int64).sum()) + self.B * self.N

    def kv_bytes_per_token(self) -> int:
        return 2 * self.H_kv * self.head_dim * 2


def make_tree_verify(B: int, N: int, H_q: int, H_kv: int, head_dim: int = 128,
                     page_size: int = 16, L: Optional[int] = None,
                     L_range: Optional[tuple[int, int]] = None, prefix_lens=None,
                     parents=None, n_roots: int = 1, max_children: int = 4, seed: int = 0,
                     perm_seed: Optional[int] = None, pad_fill: str = "random",
                     keep_logical: bool = False) -> TreeWorkload:
    """Build one tree-verify workload.

    ``parents`` (int ``[N]`` shared by every request, or ``[B, N]``) fixes
    the trees; otherwise each request draws its own ``random_bfs_tree``.
    Logical contents depend only on ``seed``, page placement only on
    ``perm_seed``.
    """
    rng = np.random.default_rng(seed)
    if prefix_lens is not None:
        lens = np.asarray(prefix_lens, dtype=np.int32).copy()
        assert lens.shape == (B,)
    elif L_range is not None:
        lens = rng.integers(L_range[0], L_range[1] + 1, size=B).astype(np.int32)
    else:
        assert L is not None
        lens = np.full(B, L, dtype=np.int32)
    if parents is None:
        par = np.stack([random_bfs_tree(rng, N, n_roots, max_children) for _ in range(B)])
    else:
        par = np.asarray(parents, dtype=np.int32)
        par = np.broadcast_to(par, (B, N)).copy() if par.ndim == 1 else par.copy()
    assert par.shape == (B, N)
    P = page_size
    d = head_dim
    q = _normal_bf16(rng, (B * N, H_q, d))
    pk = [_normal_bf16(rng, (int(lens[b]), H_kv, d)) for b in range(B)]
    pv = [_normal_bf16(rng, (int(lens[b]), H_kv, d)) for b in range(B)]
    tk = [_normal_bf16(rng, (N, H_kv, d)) for _ in range(B)]
    tv = [_normal_bf16(rng, (N, H_kv, d)) for _ in range(B)]
    perm_rng = np.random.default_rng(seed * 7919 + 17 if perm_seed is None else perm_seed)
    k_pages, v_pages, tables = build_pool(pk + tk, pv + tv, P, perm_rng, pad_fill)
    max_prefix_len = int(lens.max()) if B > 0 else 0
    wl = TreeWorkload(B=B, N=N, H_q=H_q, H_kv=H_kv, head_dim=d, page_size=P, prefix_lens=lens,
                      parents=par, q=q, k_pages=k_pages, v_pages=v_pages,
                      prefix_page_table=table_matrix(tables[:B], (max_prefix_len + P - 1) // P),
                      tree_page_table=table_matrix(tables[B:], (N + P - 1) // P),
                      max_prefix_len=max_prefix_len)
    if keep_logical:
        wl.prefix_k, wl.prefix_v, wl.tree_k, wl.tree_v = pk, pv, tk, tv
    return wl


def e4m3_codes(rng: np.random.Generator, shape, exp_lo: int = 5, exp_hi: int = 8) -> np.ndarray:
    """Random FP8 E4M3 codes with magnitudes of order one.

    Codes are drawn field by field, with no arithmetic on values: a random
    sign bit, an exponent field uniform in [exp_lo, exp_hi] (bias 7, so about
    0.25 to 3.75 for the defaults) and a uniform 3-bit mantissa.  A few codes
    are replaced by zero and by subnormals so that those encodings appear too.
    """
    n = int(np.prod(shape))
    sign = rng.integers(0, 2, size=n, dtype=np.uint8) << np.uint8(7)
    expo = rng.integers(exp_lo, exp_hi + 1, size=n, dtype=np.uint8) << np.uint8(3)
    mant = rng.integers(0, 8, size=n, dtype=np.uint8)
    codes = sign | expo | mant
    special = rng.random(n) < 0.01
    codes[special] = sign[special] | mant[special]  # exponent field 0: zero or subnormal
    return codes.reshape(shape)


@dataclasses.dataclass
class Fp8VerifyWorkload:
    """A verify workload whose K/V pools hold FP8 E4M3 codes with scales."""

    B: int
    topk: int
    S: int
    H_q: int
    H_kv: int
    head_dim: int
    page_size: int
    prefix_lens: np.ndarray
    q: np.ndarray                    # uint16 bf16 bits [B*topk*S, H_q, d]
    k_pages: np.ndarray              # uint8 E4M3 codes [num_pages, P, H_kv, d]
    v_pages: np.ndarray
    k_scale: np.ndarray              # float32 [1] or [H_kv, d]
    v_scale: np.ndarray
    prefix_page_table: np.ndarray
    draft_page_table: np.ndarray
    max_prefix_len: int

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def n_tokens(self) -> int:
        return self.B * self.topk * self.S

    def unique_kv_tokens(self) -> int:
        return int(self.prefix_lens.astype(np.int64).sum()) + self.B * self.topk * self.S

    def kv_bytes_per_token(self) -> int:
        return 2 * self.H_kv * self.head_dim


def make_verify_fp8(B: int, topk: int, S: int, H_q: int, H_kv: int, head_dim: int = 128,
                    page_size: int = 16, L: Optional[int] = None, prefix_lens=None,
                    scales: str = "tensor", seed: int = 0,
                    perm_seed: Optional[int] = None,
                    pad_code: Optional[int] = None) -> Fp8VerifyWorkload:
    """Build a verify workload over FP8 pools.

    ``scales``: ``"tensor"`` (one random K and one random V scale), ``"channel"``
    (one per KV head and channel), ``"unit"`` (both 1.0) or ``"pow2"`` (per
    channel, random powers of two).  Unused page slots hold random codes, or
    the byte ``pad_code`` when it is given (e.g. 0x7F, a NaN code).
    """
    rng = np.random.default_rng(seed)
    if prefix_lens is not None:
        lens = np.asarray(prefix_lens, dtype=np.int32).copy()
    else:
        lens = np.full(B, L, dtype=np.int32)
    P, d = page_size, head_dim
    q = _normal_bf16(rng, (B * topk * S, H_q, d))
    seqs = [int(x) for x in lens] + [S] * (B * topk)
    counts = [(n + P - 1) // P for n in seqs]
    perm_rng = np.random.default_rng(seed * 7919 + 17 if perm_seed is None else perm_seed)
    perm = perm_rng.permutation(int(sum(counts))).astype(np.int32)
    # codes are drawn in logical page order (sequence by sequence), then page i
    # of that order is placed at physical page perm[i]: the logical contents
    # depend only on `seed`, the placement only on `perm_seed`
    k_logical = e4m3_codes(rng, (int(sum(counts)), P, H_kv, d))
    v_logical = e4m3_codes(rng, (int(sum(counts)), P, H_kv, d))
    k_pages = np.empty_like(k_logical)
    v_pages = np.empty_like(v_logical)
    k_pages[perm] = k_logical
    v_pages[perm] = v_logical
    tables, cur = [], 0
    for n in counts:
        tables.append(perm[cur:cur + n].copy())
        cur += n
    if pad_code is not None:
        for tab, n in zip(tables, seqs):
            pos = np.arange(n, len(tab) * P)
            k_pages[tab[pos // P], pos % P] = np.uint8(pad_code)
            v_pages[tab[pos // P], pos % P] = np.uint8(pad_code)
    # scales keep the values (codes of magnitude 0.25 .. 3.75 times the scale)
    # at the N(0,1) magnitude of the bf16 workloads: |value| < 3
    if scales == "tensor":
        k_scale = rng.uniform(0.25, 0.75, size=1).astype(np.float32)
        v_scale = rng.uniform(0.25, 0.75, size=1).astype(np.float32)
    elif scales == "channel":
        k_scale = rng.uniform(0.25, 0.75, size=(H_kv, d)).astype(np.float32)
        v_scale = rng.uniform(0.25, 0.75, size=(H_kv, d)).astype(np.float32)
    elif scales == "unit":
        k_scale = np.ones(1, np.float32)
        v_scale = np.ones(1, np.float32)
    elif scales == "pow2":
        k_scale = np.exp2(rng.integers(-2, 2, size=(H_kv, d))).astype(np.float32)
        v_scale = np.exp2(rng.integers(-2, 2, size=(H_kv, d))).astype(np.float32)
    else:
        raise ValueError(scales)
    max_prefix_len = int(lens.max()) if B > 0 else 0
    return Fp8VerifyWorkload(B=B, topk=topk, S=S, H_q=H_q, H_kv=H_kv, head_dim=d, page_size=P,
                             prefix_lens=lens, q=q, k_pages=k_pages, v_pages=v_pages,
                             k_scale=k_scale, v_scale=v_scale,
                             prefix_page_table=table_matrix(tables[:B],
                                                            (max_prefix_len + P - 1) // P),
                             draft_page_table=table_matrix(tables[B:], (S + P - 1) // P),
                             max_prefix_len=max_prefix_len)


@dataclasses.dataclass
class SharedWorkload:
    """Multi-level verify inputs: groups of consecutive requests share one prefix.

    Request b (group ``b // (B // n_groups)``) holds the group's shared prefix
    of ``shared_len`` tokens, then its own prefix of ``prefix_lens[b]`` tokens,
    then topk branches of S drafts.
    """

    B: int
    n_groups: int
    shared_len: int
    topk: int
    S: int
    H_q: int
    H_kv: int
    head_dim: int
    page_size: int
    prefix_lens: np.ndarray          # int32 [B], own prefix lengths
    q: np.ndarray                    # uint16 [B*topk*S, H_q, d]
    k_pages: np.ndarray
    v_pages: np.ndarray
    shared_page_table: np.ndarray    # int32 [n_groups, ceil(shared_len/P)]
    prefix_page_table: np.ndarray    # int32 [B, ceil(max own len/P)]
    draft_page_table: np.ndarray     # int32 [B*topk, ceil(S/P)]
    max_prefix_len: int
    shared_k: Optional[list] = None  # logical K/V (optional)
    shared_v: Optional[list] = None
    prefix_k: Optional[list] = None
    prefix_v: Optional[list] = None
    draft_k: Optional[list] = None
    draft_v: Optional[list] = None

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def n_tokens(self) -> int:
        return self.B * self.topk * self.S

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def unique_kv_tokens(self) -> int:
        """Each shared prefix once, each own prefix once, every branch's drafts."""
        return (self.n_groups * self.shared_len + int(self.prefix_lens.astype(np.int64).sum())
                + self.B * self.topk * self.S)

    def kv_bytes_per_token(self) -> int:
        return 2 * self.H_kv * self.head_dim * 2


def make_shared_verify(B: int, n_groups: int, shared_len: int, topk: int, S: int, H_q: int,
                       H_kv: int, head_dim: int = 128, page_size: int = 16,
                       L: Optional[int] = None, prefix_lens=None, seed: int = 0,
                       perm_seed: Optional[int] = None, pad_fill: str = "random",
                       keep_logical: bool = False) -> SharedWorkload:
    """Build one multi-level verify workload (``L`` / ``prefix_lens``: own prefix lengths)."""
    assert B % n_groups == 0
    rng = np.random.default_rng(seed)
    if prefix_lens is not None:
        lens = np.asarray(prefix_lens, dtype=np.int32).copy()
        assert lens.shape == (B,)
    else:
        assert L is not None
        lens = np.full(B, L, dtype=np.int32)
    P = page_size
    d = head_dim
    q = _normal_bf16(rng, (B * topk * S, H_q, d))
    sk = [_normal_bf16(rng, (shared_len, H_kv, d)) for _ in range(n_groups)]
    sv = [_normal_bf16(rng, (shared_len, H_kv, d)) for _ in range(n_groups)]
    pk = [_normal_bf16(rng, (int(lens[b]), H_kv, d)) for b in range(B)]
    pv = [_normal_bf16(rng, (int(lens[b]), H_kv, d)) for b in range(B)]
    dk = [_normal_bf16(rng, (S, H_kv, d)) for _ in range(B * topk)]
    dv = [_normal_bf16(rng, (S, H_kv, d)) for _ in range(B * topk)]
    perm_rng = np.random.default_rng(seed * 7919 + 17 if perm_seed is None else perm_seed)
    k_pages, v_pages, tables = build_pool(sk + pk + dk, sv + pv + dv, P, perm_rng, pad_fill)
    max_prefix_len = int(lens.max()) if B > 0 else 0
    G_ = n_groups
    wl = SharedWorkload(B=B, n_groups=n_groups, shared_len=shared_len, topk=topk, S=S, H_q=H_q,
                        H_kv=H_kv, head_dim=d, page_size=P, prefix_lens=lens, q=q,
                        k_pages=k_pages, v_pages=v_pages,
                        shared_page_table=table_matrix(tables[:G_], (shared_len + P - 1) // P),
                        prefix_page_table=table_matrix(tables[G_:G_ + B],
                                                       (max_prefix_len + P - 1) // P),
                        draft_page_table=table_matrix(tables[G_ + B:], (S + P - 1) // P),
                        max_prefix_len=max_prefix_len)
    if keep_logical:
        wl.shared_k, wl.shared_v = sk, sv
        wl.prefix_k, wl.prefix_v, wl.draft_k, wl.draft_v = pk, pv, dk, dv
    return wl


# The five workloads the method is exercised on, by name.  Verify shapes come
# from the pages' example (L=2000, topk=4, S=5) and its neighbours.
VERIFY_CONFIGS = {
    "tiny": dict(B=2, topk=2, S=3, L=64, H_q=8, H_kv=2, page_size=16, seed=1),
    "llama3_8b": dict(B=32, topk=4, S=3, L=1000, H_q=32, H_kv=8, page_size=16, seed=2),
    "pages_example": dict(B=64, topk=4, S=5, L=2000, H_q=32, H_kv=8, page_size=16, seed=3),
    "long_variable": dict(B=16, topk=8, S=4, L_range=(1024, 32768), H_q=64, H_kv=8,
                          page_size=64, seed=4),
}
# Draft-tree verify: the pages' example request shape (L=2000, H_q=32,
# H_kv=8) with one 20-node tree per request in place of 4 chains of 5, and a
# 60-node tree.
TREE_CONFIGS = {
    "tree_tiny": dict(B=2, N=7, L=64, H_q=8, H_kv=2, page_size=16, seed=11),
    "tree_pages_example": dict(B=64, N=20, L=2000, H_q=32, H_kv=8, page_size=16, seed=12),
    "tree_60": dict(B=64, N=60, L=2000, H_q=32, H_kv=8, page_size=16, seed=13),
}
# Multi-level verify: the pages' example request shape (topk=4, S=5, 2000
# prefix tokens per request) with the first 1024 tokens shared by all 64
# requests (one system prompt) and 976 tokens of each request's own.
SHARED_CONFIGS = {
    "shared_tiny": dict(B=4, n_groups=2, shared_len=40, topk=2, S=3, L=25, H_q=8, H_kv=2,
                        page_size=16, seed=15),
    "shared_pages_example": dict(B=64, n_groups=1, shared_len=1024, topk=4, S=5, L=976, H_q=32,
                                 H_kv=8, page_size=16, seed=14),
}
PREFILL_CONFIG = dict(B=8, N=8192, H_q=32, H_kv=8, page_size=16, seed=5, hits=(0.0, 0.5, 0.75))
