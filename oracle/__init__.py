"""fp64 CPU oracle for cascade verify and prefix-hit prefill.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``cascade_paged_attention_gb300``) never imports, links or calls it, and
this package never imports the product path.

What is computed, and from which passage:

* ``verify``: one full masked attention per (draft token, query head), the
  definition o = softmax(q K^T / sqrt d) V with LSE = log sum exp(q k / sqrt d)
  from the "Cascade attention" page (split-property section).  Draft token s
  of branch k sees its request's prefix and its own branch drafts 0..s
  ("Topk > 1" section of the same page).  ``part="prefix"`` / ``"draft"``
  restrict the key set to the Pass A / Pass B piece of the same page's
  two-segment decomposition.
* ``verify_shared``: multi-level verify.  Requests whose block tables start
  with the same physical pages share that prefix (KV-cache tutorial, the
  block-table example of section 5.3 and ``share_prefix`` of 6.2); a group of
  consecutive requests has one shared prefix, each request its own prefix
  after it, each branch its own drafts.  Draft s of branch k sees all of the
  shared prefix, all of its request's own prefix and drafts 0..s of branch k;
  ``part`` picks one piece (``"shared"``, ``"own"``, ``"draft"``), both
  prefixes (``"prefix"``) or everything.
* ``verify_fp8``: verify over FP8 KV pools (KV-cache tutorial, section 4.5,
  "FP8 KV", per-tensor or per-channel scale): each K/V element is its E4M3
  code decoded exactly (``e4m3_decode``, from the format definition) times
  its scale; the attention is then the definition above.
* ``ancestor_masks``: the tree-attention mask of the KV-cache tutorial
  (section 8.2 tip box; interview question Q14): tree nodes flattened in BFS
  order, A(i) = the ancestors of node i with i itself, M[i, j] = 1 iff j is in
  A(i).  Built bottom-up, A(i) = {i} plus A(parent(i)).
* ``tree_verify``: verify over a general draft tree: node i of request b sees
  the request's prefix and the nodes of A(i).  ``part="prefix"`` /
  ``"draft"`` restrict it to the prefix / the tree nodes, as for ``verify``.
* ``prefill``: suffix query i of a prefix-hit prefill sees keys 0..H+i
  (rectangle 0..H-1 plus triangle H..H+i), "Causal Attention ... KV hit area"
  page, sections 1-2.
* ``merge_state``: the LSE merge identity of the cascade page.
* ``kv_reads_naive`` / ``kv_reads_cascade``: brute-force enumeration of the
  KV tokens each strategy reads (cascade page, "Naive Expand" and "Cascade"
  sections).
* ``visible_pairs``: brute-force count of the visible query-key pairs of the
  prefix-hit mask (hit-area page, sections 1-3).

Parity is pinned for every function here by tests under ``tests/`` (closed
forms, the pages' worked numbers, brute force on tiny inputs, a library
softmax special case).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

_lib = None

PART_CODES = {"full": 0, "prefix": 1, "draft": 2, "rect": 1, "tri": 2, "shared": 3, "own": 4}


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_verify.restype = i32
        lib.oracle_verify.argtypes = [P, P, P, i64, P, i32, P, i32, P, i32, i32, i32, i32, i32,
                                      i32, i32, i32, f64, P, i64, P, P, i32]
        lib.oracle_prefill.restype = i32
        lib.oracle_prefill.argtypes = [P, P, P, i64, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                       i32, f64, P, i64, P, P, i32]
        lib.oracle_tree_verify.restype = i32
        lib.oracle_tree_verify.argtypes = [P, P, P, i64, P, i32, P, i32, P, P, i32, i32, i32,
                                           i32, i32, i32, i32, f64, P, i64, P, P, i32]
        lib.oracle_verify_shared.restype = i32
        lib.oracle_verify_shared.argtypes = [P, P, P, i64, P, i32, i32, i32, P, i32, P, i32, P,
                                             i32, i32, i32, i32, i32, i32, i32, i32, f64, P, i64,
                                             P, P, i32]
        lib.oracle_verify_fp8.restype = i32
        lib.oracle_verify_fp8.argtypes = [P, P, P, P, P, i32, i64, P, i32, P, i32, P, i32, i32,
                                          i32, i32, i32, i32, i32, i32, f64, P, i64, P, P, i32]
        lib.oracle_e4m3_decode.restype = None
        lib.oracle_e4m3_decode.argtypes = [P, i64, P]
        lib.oracle_merge_state.restype = None
        lib.oracle_merge_state.argtypes = [P, P, P, P, i64, i32, P, P]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows_arg(rows):
    if rows is None:
        return None, None, 0
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, _ptr(r), int(r.size)


_ERR = {1: "bad argument", 2: "page id out of range", 3: "out of memory"}


def verify(q, k_pages, v_pages, prefix_page_table, draft_page_table, prefix_lens, topk: int,
           S: int, H_q: int, H_kv: int, scale: Optional[float] = None, part: str = "full",
           rows: Optional[Sequence[int]] = None, threads: int = 0):
    """fp64 verify attention.  Returns (o [n_rows, d] float64, lse [n_rows] float64).

    Rows are ``token * H_q + head`` with token ``(b*topk + k)*S + s``; ``rows=None``
    means all rows in that order.  Inputs are bf16 bit patterns (uint16).
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kp = np.ascontiguousarray(k_pages, dtype=np.uint16)
    vp = np.ascontiguousarray(v_pages, dtype=np.uint16)
    ppt = np.ascontiguousarray(prefix_page_table, dtype=np.int32)
    dpt = np.ascontiguousarray(draft_page_table, dtype=np.int32)
    lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    B = int(lens.shape[0])
    d = int(q.shape[-1])
    P = int(kp.shape[1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r, rp, nr = _rows_arg(rows)
    n = nr if r is not None else B * topk * S * H_q
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    err = lib.oracle_verify(_ptr(q), _ptr(kp), _ptr(vp), int(kp.shape[0]), _ptr(ppt),
                            int(ppt.shape[1]), _ptr(dpt), int(dpt.shape[1]), _ptr(lens), B,
                            topk, S, H_q, H_kv, d, P, PART_CODES[part], float(scale), rp, nr,
                            _ptr(o), _ptr(lse), threads)
    if err:
        raise ValueError(f"oracle_verify: {_ERR.get(err, err)}")
    return o, lse


def verify_wl(wl, part: str = "full", rows=None, threads: int = 0):
    """``verify`` on a ``cpa_synth.VerifyWorkload``-shaped object."""
    return verify(wl.q, wl.k_pages, wl.v_pages, wl.prefix_page_table, wl.draft_page_table,
                  wl.prefix_lens, wl.topk, wl.S, wl.H_q, wl.H_kv, part=part, rows=rows,
                  threads=threads)


def verify_shared(q, k_pages, v_pages, shared_page_table, shared_len: int, prefix_page_table,
                  draft_page_table, prefix_lens, topk: int, S: int, H_q: int, H_kv: int,
                  scale: Optional[float] = None, part: str = "full",
                  rows: Optional[Sequence[int]] = None, threads: int = 0):
    """fp64 multi-level verify; rows and tokens as in ``verify``.

    ``shared_page_table`` is int32 ``[n_groups, stride]``; request b belongs to
    group ``b // (B // n_groups)``.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kp = np.ascontiguousarray(k_pages, dtype=np.uint16)
    vp = np.ascontiguousarray(v_pages, dtype=np.uint16)
    spt = np.ascontiguousarray(shared_page_table, dtype=np.int32)
    ppt = np.ascontiguousarray(prefix_page_table, dtype=np.int32)
    dpt = np.ascontiguousarray(draft_page_table, dtype=np.int32)
    lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    B = int(lens.shape[0])
    n_groups = int(spt.shape[0])
    if n_groups < 1 or B % n_groups:
        raise ValueError("B must be a multiple of the number of groups")
    d = int(q.shape[-1])
    P = int(kp.shape[1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r, rp, nr = _rows_arg(rows)
    n = nr if r is not None else B * topk * S * H_q
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    err = lib.oracle_verify_shared(_ptr(q), _ptr(kp), _ptr(vp), int(kp.shape[0]), _ptr(spt),
                                   int(spt.shape[1]), int(shared_len), B // n_groups, _ptr(ppt),
                                   int(ppt.shape[1]), _ptr(dpt), int(dpt.shape[1]), _ptr(lens), B,
                                   topk, S, H_q, H_kv, d, P, PART_CODES[part], float(scale), rp,
                                   nr, _ptr(o), _ptr(lse), threads)
    if err:
        raise ValueError(f"oracle_verify_shared: {_ERR.get(err, err)}")
    return o, lse


def verify_shared_wl(wl, part: str = "full", rows=None, threads: int = 0):
    """``verify_shared`` on a ``cpa_synth.SharedWorkload``-shaped object."""
    return verify_shared(wl.q, wl.k_pages, wl.v_pages, wl.shared_page_table, wl.shared_len,
                         wl.prefix_page_table, wl.draft_page_table, wl.prefix_lens, wl.topk,
                         wl.S, wl.H_q, wl.H_kv, part=part, rows=rows, threads=threads)


def e4m3_decode(codes) -> np.ndarray:
    """Exact values (float64) of FP8 E4M3 codes (uint8); NaN for the NaN codes."""
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(c.shape, dtype=np.float64)
    lib.oracle_e4m3_decode(_ptr(c), int(c.size), _ptr(out))
    return out


def verify_fp8(q, k_codes, v_codes, k_scale, v_scale, prefix_page_table, draft_page_table,
               prefix_lens, topk: int, S: int, H_q: int, H_kv: int,
               scale: Optional[float] = None, part: str = "full",
               rows: Optional[Sequence[int]] = None, threads: int = 0):
    """fp64 verify over E4M3 K/V pools; ``k_scale`` / ``v_scale`` hold 1 value or [H_kv, d]."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float64).reshape(-1)
    vs = np.ascontiguousarray(v_scale, dtype=np.float64).reshape(-1)
    d = int(q.shape[-1])
    if ks.size != vs.size or ks.size not in (1, H_kv * d):
        raise ValueError("scales must hold 1 or H_kv * d values")
    ppt = np.ascontiguousarray(prefix_page_table, dtype=np.int32)
    dpt = np.ascontiguousarray(draft_page_table, dtype=np.int32)
    lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    B = int(lens.shape[0])
    P = int(kc.shape[1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r, rp, nr = _rows_arg(rows)
    n = nr if r is not None else B * topk * S * H_q
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    err = lib.oracle_verify_fp8(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                                int(ks.size > 1), int(kc.shape[0]), _ptr(ppt), int(ppt.shape[1]),
                                _ptr(dpt), int(dpt.shape[1]), _ptr(lens), B, topk, S, H_q, H_kv,
                                d, P, PART_CODES[part], float(scale), rp, nr, _ptr(o), _ptr(lse),
                                threads)
    if err:
        raise ValueError(f"oracle_verify_fp8: {_ERR.get(err, err)}")
    return o, lse


def verify_fp8_wl(wl, part: str = "full", rows=None, threads: int = 0):
    """``verify_fp8`` on a ``cpa_synth.make_verify_fp8`` workload."""
    return verify_fp8(wl.q, wl.k_pages, wl.v_pages, wl.k_scale, wl.v_scale,
                      wl.prefix_page_table, wl.draft_page_table, wl.prefix_lens, wl.topk, wl.S,
                      wl.H_q, wl.H_kv, part=part, rows=rows, threads=threads)


def ancestor_masks(parents) -> np.ndarray:
    """Ancestor-or-self bitmasks of BFS-flattened draft trees.

    ``parents`` is int ``[N]`` or ``[B, N]``: ``parents[i]`` is the BFS index
    of node i's parent, or -1 for a root (a node whose parent is the last
    prefix token).  BFS flattening lists every parent before its children, so
    ``parents[i] < i`` is required.  Returns uint64 of the same shape whose
    bit j is M[i, j]: 1 when j is i or an ancestor of i (KV-cache tutorial,
    section 8.2 tip box and Q14).  N <= 64.
    """
    par = np.asarray(parents, dtype=np.int64)
    flat = par.reshape(-1, par.shape[-1])
    N = flat.shape[1]
    if N < 1 or N > 64:
        raise ValueError("a tree has 1..64 nodes")
    out = np.zeros(flat.shape, dtype=np.uint64)
    for r in range(flat.shape[0]):
        for i in range(N):
            pi = int(flat[r, i])
            if pi < -1 or pi >= i:
                raise ValueError(f"parent of node {i} is {pi}: not a BFS-flattened tree")
            # A(i) = {i} together with A(parent(i)); the parent's set is already built
            mask = 1 << i
            if pi >= 0:
                mask |= int(out[r, pi])
            out[r, i] = np.uint64(mask)
    return out.reshape(par.shape)


def tree_verify(q, k_pages, v_pages, prefix_page_table, tree_page_table, prefix_lens, parents,
                H_q: int, H_kv: int, scale: Optional[float] = None, part: str = "full",
                rows: Optional[Sequence[int]] = None, threads: int = 0):
    """fp64 verify attention over general draft trees.

    ``parents`` int ``[B, N]`` (BFS order, see ``ancestor_masks``); ``q`` is
    ``[B*N, H_q, d]`` with token ``b*N + i`` node i of request b; tree node j
    of request b sits at logical position j of ``tree_page_table[b]``.  Rows
    are ``token * H_q + head``.  Returns (o [n_rows, d], lse [n_rows]).
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kp = np.ascontiguousarray(k_pages, dtype=np.uint16)
    vp = np.ascontiguousarray(v_pages, dtype=np.uint16)
    ppt = np.ascontiguousarray(prefix_page_table, dtype=np.int32)
    tpt = np.ascontiguousarray(tree_page_table, dtype=np.int32)
    lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    par = np.asarray(parents)
    B = int(lens.shape[0])
    N = int(par.shape[-1])
    masks = np.ascontiguousarray(ancestor_masks(par.reshape(B, N)).reshape(-1))
    d = int(q.shape[-1])
    P = int(kp.shape[1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r, rp, nr = _rows_arg(rows)
    n = nr if r is not None else B * N * H_q
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    err = lib.oracle_tree_verify(_ptr(q), _ptr(kp), _ptr(vp), int(kp.shape[0]), _ptr(ppt),
                                 int(ppt.shape[1]), _ptr(tpt), int(tpt.shape[1]), _ptr(lens),
                                 _ptr(masks), B, N, H_q, H_kv, d, P, PART_CODES[part],
                                 float(scale), rp, nr, _ptr(o), _ptr(lse), threads)
    if err:
        raise ValueError(f"oracle_tree_verify: {_ERR.get(err, err)}")
    return o, lse


def tree_verify_wl(wl, part: str = "full", rows=None, threads: int = 0):
    """``tree_verify`` on a ``cpa_synth.TreeWorkload``-shaped object."""
    return tree_verify(wl.q, wl.k_pages, wl.v_pages, wl.prefix_page_table, wl.tree_page_table,
                       wl.prefix_lens, wl.parents, wl.H_q, wl.H_kv, part=part, rows=rows,
                       threads=threads)


def prefill(q, k_pages, v_pages, page_table, B: int, N: int, H: int, H_q: int, H_kv: int,
            scale: Optional[float] = None, part: str = "full", rows=None, threads: int = 0):
    """fp64 prefix-hit prefill attention over suffix tokens ``b*M + i`` (M = N - H)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kp = np.ascontiguousarray(k_pages, dtype=np.uint16)
    vp = np.ascontiguousarray(v_pages, dtype=np.uint16)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    d = int(q.shape[-1])
    P = int(kp.shape[1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r, rp, nr = _rows_arg(rows)
    n = nr if r is not None else B * (N - H) * H_q
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    err = lib.oracle_prefill(_ptr(q), _ptr(kp), _ptr(vp), int(kp.shape[0]), _ptr(pt),
                             int(pt.shape[1]), B, N, H, H_q, H_kv, d, P, PART_CODES[part],
                             float(scale), rp, nr, _ptr(o), _ptr(lse), threads)
    if err:
        raise ValueError(f"oracle_prefill: {_ERR.get(err, err)}")
    return o, lse


def prefill_wl(wl, part: str = "full", rows=None, threads: int = 0):
    return prefill(wl.q, wl.k_pages, wl.v_pages, wl.page_table, wl.B, wl.N, wl.H, wl.H_q,
                   wl.H_kv, part=part, rows=rows, threads=threads)


def merge_state(o_a, lse_a, o_b, lse_b):
    """fp64 merge of two partial attentions by the LSE identity."""
    lib = _load()
    o_a = np.ascontiguousarray(o_a, dtype=np.float64)
    o_b = np.ascontiguousarray(o_b, dtype=np.float64)
    lse_a = np.ascontiguousarray(lse_a, dtype=np.float64)
    lse_b = np.ascontiguousarray(lse_b, dtype=np.float64)
    n = int(lse_a.size)
    d = int(o_a.size // max(n, 1)) if n else 0
    o = np.zeros_like(o_a)
    lse = np.zeros_like(lse_a)
    lib.oracle_merge_state(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), n, d, _ptr(o),
                           _ptr(lse))
    return o, lse


def kv_reads_naive(prefix_lens, topk: int, S: int) -> int:
    """KV tokens read when every branch is expanded into its own request.

    Enumerates the reads: virtual request (b, k) walks prefix positions
    0..L_b-1 and then its own drafts 0..S-1 (cascade page, "Naive Expand").
    """
    reads = 0
    for L in prefix_lens:
        for _k in range(topk):
            for _pos in range(int(L)):
                reads += 1
            for _j in range(S):
                reads += 1
    return reads


def kv_reads_cascade(prefix_lens, topk: int, S: int) -> int:
    """KV tokens read by cascade: each prefix once (Pass A), each branch's drafts once (Pass B)."""
    seen = set()
    reads = 0
    for b, L in enumerate(prefix_lens):
        for pos in range(int(L)):
            key = ("prefix", b, pos)
            assert key not in seen
            seen.add(key)
            reads += 1
        for k in range(topk):
            for j in range(S):
                key = ("draft", b, k, j)
                assert key not in seen
                seen.add(key)
                reads += 1
    return reads


def visible_pairs(N: int, H: int) -> int:
    """Count visible (suffix query, key) pairs of the prefix-hit causal mask by enumeration."""
    count = 0
    for qpos in range(H, N):          # suffix queries, 0-based absolute positions
        for kpos in range(N):
            if kpos <= qpos:
                count += 1
    return count


def visible_pairs_full(N: int) -> int:
    """Visible pairs of the no-hit causal prompt (the whole lower triangle), by enumeration."""
    return sum(1 for qpos in range(N) for kpos in range(N) if kpos <= qpos)
