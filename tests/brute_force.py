"""A second, independent fp64 attention for tiny inputs, in pure Python.

It is used only to pin the oracle.  Unlike the oracle it never touches a page
table: it works on the logical (de-paged) sequences that the input generator
keeps, expands KV heads to query heads by repetition (the repeat_interleave
grouping of the KV-cache tutorial, section 6.3), builds an explicit boolean
mask over the whole key sequence and takes softmax over full rows with
masked scores at -inf.
"""
from __future__ import annotations

import math

import numpy as np

from cpa_synth import f32_from_bf16_bits


def _f64(bits) -> np.ndarray:
    return f32_from_bf16_bits(np.asarray(bits)).astype(np.float64)


def _expand_heads(kv: np.ndarray, H_q: int) -> np.ndarray:
    """[n, H_kv, d] -> [n, H_q, d] by repeating each KV head H_q / H_kv times."""
    return np.repeat(kv, H_q // kv.shape[1], axis=1)


def _softmax_row(q, keys, vals, mask, scale):
    n = len(keys)
    scores = []
    for j in range(n):
        if mask[j]:
            scores.append(sum(float(a) * float(b) for a, b in zip(q, keys[j])) * scale)
        else:
            scores.append(-math.inf)
    m = max(scores) if n else -math.inf
    d = len(q)
    if m == -math.inf:
        return [0.0] * d, -math.inf
    w = [math.exp(s - m) if s != -math.inf else 0.0 for s in scores]
    z = sum(w)
    out = [0.0] * d
    for j in range(n):
        if w[j] != 0.0:
            for c in range(d):
                out[c] += w[j] / z * float(vals[j][c])
    return out, m + math.log(z)


def verify(wl, part: str = "full"):
    """Rows in oracle order: token (b*topk+k)*S+s, then head."""
    H_q, S, topk = wl.H_q, wl.S, wl.topk
    d = wl.head_dim
    scale = 1.0 / math.sqrt(d)
    q = _f64(wl.q)
    o_rows, lse_rows = [], []
    for b in range(wl.B):
        L = int(wl.prefix_lens[b])
        pk = _expand_heads(_f64(wl.prefix_k[b]), H_q)
        pv = _expand_heads(_f64(wl.prefix_v[b]), H_q)
        for k in range(topk):
            # the whole sequence a virtual request (b, k) would hold: prefix then its drafts
            dk = _expand_heads(_f64(wl.draft_k[b * topk + k]), H_q)
            dv = _expand_heads(_f64(wl.draft_v[b * topk + k]), H_q)
            seq_k = np.concatenate([pk, dk], axis=0)
            seq_v = np.concatenate([pv, dv], axis=0)
            for s in range(S):
                t = (b * topk + k) * S + s
                mask = [False] * (L + S)
                for j in range(L + S):
                    is_prefix = j < L
                    if part == "prefix":
                        mask[j] = is_prefix
                    elif part == "draft":
                        mask[j] = (not is_prefix) and (j - L) <= s
                    else:
                        mask[j] = is_prefix or (j - L) <= s
                for h in range(H_q):
                    o, lse = _softmax_row(q[t, h], seq_k[:, h], seq_v[:, h], mask, scale)
                    o_rows.append(o)
                    lse_rows.append(lse)
    return np.array(o_rows, dtype=np.float64).reshape(-1, d), np.array(lse_rows)


def prefill(wl, part: str = "full"):
    """Rows in oracle order: suffix token b*M+i, then head."""
    H_q, N, H = wl.H_q, wl.N, wl.H
    M = N - H
    d = wl.head_dim
    scale = 1.0 / math.sqrt(d)
    q = _f64(wl.q)
    o_rows, lse_rows = [], []
    for b in range(wl.B):
        sk = _expand_heads(_f64(wl.seq_k[b]), H_q)
        sv = _expand_heads(_f64(wl.seq_v[b]), H_q)
        for i in range(M):
            qpos = H + i
            mask = []
            for j in range(N):
                causal = j <= qpos
                if part == "rect":
                    mask.append(causal and j < H)
                elif part == "tri":
                    mask.append(causal and j >= H)
                else:
                    mask.append(causal)
            for h in range(H_q):
                o, lse = _softmax_row(q[b * M + i, h], sk[:, h], sv[:, h], mask, scale)
                o_rows.append(o)
                lse_rows.append(lse)
    return np.array(o_rows, dtype=np.float64).reshape(-1, d), np.array(lse_rows)


def attend_subset(q_vec, keys, vals, subset, scale):
    """Attention of one query over an arbitrary subset of key indices."""
    n = keys.shape[0]
    mask = [j in subset for j in range(n)]
    o, lse = _softmax_row(q_vec, keys, vals, mask, scale)
    return np.array(o), lse


def tree_visible(parents) -> np.ndarray:
    """Tree-attention mask, built top-down: M[i, j] = True iff i is j or lies below j.

    Children lists are read off the parent array and each node's subtree is
    walked from the node down, the reverse direction of the oracle's
    bottom-up ancestor sets.
    """
    N = len(parents)
    children = [[] for _ in range(N)]
    for i, p in enumerate(parents):
        if p >= 0:
            children[int(p)].append(i)
    vis = np.zeros((N, N), dtype=bool)
    for j in range(N):
        stack = [j]
        while stack:
            i = stack.pop()
            vis[i, j] = True
            stack.extend(children[i])
    return vis


def tree_verify(wl, part: str = "full"):
    """Rows in oracle order: token b*N+i, then head."""
    H_q, N = wl.H_q, wl.N
    d = wl.head_dim
    scale = 1.0 / math.sqrt(d)
    q = _f64(wl.q)
    o_rows, lse_rows = [], []
    for b in range(wl.B):
        L = int(wl.prefix_lens[b])
        vis = tree_visible([int(x) for x in wl.parents[b]])
        seq_k = np.concatenate([_expand_heads(_f64(wl.prefix_k[b]), H_q),
                                _expand_heads(_f64(wl.tree_k[b]), H_q)], axis=0)
        seq_v = np.concatenate([_expand_heads(_f64(wl.prefix_v[b]), H_q),
                                _expand_heads(_f64(wl.tree_v[b]), H_q)], axis=0)
        for i in range(N):
            mask = [False] * (L + N)
            for j in range(L + N):
                if j < L:
                    mask[j] = part != "draft"
                else:
                    mask[j] = part != "prefix" and bool(vis[i, j - L])
            for h in range(H_q):
                o, lse = _softmax_row(q[b * N + i, h], seq_k[:, h], seq_v[:, h], mask, scale)
                o_rows.append(o)
                lse_rows.append(lse)
    return np.array(o_rows, dtype=np.float64).reshape(-1, d), np.array(lse_rows)


def verify_shared(wl, part: str = "full"):
    """Multi-level verify on logical sequences; rows in oracle order."""
    H_q, S, topk = wl.H_q, wl.S, wl.topk
    d = wl.head_dim
    scale = 1.0 / math.sqrt(d)
    q = _f64(wl.q)
    R = wl.B // wl.n_groups
    Ls = wl.shared_len
    o_rows, lse_rows = [], []
    for b in range(wl.B):
        g = b // R
        L = int(wl.prefix_lens[b])
        for k in range(topk):
            # the sequence this branch would hold: shared prefix, own prefix, own drafts
            parts_k = [wl.shared_k[g], wl.prefix_k[b], wl.draft_k[b * topk + k]]
            parts_v = [wl.shared_v[g], wl.prefix_v[b], wl.draft_v[b * topk + k]]
            seq_k = np.concatenate([_expand_heads(_f64(x), H_q) for x in parts_k], axis=0)
            seq_v = np.concatenate([_expand_heads(_f64(x), H_q) for x in parts_v], axis=0)
            for s in range(S):
                t = (b * topk + k) * S + s
                mask = []
                for j in range(Ls + L + S):
                    if j < Ls:
                        mask.append(part in ("full", "prefix", "shared"))
                    elif j < Ls + L:
                        mask.append(part in ("full", "prefix", "own"))
                    else:
                        mask.append(part in ("full", "draft") and (j - Ls - L) <= s)
                for h in range(H_q):
                    o, lse = _softmax_row(q[t, h], seq_k[:, h], seq_v[:, h], mask, scale)
                    o_rows.append(o)
                    lse_rows.append(lse)
    return np.array(o_rows, dtype=np.float64).reshape(-1, d), np.array(lse_rows)
