"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: the pages' worked
numbers and figures (tests/golden/), closed forms, a library softmax /
scaled-dot-product attention in the special cases where the method reduces
to it, and a pure-Python brute force that never touches a page table.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import cpa_synth
import oracle
from tests import brute_force

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f64(bits):
    return cpa_synth.f32_from_bf16_bits(np.asarray(bits)).astype(np.float64)


TINY_VERIFY = [
    # (B, topk, S, H_q, H_kv, P, lens)
    (2, 2, 3, 4, 2, 4, [10, 7]),       # GQA, partial last page
    (1, 4, 3, 2, 1, 4, [8]),           # MQA, L a multiple of P, the pages' topk=4/S=3 shape
    (2, 1, 2, 2, 2, 8, [5, 0]),        # MHA, topk=1, an empty prefix
    (3, 3, 1, 4, 4, 2, [1, 4, 3]),     # S=1, tiny pages
]


@pytest.mark.parametrize("case", TINY_VERIFY)
@pytest.mark.parametrize("part", ["full", "prefix", "draft"])
def test_verify_matches_brute_force(case, part):
    B, topk, S, H_q, H_kv, P, lens = case
    wl = cpa_synth.make_verify(B=B, topk=topk, S=S, H_q=H_q, H_kv=H_kv, head_dim=16,
                               page_size=P, prefix_lens=lens, seed=11, keep_logical=True)
    o, lse = oracle.verify_wl(wl, part=part)
    ob, lseb = brute_force.verify(wl, part=part)
    assert o.shape == ob.shape
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    finite = np.isfinite(lseb)
    assert np.array_equal(finite, np.isfinite(lse))
    np.testing.assert_allclose(lse[finite], lseb[finite], rtol=0, atol=1e-12)
    assert np.all(lse[~finite] == -np.inf)


TINY_PREFILL = [
    # (B, N, H, H_q, H_kv, P)
    (2, 9, 4, 4, 2, 4),
    (1, 7, 0, 2, 1, 4),    # no hit: plain causal prompt
    (2, 6, 5, 2, 2, 2),    # a single suffix token
    (1, 10, 3, 4, 1, 8),   # hit not on a page boundary
]


@pytest.mark.parametrize("case", TINY_PREFILL)
@pytest.mark.parametrize("part", ["full", "rect", "tri"])
def test_prefill_matches_brute_force(case, part):
    B, N, H, H_q, H_kv, P = case
    wl = cpa_synth.make_prefill(B=B, N=N, H=H, H_q=H_q, H_kv=H_kv, head_dim=16, page_size=P,
                                seed=5, keep_logical=True)
    o, lse = oracle.prefill_wl(wl, part=part)
    ob, lseb = brute_force.prefill(wl, part=part)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    finite = np.isfinite(lseb)
    assert np.array_equal(finite, np.isfinite(lse))
    np.testing.assert_allclose(lse[finite], lseb[finite], rtol=0, atol=1e-12)


def test_full_visibility_is_textbook_softmax():
    """topk=1, S=1: each draft sees its whole sequence, so o = softmax(q K^T / sqrt d) V."""
    B, H_q, H_kv, d = 3, 4, 2, 32
    wl = cpa_synth.make_verify(B=B, topk=1, S=1, H_q=H_q, H_kv=H_kv, head_dim=d, page_size=4,
                               prefix_lens=[13, 1, 6], seed=3, keep_logical=True)
    o, lse = oracle.verify_wl(wl)
    q = torch.from_numpy(_f64(wl.q))                      # [B, H_q, d]
    for b in range(B):
        k = torch.from_numpy(np.concatenate([_f64(wl.prefix_k[b]), _f64(wl.draft_k[b])]))
        v = torch.from_numpy(np.concatenate([_f64(wl.prefix_v[b]), _f64(wl.draft_v[b])]))
        k = k.repeat_interleave(H_q // H_kv, dim=1).transpose(0, 1)   # [H_q, n, d]
        v = v.repeat_interleave(H_q // H_kv, dim=1).transpose(0, 1)
        scores = torch.einsum("hd,hnd->hn", q[b], k) / math.sqrt(d)
        ref = torch.einsum("hn,hnd->hd", torch.softmax(scores, dim=-1), v)
        ref_lse = torch.logsumexp(scores, dim=-1)
        np.testing.assert_allclose(o[b * H_q:(b + 1) * H_q], ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b * H_q:(b + 1) * H_q], ref_lse.numpy(), rtol=0,
                                   atol=1e-12)


def _sdpa_with_mask(q, k, v, mask):
    """fp64 torch scaled_dot_product_attention; q [Lq, H, d], k/v [Lk, H, d]."""
    out = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), attn_mask=mask)
    return out.transpose(0, 1)


@pytest.mark.parametrize("H", [0, 3, 8])
def test_prefill_is_library_causal_attention(H):
    """Suffix queries with the cached-prefill mask tril(ones(L_new, L_total), diagonal=L_total-L_new)."""
    N, H_q, H_kv, d = 12, 4, 2, 16
    wl = cpa_synth.make_prefill(B=2, N=N, H=H, H_q=H_q, H_kv=H_kv, head_dim=d, page_size=4,
                                seed=9, keep_logical=True)
    o, _ = oracle.prefill_wl(wl)
    M = N - H
    mask = torch.tril(torch.ones(M, N, dtype=torch.bool), diagonal=N - M)
    for b in range(2):
        q = torch.from_numpy(_f64(wl.q[b * M:(b + 1) * M]))
        k = torch.from_numpy(_f64(wl.seq_k[b])).repeat_interleave(H_q // H_kv, dim=1)
        v = torch.from_numpy(_f64(wl.seq_v[b])).repeat_interleave(H_q // H_kv, dim=1)
        ref = _sdpa_with_mask(q, k, v, mask)
        if H == 0:
            ref2 = torch.nn.functional.scaled_dot_product_attention(
                q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), is_causal=True
            ).transpose(0, 1)
            np.testing.assert_allclose(ref.numpy(), ref2.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(o[b * M * H_q:(b + 1) * M * H_q].reshape(M, H_q, d),
                                   ref.numpy(), rtol=0, atol=1e-12)


def test_topk1_equals_one_kvcache_call():
    """topk=1: one attention over L+S cached keys with a causal tail (cache_seqlens = L+S)."""
    L, S, H_q, H_kv, d = 9, 4, 4, 2, 16
    wl = cpa_synth.make_verify(B=1, topk=1, S=S, H_q=H_q, H_kv=H_kv, head_dim=d, page_size=4,
                               prefix_lens=[L], seed=21, keep_logical=True)
    o, _ = oracle.verify_wl(wl)
    k = np.concatenate([_f64(wl.prefix_k[0]), _f64(wl.draft_k[0])])
    v = np.concatenate([_f64(wl.prefix_v[0]), _f64(wl.draft_v[0])])
    k = torch.from_numpy(k).repeat_interleave(H_q // H_kv, dim=1)
    v = torch.from_numpy(v).repeat_interleave(H_q // H_kv, dim=1)
    mask = torch.tril(torch.ones(S, L + S, dtype=torch.bool), diagonal=L)
    ref = _sdpa_with_mask(torch.from_numpy(_f64(wl.q)), k, v, mask)
    np.testing.assert_allclose(o.reshape(S, H_q, d), ref.numpy(), rtol=0, atol=1e-12)


def test_merge_identity_on_random_splits():
    """merge_state(attn(A), attn(B)) == attn(A u B) for disjoint A, B (cascade page)."""
    rng = np.random.default_rng(0)
    d = 8
    for trial in range(40):
        n = int(rng.integers(1, 12))
        q = rng.standard_normal(d) * 2
        keys = rng.standard_normal((n, d)) * 2
        vals = rng.standard_normal((n, d))
        members = rng.integers(0, 2, size=n)
        if trial % 10 == 0:
            members[:] = 0          # A empty
        elif trial % 10 == 1:
            members[:] = 1          # B empty
        A = {j for j in range(n) if members[j] == 1}
        Bset = {j for j in range(n) if members[j] == 0}
        scale = 1 / math.sqrt(d)
        oa, la = brute_force.attend_subset(q, keys, vals, A, scale)
        ob, lb = brute_force.attend_subset(q, keys, vals, Bset, scale)
        of, lf = brute_force.attend_subset(q, keys, vals, A | Bset, scale)
        om, lm = oracle.merge_state(oa[None], np.array([la]), ob[None], np.array([lb]))
        np.testing.assert_allclose(om[0], of, rtol=0, atol=1e-12)
        assert abs(lm[0] - lf) < 1e-12


def test_merge_edge_cases():
    d = 4
    x = np.arange(d, dtype=np.float64)[None]
    y = -np.ones((1, d))
    # one side empty returns the other side exactly
    o, l = oracle.merge_state(x, np.array([-np.inf]), y, np.array([0.3]))
    assert np.array_equal(o, y) and l[0] == 0.3
    o, l = oracle.merge_state(x, np.array([1.7]), y, np.array([-np.inf]))
    assert np.array_equal(o, x) and l[0] == 1.7
    # both empty: zero output, -inf, no NaN
    o, l = oracle.merge_state(x, np.array([-np.inf]), y, np.array([-np.inf]))
    assert np.array_equal(o, np.zeros((1, d))) and l[0] == -np.inf
    # huge gaps do not overflow
    o, l = oracle.merge_state(x, np.array([1000.0]), y, np.array([-1000.0]))
    np.testing.assert_allclose(o, x, atol=1e-300)
    assert abs(l[0] - 1000.0) < 1e-12
    # equal halves average
    o, l = oracle.merge_state(x, np.array([2.0]), y, np.array([2.0]))
    np.testing.assert_allclose(o, (x + y) / 2, atol=1e-15)
    assert abs(l[0] - (2.0 + math.log(2))) < 1e-15


@pytest.mark.parametrize("kind", ["verify", "prefill"])
def test_parts_merge_to_full(kind):
    """Pass A + Pass B (or rectangle + triangle) merged equals the full attention."""
    if kind == "verify":
        wl = cpa_synth.make_verify(B=2, topk=3, S=4, H_q=4, H_kv=2, head_dim=32, page_size=4,
                                   prefix_lens=[9, 0], seed=2)
        a = oracle.verify_wl(wl, part="prefix")
        b = oracle.verify_wl(wl, part="draft")
        f = oracle.verify_wl(wl, part="full")
    else:
        wl = cpa_synth.make_prefill(B=2, N=11, H=5, H_q=4, H_kv=2, head_dim=32, page_size=4,
                                    seed=2)
        a = oracle.prefill_wl(wl, part="rect")
        b = oracle.prefill_wl(wl, part="tri")
        f = oracle.prefill_wl(wl, part="full")
    o, lse = oracle.merge_state(a[0], a[1], b[0], b[1])
    np.testing.assert_allclose(o, f[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, f[1], rtol=0, atol=1e-12)


def _one_hot_bits(n, d):
    """bf16 bits of one-hot rows: key j gets a 1.0 in dimension j."""
    v = np.zeros((n, 1, d), dtype=np.uint16)
    for j in range(n):
        v[j, 0, j] = 0x3F80
    return v


def test_branch_mask_matches_page_figure():
    """With q = 0 every visible key gets equal weight; one-hot V rows reveal the visible set."""
    g = _golden("branch_visibility.json")
    topk, S, L = g["topk"], g["S"], 5
    d = L + topk * S
    ids = np.arange(d)
    # key ids: prefix position p -> p; draft (k, j) -> L + k*S + j
    pk = [np.zeros((L, 1, d), np.uint16)]
    pv = [_one_hot_bits(d, d)[:L]]
    dk, dv = [], []
    for k in range(topk):
        dk.append(np.zeros((S, 1, d), np.uint16))
        dv.append(_one_hot_bits(d, d)[L + k * S: L + (k + 1) * S])
    rng = np.random.default_rng(4)
    kp, vp, tabs = cpa_synth.build_pool(pk + dk, pv + dv, 2, rng)
    ppt = cpa_synth.table_matrix(tabs[:1], (L + 1) // 2)
    dpt = cpa_synth.table_matrix(tabs[1:], (S + 1) // 2)
    q = np.zeros((topk * S, 1, d), np.uint16)
    o, lse = oracle.verify(q, kp, vp, ppt, dpt, [L], topk, S, 1, 1)
    for k in range(topk):
        for j in range(S):
            row = o[k * S + j]
            vis = set(ids[row > 0].tolist())
            want = set(range(L)) | {L + kk * S + jj for kk, jj in g["visible_drafts"][f"d_{k}{j}"]}
            assert vis == want
            np.testing.assert_allclose(row[row > 0], 1.0 / len(want), rtol=0, atol=1e-15)
            assert abs(lse[k * S + j] - math.log(len(want))) < 1e-15


def test_prefix_hit_mask_matches_page_figure():
    g = _golden("prefix_hit_8tok.json")
    N, H = g["N"], g["H"]
    d = N
    seq_k = [np.zeros((N, 1, d), np.uint16)]
    seq_v = [_one_hot_bits(N, d)]
    kp, vp, tabs = cpa_synth.build_pool(seq_k, seq_v, 4, np.random.default_rng(1))
    pt = cpa_synth.table_matrix(tabs, N // 4)
    M = N - H
    q = np.zeros((M, 1, d), np.uint16)
    o, lse = oracle.prefill(q, kp, vp, pt, 1, N, H, 1, 1)
    vis = (o > 0).astype(int)
    assert vis.tolist() == g["suffix_visible"]
    assert int(vis.sum()) == g["W_hit"]
    o_r, _ = oracle.prefill(q, kp, vp, pt, 1, N, H, 1, 1, part="rect")
    o_t, _ = oracle.prefill(q, kp, vp, pt, 1, N, H, 1, 1, part="tri")
    assert int((o_r > 0).sum()) == g["rectangle"]
    assert int((o_t > 0).sum()) == g["triangle"]
    np.testing.assert_allclose(lse, np.log(vis.sum(axis=1)), rtol=0, atol=1e-15)


def test_kv_reads_worked_example():
    g = _golden("cascade_kv_reads.json")["worked_example"]
    naive = oracle.kv_reads_naive([g["L"]], g["topk"], g["S"])
    casc = oracle.kv_reads_cascade([g["L"]], g["topk"], g["S"])
    assert naive == g["naive_tokens_per_request"] == 8020
    assert casc == g["cascade_tokens_per_request"] == 2020
    assert 3.9 < naive / casc < 4.0


def test_kv_reads_closed_forms():
    rng = np.random.default_rng(1)
    for _ in range(20):
        B = int(rng.integers(1, 6))
        topk = int(rng.integers(1, 6))
        S = int(rng.integers(1, 6))
        L = int(rng.integers(0, 60))
        lens = [L] * B
        assert oracle.kv_reads_naive(lens, topk, S) == B * topk * (L + S)
        assert oracle.kv_reads_cascade(lens, topk, S) == B * L + B * topk * S
    # variable lengths: the same formulas summed per request
    lens = [3, 17, 0, 9]
    assert oracle.kv_reads_naive(lens, 3, 2) == sum(3 * (L + 2) for L in lens)
    assert oracle.kv_reads_cascade(lens, 3, 2) == sum(L + 3 * 2 for L in lens)


def test_w_hit_closed_forms_by_enumeration():
    for N in range(0, 65):
        assert oracle.visible_pairs_full(N) == N * (N + 1) // 2
        for H in range(0, N + 1):
            M = N - H
            w = oracle.visible_pairs(N, H)
            assert w == (N * (N + 1) - H * (H + 1)) // 2
            assert w == M * H + M * (M + 1) // 2
    g = _golden("prefix_hit_8tok.json")
    assert oracle.visible_pairs(g["N"], g["H"]) == g["W_hit"]
    assert oracle.visible_pairs_full(g["N"]) == g["W_0"]


def test_hit_ratio_example():
    g = _golden("hit_ratio.json")
    N = 8192
    H = int(g["h"] * N)
    exact = 1 - H * (H + 1) / (N * (N + 1))
    assert abs(exact - g["dense_causal_remaining"]) < 1e-4
    assert abs((1 - g["h"]) - g["token_linear_remaining"]) < 1e-15
    # spot-check the exact ratio against enumeration at a size that enumerates fast
    n, h = 200, 100
    assert oracle.visible_pairs(n, h) / oracle.visible_pairs_full(n) == pytest.approx(
        1 - h * (h + 1) / (n * (n + 1)), abs=0)


def test_page_permutation_does_not_change_result():
    kw = dict(B=2, topk=2, S=3, H_q=4, H_kv=2, head_dim=32, page_size=4, prefix_lens=[11, 6],
              seed=8)
    a = cpa_synth.make_verify(perm_seed=1, **kw)
    b = cpa_synth.make_verify(perm_seed=2, **kw)
    assert not np.array_equal(a.prefix_page_table, b.prefix_page_table)
    oa, la = oracle.verify_wl(a)
    ob, lb = oracle.verify_wl(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_row_subset_matches_full_rows():
    wl = cpa_synth.make_verify(B=2, topk=2, S=2, H_q=4, H_kv=1, head_dim=16, page_size=4,
                               prefix_lens=[7, 3], seed=6)
    o, lse = oracle.verify_wl(wl)
    rows = [0, 5, 13, 31]
    os_, ls_ = oracle.verify_wl(wl, rows=rows)
    assert np.array_equal(os_, o[rows]) and np.array_equal(ls_, lse[rows])


def test_bad_page_id_is_reported():
    wl = cpa_synth.make_verify(B=1, topk=1, S=1, H_q=2, H_kv=1, head_dim=16, page_size=4,
                               prefix_lens=[6], seed=6)
    wl.prefix_page_table[0, 1] = wl.num_pages + 3
    with pytest.raises(ValueError, match="page id"):
        oracle.verify_wl(wl)
