"""Pins of the oracle's draft-tree verify.

Tree attention (KV-cache tutorial, section 8.2 tip box and Q14): the draft
tree is flattened in BFS order, A(i) is node i's ancestors together with i,
and node i attends key j of the tree iff j is in A(i), on top of the whole
prefix.  Each test ties the oracle to something other than itself: a
hand-drawn tree, a top-down construction of the mask, a pure-Python brute
force on logical (de-paged) data, and the two special cases that reduce to
functions pinned elsewhere (a forest of chains is chain-per-branch verify; a
single chain is prefix-hit prefill).
"""
import json
import math
import os

import numpy as np
import pytest

import cpa_synth
import oracle
from tests import brute_force

# A small Medusa-style static tree, drawn by hand:
#
#            0
#          /   \
#         1     2
#        / \     \
#       3   4     5
#       |
#       6
HAND_PARENTS = [-1, 0, 0, 1, 1, 2, 3]
HAND_ANCESTORS = [{0}, {0, 1}, {0, 2}, {0, 1, 3}, {0, 1, 4}, {0, 2, 5}, {0, 1, 3, 6}]


def _bits_to_sets(masks, N):
    return [{j for j in range(N) if (int(m) >> j) & 1} for m in masks]


def test_ancestor_masks_hand_drawn_tree():
    got = _bits_to_sets(oracle.ancestor_masks(HAND_PARENTS), len(HAND_PARENTS))
    assert got == HAND_ANCESTORS


def test_branch_example_of_the_pages_as_a_forest():
    """The cascade page's 4 branches of 3 drafts, flattened in BFS order, give its visible sets."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "branch_visibility.json")))
    topk, S = g["topk"], g["S"]
    masks = oracle.ancestor_masks(cpa_synth.chain_forest(topk, S))
    node = lambda k, j: j * topk + k  # BFS: level j holds draft j of every branch
    for k in range(topk):
        for j in range(S):
            want = {node(kk, jj) for kk, jj in g["visible_drafts"][f"d_{k}{j}"]}
            assert _bits_to_sets([masks[node(k, j)]], topk * S)[0] == want


def test_ancestor_masks_of_a_chain_are_causal():
    """On a single chain the tree mask is the lower-triangular causal mask (Q14)."""
    N = 64
    masks = oracle.ancestor_masks([-1] + list(range(N - 1)))
    for i, m in enumerate(masks):
        assert _bits_to_sets([m], N)[0] == set(range(i + 1))


@pytest.mark.parametrize("seed", range(6))
def test_ancestor_masks_agree_with_top_down_construction(seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(1, 65))
    par = cpa_synth.random_bfs_tree(rng, N, n_roots=int(rng.integers(1, min(N, 4) + 1)))
    vis = brute_force.tree_visible([int(x) for x in par])
    masks = oracle.ancestor_masks(par)
    for i in range(N):
        assert _bits_to_sets([masks[i]], N)[0] == set(np.nonzero(vis[i])[0].tolist())
    # one bit per tree level on the path: |A(i)| = depth(i) + 1
    depth = [0] * N
    for i in range(N):
        depth[i] = 0 if par[i] < 0 else depth[par[i]] + 1
        assert bin(int(masks[i])).count("1") == depth[i] + 1


def test_ancestor_masks_reject_a_parent_after_its_child():
    with pytest.raises(ValueError):
        oracle.ancestor_masks([-1, 2, 0])
    with pytest.raises(ValueError):
        oracle.ancestor_masks([0])
    with pytest.raises(ValueError):
        oracle.ancestor_masks([-1] * 65)


def test_random_bfs_tree_is_bfs_ordered():
    rng = np.random.default_rng(7)
    for _ in range(20):
        N = int(rng.integers(1, 65))
        par = cpa_synth.random_bfs_tree(rng, N, n_roots=1)
        assert par[0] == -1 and (par[1:] >= 0).all()
        assert (par[1:] < np.arange(1, N)).all()
        assert (np.diff(par[1:]) >= 0).all()  # children of earlier nodes come first


def _one_hot_bits(n, d):
    v = np.zeros((n, 1, d), dtype=np.uint16)
    for j in range(n):
        v[j, 0, j] = 0x3F80
    return v


def test_hand_drawn_tree_visible_sets():
    """q = 0 gives every visible key the same weight; one-hot V rows reveal the set."""
    N, L = len(HAND_PARENTS), 3
    d = L + N
    pv = [_one_hot_bits(d, d)[:L]]
    tv = [_one_hot_bits(d, d)[L:]]
    pk = [np.zeros((L, 1, d), np.uint16)]
    tk = [np.zeros((N, 1, d), np.uint16)]
    kp, vp, tabs = cpa_synth.build_pool(pk + tk, pv + tv, 2, np.random.default_rng(5))
    ppt = cpa_synth.table_matrix(tabs[:1], 2)
    tpt = cpa_synth.table_matrix(tabs[1:], 4)
    q = np.zeros((N, 1, d), np.uint16)
    o, lse = oracle.tree_verify(q, kp, vp, ppt, tpt, [L], [HAND_PARENTS], 1, 1)
    for i in range(N):
        vis = set(np.nonzero(o[i] > 0)[0].tolist())
        want = set(range(L)) | {L + j for j in HAND_ANCESTORS[i]}
        assert vis == want
        np.testing.assert_allclose(o[i][o[i] > 0], 1.0 / len(want), rtol=0, atol=1e-15)
        assert abs(lse[i] - math.log(len(want))) < 1e-15


TINY_TREES = [
    # (B, N, H_q, H_kv, P, lens, n_roots)
    (2, 7, 4, 2, 4, [10, 7], 1),
    (1, 9, 2, 1, 4, [8], 3),
    (2, 5, 2, 2, 8, [5, 0], 2),
]


@pytest.mark.parametrize("case", TINY_TREES)
@pytest.mark.parametrize("part", ["full", "prefix", "draft"])
def test_tree_verify_matches_brute_force(case, part):
    B, N, H_q, H_kv, P, lens, n_roots = case
    wl = cpa_synth.make_tree_verify(B=B, N=N, H_q=H_q, H_kv=H_kv, head_dim=16, page_size=P,
                                    prefix_lens=lens, n_roots=n_roots, seed=N,
                                    keep_logical=True)
    o, lse = oracle.tree_verify_wl(wl, part=part)
    bo, blse = brute_force.tree_verify(wl, part=part)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, blse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("topk,S", [(4, 5), (3, 2), (1, 6)])
def test_forest_of_chains_is_chain_per_branch_verify(topk, S):
    """topk chains of S drafts flattened in BFS order give the chain verify result exactly."""
    vw = cpa_synth.make_verify(B=2, topk=topk, S=S, H_q=4, H_kv=2, head_dim=32, page_size=4,
                               prefix_lens=[9, 4], seed=3, keep_logical=True)
    B, N, H_q = vw.B, topk * S, vw.H_q
    # draft s of branch k becomes BFS node s*topk + k
    bfs = [(s, k) for s in range(S) for k in range(topk)]
    tk = [np.stack([vw.draft_k[b * topk + k][s] for s, k in bfs]) for b in range(B)]
    tv = [np.stack([vw.draft_v[b * topk + k][s] for s, k in bfs]) for b in range(B)]
    kp, vp, tabs = cpa_synth.build_pool(vw.prefix_k + tk, vw.prefix_v + tv, 4,
                                        np.random.default_rng(9))
    ppt = cpa_synth.table_matrix(tabs[:B], 3)
    tpt = cpa_synth.table_matrix(tabs[B:], (N + 3) // 4)
    chain_tok = [(b * topk + k) * S + s for b in range(B) for s, k in bfs]
    q = vw.q[chain_tok]
    par = np.broadcast_to(cpa_synth.chain_forest(topk, S), (B, N))
    for part in ("full", "prefix", "draft"):
        o, lse = oracle.tree_verify(q, kp, vp, ppt, tpt, vw.prefix_lens, par, H_q, vw.H_kv,
                                    part=part)
        co, clse = oracle.verify_wl(vw, part=part)
        rows = (np.asarray(chain_tok)[:, None] * H_q + np.arange(H_q)[None, :]).reshape(-1)
        np.testing.assert_array_equal(o, co[rows])
        np.testing.assert_array_equal(lse, clse[rows])


def test_single_chain_is_prefix_hit_prefill():
    """One chain of n nodes after an L-token prefix is the causal suffix of an L+n prefill."""
    B, n, L, P, H_q, H_kv = 2, 11, 16, 8, 4, 2
    wl = cpa_synth.make_tree_verify(B=B, N=n, H_q=H_q, H_kv=H_kv, head_dim=32, page_size=P, L=L,
                                    parents=[-1] + list(range(n - 1)), seed=21)
    o, lse = oracle.tree_verify_wl(wl)
    # L is a multiple of P, so logical position L + j is tree page j // P, slot j % P
    pt = np.concatenate([wl.prefix_page_table, wl.tree_page_table], axis=1)
    po, plse = oracle.prefill(wl.q, wl.k_pages, wl.v_pages, pt, B, L + n, L, H_q, H_kv)
    np.testing.assert_array_equal(o, po)
    np.testing.assert_array_equal(lse, plse)


def test_tree_parts_merge_to_full():
    wl = cpa_synth.make_tree_verify(B=3, N=13, H_q=4, H_kv=2, head_dim=32, page_size=4,
                                    prefix_lens=[9, 0, 17], n_roots=2, seed=4)
    a = oracle.tree_verify_wl(wl, part="prefix")
    b = oracle.tree_verify_wl(wl, part="draft")
    f = oracle.tree_verify_wl(wl, part="full")
    o, lse = oracle.merge_state(a[0], a[1], b[0], b[1])
    np.testing.assert_allclose(o, f[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, f[1], rtol=0, atol=1e-12)
    # an empty prefix leaves Pass A empty: lse = -inf, o = 0
    rows0 = slice(13 * 4, 26 * 4)
    assert np.all(np.isneginf(a[1][rows0])) and not np.any(a[0][rows0])


def test_tree_page_permutation_does_not_change_result():
    kw = dict(B=2, N=10, H_q=4, H_kv=2, head_dim=32, page_size=4, prefix_lens=[13, 6], seed=8)
    a = oracle.tree_verify_wl(cpa_synth.make_tree_verify(perm_seed=1, **kw))
    b = oracle.tree_verify_wl(cpa_synth.make_tree_verify(perm_seed=2, **kw))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_tree_bad_page_is_reported():
    wl = cpa_synth.make_tree_verify(B=1, N=4, H_q=2, H_kv=1, head_dim=16, page_size=4, L=4,
                                    seed=1)
    wl.tree_page_table[0, 0] = wl.num_pages
    with pytest.raises(ValueError):
        oracle.tree_verify_wl(wl)
