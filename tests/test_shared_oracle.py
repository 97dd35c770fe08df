"""Pins of the oracle's multi-level verify (a prefix shared by a group of requests).

The KV-cache tutorial's block-table example (section 5.3) has two requests
whose tables begin with the same physical pages; ``share_prefix`` (section
6.2) makes such tables by copying whole pages.  A request's keys are then the
shared prefix, its own prefix and its branch's drafts.  The pins: the pages'
two-request example, equality with the single-level ``verify`` on the
concatenated block table, brute force on logical data, and the merge of the
three pieces.
"""
import json
import os

import numpy as np
import pytest

import cpa_synth
import oracle
from tests import brute_force

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _concat_tables(wl):
    """Each request's single-level block table: its group's shared pages, then its own."""
    R = wl.B // wl.n_groups
    n_shared = wl.shared_page_table.shape[1]
    out = np.full((wl.B, n_shared + wl.prefix_page_table.shape[1]), -1, dtype=np.int32)
    for b in range(wl.B):
        out[b, :n_shared] = wl.shared_page_table[b // R]
        out[b, n_shared:] = wl.prefix_page_table[b]
    return out


def test_block_table_example_of_the_pages():
    """Requests A = [12, 7, 34, 19] and B = [12, 7, 5] share pages 12 and 7 (32 tokens)."""
    g = json.load(open(os.path.join(GOLDEN, "block_table_sharing.json")))
    P = g["page_size"]
    A, Bt = g["request_A_physical"], g["request_B_physical"]
    n_shared = g["shared_tokens"] // P
    assert A[:n_shared] == Bt[:n_shared] and A[n_shared] != Bt[n_shared]
    H_kv, H_q, d, topk, S = 1, 2, 16, 2, 3
    rng = np.random.default_rng(0)
    n_pages = 40
    bits = lambda shape: cpa_synth.bf16_bits_from_f32(rng.standard_normal(shape, dtype=np.float32))
    kp = bits((n_pages, P, H_kv, d))
    vp = bits((n_pages, P, H_kv, d))
    draft_pages = np.array([[30], [31], [32], [33]], dtype=np.int32)  # B*topk branches
    q = bits((2 * topk * S, H_q, d))
    # single level: each request's whole block table
    full_pt = np.full((2, 4), -1, dtype=np.int32)
    full_pt[0, :4] = A
    full_pt[1, :3] = Bt
    ref = oracle.verify(q, kp, vp, full_pt, draft_pages, [4 * P, 3 * P], topk, S, H_q, H_kv)
    # multi-level: the shared pages once for the group, then each request's own pages
    own = np.full((2, 2), -1, dtype=np.int32)
    own[0, :2] = A[n_shared:]
    own[1, :1] = Bt[n_shared:]
    got = oracle.verify_shared(q, kp, vp, np.array([A[:n_shared]], dtype=np.int32),
                               n_shared * P, own, draft_pages, [2 * P, 1 * P], topk, S, H_q,
                               H_kv)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])


@pytest.mark.parametrize("n_groups,shared_len", [(1, 32), (2, 48), (4, 16)])
def test_whole_page_sharing_equals_single_level_verify(n_groups, shared_len):
    wl = cpa_synth.make_shared_verify(B=4, n_groups=n_groups, shared_len=shared_len, topk=3, S=2,
                                      H_q=4, H_kv=2, head_dim=32, page_size=16,
                                      prefix_lens=[7, 0, 33, 16], seed=n_groups)
    lens = wl.prefix_lens + shared_len
    # shared_len is a multiple of the page size, so own position j is concatenated position
    # shared_len + j of the single-level table
    for part_ml, part_sl in (("full", "full"), ("prefix", "prefix"), ("draft", "draft")):
        got = oracle.verify_shared_wl(wl, part=part_ml)
        ref = oracle.verify(wl.q, wl.k_pages, wl.v_pages, _concat_tables(wl),
                            wl.draft_page_table, lens, wl.topk, wl.S, wl.H_q, wl.H_kv,
                            part=part_sl)
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_array_equal(got[1], ref[1])


@pytest.mark.parametrize("part", ["full", "prefix", "draft", "shared", "own"])
def test_shared_matches_brute_force(part):
    wl = cpa_synth.make_shared_verify(B=4, n_groups=2, shared_len=13, topk=2, S=3, H_q=4,
                                      H_kv=2, head_dim=16, page_size=4,
                                      prefix_lens=[5, 0, 9, 2], seed=3, keep_logical=True)
    o, lse = oracle.verify_shared_wl(wl, part=part)
    bo, blse = brute_force.verify_shared(wl, part=part)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, blse, rtol=0, atol=1e-12)


def test_three_pieces_merge_to_full():
    wl = cpa_synth.make_shared_verify(B=6, n_groups=3, shared_len=21, topk=2, S=4, H_q=4,
                                      H_kv=1, head_dim=32, page_size=8,
                                      prefix_lens=[3, 0, 40, 8, 1, 17], seed=5)
    sh = oracle.verify_shared_wl(wl, part="shared")
    ow = oracle.verify_shared_wl(wl, part="own")
    dr = oracle.verify_shared_wl(wl, part="draft")
    full = oracle.verify_shared_wl(wl)
    pre = oracle.merge_state(sh[0], sh[1], ow[0], ow[1])
    np.testing.assert_allclose(pre[0], oracle.verify_shared_wl(wl, part="prefix")[0], atol=1e-12,
                               rtol=0)
    o, lse = oracle.merge_state(pre[0], pre[1], dr[0], dr[1])
    np.testing.assert_allclose(o, full[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, full[1], rtol=0, atol=1e-12)


def test_empty_shared_prefix_is_single_level_verify():
    wl = cpa_synth.make_shared_verify(B=2, n_groups=1, shared_len=0, topk=2, S=2, H_q=2, H_kv=1,
                                      head_dim=16, page_size=4, prefix_lens=[6, 3], seed=6)
    got = oracle.verify_shared_wl(wl)
    ref = oracle.verify(wl.q, wl.k_pages, wl.v_pages, wl.prefix_page_table,
                        wl.draft_page_table, wl.prefix_lens, wl.topk, wl.S, wl.H_q, wl.H_kv)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])


def test_kv_reads_of_the_three_levels():
    """Unique KV of multi-level cascade: each shared prefix once per group, not per request."""
    wl = cpa_synth.make_shared_verify(**cpa_synth.SHARED_CONFIGS["shared_tiny"])
    per_request = int((wl.prefix_lens + wl.shared_len).sum()) + wl.B * wl.topk * wl.S
    assert wl.unique_kv_tokens() == per_request - (wl.B - wl.n_groups) * wl.shared_len
