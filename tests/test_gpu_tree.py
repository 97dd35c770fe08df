"""GPU parity of draft-tree verify (cpa_tree_verify, cpa_tree_pass_b) against the fp64 oracle.

Same tolerances as the chain verify: max|do| <= 1e-2, max|dlse| <= 1e-3;
page-table indexing bit-exact (two physical page permutations give the same
output bits).
"""
import numpy as np
import pytest
import torch

import cascade_paged_attention_gb300 as cpa
import cpa_synth
import oracle
from tests.gpu_util import TreeDev, VerifyDev, compare, dev_bf16, dev_i32, sample_rows

pytestmark = pytest.mark.gpu

SMALL_TREES = {
    "tiny": dict(cpa_synth.TREE_CONFIGS["tree_tiny"]),
    # forest of 3 roots, partial last prefix page, an empty prefix
    "forest_partial_page": dict(B=3, N=23, H_q=8, H_kv=2, page_size=16,
                                prefix_lens=[100, 0, 37], n_roots=3, seed=71),
    # 64 nodes (the widest mask) with G = 4: 256 query rows, two M tiles in the prefix pass
    "n64_two_mtiles": dict(B=2, N=64, H_q=8, H_kv=2, page_size=16, prefix_lens=[500, 129],
                           seed=72),
    # MQA, large pages, a tree that spans several tree pages
    "mqa_pages8": dict(B=2, N=40, H_q=4, H_kv=1, page_size=8, prefix_lens=[77, 8], n_roots=2,
                       seed=73),
    "pages64_g8": dict(B=2, N=20, H_q=64, H_kv=8, page_size=64, prefix_lens=[1000, 64],
                       seed=74),
    "single_node": dict(B=3, N=1, H_q=32, H_kv=8, page_size=16, prefix_lens=[16, 1, 0],
                        seed=75),
}


def _tree(key, **over):
    spec = dict(SMALL_TREES[key])
    spec.update(over)
    return cpa_synth.make_tree_verify(**spec)


@pytest.mark.parametrize("key", list(SMALL_TREES))
def test_tree_verify_matches_oracle(cuda_device, key):
    wl = _tree(key)
    d = TreeDev(wl)
    o, lse = cpa.cpa_tree_verify(*d.args(), max_prefix_len=wl.max_prefix_len)
    torch.cuda.synchronize()
    compare(o, lse, *oracle.tree_verify_wl(wl))


@pytest.mark.parametrize("key", ["tiny", "forest_partial_page", "n64_two_mtiles", "mqa_pages8"])
def test_tree_pass_b_matches_oracle(cuda_device, key):
    wl = _tree(key)
    d = TreeDev(wl)
    o_b, lse_b = cpa.cpa_tree_pass_b(d.q, d.k, d.v, d.tpt, d.parents)
    torch.cuda.synchronize()
    compare(o_b, lse_b, *oracle.tree_verify_wl(wl, part="draft"))


def test_tree_prefix_part_matches_oracle(cuda_device):
    """The prefix pass of a tree is Pass A with the N nodes as one query block."""
    wl = _tree("n64_two_mtiles")
    d = TreeDev(wl)
    o_a, lse_a = cpa.cpa_cascade_pass_a(d.q, d.k, d.v, d.ppt, d.lens, 1, wl.N,
                                        max_prefix_len=wl.max_prefix_len)
    torch.cuda.synchronize()
    compare(o_a, lse_a, *oracle.tree_verify_wl(wl, part="prefix"))


def test_chain_forest_tree_equals_cascade_verify(cuda_device):
    """topk chains given as a tree agree with the chain-per-branch cascade kernel."""
    topk, S = 4, 5
    vw = cpa_synth.make_verify(B=4, topk=topk, S=S, H_q=32, H_kv=8, page_size=16, L=300,
                               seed=76, keep_logical=True)
    B, N = vw.B, topk * S
    bfs = [(s, k) for s in range(S) for k in range(topk)]
    tk = [np.stack([vw.draft_k[b * topk + k][s] for s, k in bfs]) for b in range(B)]
    tv = [np.stack([vw.draft_v[b * topk + k][s] for s, k in bfs]) for b in range(B)]
    kp, vp, tabs = cpa_synth.build_pool(vw.prefix_k + tk, vw.prefix_v + tv, 16,
                                        np.random.default_rng(3))
    ppt = cpa_synth.table_matrix(tabs[:B], (300 + 15) // 16)
    tpt = cpa_synth.table_matrix(tabs[B:], (N + 15) // 16)
    chain_tok = np.array([(b * topk + k) * S + s for b in range(B) for s, k in bfs])
    par = np.ascontiguousarray(np.broadcast_to(cpa_synth.chain_forest(topk, S), (B, N)))
    o, lse = cpa.cpa_tree_verify(dev_bf16(vw.q[chain_tok]), dev_bf16(kp), dev_bf16(vp),
                                 dev_i32(ppt), dev_i32(tpt), dev_i32(vw.prefix_lens),
                                 dev_i32(par))
    vd = VerifyDev(vw)
    co, cl = cpa.cpa_cascade_verify(*vd.args())
    torch.cuda.synchronize()
    idx = torch.as_tensor(chain_tok, device=cuda_device)
    assert (o.float() - co[idx].float()).abs().max().item() <= 1e-2
    assert (lse - cl[idx]).abs().max().item() <= 1e-3
    # and both against the chain oracle
    rows = (chain_tok[:, None] * vw.H_q + np.arange(vw.H_q)[None, :]).reshape(-1)
    ref_o, ref_l = oracle.verify_wl(vw)
    compare(o, lse, ref_o[rows], ref_l[rows])


def test_tree_page_permutation_is_bit_exact(cuda_device):
    kw = dict(B=4, N=30, H_q=32, H_kv=8, page_size=16, L=700, n_roots=2, seed=77)
    a = TreeDev(cpa_synth.make_tree_verify(perm_seed=1, **kw))
    b = TreeDev(cpa_synth.make_tree_verify(perm_seed=2, **kw))
    assert not torch.equal(a.ppt, b.ppt)
    oa, la = cpa.cpa_tree_verify(*a.args())
    oa, la = oa.clone(), la.clone()
    ob, lb = cpa.cpa_tree_verify(*b.args())
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la.view(torch.int32), lb.view(torch.int32))


def test_unused_tree_slots_are_never_read(cuda_device):
    wl = cpa_synth.make_tree_verify(B=3, N=21, H_q=32, H_kv=8, page_size=16,
                                    prefix_lens=[1, 17, 200], n_roots=2, seed=78,
                                    pad_fill="nan")
    d = TreeDev(wl)
    o, lse = cpa.cpa_tree_verify(*d.args())
    torch.cuda.synchronize()
    compare(o, lse, *oracle.tree_verify_wl(wl))


@pytest.mark.parametrize("name", ["tree_pages_example", "tree_60"])
def test_tree_full_size_sampled_rows(cuda_device, name):
    wl = cpa_synth.make_tree_verify(**cpa_synth.TREE_CONFIGS[name])
    d = TreeDev(wl)
    n_rows = wl.n_tokens * wl.H_q
    rows = sample_rows(n_rows, 2048, seed=5,
                       always=[0, n_rows - 1, wl.N * wl.H_q - 1, wl.N * wl.H_q])
    ref = oracle.tree_verify_wl(wl, rows=rows)
    o, lse = cpa.cpa_tree_verify(*d.args(), max_prefix_len=wl.max_prefix_len)
    torch.cuda.synchronize()
    compare(o, lse, *ref, rows=rows)


def test_bad_tree_parent_is_reported(cuda_device):
    wl = _tree("tiny")
    wl.parents[1, 3] = 5  # a parent after its child
    d = TreeDev(wl)
    ws = torch.zeros(cpa.cpa_tree_verify_workspace_size(wl.B, wl.N, wl.H_q, wl.H_kv, 128, 16),
                     dtype=torch.uint8, device=cuda_device)
    cpa.cpa_tree_verify(*d.args(), workspace=ws)
    st, word = cpa.cpa_get_device_status(ws)
    assert st == 9 and word & 8
    d.parents.copy_(dev_i32(_tree("tiny").parents))
    o, lse = cpa.cpa_tree_verify(*d.args(), workspace=ws)
    st, word = cpa.cpa_get_device_status(ws)
    assert st == 0 and word == 0
    compare(o, lse, *oracle.tree_verify_wl(_tree("tiny")))


def test_bad_tree_page_is_reported(cuda_device):
    wl = _tree("forest_partial_page")
    wl.tree_page_table[2, 1] = wl.num_pages
    d = TreeDev(wl)
    ws = torch.zeros(cpa.cpa_status_workspace_size(), dtype=torch.uint8, device=cuda_device)
    cpa.cpa_tree_pass_b(d.q, d.k, d.v, d.tpt, d.parents, workspace=ws)
    st, word = cpa.cpa_get_device_status(ws)
    assert st == 5 and word & 1


def test_tree_host_checks(cuda_device):
    wl = _tree("tiny")
    d = TreeDev(wl)
    with pytest.raises(cpa.CpaError) as e:  # 65 nodes
        big = cpa_synth.make_tree_verify(B=1, N=64, H_q=2, H_kv=2, page_size=16, L=16, seed=1)
        bd = TreeDev(big)
        par = torch.cat([bd.parents, bd.parents[:, :1]], dim=1)
        q = torch.cat([bd.q, bd.q[:1]], dim=0)
        tpt = torch.cat([bd.tpt, bd.tpt[:, :1]], dim=1)
        cpa.cpa_tree_verify(q, bd.k, bd.v, bd.ppt, tpt, bd.lens, par,
                            workspace=torch.zeros(1 << 20, dtype=torch.uint8, device=cuda_device))
    assert e.value.status == 2
    with pytest.raises(cpa.CpaError) as e:  # tree table too narrow
        cpa.cpa_tree_verify(d.q, d.k, d.v, d.ppt, d.tpt[:, :0].contiguous(), d.lens, d.parents)
    assert e.value.status == 1
