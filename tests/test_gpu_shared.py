"""GPU parity of multi-level cascade verify (cpa_cascade_verify_shared) against the fp64 oracle.

Same tolerances as the other verify calls: max|do| <= 1e-2, max|dlse| <= 1e-3;
page-table indexing bit-exact under a different physical page permutation.
"""
import pytest
import torch

import cascade_paged_attention_gb300 as cpa
import cpa_synth
import oracle
from tests.gpu_util import compare, dev_bf16, dev_i32, sample_rows

pytestmark = pytest.mark.gpu


class SharedDev:
    def __init__(self, wl, device="cuda:0"):
        self.wl = wl
        self.q = dev_bf16(wl.q, device)
        self.k = dev_bf16(wl.k_pages, device)
        self.v = dev_bf16(wl.v_pages, device)
        self.spt = dev_i32(wl.shared_page_table, device)
        self.ppt = dev_i32(wl.prefix_page_table, device)
        self.dpt = dev_i32(wl.draft_page_table, device)
        self.lens = dev_i32(wl.prefix_lens, device)

    def call(self, **kw):
        wl = self.wl
        return cpa.cpa_cascade_verify_shared(self.q, self.k, self.v, self.spt, wl.shared_len,
                                             self.ppt, self.dpt, self.lens, wl.topk, wl.S,
                                             max_prefix_len=wl.max_prefix_len, **kw)


SMALL_SHARED = {
    "tiny": dict(cpa_synth.SHARED_CONFIGS["shared_tiny"]),
    # one system prompt for 8 requests: 160 queries in one group, 5 q tiles
    "one_group": dict(B=8, n_groups=1, shared_len=1024, topk=4, S=5, H_q=32, H_kv=8,
                      page_size=16, prefix_lens=[976, 0, 13, 500, 976, 1, 700, 129], seed=81),
    # shared length not a page multiple, MQA, an empty own prefix
    "ragged_shared_mqa": dict(B=6, n_groups=3, shared_len=333, topk=2, S=3, H_q=16, H_kv=1,
                              page_size=32, prefix_lens=[0, 47, 300, 2, 64, 0], seed=82),
    # 256-row own units (two M tiles), G = 8, large pages
    "two_mtiles_p64": dict(B=4, n_groups=2, shared_len=700, topk=8, S=4, H_q=64, H_kv=8,
                           page_size=64, prefix_lens=[200, 1500, 0, 64], seed=83),
    "no_shared": dict(B=4, n_groups=2, shared_len=0, topk=3, S=2, H_q=8, H_kv=2, page_size=16,
                      prefix_lens=[100, 17, 0, 64], seed=84),
    # whole shared pages (one launch) with two M tiles, groups of two requests
    "paged_two_mtiles": dict(B=6, n_groups=3, shared_len=640, topk=8, S=4, H_q=64, H_kv=8,
                             page_size=64, prefix_lens=[0, 1000, 64, 333, 1, 700], seed=85),
    # whole shared pages, ragged own prefixes, one M tile, GQA 4
    "paged_ragged_own": dict(B=6, n_groups=2, shared_len=128, topk=3, S=4, H_q=16, H_kv=4,
                             page_size=16, prefix_lens=[5, 0, 250, 127, 128, 1], seed=86),
}


def test_shared_paths_cover_both_schedules():
    """Whole shared pages take the one-launch schedule, a shared prefix that
    ends inside a page the two-launch one: both are among the cases above."""
    aligned = [k for k, c in SMALL_SHARED.items()
               if c["shared_len"] > 0 and c["shared_len"] % c["page_size"] == 0]
    ragged = [k for k, c in SMALL_SHARED.items() if c["shared_len"] % c["page_size"] != 0]
    assert len(aligned) >= 2 and len(ragged) >= 2


@pytest.mark.parametrize("key", list(SMALL_SHARED))
def test_shared_verify_matches_oracle(cuda_device, key):
    wl = cpa_synth.make_shared_verify(**SMALL_SHARED[key])
    d = SharedDev(wl)
    o, lse = d.call()
    torch.cuda.synchronize()
    compare(o, lse, *oracle.verify_shared_wl(wl))


def test_shared_verify_full_size_sampled_rows(cuda_device):
    wl = cpa_synth.make_shared_verify(**cpa_synth.SHARED_CONFIGS["shared_pages_example"])
    d = SharedDev(wl)
    n_rows = wl.n_tokens * wl.H_q
    rows = sample_rows(n_rows, 2048, seed=6, always=[0, n_rows - 1, 20 * wl.H_q - 1])
    o, lse = d.call()
    torch.cuda.synchronize()
    compare(o, lse, *oracle.verify_shared_wl(wl, rows=rows), rows=rows)


def test_shared_page_permutation_is_bit_exact(cuda_device):
    kw = dict(SMALL_SHARED["one_group"])
    kw.pop("seed")
    a = SharedDev(cpa_synth.make_shared_verify(seed=85, perm_seed=1, **kw))
    b = SharedDev(cpa_synth.make_shared_verify(seed=85, perm_seed=2, **kw))
    assert not torch.equal(a.spt, b.spt)
    oa, la = a.call()
    oa, la = oa.clone(), la.clone()
    ob, lb = b.call()
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la.view(torch.int32), lb.view(torch.int32))


def test_bad_shared_page_is_reported(cuda_device):
    """The first launch's status bit survives the second launch of the call."""
    wl = cpa_synth.make_shared_verify(**SMALL_SHARED["tiny"])
    wl.shared_page_table[1, 0] = wl.num_pages + 3
    d = SharedDev(wl)
    nbytes = cpa.cpa_cascade_verify_shared_workspace_size(wl.B, wl.n_groups, wl.topk, wl.S,
                                                          wl.H_q, wl.H_kv, 128, wl.page_size)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=cuda_device)
    d.call(workspace=ws)
    st, word = cpa.cpa_get_device_status(ws)
    assert st == 5 and word & 1
