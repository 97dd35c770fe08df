"""The static-scratch cascade verify (cpa_cascade_verify_noalloc).

Callers that cannot call cudaMalloc -- an engine that reserved its HBM for
the KV pool up front, a decode loop that cannot afford the allocator's
device-wide synchronisation, a plugin whose host owns all device memory --
use this entry point: its scratch is a fixed array inside the library, so
nothing is allocated per call.  It must give the same result as the
workspace-taking cpa_cascade_verify, call after call, although every call
reuses the same scratch.  This file is collected last on purpose.
"""
import pytest
import torch

import cascade_paged_attention_gb300 as cpa
import cpa_synth
from tests.gpu_util import TOL_LSE, TOL_O, VerifyDev

pytestmark = pytest.mark.gpu


def _max_diff(a, b):
    return float((a.float() - b.float()).abs().max())


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row(cuda_device):
    wl = cpa_synth.make_verify(**cpa_synth.VERIFY_CONFIGS["llama3_8b"])
    d = VerifyDev(wl)
    ref_o, ref_lse = cpa.cpa_cascade_verify(*d.args(), max_prefix_len=wl.max_prefix_len,
                                            check=True)
    torch.cuda.synchronize()
    ref_o, ref_lse = ref_o.clone(), ref_lse.clone()
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        cpa.cpa_cascade_verify_noalloc(*d.args(), o=o, lse=lse,
                                       max_prefix_len=wl.max_prefix_len, check=True)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())
        # within the tolerance of every other GPU test ...
        assert _max_diff(o, ref_o) <= TOL_O
        assert _max_diff(lse, ref_lse) <= TOL_LSE
        # ... and in fact bit for bit: the same kernel with the same work partition
        # and merge order, only the scratch memory differs
        assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))


def test_noalloc_reports_a_bad_page_through_its_status_word(cuda_device):
    wl = cpa_synth.make_verify(B=2, topk=2, S=3, H_q=8, H_kv=2, page_size=16,
                               prefix_lens=[40, 40], seed=60)
    good = int(wl.prefix_page_table[1, 1])
    wl.prefix_page_table[1, 1] = wl.num_pages + 5
    d = VerifyDev(wl)
    o = torch.empty_like(d.q)
    lse = torch.empty(d.q.shape[0], wl.H_q, dtype=torch.float32, device=cuda_device)
    cpa.cpa_cascade_verify_noalloc(*d.args(), o=o, lse=lse)
    st, word = cpa.cpa_noalloc_device_status()
    assert st == 5 and word & 1  # CPA_ERR_BAD_PAGE, CPA_DEV_BAD_PAGE
    with pytest.raises(cpa.CpaError):
        cpa.cpa_cascade_verify_noalloc(*d.args(), o=o, lse=lse, check=True)
    # the next clean call clears the word
    d.ppt[1, 1] = good
    cpa.cpa_cascade_verify_noalloc(*d.args(), o=o, lse=lse)
    assert cpa.cpa_noalloc_device_status() == (0, 0)


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_device):
    # a batch whose merge counters alone push the scratch need past the fixed
    # array: rejected on the host before anything is launched or read.  With
    # topk = 1 the cascade launch has as many work units as the general
    # workspace query assumes, so that query gives the size the call needs.
    topk, S, H_q, H_kv = 1, 1, 8, 8
    B = 1024
    while cpa.cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, 128, 16) <= 48 * 2**20:
        B *= 2
    assert B < 2**21
    q = torch.zeros(8, 16, dtype=torch.bfloat16, device=cuda_device)
    i = torch.zeros(8, dtype=torch.int32, device=cuda_device)
    lib = cpa.lib()
    p = lambda t: t.data_ptr()
    st = lib.cpa_cascade_verify_noalloc(p(q), p(q), p(q), p(i), 1, p(i), 1, p(i), B, topk, S,
                                        H_q, H_kv, 128, 16, 1, 16, 0.088, p(q), p(i), None)
    assert st == 3  # CPA_ERR_WORKSPACE
    assert cpa.cpa_status_string(st) == "workspace missing or too small"
    # a shape that fits is not rejected by the size check: a bad argument of
    # another kind reports its own error
    st = lib.cpa_cascade_verify_noalloc(p(q), p(q), p(q), p(i), 1, p(i), 1, p(i), 2, topk, S,
                                        H_q, H_kv, 96, 16, 1, 16, 0.088, p(q), p(i), None)
    assert st == 2  # CPA_ERR_UNSUPPORTED (head_dim 96)
