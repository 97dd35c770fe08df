"""The static-scratch cascade verify (cpa_cascade_verify_noalloc).

Callers that cannot call cudaMalloc -- an engine that reserved its HBM for
the KV pool up front, a decode loop that cannot afford the allocator's
device-wide synchronisation, a plugin whose host owns all device memory --
use this entry point: its scratch is a fixed array inside the library, so
nothing is allocated per call.  It must give the same result as the
workspace-taking cpa_cascade_verify, call after call, although every call
reuses the same scratch.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import cascade_paged_attention_gb300 as cpa
import cpa_synth
import oracle
from tests.gpu_util import TOL_LSE, TOL_O, VerifyDev, compare
from tests.test_gpu_graph import _load, _static_buffers

pytestmark = pytest.mark.gpu


def _max_diff(a, b):
    return float((a.float() - b.float()).abs().max())


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row(cuda_device):
    wl = cpa_synth.make_verify(**cpa_synth.VERIFY_CONFIGS["llama3_8b"])
    d = VerifyDev(wl)
    ref_o, ref_lse = cpa.cpa_cascade_verify(*d.args(), max_prefix_len=wl.max_prefix_len)
    torch.cuda.synchronize()
    ref_o, ref_lse = ref_o.clone(), ref_lse.clone()
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        cpa.cpa_cascade_verify_noalloc(*d.args(), o=o, lse=lse,
                                       max_prefix_len=wl.max_prefix_len)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())
        assert _max_diff(o, ref_o) <= TOL_O
        assert _max_diff(lse, ref_lse) <= TOL_LSE


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_device):
    # a batch whose merge counters alone push the workspace past the fixed scratch:
    # rejected on the host before anything is launched or read
    topk, S, H_q, H_kv = 4, 1, 8, 8
    B = 1024
    while cpa.cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, 128, 16) <= 48 * 2**20:
        B *= 2
    assert B < 2**22
    q = torch.zeros(8, 16, dtype=torch.bfloat16, device=cuda_device)
    i = torch.zeros(8, dtype=torch.int32, device=cuda_device)
    lib = cpa.lib()
    p = lambda t: t.data_ptr()
    st = lib.cpa_cascade_verify_noalloc(p(q), p(q), p(q), p(i), 1, p(i), 1, p(i), B, topk, S,
                                        H_q, H_kv, 128, 16, 1, 16, 0.088, p(q), p(i), None)
    assert st == 3  # CPA_ERR_WORKSPACE
    assert cpa.cpa_status_string(st) == "workspace missing or too small"


def test_noalloc_graph_replay(cuda_device):
    """The static-scratch call captured once and replayed over new lengths."""
    B, topk, S, H_q, H_kv, P, max_len = 4, 2, 3, 16, 4, 16, 600
    steps = [cpa_synth.make_verify(B=B, topk=topk, S=S, H_q=H_q, H_kv=H_kv, page_size=P,
                                   prefix_lens=lens, seed=300 + i)
             for i, lens in enumerate([[600, 1, 0, 333], [17, 600, 250, 5]])]
    bufs, _ = _static_buffers(steps, cuda_device)
    o = torch.empty_like(bufs["q"])
    lse = torch.empty(bufs["q"].shape[0], H_q, dtype=torch.float32, device=cuda_device)

    def call():
        cpa.cpa_cascade_verify_noalloc(bufs["q"], bufs["k"], bufs["v"], bufs["ppt"], bufs["dpt"],
                                       bufs["lens"], topk, S, o, lse, max_prefix_len=max_len)

    _load(bufs, steps[0])
    call()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    for wl in steps:
        _load(bufs, wl)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        compare(o, lse, *oracle.verify_wl(wl))
