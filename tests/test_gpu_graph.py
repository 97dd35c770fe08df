"""Verify replayed from one captured CUDA graph while the page tables, prefix
lengths, queries and KV pool change in place between replays.

This is how a decode loop runs the call (KV-cache tutorial, section 5.2:
the block table is what changes from step to step; the cascade page's
topk = 1 case is plain decode over L + S keys).  The call takes no host
synchronisation and reads every length and page id on the device, so one
capture serves every step whose lengths stay within max_prefix_len.
"""
import numpy as np
import pytest
import torch

import cascade_paged_attention_gb300 as cpa
import cpa_synth
import oracle
from tests.gpu_util import compare

pytestmark = pytest.mark.gpu


def _static_buffers(wls, device):
    """Device buffers big enough for every workload of the list."""
    w0 = wls[0]
    n_pages = max(w.num_pages for w in wls)
    ppt_w = max(w.prefix_page_table.shape[1] for w in wls)
    dpt_w = max(w.draft_page_table.shape[1] for w in wls)
    P, H_kv, d = w0.page_size, w0.H_kv, w0.head_dim
    bufs = dict(
        q=torch.zeros(w0.q.shape, dtype=torch.bfloat16, device=device),
        k=torch.zeros((n_pages, P, H_kv, d), dtype=torch.bfloat16, device=device),
        v=torch.zeros((n_pages, P, H_kv, d), dtype=torch.bfloat16, device=device),
        ppt=torch.full((w0.B, ppt_w), -1, dtype=torch.int32, device=device),
        dpt=torch.full((w0.B * w0.topk, dpt_w), -1, dtype=torch.int32, device=device),
        lens=torch.zeros(w0.B, dtype=torch.int32, device=device),
    )
    return bufs, n_pages


def _load(bufs, wl):
    """Copy one workload into the static buffers (in place, same addresses)."""
    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16)

    bufs["q"].copy_(bf(wl.q))
    bufs["k"][:wl.num_pages].copy_(bf(wl.k_pages))
    bufs["v"][:wl.num_pages].copy_(bf(wl.v_pages))
    bufs["ppt"].fill_(-1)
    bufs["ppt"][:, :wl.prefix_page_table.shape[1]].copy_(torch.from_numpy(wl.prefix_page_table))
    bufs["dpt"].fill_(-1)
    bufs["dpt"][:, :wl.draft_page_table.shape[1]].copy_(torch.from_numpy(wl.draft_page_table))
    bufs["lens"].copy_(torch.from_numpy(wl.prefix_lens))


@pytest.mark.parametrize("topk,S", [(1, 1), (4, 5)])
def test_graph_replay_with_in_place_updates(cuda_device, topk, S):
    B, H_q, H_kv, P, max_len = 8, 32, 8, 16, 1200
    rng = np.random.default_rng(90 + topk)
    steps = []
    for s in range(4):
        lens = rng.integers(0, max_len + 1, size=B)
        lens[0] = max_len if s == 0 else lens[0]  # the largest pool first
        steps.append(cpa_synth.make_verify(B=B, topk=topk, S=S, H_q=H_q, H_kv=H_kv,
                                           page_size=P, prefix_lens=lens, seed=200 + s))
    bufs, n_pages = _static_buffers(steps, cuda_device)
    o = torch.empty_like(bufs["q"])
    lse = torch.empty(bufs["q"].shape[0], H_q, dtype=torch.float32, device=cuda_device)
    ws = torch.zeros(cpa.cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, 128, P),
                     dtype=torch.uint8, device=cuda_device)

    def call():
        cpa.cpa_cascade_verify(bufs["q"], bufs["k"], bufs["v"], bufs["ppt"], bufs["dpt"],
                               bufs["lens"], topk, S, max_prefix_len=max_len, o=o, lse=lse,
                               workspace=ws)

    _load(bufs, steps[0])
    call()  # outside capture first: loads the library and sets kernel attributes
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
        st, word = cpa.cpa_get_device_status(ws)
        assert st == 0 and word == 0
