"""GPU parity of the FP8 KV-page path (cpa_cascade_verify_fp8,
cpa_cascade_pass_a_fp8) against the fp64 oracle over the same E4M3 codes
and scales (KV-cache tutorial, section 4.5 "FP8 KV").

Tolerance: the same max|do| <= 1e-2, max|dlse| <= 1e-3 as the bf16 path.  The
codes are exact on chip; what rounds is q * k_scale (once, to f16) and P
(f16), with fp32 accumulation.
"""
import numpy as np
import pytest
import torch

import cascade_paged_attention_gb300 as cpa
import cpa_synth
import oracle
from tests.gpu_util import compare, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


class Fp8Dev:
    def __init__(self, wl, device="cuda:0"):
        self.wl = wl
        self.q = dev_bf16(wl.q, device)
        self.k = torch.from_numpy(np.ascontiguousarray(wl.k_pages)).to(device)
        self.v = torch.from_numpy(np.ascontiguousarray(wl.v_pages)).to(device)
        self.ks = torch.from_numpy(np.ascontiguousarray(wl.k_scale, dtype=np.float32)).to(device)
        self.vs = torch.from_numpy(np.ascontiguousarray(wl.v_scale, dtype=np.float32)).to(device)
        self.ppt = dev_i32(wl.prefix_page_table, device)
        self.dpt = dev_i32(wl.draft_page_table, device)
        self.lens = dev_i32(wl.prefix_lens, device)

    def verify(self, **kw):
        wl = self.wl
        return cpa.cpa_cascade_verify_fp8(self.q, self.k, self.v, self.ks, self.vs, self.ppt,
                                          self.dpt, self.lens, wl.topk, wl.S,
                                          max_prefix_len=wl.max_prefix_len, check=True, **kw)

    def pass_a(self):
        wl = self.wl
        return cpa.cpa_cascade_pass_a_fp8(self.q, self.k, self.v, self.ks, self.vs, self.ppt,
                                          self.lens, wl.topk, wl.S,
                                          max_prefix_len=wl.max_prefix_len, check=True)


SMALL = {
    "tiny": dict(B=2, topk=2, S=3, L=64, H_q=8, H_kv=2, page_size=16, seed=71),
    "gqa_partial_page": dict(B=3, topk=3, S=2, H_q=8, H_kv=2, page_size=16,
                             prefix_lens=[100, 17, 64], seed=72),
    "mqa_empty_prefix": dict(B=3, topk=2, S=4, H_q=16, H_kv=1, page_size=32,
                             prefix_lens=[0, 300, 5], seed=73),
    "mha_pages8": dict(B=2, topk=1, S=1, H_q=4, H_kv=4, page_size=8, prefix_lens=[129, 1],
                       seed=74),
    "pages64": dict(B=2, topk=4, S=4, H_q=32, H_kv=8, page_size=64, prefix_lens=[700, 1500],
                    seed=75),
    "topk16_s5": dict(B=2, topk=16, S=5, H_q=8, H_kv=8, page_size=16,
                      prefix_lens=[200, 1000], seed=76),
    "topk8_s12": dict(B=2, topk=8, S=12, H_q=8, H_kv=8, page_size=16, prefix_lens=[300, 40],
                      seed=77),
}


@pytest.mark.parametrize("scales", ["tensor", "channel"])
@pytest.mark.parametrize("key", list(SMALL))
def test_fp8_cascade_verify_matches_oracle(cuda_device, key, scales):
    wl = cpa_synth.make_verify_fp8(scales=scales, **SMALL[key])
    d = Fp8Dev(wl)
    o, lse = d.verify()
    torch.cuda.synchronize()
    compare(o, lse, *oracle.verify_fp8_wl(wl))


@pytest.mark.parametrize("scales", ["tensor", "channel"])
@pytest.mark.parametrize("key", ["tiny", "gqa_partial_page", "mqa_empty_prefix", "pages64"])
def test_fp8_pass_a_matches_oracle(cuda_device, key, scales):
    wl = cpa_synth.make_verify_fp8(scales=scales, **SMALL[key])
    d = Fp8Dev(wl)
    o_a, lse_a = d.pass_a()
    torch.cuda.synchronize()
    compare(o_a, lse_a, *oracle.verify_fp8_wl(wl, part="prefix"))


@pytest.mark.parametrize("scales", ["tensor", "channel"])
@pytest.mark.parametrize("name", ["llama3_8b", "pages_example"])
def test_fp8_full_config_all_rows(cuda_device, name, scales):
    cfg = dict(cpa_synth.VERIFY_CONFIGS[name])
    wl = cpa_synth.make_verify_fp8(scales=scales, **cfg)
    d = Fp8Dev(wl)
    o, lse = d.verify()
    torch.cuda.synchronize()
    compare(o, lse, *oracle.verify_fp8_wl(wl))


def test_fp8_unused_slots_hold_nan_codes(cuda_device):
    """Slots past every sequence end hold the NaN code 0x7F: never seen by any row."""
    wl = cpa_synth.make_verify_fp8(B=4, topk=3, S=5, H_q=32, H_kv=8, page_size=16,
                                   prefix_lens=[1, 15, 17, 200], seed=78, scales="channel",
                                   pad_code=0x7F)
    d = Fp8Dev(wl)
    o, lse = d.verify()
    torch.cuda.synchronize()
    compare(o, lse, *oracle.verify_fp8_wl(wl))


def test_fp8_page_permutation_is_bit_exact(cuda_device):
    kw = dict(B=8, topk=4, S=3, H_q=32, H_kv=8, page_size=16, L=1000, seed=79,
              scales="channel")
    a = Fp8Dev(cpa_synth.make_verify_fp8(perm_seed=1, **kw))
    b = Fp8Dev(cpa_synth.make_verify_fp8(perm_seed=2, **kw))
    assert not torch.equal(a.ppt, b.ppt)
    oa, la = a.verify()
    ob, lb = b.verify()
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la.view(torch.int32), lb.view(torch.int32))


def test_fp8_unit_scales_equal_the_bf16_path_on_the_same_values(cuda_device):
    """Codes with unit scales are exactly representable in bf16: the FP8 call and
    the bf16 call on the decoded pools compute the same attention (within the
    tolerance: the two paths round P differently)."""
    wl = cpa_synth.make_verify_fp8(B=4, topk=4, S=5, H_q=32, H_kv=8, page_size=16, L=700,
                                   seed=80, scales="unit")
    d = Fp8Dev(wl)
    o8, l8 = d.verify()
    kb = torch.from_numpy(np.ascontiguousarray(wl.k_pages)).view(torch.float8_e4m3fn)
    vb = torch.from_numpy(np.ascontiguousarray(wl.v_pages)).view(torch.float8_e4m3fn)
    kb = kb.float().to(torch.bfloat16).to(cuda_device)
    vb = vb.float().to(torch.bfloat16).to(cuda_device)
    o16, l16 = cpa.cpa_cascade_verify(d.q, kb, vb, d.ppt, d.dpt, d.lens, wl.topk, wl.S,
                                      max_prefix_len=wl.max_prefix_len, check=True)
    torch.cuda.synchronize()
    assert float((o8.float() - o16.float()).abs().max()) <= 1e-2
    assert float((l8 - l16).abs().max()) <= 1e-3


def test_fp8_two_m_tiles_are_refused(cuda_device):
    wl = cpa_synth.make_verify_fp8(B=1, topk=8, S=4, H_q=64, H_kv=8, page_size=16, L=64,
                                   seed=81)
    d = Fp8Dev(wl)
    with pytest.raises(cpa.CpaError) as e:
        d.verify()
    assert e.value.status == 2  # CPA_ERR_UNSUPPORTED
