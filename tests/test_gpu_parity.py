"""GPU parity: every entry point of libcpa.so against the fp64 oracle.

Tolerance (bf16 inputs, fp32 accumulation): max|do| <= 1e-2, max|dlse| <= 1e-3;
page-table indexing is checked bit-exactly (same logical data under two
physical page permutations gives identical output bits).
"""
import numpy as np
import pytest
import torch

import cascade_paged_attention_gb300 as cpa
import cpa_synth
import oracle
from tests.gpu_util import PrefillDev, VerifyDev, compare, dev_bf16, sample_rows

pytestmark = pytest.mark.gpu


def _verify_wl(name, **over):
    cfg = dict(cpa_synth.VERIFY_CONFIGS[name])
    cfg.update(over)
    return cpa_synth.make_verify(**cfg)


SMALL_VERIFY = {
    "tiny": dict(name="tiny"),
    "gqa_partial_page": dict(B=3, topk=3, S=2, H_q=8, H_kv=2, page_size=16,
                             prefix_lens=[100, 17, 64], seed=31),
    "mqa_empty_prefix": dict(B=3, topk=2, S=4, H_q=16, H_kv=1, page_size=32,
                             prefix_lens=[0, 300, 5], seed=32),
    "mha_pages8": dict(B=2, topk=1, S=1, H_q=4, H_kv=4, page_size=8, prefix_lens=[129, 1],
                       seed=33),
    "two_mtiles": dict(B=2, topk=8, S=4, H_q=64, H_kv=8, page_size=64,
                       prefix_lens=[700, 1500], seed=34),
    "pages128": dict(B=2, topk=2, S=3, H_q=32, H_kv=8, page_size=128,
                     prefix_lens=[1000, 257], seed=35),
    # the widest draft tiles: 16 branches of 8-row blocks, 8 branches of 16-row blocks
    "topk16_s5": dict(B=2, topk=16, S=5, H_q=8, H_kv=8, page_size=16,
                      prefix_lens=[200, 1000], seed=36),
    "topk8_s12_two_mtiles": dict(B=2, topk=8, S=12, H_q=16, H_kv=8, page_size=16,
                                 prefix_lens=[300, 40], seed=37),
    # 64 units of 17 tiles over about 7 tiles per CTA (152 SMs): units split over
    # three or four CTAs, so the final merges take two or three other parts, the
    # staged (one bulk copy per part) and the unstaged forms
    "split3": dict(B=8, topk=4, S=5, H_q=32, H_kv=8, page_size=16,
                   prefix_lens=[2000, 1999, 2000, 1873, 2000, 2000, 1024, 2000], seed=38),
}


def _make_small(key, **over):
    spec = dict(SMALL_VERIFY[key])
    if "name" in spec:
        return _verify_wl(spec.pop("name"), **over)
    spec.update(over)
    return cpa_synth.make_verify(**spec)


# ------------------------------------------------------------------ merge_state
def test_merge_state_matches_oracle(cuda_device):
    rng = np.random.default_rng(0)
    n, H, d = 257, 8, 128
    # partial outputs are convex combinations of V rows ~ N(0, 1): keep them in that range,
    # where the final bf16 rounding (half an ulp) stays below the 1e-2 tolerance
    o_a = np.clip(rng.standard_normal((n, H, d)) * 0.5, -1.9, 1.9)
    o_b = np.clip(rng.standard_normal((n, H, d)) * 0.5, -1.9, 1.9)
    lse_a = rng.standard_normal((n, H)) * 3
    lse_b = rng.standard_normal((n, H)) * 3
    lse_a[0, :] = -np.inf                       # empty A
    lse_b[1, :] = -np.inf                       # empty B
    lse_a[2, :] = -np.inf
    lse_b[2, :] = -np.inf                       # both empty
    lse_a[3, :] = 80.0
    lse_b[3, :] = -80.0                         # huge gap
    ref_o, ref_l = oracle.merge_state(o_a.reshape(-1, d), lse_a.reshape(-1),
                                      o_b.reshape(-1, d), lse_b.reshape(-1))
    t = lambda a: torch.tensor(a, dtype=torch.float32, device=cuda_device)
    o, lse = cpa.cpa_merge_state(t(o_a), t(lse_a), t(o_b), t(lse_b))
    torch.cuda.synchronize()
    compare(o, lse, ref_o, ref_l)
    assert torch.all(o.float()[2] == 0)


# ------------------------------------------------------------------ Pass B
@pytest.mark.parametrize("key", ["tiny", "gqa_partial_page", "mqa_empty_prefix", "two_mtiles"])
def test_pass_b_matches_oracle(cuda_device, key):
    wl = _make_small(key)
    d = VerifyDev(wl)
    o_b, lse_b = cpa.cpa_cascade_pass_b(d.q, d.k, d.v, d.dpt, wl.B, wl.topk, wl.S, check=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.verify_wl(wl, part="draft")
    compare(o_b, lse_b, ref_o, ref_l)


# ------------------------------------------------------------------ Pass A
@pytest.mark.parametrize("key", list(SMALL_VERIFY))
def test_pass_a_matches_oracle(cuda_device, key):
    wl = _make_small(key)
    d = VerifyDev(wl)
    o_a, lse_a = cpa.cpa_cascade_pass_a(d.q, d.k, d.v, d.ppt, d.lens, wl.topk, wl.S,
                                        max_prefix_len=wl.max_prefix_len, check=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.verify_wl(wl, part="prefix")
    compare(o_a, lse_a, ref_o, ref_l)


# ------------------------------------------------------------------ cascade verify
@pytest.mark.parametrize("key", list(SMALL_VERIFY))
def test_cascade_verify_matches_oracle(cuda_device, key):
    wl = _make_small(key)
    d = VerifyDev(wl)
    o, lse = cpa.cpa_cascade_verify(*d.args(), max_prefix_len=wl.max_prefix_len, check=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.verify_wl(wl)
    compare(o, lse, ref_o, ref_l)


@pytest.mark.parametrize("key", list(SMALL_VERIFY))
def test_naive_expand_matches_oracle(cuda_device, key):
    wl = _make_small(key)
    d = VerifyDev(wl)
    o, lse = cpa.cpa_naive_expand_verify(*d.args(), max_prefix_len=wl.max_prefix_len,
                                         check=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.verify_wl(wl)
    compare(o, lse, ref_o, ref_l)


def test_pass_a_b_merge_composition(cuda_device):
    """Pass A, Pass B and merge_state as three calls equal the fused cascade."""
    wl = _make_small("gqa_partial_page")
    d = VerifyDev(wl)
    o_a, l_a = cpa.cpa_cascade_pass_a(d.q, d.k, d.v, d.ppt, d.lens, wl.topk, wl.S)
    o_b, l_b = cpa.cpa_cascade_pass_b(d.q, d.k, d.v, d.dpt, wl.B, wl.topk, wl.S)
    o, lse = cpa.cpa_merge_state(o_a, l_a, o_b, l_b)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.verify_wl(wl)
    compare(o, lse, ref_o, ref_l)


def test_unused_page_slots_are_never_read(cuda_device):
    """Slots past every sequence end are NaN: results must stay finite and correct."""
    wl = cpa_synth.make_verify(B=4, topk=3, S=5, H_q=32, H_kv=8, page_size=16,
                               prefix_lens=[1, 15, 17, 200], seed=40, pad_fill="nan")
    d = VerifyDev(wl)
    ref = oracle.verify_wl(wl)
    for fn in (cpa.cpa_cascade_verify, cpa.cpa_naive_expand_verify):
        o, lse = fn(*d.args())
        torch.cuda.synchronize()
        compare(o, lse, *ref)
    o_a, l_a = cpa.cpa_cascade_pass_a(d.q, d.k, d.v, d.ppt, d.lens, wl.topk, wl.S)
    torch.cuda.synchronize()
    compare(o_a, l_a, *oracle.verify_wl(wl, part="prefix"))


def test_page_permutation_is_bit_exact(cuda_device):
    kw = dict(B=8, topk=4, S=3, H_q=32, H_kv=8, page_size=16, L=1000, seed=41)
    a = VerifyDev(cpa_synth.make_verify(perm_seed=1, **kw))
    b = VerifyDev(cpa_synth.make_verify(perm_seed=2, **kw))
    assert not torch.equal(a.ppt, b.ppt)
    for fn in (cpa.cpa_cascade_verify, cpa.cpa_naive_expand_verify):
        oa, la = fn(*a.args())
        ob, lb = fn(*b.args())
        torch.cuda.synchronize()
        assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
        assert torch.equal(la.view(torch.int32), lb.view(torch.int32))


def test_repeated_calls_are_deterministic(cuda_device):
    wl = _make_small("two_mtiles")
    d = VerifyDev(wl)
    o1, l1 = cpa.cpa_cascade_verify(*d.args())
    o1 = o1.clone()
    l1 = l1.clone()
    o2, l2 = cpa.cpa_cascade_verify(*d.args())
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


# ------------------------------------------------------------------ full-size configs
@pytest.mark.parametrize("name", ["llama3_8b", "pages_example"])
def test_full_config_all_rows(cuda_device, name):
    wl = _verify_wl(name)
    d = VerifyDev(wl)
    ref = oracle.verify_wl(wl)
    o, lse = cpa.cpa_cascade_verify(*d.args(), max_prefix_len=wl.max_prefix_len, check=True)
    torch.cuda.synchronize()
    compare(o, lse, *ref)
    o, lse = cpa.cpa_naive_expand_verify(*d.args(), max_prefix_len=wl.max_prefix_len,
                                         check=True)
    torch.cuda.synchronize()
    compare(o, lse, *ref)


@pytest.mark.slow
def test_long_variable_config_all_rows(cuda_device):
    """Config 4 (per-request L uniform in [1024, 32768], two M tiles): every row."""
    wl = _verify_wl("long_variable")
    d = VerifyDev(wl)
    ref = oracle.verify_wl(wl)
    o, lse = cpa.cpa_cascade_verify(*d.args(), max_prefix_len=wl.max_prefix_len, check=True)
    torch.cuda.synchronize()
    compare(o, lse, *ref)
    o, lse = cpa.cpa_naive_expand_verify(*d.args(), max_prefix_len=wl.max_prefix_len,
                                         check=True)
    torch.cuda.synchronize()
    compare(o, lse, *ref)


# ------------------------------------------------------------------ prefix-hit prefill
PREFILL_SMALL = [
    dict(B=2, N=300, H=0, H_q=8, H_kv=2, page_size=16, seed=51),
    dict(B=2, N=300, H=128, H_q=8, H_kv=2, page_size=16, seed=52),
    dict(B=1, N=333, H=201, H_q=32, H_kv=8, page_size=16, seed=53),
    dict(B=3, N=97, H=96, H_q=4, H_kv=4, page_size=8, seed=54),
]


@pytest.mark.parametrize("cfg", PREFILL_SMALL)
@pytest.mark.parametrize("part", [cpa.PREFILL_FULL, cpa.PREFILL_RECT, cpa.PREFILL_TRI])
def test_prefill_hit_matches_oracle(cuda_device, cfg, part):
    wl = cpa_synth.make_prefill(**cfg)
    d = PrefillDev(wl)
    o, lse = cpa.cpa_prefill_hit(d.q, d.k, d.v, d.pt, wl.B, wl.N, wl.H, part=part, check=True)
    torch.cuda.synchronize()
    ref = oracle.prefill_wl(wl, part={0: "full", 1: "rect", 2: "tri"}[part])
    compare(o, lse, *ref)


def test_prefill_rect_tri_merge_equals_full(cuda_device):
    wl = cpa_synth.make_prefill(B=2, N=520, H=260, H_q=8, H_kv=2, page_size=16, seed=55)
    d = PrefillDev(wl)
    o_r, l_r = cpa.cpa_prefill_hit(d.q, d.k, d.v, d.pt, wl.B, wl.N, wl.H, part=cpa.PREFILL_RECT)
    o_t, l_t = cpa.cpa_prefill_hit(d.q, d.k, d.v, d.pt, wl.B, wl.N, wl.H, part=cpa.PREFILL_TRI)
    o, lse = cpa.cpa_merge_state(o_r, l_r, o_t, l_t)
    torch.cuda.synchronize()
    compare(o, lse, *oracle.prefill_wl(wl))


def prefill_check_rows(B, M, H, H_q, H_kv, seed, per_request=256):
    """Rows (token * H_q + head) checked at the full prefill size.

    Every request: `per_request` random suffix tokens with all H_q heads, plus
    its first and last suffix token.  One (request, KV head) group -- the last
    request, the last KV head -- additionally gets, for all of its heads, the
    first and last token of every q tile (so both members of every dealt pair
    (j, QT-1-j)) and the tokens whose key range ends on a 128-key tile boundary
    (the diagonal rows of the masked tiles).
    """
    G = H_q // H_kv
    TS = 128 // G
    rng = np.random.default_rng(seed)
    toks = set()
    for b in range(B):
        pick = rng.choice(M, size=min(per_request, M), replace=False)
        toks.update(int(b * M + i) for i in pick)
        toks.update((b * M, b * M + M - 1))
    rows = set(t * H_q + h for t in toks for h in range(H_q))
    b, hk = B - 1, H_kv - 1
    group_toks = set()
    for p0 in range(0, M, TS):
        group_toks.update((p0, min(p0 + TS, M) - 1))
    for i in range(M):
        if (H + i) % 128 in (0, 127):
            group_toks.add(i)
    for i in group_toks:
        rows.update((b * M + i) * H_q + hk * G + g for g in range(G))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.slow
@pytest.mark.parametrize("h", [0.0, 0.5, 0.75])
def test_prefill_full_size_rows(cuda_device, h):
    """Config 5 (B=8, N=8192): >= 256 suffix rows per request x all heads, and
    every q tile's boundary and diagonal rows of one (request, KV head) group."""
    c = cpa_synth.PREFILL_CONFIG
    N = c["N"]
    H = int(h * N)
    wl = cpa_synth.make_prefill(B=c["B"], N=N, H=H, H_q=c["H_q"], H_kv=c["H_kv"],
                                page_size=c["page_size"], seed=c["seed"])
    d = PrefillDev(wl)
    M = N - H
    rows = prefill_check_rows(wl.B, M, H, wl.H_q, wl.H_kv, seed=int(h * 100))
    assert len(rows) >= wl.B * 256 * wl.H_q
    ref = oracle.prefill_wl(wl, rows=rows)
    o, lse = cpa.cpa_prefill_hit(d.q, d.k, d.v, d.pt, wl.B, wl.N, wl.H, check=True)
    torch.cuda.synchronize()
    compare(o, lse, *ref, rows=rows)


# ------------------------------------------------------------------ device-detected errors
def test_bad_page_id_is_reported(cuda_device):
    wl = cpa_synth.make_verify(B=2, topk=2, S=3, H_q=8, H_kv=2, page_size=16,
                               prefix_lens=[40, 40], seed=60)
    wl.prefix_page_table[1, 1] = wl.num_pages + 5
    d = VerifyDev(wl)
    ws = torch.zeros(cpa.cpa_cascade_verify_workspace_size(2, 2, 3, 8, 2, 128, 16),
                     dtype=torch.uint8, device=cuda_device)
    cpa.cpa_cascade_verify(*d.args(), workspace=ws)
    st, word = cpa.cpa_get_device_status(ws)
    assert st == 5 and word & 1
    # the context is still usable and a clean call clears the word
    d.ppt[1, 1] = int(wl.prefix_page_table[0, 0])
    cpa.cpa_cascade_verify(*d.args(), workspace=ws)
    st, word = cpa.cpa_get_device_status(ws)
    assert st == 0 and word == 0


def test_prefix_length_over_bound_is_reported(cuda_device):
    wl = cpa_synth.make_verify(B=2, topk=1, S=2, H_q=8, H_kv=2, page_size=16,
                               prefix_lens=[40, 40], seed=61)
    d = VerifyDev(wl)
    ws = torch.zeros(cpa.cpa_cascade_verify_workspace_size(2, 1, 2, 8, 2, 128, 16),
                     dtype=torch.uint8, device=cuda_device)
    cpa.cpa_cascade_verify(*d.args(), max_prefix_len=32, workspace=ws)
    st, word = cpa.cpa_get_device_status(ws)
    assert st == 8 and word & 4


def test_bounded_wait_gives_up_and_context_survives(cuda_device):
    ws = torch.zeros(cpa.cpa_status_workspace_size(), dtype=torch.uint8, device=cuda_device)
    cpa.cpa_debug_wait_timeout(ws, 2000)
    st, word = cpa.cpa_get_device_status(ws)
    assert st == 6 and word & 2
    wl = _make_small("tiny")
    d = VerifyDev(wl)
    o, lse = cpa.cpa_cascade_verify(*d.args())
    torch.cuda.synchronize()
    compare(o, lse, *oracle.verify_wl(wl))
