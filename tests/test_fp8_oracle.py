"""Pins of the oracle's FP8 KV verify (KV-cache tutorial, section 4.5: FP8 KV with a
per-tensor or per-channel scale).

Each K/V element is its E4M3 code decoded exactly, times its scale.  Pins:
the decoder against the library's float8_e4m3fn conversion for all 256
codes and against the format's closed-form values; with scales that keep
every product exactly representable in bf16 (1, or powers of two), the FP8
verify equals the already pinned bf16 verify on those values bit for bit;
brute force with arbitrary per-channel scales; the parts merge to the full
result.
"""
import math

import numpy as np
import pytest
import torch

import cpa_synth
import oracle


def test_e4m3_decoder_matches_library_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    keep = ~np.isnan(ref)
    np.testing.assert_array_equal(got[keep], ref[keep])


def test_e4m3_closed_form_values():
    v = lambda c: float(oracle.e4m3_decode(np.array([c], dtype=np.uint8))[0])
    assert v(0x38) == 1.0                   # exponent field 7 = bias
    assert v(0x7E) == 448.0                 # largest finite: 1.75 * 2^8
    assert v(0xFE) == -448.0
    assert v(0x01) == 2.0 ** -9             # smallest subnormal
    assert v(0x07) == 7 * 2.0 ** -9         # largest subnormal
    assert v(0x08) == 2.0 ** -6             # smallest normal
    assert v(0x00) == 0.0 and math.copysign(1.0, v(0x80)) == -1.0
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))
    assert v(0x3C) == 1.5 and v(0x40) == 2.0


def _bf16_pools(wl):
    """The same values as bf16 bit patterns (exact when every product is representable)."""
    def conv(codes, scale):
        vals = oracle.e4m3_decode(codes)
        sc = np.asarray(scale, dtype=np.float64)
        vals = vals * (sc if sc.size == 1 else sc.reshape(1, 1, wl.H_kv, wl.head_dim))
        f32 = vals.astype(np.float32)
        assert np.array_equal(f32.astype(np.float64), vals)
        bits = cpa_synth.bf16_bits_from_f32(f32)
        assert np.array_equal(cpa_synth.f32_from_bf16_bits(bits), f32)
        return bits
    return conv(wl.k_pages, wl.k_scale), conv(wl.v_pages, wl.v_scale)


@pytest.mark.parametrize("scales", ["unit", "pow2"])
def test_representable_scales_equal_bf16_verify(scales):
    wl = cpa_synth.make_verify_fp8(B=3, topk=2, S=4, H_q=4, H_kv=2, head_dim=32, page_size=8,
                                   prefix_lens=[13, 0, 40], scales=scales, seed=7)
    kb, vb = _bf16_pools(wl)
    for part in ("full", "prefix", "draft"):
        got = oracle.verify_fp8_wl(wl, part=part)
        ref = oracle.verify(wl.q, kb, vb, wl.prefix_page_table, wl.draft_page_table,
                            wl.prefix_lens, wl.topk, wl.S, wl.H_q, wl.H_kv, part=part)
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_array_equal(got[1], ref[1])


def _brute_fp8(wl):
    """Pure-Python attention: decode through the library's float8 type, de-page by hand."""
    d, P, H_q, H_kv = wl.head_dim, wl.page_size, wl.H_q, wl.H_kv
    G = H_q // H_kv
    dec = lambda c: torch.from_numpy(np.ascontiguousarray(c)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    kv_k, kv_v = dec(wl.k_pages), dec(wl.v_pages)
    ks = np.asarray(wl.k_scale, np.float64)
    vs = np.asarray(wl.v_scale, np.float64)
    kscale = lambda h: ks[0] if ks.size == 1 else ks.reshape(H_kv, d)[h]
    vscale = lambda h: vs[0] if vs.size == 1 else vs.reshape(H_kv, d)[h]
    q = cpa_synth.f32_from_bf16_bits(wl.q).astype(np.float64)
    scale = 1.0 / math.sqrt(d)
    o_rows, l_rows = [], []
    for b in range(wl.B):
        L = int(wl.prefix_lens[b])
        for k in range(wl.topk):
            for s in range(wl.S):
                t = (b * wl.topk + k) * wl.S + s
                keys = [(wl.prefix_page_table[b], pos) for pos in range(L)]
                keys += [(wl.draft_page_table[b * wl.topk + k], j) for j in range(s + 1)]
                for hq in range(H_q):
                    h = hq // G
                    scores, vals = [], []
                    for tab, pos in keys:
                        pg, slot = tab[pos // P], pos % P
                        kr = kv_k[pg, slot, h] * kscale(h)
                        vals.append(kv_v[pg, slot, h] * vscale(h))
                        scores.append(sum(a * c for a, c in zip(q[t, hq], kr)) * scale)
                    m = max(scores)
                    w = [math.exp(x - m) for x in scores]
                    z = sum(w)
                    o_rows.append(sum(wi / z * vi for wi, vi in zip(w, vals)))
                    l_rows.append(m + math.log(z))
    return np.array(o_rows), np.array(l_rows)


@pytest.mark.parametrize("scales", ["tensor", "channel"])
def test_fp8_verify_matches_brute_force(scales):
    wl = cpa_synth.make_verify_fp8(B=2, topk=2, S=3, H_q=4, H_kv=2, head_dim=16, page_size=4,
                                   prefix_lens=[9, 2], scales=scales, seed=11)
    o, lse = oracle.verify_fp8_wl(wl)
    bo, bl = _brute_fp8(wl)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


def test_fp8_parts_merge_to_full():
    wl = cpa_synth.make_verify_fp8(B=2, topk=3, S=2, H_q=8, H_kv=2, head_dim=32, page_size=4,
                                   prefix_lens=[17, 0], scales="channel", seed=12)
    a = oracle.verify_fp8_wl(wl, part="prefix")
    b = oracle.verify_fp8_wl(wl, part="draft")
    f = oracle.verify_fp8_wl(wl)
    o, lse = oracle.merge_state(a[0], a[1], b[0], b[1])
    np.testing.assert_allclose(o, f[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, f[1], rtol=0, atol=1e-12)


def test_fp8_scales_are_validated():
    wl = cpa_synth.make_verify_fp8(B=1, topk=1, S=1, H_q=2, H_kv=1, head_dim=16, page_size=4,
                                   L=3, seed=13)
    with pytest.raises(ValueError):
        oracle.verify_fp8(wl.q, wl.k_pages, wl.v_pages, np.ones(3), np.ones(3),
                          wl.prefix_page_table, wl.draft_page_table, wl.prefix_lens, 1, 1, 2, 1)
