"""Invariants of the seeded input generator (host logic, no GPU)."""
import numpy as np

import cpa_synth


def _used_pages(wl):
    used = []
    P = wl.page_size
    for b in range(wl.B):
        n = (int(wl.prefix_lens[b]) + P - 1) // P
        used.extend(wl.prefix_page_table[b, :n].tolist())
        assert np.all(wl.prefix_page_table[b, n:] == -1)
    nd = (wl.S + P - 1) // P
    for v in range(wl.B * wl.topk):
        used.extend(wl.draft_page_table[v, :nd].tolist())
    return used


def test_page_tables_are_a_permutation():
    wl = cpa_synth.make_verify(B=5, topk=3, S=4, H_q=4, H_kv=2, head_dim=8, page_size=4,
                               L_range=(0, 30), seed=3)
    used = _used_pages(wl)
    assert len(used) == len(set(used)) == wl.num_pages
    assert min(used) >= 0 and max(used) < wl.num_pages


def test_logical_content_independent_of_placement():
    kw = dict(B=3, topk=2, S=3, H_q=4, H_kv=2, head_dim=8, page_size=4, L=13, seed=7,
              keep_logical=True)
    a = cpa_synth.make_verify(perm_seed=1, **kw)
    b = cpa_synth.make_verify(perm_seed=99, **kw)
    assert np.array_equal(a.q, b.q)
    for x, y in zip(a.prefix_k + a.draft_v, b.prefix_k + b.draft_v):
        assert np.array_equal(x, y)
    assert not np.array_equal(a.prefix_page_table, b.prefix_page_table)
    # the pages hold the logical tokens at table[pos // P], slot pos % P
    P = a.page_size
    for bb in range(a.B):
        for pos in range(int(a.prefix_lens[bb])):
            page = a.prefix_page_table[bb, pos // P]
            assert np.array_equal(a.k_pages[page, pos % P], a.prefix_k[bb][pos])


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    bits = cpa_synth.bf16_bits_from_f32(x)
    back = cpa_synth.f32_from_bf16_bits(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins
    assert back[0] == 1.0 and back[1] == 1.0
    assert back[2] == np.float32(1.015625)
    assert back[3] == -2.5


def test_prefill_layout():
    wl = cpa_synth.make_prefill(B=2, N=21, H=8, H_q=4, H_kv=2, head_dim=8, page_size=4, seed=1,
                                keep_logical=True)
    assert wl.q.shape == (2 * 13, 4, 8)
    assert wl.page_table.shape == (2, 6)
    flat = wl.page_table.ravel()
    assert len(set(flat.tolist())) == flat.size == wl.num_pages
    assert wl.visible_pairs() == (21 * 22 - 8 * 9) // 2


def test_nan_padding_only_outside_sequences():
    wl = cpa_synth.make_verify(B=2, topk=1, S=2, H_q=2, H_kv=1, head_dim=8, page_size=4,
                               prefix_lens=[5, 3], seed=2, pad_fill="nan", keep_logical=True)
    P = wl.page_size
    for b in range(2):
        L = int(wl.prefix_lens[b])
        last = wl.prefix_page_table[b, (L - 1) // P]
        for slot in range(P):
            pos = ((L - 1) // P) * P + slot
            is_nan = np.all(wl.k_pages[last, slot] == 0x7FC0)
            assert is_nan == (pos >= L)


def test_tree_workload_layout():
    wl = cpa_synth.make_tree_verify(B=3, N=11, H_q=4, H_kv=2, head_dim=8, page_size=4,
                                    prefix_lens=[7, 0, 12], n_roots=2, seed=4, keep_logical=True)
    assert wl.q.shape == (3 * 11, 4, 8) and wl.parents.shape == (3, 11)
    assert wl.tree_page_table.shape == (3, 3)
    used = []
    for b in range(3):
        n = (int(wl.prefix_lens[b]) + 3) // 4
        used += wl.prefix_page_table[b, :n].tolist() + wl.tree_page_table[b].tolist()
        # every parent precedes its child; exactly n_roots roots
        par = wl.parents[b]
        assert (par[par >= 0] < np.nonzero(par >= 0)[0]).all()
        assert int((par == -1).sum()) == 2
        for j in range(11):
            page = wl.tree_page_table[b, j // 4]
            assert np.array_equal(wl.k_pages[page, j % 4], wl.tree_k[b][j])
    assert len(used) == len(set(used)) == wl.num_pages


def test_shared_workload_layout():
    wl = cpa_synth.make_shared_verify(B=4, n_groups=2, shared_len=9, topk=2, S=3, H_q=4, H_kv=2,
                                      head_dim=8, page_size=4, prefix_lens=[5, 0, 8, 1], seed=5,
                                      keep_logical=True)
    assert wl.shared_page_table.shape == (2, 3)
    for g in range(2):
        for pos in range(9):
            page = wl.shared_page_table[g, pos // 4]
            assert np.array_equal(wl.v_pages[page, pos % 4], wl.shared_v[g][pos])
    assert wl.unique_kv_tokens() == 2 * 9 + 14 + 4 * 2 * 3


def test_fp8_codes_have_no_nan_and_order_one_magnitudes():
    rng = np.random.default_rng(0)
    c = cpa_synth.e4m3_codes(rng, (4096,))
    assert not np.any((c & 0x7F) == 0x7F)
    expo = (c >> 3) & 0xF
    assert set(np.unique(expo).tolist()) <= {0, 5, 6, 7, 8}
    assert (expo == 0).mean() < 0.05


def test_fp8_logical_contents_do_not_depend_on_placement():
    """The FP8 generator keeps the logical K/V of every sequence fixed by `seed`
    whatever the page permutation (`perm_seed`), like the bf16 generator."""
    kw = dict(B=3, topk=2, S=3, H_q=8, H_kv=2, page_size=8, prefix_lens=[20, 0, 9], seed=5)
    a = cpa_synth.make_verify_fp8(perm_seed=1, **kw)
    b = cpa_synth.make_verify_fp8(perm_seed=2, **kw)
    assert not np.array_equal(a.prefix_page_table, b.prefix_page_table)

    def logical(wl, tab, n):
        pos = np.arange(n)
        return wl.k_pages[tab[pos // wl.page_size], pos % wl.page_size], \
            wl.v_pages[tab[pos // wl.page_size], pos % wl.page_size]

    for r in range(kw["B"]):
        n = int(a.prefix_lens[r])
        for x, y in zip(logical(a, a.prefix_page_table[r], n), logical(b, b.prefix_page_table[r], n)):
            assert np.array_equal(x, y)
    for v in range(kw["B"] * kw["topk"]):
        for x, y in zip(logical(a, a.draft_page_table[v], kw["S"]),
                        logical(b, b.draft_page_table[v], kw["S"])):
            assert np.array_equal(x, y)
    assert np.array_equal(a.q, b.q)
    assert np.array_equal(a.k_scale, b.k_scale)
