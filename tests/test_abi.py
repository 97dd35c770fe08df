"""The C ABI on the CPU: the library loads, exports everything include/cpa.h
declares, and its host-side logic (argument checks, work partition) behaves.
No compute call runs here."""
import ctypes

import numpy as np
import pytest

import cascade_paged_attention_gb300 as cpa


@pytest.fixture(scope="module")
def L():
    cpa.build_library()
    return cpa.lib()


def test_every_declared_function_is_exported(L):
    names = cpa.declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/cpa.h but not exported"
    for n in ("cpa_cascade_verify", "cpa_merge_state", "cpa_naive_expand_verify",
              "cpa_cascade_pass_a", "cpa_cascade_pass_b", "cpa_prefill_hit",
              "cpa_get_device_status"):
        assert n in names


def test_python_binding_covers_the_header(L):
    for n in cpa.declared_functions():
        assert hasattr(cpa, n), f"binding lacks {n}"


def test_status_strings(L):
    assert cpa.cpa_status_string(0) == "ok"
    seen = {cpa.cpa_status_string(i) for i in range(10)}
    assert len(seen) == 10
    assert cpa.cpa_status_string(99) == "unknown status"
    assert cpa.cpa_version() >= 100


def test_null_pointers_are_rejected_before_any_launch(L):
    null = None
    st = L.cpa_cascade_verify(null, null, null, null, 1, null, 1, null, 1, 1, 1, 8, 2, 128, 16,
                              1, 16, 0.088, null, null, null, 0, null)
    assert st == 1
    st = L.cpa_merge_state(null, null, null, null, 1, 1, 128, null, null, null)
    assert st == 1
    st = L.cpa_prefill_hit(null, null, null, null, 1, 1, 8, 0, 8, 2, 128, 16, 1, 0.088, 0, null,
                           null, null, 0, null)
    assert st == 1
    st = L.cpa_get_device_status(null, None, null)
    assert st == 1
    st = L.cpa_tree_verify(null, null, null, null, 1, null, 1, null, null, 1, 7, 8, 2, 128, 16,
                           1, 16, 0.088, null, null, null, 0, null)
    assert st == 1
    st = L.cpa_tree_pass_b(null, null, null, null, 1, null, 1, 7, 8, 2, 128, 16, 1, 0.088, null,
                           null, null, 0, null)
    assert st == 1


def test_shared_verify_checks_before_any_launch(L):
    """Multi-level verify: bad groupings and tables fail their host checks, nothing launches."""
    buf = (ctypes.c_uint8 * 4352)()
    p = ctypes.c_void_p((ctypes.addressof(buf) + 255) // 256 * 256)
    null = None
    # null q
    st = L.cpa_cascade_verify_shared(null, p, p, p, 4, 1, 64, p, 1, p, 1, p, 4, 2, 3, 8, 2, 128,
                                     16, 8, 16, 0.088, p, p, p, 4096, None)
    assert st == 1
    # B = 4 is not a multiple of 3 groups
    st = L.cpa_cascade_verify_shared(p, p, p, p, 4, 3, 64, p, 1, p, 1, p, 4, 2, 3, 8, 2, 128, 16,
                                     8, 16, 0.088, p, p, p, 4096, None)
    assert st == 1
    # shared table narrower than ceil(shared_len / page_size)
    st = L.cpa_cascade_verify_shared(p, p, p, p, 3, 2, 64, p, 1, p, 1, p, 4, 2, 3, 8, 2, 128, 16,
                                     8, 16, 0.088, p, p, p, 4096, None)
    assert st == 1
    # negative shared length
    st = L.cpa_cascade_verify_shared(p, p, p, p, 4, 2, -1, p, 1, p, 1, p, 4, 2, 3, 8, 2, 128, 16,
                                     8, 16, 0.088, p, p, p, 4096, None)
    assert st == 1
    # head_dim 64
    st = L.cpa_cascade_verify_shared(p, p, p, p, 4, 2, 64, p, 1, p, 1, p, 4, 2, 3, 8, 2, 64, 16,
                                     8, 16, 0.088, p, p, p, 4096, None)
    assert st == 2
    assert cpa.cpa_cascade_verify_shared_workspace_size(4, 3, 2, 3, 8, 2, 128, 16) == 0
    assert cpa.cpa_cascade_verify_shared_workspace_size(4, 0, 2, 3, 8, 2, 128, 16) == 0


def test_tree_shape_checks_before_any_launch(L):
    """Non-null dummy pointers that are never dereferenced: every call fails its host checks."""
    buf = (ctypes.c_uint8 * 4352)()
    base = ctypes.addressof(buf)
    p = ctypes.c_void_p((base + 255) // 256 * 256)
    # 65 nodes
    st = L.cpa_tree_pass_b(p, p, p, p, 5, p, 1, 65, 8, 2, 128, 16, 1, 0.088, p, p, p, 4096, None)
    assert st == 2
    # tree table narrower than ceil(N / page_size)
    st = L.cpa_tree_pass_b(p, p, p, p, 1, p, 1, 17, 8, 2, 128, 16, 1, 0.088, p, p, p, 4096, None)
    assert st == 1
    # head_dim 64
    st = L.cpa_tree_pass_b(p, p, p, p, 1, p, 1, 7, 8, 2, 64, 16, 1, 0.088, p, p, p, 4096, None)
    assert st == 2
    # workspace below the status word
    st = L.cpa_tree_pass_b(p, p, p, p, 1, p, 1, 7, 8, 2, 128, 16, 1, 0.088, p, p, p, 16, None)
    assert st == 3
    # tree verify: 65 nodes, then N*G > 256 rows
    st = L.cpa_tree_verify(p, p, p, p, 1, p, 5, p, p, 1, 65, 2, 2, 128, 16, 4, 16, 0.088, p, p,
                           p, 4096, None)
    assert st == 2
    st = L.cpa_tree_verify(p, p, p, p, 1, p, 4, p, p, 1, 64, 64, 8, 128, 16, 4, 16, 0.088, p, p,
                           p, 4096, None)
    assert st == 2


def test_workspace_size_rejects_bad_shapes(L):
    assert cpa.cpa_cascade_verify_workspace_size(0, 1, 1, 8, 2, 128, 16) == 0
    assert cpa.cpa_cascade_verify_workspace_size(1, 1, 1, 8, 3, 128, 16) == 0
    assert cpa.cpa_cascade_verify_workspace_size(1, 1, 1, 8, 2, 64, 16) == 0
    assert cpa.cpa_cascade_verify_workspace_size(1, 1, 1, 8, 2, 128, 12) == 0
    assert cpa.cpa_prefill_hit_workspace_size(1, 10, 11, 8, 2, 128, 16) == 0
    assert cpa.cpa_status_workspace_size() == 256
    assert cpa.cpa_tree_verify_workspace_size(1, 65, 8, 2, 128, 16) == 0
    assert cpa.cpa_tree_verify_workspace_size(1, 0, 8, 2, 128, 16) == 0
    assert cpa.cpa_tree_verify_workspace_size(1, 7, 8, 2, 64, 16) == 0


@pytest.mark.parametrize("total,n", [(16384, 152), (152, 152), (153, 152), (7, 3), (1, 1),
                                     (270848 // 64 * 8 + 5, 152)])
def test_partition_covers_every_tile_once(L, total, n):
    ranges = [cpa.cpa_plan_partition(total, n, c, 0)[1:] for c in range(n)]
    assert ranges[0][0] == 0 and ranges[-1][1] == total
    for (b0, e0), (b1, e1) in zip(ranges, ranges[1:]):
        assert e0 == b1
    sizes = [e - b for b, e in ranges]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    rng = np.random.default_rng(total)
    for t in list(rng.integers(0, total, size=200)) + [0, total - 1]:
        owner = cpa.cpa_plan_partition(total, n, 0, int(t))[0]
        b, e = ranges[owner]
        assert b <= t < e


def test_partition_split_arithmetic_forms_agree(L):
    """The 32-bit form of the split arithmetic (used where total * n < 2^31) gives the
    64-bit form's begin, end and owner: every CTA boundary and its neighbours, for sizes
    up to the 2^31 limit."""
    rng = np.random.default_rng(11)
    cases = [(16384, 152), (2 ** 31 // 152 - 1, 152), (2 ** 31 // 152 + 1, 152), (1, 1),
             (8704, 152), (2 ** 31 // 7 - 3, 7)]
    cases += [(int(rng.integers(1, 2 ** 24)), int(rng.integers(1, 300))) for _ in range(40)]
    for total, n in cases:
        n = min(n, total)
        for c in sorted({0, n - 1, n // 2, int(rng.integers(0, n))}):
            r = cpa.cpa_plan_partition(total, n, c, 0)
            assert r[0] >= 0, (total, n, c)
            for t in {r[1], r[2] - 1, max(r[1] - 1, 0), min(r[2], total - 1)}:
                assert cpa.cpa_plan_partition(total, n, c, int(t))[0] >= 0, (total, n, t)


def test_partition_split_units_are_merged_once(L):
    """Every unit split over CTAs is owned by a contiguous CTA run, each with a nonempty piece,
    and the two partial slots per CTA never collide."""
    rng = np.random.default_rng(7)
    for _ in range(30):
        tiles = rng.integers(1, 60, size=int(rng.integers(1, 40)))
        total = int(tiles.sum())
        n = int(rng.integers(1, min(total, 200) + 1))
        begins = [cpa.cpa_plan_partition(total, n, c, 0)[1] for c in range(n)] + [total]
        slots = {}
        ustart = 0
        for u, t in enumerate(tiles):
            uend = ustart + int(t)
            ca = cpa.cpa_plan_partition(total, n, 0, ustart)[0]
            cb = cpa.cpa_plan_partition(total, n, 0, uend - 1)[0]
            for c in range(ca, cb + 1):
                piece = (max(ustart, begins[c]), min(uend, begins[c + 1]))
                assert piece[0] < piece[1]
                if ca != cb:
                    slot = 2 * c + (1 if begins[c] < ustart else 0)
                    assert slot not in slots, (slot, slots.get(slot), u)
                    slots[slot] = u
            ustart = uend


def test_invalid_prefill_part(L):
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, ctypes.c_void_p)
    st = L.cpa_prefill_hit(p, p, p, p, 1, 1, 8, 0, 8, 2, 128, 16, 1, 0.088, 7, p, p, p, 0, None)
    assert st == 1
