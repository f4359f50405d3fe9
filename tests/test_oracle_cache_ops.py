"""Pins for the oracle's new-token write and block copy (CPU only).

Address translation (ricepunchb garden, section 3.2) is checked against a
brute-force search written independently: walk the table block by block
subtracting B until the position falls inside one.
"""
import numpy as np
import pytest

import oracle


def brute_force_location(table, pos, B):
    """Find (physical block, offset) of a position by walking the table."""
    remaining = pos
    for phys in table:
        if remaining < B:
            return phys, remaining
        remaining -= B
    raise IndexError(pos)


@pytest.mark.parametrize("B", [1, 4, 8, 16, 64])
def test_reshape_and_cache_places_tokens_at_translated_address(B):
    rs = np.random.default_rng(20 + B)
    H, D, nb = 3, 16, 40
    table = list(rs.permutation(nb)[:6])
    n = min(6 * B, 37)
    positions = rs.permutation(n)[:min(n, 12)]
    slots = np.array([table[p // B] * B + p % B for p in positions], dtype=np.int64)
    k = rs.integers(0, 65536, size=(len(slots), H, D), dtype=np.uint16)
    v = rs.integers(0, 65536, size=(len(slots), H, D), dtype=np.uint16)
    kc = rs.integers(0, 65536, size=(nb, H, B, D), dtype=np.uint16)
    vc = rs.integers(0, 65536, size=(nb, H, B, D), dtype=np.uint16)
    kc0, vc0 = kc.copy(), vc.copy()
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    touched = np.zeros((nb, B), bool)
    for t, p in enumerate(positions):
        phys, off = brute_force_location(table, int(p), B)
        assert np.array_equal(kc[phys, :, off, :], k[t])
        assert np.array_equal(vc[phys, :, off, :], v[t])
        touched[phys, off] = True
    # every other word unchanged (bit patterns compared, NaN encodings included)
    mask = ~touched[:, None, :, None].repeat(H, 1).repeat(D, 3)
    assert np.array_equal(kc[mask], kc0[mask]) and np.array_equal(vc[mask], vc0[mask])


def test_reshape_and_cache_negative_slot_skips():
    rs = np.random.default_rng(30)
    kc = rs.integers(0, 65536, size=(4, 2, 8, 8), dtype=np.uint16)
    vc = kc.copy()
    before = kc.copy()
    k = rs.integers(0, 65536, size=(2, 2, 8), dtype=np.uint16)
    oracle.reshape_and_cache(k, k, kc, vc, np.array([-1, -1]))
    assert np.array_equal(kc, before)


def test_reshape_and_cache_rejects_out_of_pool_slot():
    kc = np.zeros((2, 1, 4, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(np.zeros((1, 1, 8), np.uint16), np.zeros((1, 1, 8), np.uint16),
                                 kc, kc.copy(), np.array([8]))


def test_copy_blocks_copies_whole_blocks_only():
    rs = np.random.default_rng(31)
    nb, H, B, D = 12, 3, 16, 8
    kc = rs.integers(0, 65536, size=(nb, H, B, D), dtype=np.uint16)
    vc = rs.integers(0, 65536, size=(nb, H, B, D), dtype=np.uint16)
    kc0, vc0 = kc.copy(), vc.copy()
    pairs = np.array([[2, 9], [5, 0], [11, 7]], dtype=np.int32)
    oracle.copy_blocks(kc, vc, pairs)
    dsts = set(pairs[:, 1].tolist())
    for src, dst in pairs:
        assert np.array_equal(kc[dst], kc0[src]) and np.array_equal(vc[dst], vc0[src])
    for b in range(nb):
        if b not in dsts:
            assert np.array_equal(kc[b], kc0[b]) and np.array_equal(vc[b], vc0[b])


def test_copy_blocks_rejects_bad_ids():
    kc = np.zeros((3, 1, 4, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.copy_blocks(kc, kc.copy(), np.array([[0, 3]]))


def test_swap_blocks_between_two_pools():
    rs = np.random.default_rng(32)
    H, B, D = 2, 8, 16
    gpu = rs.integers(0, 65536, size=(10, H, B, D), dtype=np.uint16)
    gpv = rs.integers(0, 65536, size=(10, H, B, D), dtype=np.uint16)
    cpu = np.zeros((6, H, B, D), np.uint16)
    cpv = np.zeros_like(cpu)
    pairs = np.array([[7, 2], [1, 5], [9, 0]], np.int32)
    oracle.swap_blocks(cpu, cpv, gpu, gpv, pairs)
    for s, d in pairs:
        assert np.array_equal(cpu[d], gpu[s]) and np.array_equal(cpv[d], gpv[s])
    untouched = [b for b in range(6) if b not in pairs[:, 1]]
    assert not cpu[untouched].any() and not cpv[untouched].any()
    back = np.zeros_like(gpu)
    backv = np.zeros_like(gpv)
    oracle.swap_blocks(back, backv, cpu, cpv, pairs[:, ::-1])
    for s, _ in pairs:
        assert np.array_equal(back[s], gpu[s]) and np.array_equal(backv[s], gpv[s])
    with pytest.raises(ValueError):
        oracle.swap_blocks(cpu, cpv, gpu, gpv, np.array([[10, 0]]))
