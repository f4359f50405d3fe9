"""Pins for the block manager's policy model (CPU only).

Checked against: the copy-on-write walkthrough of the wywy.jp notes (parallel
sampling, paper section 4.4), the sharing diagram of the ricepunchb garden
(section 5.1), the waste bound of the detail page's KV Cache Manager paragraph,
bookkeeping invariants, and the published SplitMix64 reference outputs.
"""
import json
import os

import numpy as np
import pytest

from oracle.block_manager import (BlockManagerModel, InvalidRequest, OutOfBlocks,
                                  seeded_permutation, splitmix64_stream)

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "pages_facts.json")))


def test_splitmix64_reference_outputs():
    # Reference outputs of SplitMix64 (Steele, Lea, Flood 2014; Vigna's public
    # domain splitmix64.c) for seeds 0 and 1234567.
    g = splitmix64_stream(0)
    assert [next(g) for _ in range(3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                          0x06C45D188009454F]
    g = splitmix64_stream(1234567)
    assert [next(g) for _ in range(2)] == [6457827717110365317, 3203168211198807973]


def test_seeded_permutation_is_a_permutation_and_seeded():
    for n in (1, 2, 17, 1000):
        p = seeded_permutation(n, 5)
        assert sorted(p) == list(range(n))
    assert seeded_permutation(100, 1) != seeded_permutation(100, 2)
    assert seeded_permutation(100, 3) == seeded_permutation(100, 3)


def check_invariants(bm: BlockManagerModel):
    B = bm.B
    refsum = 0
    for sid, table in bm.tables.items():
        n = bm.ctx[sid]
        waste = len(table) * B - n
        assert 0 <= waste < B or (n == 0 and len(table) == 0)
        refsum += len(table)
        assert all(bm.ref[b] >= 1 for b in table)
    assert sum(bm.ref) == refsum
    used = {b for t in bm.tables.values() for b in t}
    assert len(used) + bm.num_free() == bm.num_blocks
    assert used.isdisjoint(set(bm.free))


def test_cow_walkthrough_from_the_notes():
    f = FACTS["cow_walkthrough"]
    B = f["block_size"]
    bm = BlockManagerModel(16, B, seed=1)
    bm.add_sequence(1, f["prompt_len"])          # sample A1 holds the prompt
    bm.fork(1, 2)                                # sample A2 shares every block
    shared_last = bm.block_table(1)[-1]
    assert bm.refcount(shared_last) == f["shared_last_block_refcount_before"]
    slot, src, dst = bm.append_slot(1)           # A1 writes its last logical block
    assert f["first_writer"]["copies"] and (src, dst) != (-1, -1)
    assert src == shared_last and dst != shared_last
    assert bm.refcount(shared_last) == f["first_writer"]["old_block_refcount_after"]
    assert bm.block_table(1)[-1] == dst and slot == dst * B + f["prompt_len"] % B
    slot2, src2, dst2 = bm.append_slot(2)        # A2 writes in place
    assert not f["second_writer"]["copies"] and (src2, dst2) == (-1, -1)
    assert slot2 == shared_last * B + f["prompt_len"] % B
    # the full logical block 0 is still shared
    assert bm.block_table(1)[0] == bm.block_table(2)[0]
    assert bm.refcount(bm.block_table(1)[0]) == 2
    check_invariants(bm)


def test_sharing_diagram_structure():
    """Two sequences share two full prompt blocks and own a third block each."""
    f = FACTS["sharing_diagram"]
    B = 16
    bm = BlockManagerModel(32, B, seed=2)
    bm.add_sequence("A", 2 * B)
    bm.fork("A", "B")
    bm.append_slot("A")
    bm.append_slot("B")
    ta, tb = bm.block_table("A"), bm.block_table("B")
    # same pattern as the diagram: positions 0,1 equal, position 2 differs
    pat = [x == y for x, y in zip(f["table_a"], f["table_b"])]
    assert [x == y for x, y in zip(ta, tb)] == pat
    counts = {b: bm.refcount(b) for b in set(ta) | set(tb)}
    diagram = {int(k): v for k, v in f["refcounts"].items()}
    relabel = dict(zip(f["table_a"] + f["table_b"], ta + tb))
    assert {relabel[k]: v for k, v in diagram.items()} == counts
    check_invariants(bm)


def test_six_way_fork_copies_five_times_then_writes_in_place():
    B = 16
    bm = BlockManagerModel(64, B, seed=3)
    bm.add_sequence(0, 100)                 # 6 full blocks + a partial one (4 tokens)
    for c in range(1, 6):
        bm.fork(0, c)
    last = bm.block_table(0)[-1]
    assert bm.refcount(last) == 6
    pairs = [bm.append_slot(s)[1:] for s in range(6)]
    assert all(src == last for src, _ in pairs[:5]) and pairs[5] == (-1, -1)
    assert len({d for _, d in pairs[:5]}) == 5 and bm.refcount(last) == 1
    check_invariants(bm)


def test_prompt_on_block_boundary_needs_no_copy():
    bm = BlockManagerModel(16, 4, seed=4)
    bm.add_sequence(0, 8)
    bm.fork(0, 1)
    _, s0, d0 = bm.append_slot(0)
    _, s1, d1 = bm.append_slot(1)
    assert (s0, d0) == (-1, -1) and (s1, d1) == (-1, -1)
    assert bm.block_table(0)[:2] == bm.block_table(1)[:2]
    assert bm.block_table(0)[2] != bm.block_table(1)[2]


def test_allocation_follows_seeded_free_list():
    perm = seeded_permutation(20, 9)
    bm = BlockManagerModel(20, 8, seed=9)
    bm.add_sequence(0, 17)                  # 3 blocks: the first three of the free list
    assert bm.block_table(0) == perm[:3]
    slots = bm.add_sequence(1, 1)
    assert bm.block_table(1) == [perm[3]] and slots == [perm[3] * 8]


def test_free_restores_pool_and_respects_sharing():
    bm = BlockManagerModel(40, 8, seed=5)
    bm.add_sequence(0, 30)
    bm.fork(0, 1)
    for _ in range(20):
        bm.append_slot(1)
    bm.free_sequence(0)
    check_invariants(bm)
    assert all(bm.refcount(b) == 1 for b in bm.block_table(1))
    bm.free_sequence(1)
    assert bm.num_free() == 40 and sum(bm.ref) == 0


def test_out_of_blocks_leaves_state_unchanged():
    bm = BlockManagerModel(4, 4, seed=6)
    bm.add_sequence(0, 13)                  # 4 blocks, pool exhausted
    snapshot = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()},
                dict(bm.ctx))
    with pytest.raises(OutOfBlocks):
        bm.add_sequence(1, 1)
    bm.fork(0, 2)
    snapshot = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()},
                dict(bm.ctx))
    with pytest.raises(OutOfBlocks):
        bm.append_slot(2)                   # would need a CoW block
    assert snapshot == (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()},
                        dict(bm.ctx))
    with pytest.raises(InvalidRequest):
        bm.append_slot(99)


def test_random_churn_keeps_invariants():
    rs = np.random.default_rng(7)
    bm = BlockManagerModel(200, 16, seed=7)
    live = []
    nxt = 0
    for _ in range(3000):
        op = rs.integers(0, 10)
        try:
            if op < 2 or not live:
                bm.add_sequence(nxt, int(rs.integers(0, 60)))
                live.append(nxt)
                nxt += 1
            elif op < 3:
                bm.fork(live[int(rs.integers(len(live)))], nxt)
                live.append(nxt)
                nxt += 1
            elif op < 4:
                sid = live.pop(int(rs.integers(len(live))))
                bm.free_sequence(sid)
            else:
                slot, src, dst = bm.append_slot(live[int(rs.integers(len(live)))])
                assert 0 <= slot < 200 * 16
        except OutOfBlocks:
            pass
        check_invariants(bm)


# ---- swapping (wywy.jp notes: "Swapping", all-or-nothing eviction) -----------------

def groups_of(bm):
    """Sharing pattern of the live tables: sequence -> tuple of block-class labels."""
    label, out = {}, {}
    for sid in sorted(bm.tables):
        out[sid] = tuple(label.setdefault((bm.swapped[sid], b), len(label))
                         for b in bm.tables[sid])
    return out


def test_swap_round_trip_keeps_sharing_and_counts():
    bm = BlockManagerModel(64, 16, seed=8)
    bm.add_cpu_pool(64, seed=9)
    bm.add_sequence(0, 70)
    for c in (1, 2):
        bm.fork(0, c)
    bm.append_slot(1)                     # 1 gets its own copy of the partial block
    bm.add_sequence(5, 20)                # an unrelated resident sequence
    before = groups_of(bm)
    free_gpu = bm.num_free()
    pairs = bm.swap_out([0, 1, 2])
    distinct = {b for s in (0, 1, 2) for b in bm.tables[s]}
    assert len(pairs) == len(distinct) == 6
    assert all(bm.swapped[s] for s in (0, 1, 2)) and not bm.swapped[5]
    assert bm.num_free() == free_gpu + 6
    assert [bm.cpu_ref[b] for b in bm.tables[0]] == [3, 3, 3, 3, 2]
    with pytest.raises(InvalidRequest):
        bm.append_slot(0)                 # swapped-out sequences do not grow
    with pytest.raises(InvalidRequest):
        bm.fork(1, 9)
    back = bm.swap_in([0, 1, 2])
    assert [c for c, _ in back] == [n for _, n in pairs]
    assert groups_of(bm) == before
    assert [bm.ref[b] for b in bm.tables[0]] == [3, 3, 3, 3, 2]
    assert bm.cpu_free and len(bm.cpu_free) == 64


def test_swap_refuses_blocks_shared_outside_the_group():
    bm = BlockManagerModel(32, 16, seed=10)
    bm.add_cpu_pool(32, seed=11)
    bm.add_sequence(0, 40)
    bm.fork(0, 1)
    snapshot = (list(bm.free), list(bm.ref), dict(bm.swapped))
    with pytest.raises(InvalidRequest):
        bm.swap_out([0])                  # 1 still holds 0's blocks
    assert snapshot == (list(bm.free), list(bm.ref), dict(bm.swapped))
    bm.swap_out([1, 0])


def test_swap_is_all_or_nothing_on_oom():
    bm = BlockManagerModel(32, 16, seed=12)
    bm.add_cpu_pool(3, seed=13)
    bm.add_sequence(0, 64)                # 4 blocks > 3 CPU blocks
    with pytest.raises(OutOfBlocks):
        bm.swap_out([0])
    assert not bm.swapped[0] and len(bm.cpu_free) == 3 and bm.num_free() == 28


def test_freeing_a_swapped_sequence_releases_cpu_blocks():
    bm = BlockManagerModel(16, 8, seed=14)
    bm.add_cpu_pool(16, seed=15)
    bm.add_sequence(0, 20)
    bm.swap_out([0])
    assert len(bm.cpu_free) == 13
    bm.free_sequence(0)
    assert len(bm.cpu_free) == 16 and sum(bm.cpu_ref) == 0 and bm.num_free() == 16
