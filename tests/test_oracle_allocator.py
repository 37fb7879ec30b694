"""Pins of the oracle's block allocator.

The free queue is checked against a plain Python list model (brute force);
the pool and sequence manager against the worked example that the pages
print, the waste bound they state, and the semantics of their pseudocode.
"""
import json
import os

import numpy as np
import pytest

from oracle.block_pool import AllocError, BlockPool, FreeBlockQueue, NoFreeBlocks, SequenceManager

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_free_queue_matches_a_list_model():
    rng = np.random.default_rng(0)
    n = 40
    order = rng.permutation(n).tolist()
    q = FreeBlockQueue(order)
    model = list(order)
    out = []
    for step in range(3000):
        op = rng.integers(0, 4)
        if op == 0 and model:
            k = int(rng.integers(0, min(5, len(model)) + 1))
            got = q.popleft_n(k)
            assert got == model[:k]
            del model[:k]
            out.extend(got)
        elif op == 1 and model:
            b = model[int(rng.integers(0, len(model)))]
            q.remove(b)
            model.remove(b)
            out.append(b)
        elif op == 2 and out:
            k = int(rng.integers(0, min(4, len(out)) + 1))
            blocks, out = out[:k], out[k:]
            q.prepend_n(blocks)
            model = list(blocks) + model
        elif op == 3 and out:
            k = int(rng.integers(0, min(4, len(out)) + 1))
            blocks, out = out[:k], out[k:]
            q.append_n(blocks)
            model = model + list(blocks)
        assert q.to_list() == model and len(q) == len(model)


def test_worked_example_block_table_and_growth():
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    p = g["printed"]
    bs = p["block_size"]
    order = [7, 2, 5] + [b for b in range(16) if b not in (7, 2, 5)]
    m = SequenceManager(16, bs, order)
    m.add_seq(0)
    slots = m.append_slots(0, p["prefill_tokens"])
    assert m.block_table(0) == p["physical_blocks"]
    assert slots == g["derived_by_hand"]["slots_tokens_0_to_11"][:9]
    free_before = m.num_free()
    for i in range(p["decode_tokens_fitting_in_last_block"]):
        m.append_slots(0, 1)
        assert m.num_free() == free_before          # no new block while #5 has room
    assert len(m.block_table(0)) == 3
    assert m.append_slots(0, 1) == [order[3] * bs + 0]  # token index 12 needs a 4th block
    assert len(m.block_table(0)) == p["new_block_is_logical_block"] + 1


def test_waste_is_below_one_block():
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))["waste_bound"]
    rng = np.random.default_rng(1)
    m = SequenceManager(4000, g["block_size"])
    for s in range(60):
        m.add_seq(s)
        for _ in range(int(rng.integers(1, 6))):
            m.append_slots(s, int(rng.integers(0, 300)))
        assert 0 <= m.waste(s) <= g["max_unused_slots"]


def test_get_new_blocks_fails_when_short_and_changes_nothing():
    pool = BlockPool(4)
    pool.get_new_blocks(3)
    with pytest.raises(NoFreeBlocks):
        pool.get_new_blocks(2)
    assert pool.get_num_free_blocks() == 1 and pool.ref_cnt == [1, 1, 1, 0]
    m = SequenceManager(4, 4)
    m.add_seq(0)
    m.append_slots(0, 10)
    with pytest.raises(NoFreeBlocks):
        m.append_slots(0, 7)           # needs 2 more blocks, 1 free
    assert m.block_table(0) == [0, 1, 2] and m.num_tokens[0] == 10 and m.num_free() == 1


def test_free_puts_blocks_at_the_head_in_reverse_order():
    m = SequenceManager(8, 4)
    m.add_seq(0)
    m.append_slots(0, 10)              # blocks 0,1,2
    assert m.free_list() == [3, 4, 5, 6, 7]
    m.free_seq(0)
    assert m.free_list() == [2, 1, 0, 3, 4, 5, 6, 7]   # tail block reused first
    m.add_seq(1)
    m.append_slots(1, 1)
    assert m.block_table(1) == [2]


def test_shared_blocks_return_only_when_the_last_user_frees():
    m = SequenceManager(10, 4)
    m.add_seq(0)
    m.append_slots(0, 8)               # blocks 0, 1
    m.add_seq(1)
    m.share(1, 0, 8)
    assert [m.ref(0), m.ref(1)] == [2, 2]
    m.append_slots(1, 1)               # block 1 is full: fresh block 2 for seq 1
    assert m.block_table(1) == [0, 1, 2]
    m.free_seq(0)
    assert [m.ref(0), m.ref(1), m.ref(2)] == [1, 1, 1] and 0 not in m.free_list()
    m.free_seq(1)
    assert m.free_list()[:3] == [2, 1, 0]


def test_touch_revives_a_free_block_from_the_middle():
    pool = BlockPool(6)
    pool.touch([3])
    assert pool.free_block_queue.to_list() == [0, 1, 2, 4, 5] and pool.ref_cnt[3] == 1
    pool.touch([3])
    assert pool.ref_cnt[3] == 2


def test_hashed_blocks_go_to_the_tail():
    pool = BlockPool(5)
    blocks = pool.get_new_blocks(3)    # 0,1,2
    pool.block_hash[1] = 0xABC
    pool.free_blocks([2, 1, 0])
    assert pool.free_block_queue.to_list() == [2, 0, 3, 4, 1]


def test_copy_on_write_of_a_shared_partial_block():
    m = SequenceManager(10, 4)
    m.add_seq(0)
    m.append_slots(0, 6)               # blocks 0, 1 (block 1 holds 2 of 4)
    m.add_seq(1)
    m.share(1, 0, 6)
    with pytest.raises(AllocError):
        m.append_slots(1, 1)           # writing a shared block is refused
    assert m.cow(1, 1) == (1, 2)
    assert m.block_table(1) == [0, 2] and m.ref(1) == 1 and m.ref(2) == 1
    assert m.append_slots(1, 1) == [2 * 4 + 2]
    assert m.cow(0, 1) == (1, 1)       # now private: no copy
    assert m.cow_copies == 1


def test_errors_leave_state_unchanged():
    m = SequenceManager(3, 4)
    with pytest.raises(AllocError):
        m.append_slots(5, 1)
    m.add_seq(0)
    with pytest.raises(AllocError):
        m.add_seq(0)
    with pytest.raises(AllocError):
        m.cow(0, 0)
    with pytest.raises(AllocError):
        m.ref(3)
    m.append_slots(0, 12)
    m.add_seq(1)
    m.share(1, 0, 12)
    with pytest.raises(NoFreeBlocks):
        m.cow(1, 2)
    assert m.block_table(1) == [0, 1, 2] and m.ref(2) == 2
    with pytest.raises(AllocError):
        m.free_seq(9)
    with pytest.raises(AllocError):
        SequenceManager(4, 4, [0, 1, 1, 3])
