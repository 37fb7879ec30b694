"""Preemption by swapping in the oracle ("2.1 PagedAttention" §7): the
allocator's swap_out / swap_in bookkeeping and the swap_blocks copy, pinned
against free_seq, exact data round trips and the attention result."""
import numpy as np
import pytest

from oracle import paged_attention as pa
from oracle.block_pool import AllocError, NoFreeBlocks, SequenceManager

BS, HKV, D = 4, 2, 8


def _mgr(nb=16, ncpu=8, order=None):
    m = SequenceManager(nb, BS, order)
    m.enable_swap(ncpu)
    return m


def _state(m):
    return (m.free_list(), list(m.pool.ref_cnt), {s: list(t) for s, t in m.tables.items()},
            dict(m.num_tokens), m.cpu_free.to_list(), set(m.on_cpu))


def test_swap_out_releases_gpu_blocks_exactly_as_free_seq():
    order = list(np.random.default_rng(0).permutation(16))
    a, b = _mgr(order=order), _mgr(order=order)
    for m in (a, b):
        m.add_seq(0)
        m.append_slots(0, 10)
        m.add_seq(1)
        m.append_slots(1, 7)
    table = a.block_table(0)
    pairs = a.swap_out(0)
    b.free_seq(0)
    assert a.free_list() == b.free_list() and a.pool.ref_cnt == b.pool.ref_cnt
    assert [g for g, _ in pairs] == table                    # logical order
    assert [c for _, c in pairs] == [0, 1, 2]                # head of the swap pool
    assert a.block_table(0) == [0, 1, 2] and a.num_tokens[0] == 10 and 0 in a.on_cpu


def test_swap_in_takes_new_gpu_blocks_and_returns_the_swap_blocks():
    m = _mgr()
    m.add_seq(0)
    m.append_slots(0, 9)
    m.swap_out(0)
    head = m.free_list()[:3]
    pairs = m.swap_in(0)
    assert pairs == list(zip([0, 1, 2], head))
    assert m.block_table(0) == head and 0 not in m.on_cpu
    assert m.cpu_free.to_list() == [2, 1, 0, 3, 4, 5, 6, 7]  # back at the head, last block first
    assert m.append_slots(0, 3) == [head[2] * BS + k for k in range(1, 4)]   # grows again


def test_round_trip_restores_the_kv_and_the_attention_exactly():
    rng = np.random.default_rng(1)
    nb, ncpu = 16, 8
    m = _mgr(nb, ncpu, order=list(rng.permutation(nb)))
    m.add_seq(0)
    L = 11
    slots = m.append_slots(0, L)
    kc = rng.standard_normal((nb, BS, HKV, D))
    vc = rng.standard_normal((nb, BS, HKV, D))
    k, v = rng.standard_normal((L, HKV, D)), rng.standard_normal((L, HKV, D))
    kc, vc = pa.reshape_and_cache(k, v, slots, kc, vc)
    q = rng.standard_normal((1, 4, D))
    before = pa.decode(q, kc, vc, [m.block_table(0)], [L], 0.3)
    kh = np.zeros((ncpu, BS, HKV, D))
    vh = np.zeros((ncpu, BS, HKV, D))
    kh, vh = pa.swap_blocks(kc, vc, kh, vh, m.swap_out(0))
    # another request overwrites the released GPU blocks
    m.add_seq(1)
    junk = m.append_slots(1, nb * BS)
    kc, vc = pa.reshape_and_cache(np.full((len(junk), HKV, D), 7.0), np.full((len(junk), HKV, D), 7.0), junk, kc, vc)
    m.free_seq(1)
    kc, vc = pa.swap_blocks(kh, vh, kc, vc, m.swap_in(0))
    got_k = pa.gather_context(kc, m.block_table(0), L, BS)
    assert np.array_equal(got_k, k)
    after = pa.decode(q, kc, vc, [m.block_table(0)], [L], 0.3)
    assert np.array_equal(before, after)


def test_swapping_out_a_sharer_leaves_the_other_holder_alone():
    m = _mgr()
    m.add_seq(0)
    m.append_slots(0, 8)
    m.add_seq(1)
    m.share(1, 0, 8)
    shared = m.block_table(0)
    pairs = m.swap_out(1)
    assert [g for g, _ in pairs] == shared
    assert all(m.ref(b) == 1 for b in shared) and m.block_table(0) == shared
    back = m.swap_in(1)
    assert not set(g for _, g in back) & set(shared)         # private copies now


def test_shortages_and_operations_on_swapped_requests_change_nothing():
    m = _mgr(nb=8, ncpu=2)
    m.add_seq(0)
    m.append_slots(0, 12)                                    # 3 blocks > 2 swap blocks
    s0 = _state(m)
    with pytest.raises(NoFreeBlocks):
        m.swap_out(0)
    assert _state(m) == s0
    m.add_seq(1)
    m.append_slots(1, 5)
    m.swap_out(1)                                            # 2 blocks
    s1 = _state(m)
    for op, args in [("append_slots", (1, 1)), ("cow", (1, 0)), ("swap_out", (1,)), ("share", (2, 1, 4))]:
        if op == "share":
            m.add_seq(2)
            s1 = _state(m)
        with pytest.raises(AllocError):
            getattr(m, op)(*args)
        assert _state(m) == s1
    m.free_seq(2)
    m.add_seq(3)
    m.append_slots(3, 5 * BS)                                # 5 + 3 = all 8 GPU blocks in use
    s2 = _state(m)
    with pytest.raises(NoFreeBlocks):
        m.swap_in(1)
    assert _state(m) == s2
    m.free_seq(1)                                            # swapped out: returns its swap blocks
    assert m.num_free_cpu() == 2 and 1 not in m.tables


def test_cached_blocks_stay_cached_after_their_request_is_swapped_out():
    m = SequenceManager(16, BS)
    m.enable_prefix_caching()
    m.enable_swap(8)
    p = list(range(2 * BS + 1))
    m.add_seq_cached(0, p)
    m.append_tokens(0, p)
    cached = m.block_table(0)[:2]
    m.swap_out(0)
    assert m.free_list()[-2:] == list(reversed(cached))      # hashed: at the tail
    assert m.add_seq_cached(1, p) == 2 * BS                  # still hit
    back = m.swap_in(0)
    assert all(m.pool.block_hash[g] is None for _, g in back)
