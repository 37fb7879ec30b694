"""Automatic prefix caching in the allocator oracle ("Khám phá vLLM … phần 2",
prefix caching; "2.1 PagedAttention" §9.2-9.3), pinned by published hash test
vectors, the pages' worked scenario, and content-level properties that do not
depend on the hash formula."""
import random

import pytest

from oracle.block_pool import SequenceManager, block_hash, fnv1a64

BS = 4


def test_fnv1a64_published_vectors():
    # the FNV-1a 64-bit test vectors published with the algorithm
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def _mgr(nb=32):
    m = SequenceManager(nb, BS)
    m.enable_prefix_caching()
    return m


def test_second_request_with_the_same_long_prefix_reuses_its_blocks():
    # the pages' example: long_prefix = n * block_size tokens shared by two prompts
    n = 3
    prefix = list(range(100, 100 + n * BS))
    m = _mgr()
    assert m.add_seq_cached(0, prefix + [1, 2]) == 0        # first request: nothing cached yet
    m.append_tokens(0, prefix + [1, 2])
    assert len(m.pool.cached_block_hash_to_block) == n      # only the n full blocks
    got = m.add_seq_cached(1, prefix + [7, 8, 9])
    assert got == n * BS
    assert m.block_table(1) == m.block_table(0)[:n]
    assert all(m.ref(b) == 2 for b in m.block_table(0)[:n])  # request 0 still alive
    assert m.lookup_blocks == 1 + n and m.hit_blocks == n   # request 0's miss, then n hits


def test_hit_after_the_first_request_finished_takes_blocks_out_of_the_free_queue():
    n = 2
    prefix = list(range(7, 7 + n * BS))
    m = _mgr()
    m.add_seq_cached(0, prefix + [5])
    m.append_tokens(0, prefix + [5])
    cached = m.block_table(0)[:n]
    m.free_seq(0)
    free = m.free_list()
    assert all(m.ref(b) == 0 for b in cached) and set(cached) <= set(free)
    # hashed blocks at the tail, the request's first block last (evicted last)
    assert free[-n:] == list(reversed(cached))
    assert m.add_seq_cached(1, prefix + [6, 6]) == n * BS
    assert m.block_table(1) == cached
    assert all(m.ref(b) == 1 for b in cached)
    assert not set(cached) & set(m.free_list())


def test_hash_chain_same_block_after_a_different_prefix_misses():
    m = _mgr()
    a = [1, 2, 3, 4, 5, 6, 7, 8, 9]
    m.add_seq_cached(0, a)
    m.append_tokens(0, a)
    b = [0, 0, 0, 0, 5, 6, 7, 8, 9]        # block 1 equal to a's, block 0 not
    assert m.add_seq_cached(1, b) == 0


def test_salt_separates_requests():
    m = _mgr()
    p = list(range(2 * BS + 1))
    m.add_seq_cached(0, p, salt=11)
    m.append_tokens(0, p)
    assert m.add_seq_cached(1, p, salt=12) == 0
    assert m.add_seq_cached(2, p, salt=11) == 2 * BS


def test_partial_blocks_are_never_cached_and_one_token_is_left_to_compute():
    m = _mgr()
    p = list(range(3 * BS))            # exactly three full blocks
    m.add_seq_cached(0, p)
    m.append_tokens(0, p)
    assert len(m.pool.cached_block_hash_to_block) == 3
    # the same prompt again: at most floor((n-1)/bs) = 2 blocks, so the last
    # token is computed
    assert m.add_seq_cached(1, p) == 2 * BS
    q = p + [1, 2]                     # longer prompt: all three blocks hit
    assert m.add_seq_cached(2, q) == 3 * BS


def test_eviction_takes_the_last_block_first():
    n = 3
    p = list(range(50, 50 + n * BS))
    m = _mgr(nb=8)
    m.add_seq_cached(0, p + [1])
    m.append_tokens(0, p + [1])        # 4 blocks, 3 of them cached
    m.free_seq(0)
    # take every unhashed free block and one more: the hashed block at the
    # queue's front is the request's last full block
    m.add_seq(9)
    m.append_slots(9, (8 - n + 1) * BS)
    assert m.pool.evictions == 1
    assert len(m.pool.cached_block_hash_to_block) == n - 1
    assert m.add_seq_cached(1, p + [2]) == (n - 1) * BS


def test_duplicate_content_keeps_the_first_cached_block():
    m = _mgr()
    p = list(range(2 * BS + 1))
    m.add_seq_cached(0, p)
    m.add_seq_cached(1, p)             # both miss: neither has appended yet
    m.append_tokens(0, p)
    m.append_tokens(1, p)
    cmap = m.pool.cached_block_hash_to_block
    assert sorted(cmap.values()) == sorted(m.block_table(0)[:2])
    assert all(m.pool.block_hash[b] is None for b in m.block_table(1))


def test_appends_without_token_ids_end_hashing():
    m = _mgr()
    m.add_seq_cached(0, [1, 2, 3])
    m.append_tokens(0, [1, 2, 3])
    m.append_slots(0, 5)               # ids unknown
    m.append_tokens(0, [9] * 8)
    assert len(m.pool.cached_block_hash_to_block) == 0


def test_disabled_caching_changes_nothing():
    m1 = SequenceManager(16, BS)
    m2 = SequenceManager(16, BS)
    p = list(range(9))
    for m in (m1, m2):
        m.add_seq(0)
    assert m1.add_seq_cached(1, p) == 0
    m1.append_tokens(1, p)
    m2.add_seq(1)
    m2.append_slots(1, len(p))
    assert m1.free_list() == m2.free_list() and m1.block_table(1) == m2.block_table(1)
    assert m1.pool.cached_block_hash_to_block == {}


@pytest.mark.parametrize("seed", range(6))
def test_random_scripts_hits_always_hold_the_prompt_tokens(seed):
    """Content model: every slot written by append_tokens records its token id;
    a cache hit must return blocks whose recorded ids are exactly the prompt's
    tokens for those positions (and the blocks before them matched too)."""
    rng = random.Random(seed)
    nb = 40
    m = _mgr(nb)
    content = {}                       # slot -> token id
    prompts = [[rng.randrange(3) for _ in range(rng.randrange(1, 5) * BS + rng.randrange(BS))]
               for _ in range(6)]
    live = {}
    next_id = 0
    for _ in range(300):
        if live and rng.random() < 0.35:
            seq = rng.choice(sorted(live))
            m.free_seq(seq)
            del live[seq]
            continue
        base = rng.choice(prompts)
        prompt = base + [rng.randrange(3) for _ in range(rng.randrange(3))]
        seq = next_id
        next_id += 1
        try:
            got = m.add_seq_cached(seq, prompt, salt=rng.randrange(2))
        except Exception:
            raise
        table = m.block_table(seq)
        assert got == len(table) * BS and got <= max(len(prompt) - 1, 0)
        for i, b in enumerate(table):
            for k in range(BS):
                assert content.get(b * BS + k) == prompt[i * BS + k]
        try:
            slots = m.append_tokens(seq, prompt[got:])
        except Exception:               # pool exhausted: drop the request
            m.free_seq(seq)
            continue
        for s_, t in zip(slots, prompt[got:]):
            content[s_] = t
        live[seq] = prompt
        # invariants: map and block hashes agree; cached blocks are free or referenced
        for h, b in m.pool.cached_block_hash_to_block.items():
            assert m.pool.block_hash[b] == h
        refs = [0] * nb
        for q in live:
            for b in m.block_table(q):
                refs[b] += 1
        assert refs == m.pool.ref_cnt
        assert sorted(m.free_list()) == [b for b in range(nb) if refs[b] == 0]


def test_block_hash_is_chained_over_the_parent():
    # a change of parent alone changes the hash; equal inputs give equal hashes
    t = [1, 2, 3, 4]
    assert block_hash(0, t) == block_hash(0, list(t))
    assert block_hash(0, t) != block_hash(1, t)
    assert block_hash(0, t) != block_hash(0, [1, 2, 3, 5])
