"""The C++ block allocator against the oracle allocator, field by field.

Seeded random scripts (allocate, append, share, copy-on-write, free, pool
exhaustion) replay on both; refcounts, free-queue order, tables, lengths and
outputs must match exactly, and every error must leave both states unchanged.
A host ASan/UBSan build of the allocator runs the same kind of script.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle.block_pool import AllocError, NoFreeBlocks, SequenceManager
from paged_kv_cache_76_gb300 import _lib
from paged_kv_cache_76_gb300.allocator import BlockAllocator
from paged_kv_cache_76_gb300.allocator import NoFreeBlocks as CNoFree

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    try:
        _lib.lib()
    except _lib.LibraryMissing:
        from paged_kv_cache_76_gb300 import build
        build.build()


def assert_same(c: BlockAllocator, o: SequenceManager):
    assert c.num_free() == o.num_free()
    assert c.free_list() == o.free_list()
    assert [c.ref(b) for b in range(c.num_blocks)] == o.pool.ref_cnt
    assert sorted(o.tables) == sorted(s for s in o.tables)
    for s in o.tables:
        assert c.block_table(s) == o.block_table(s)
        assert c.seq_len(s) == o.num_tokens[s]
    st = c.stats()
    assert st["num_seqs"] == len(o.tables) and st["cow_copies"] == o.cow_copies
    assert st["waste_slots"] == sum(o.waste(s) for s in o.tables)


def test_worked_example_on_the_cpp_allocator():
    order = [7, 2, 5] + [b for b in range(16) if b not in (7, 2, 5)]
    c = BlockAllocator(16, 4, order)
    c.add_seq(0)
    assert c.append_slots(0, 9).tolist() == [28, 29, 30, 31, 8, 9, 10, 11, 20]
    assert c.block_table(0) == [7, 2, 5]
    assert c.append_slots(0, 3).tolist() == [21, 22, 23] and c.num_free() == 13
    assert c.append_slots(0, 1).tolist() == [order[3] * 4]      # token index 12 takes a 4th block


def _do(target, op, *args):
    try:
        return ("ok", getattr(target, op)(*args))
    except (NoFreeBlocks, CNoFree):
        return ("nofree", None)
    except (AllocError, _lib.PAError) as e:
        if isinstance(e, _lib.PAError) and e.status == _lib.PA_ERR_NO_FREE_BLOCKS:
            return ("nofree", None)
        return ("err", None)


@pytest.mark.parametrize("seed", range(6))
def test_random_scripts_match_the_oracle_bit_exactly(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(8, 80))
    bs = int(rng.choice([1, 2, 4, 16]))
    order = rng.permutation(nb).astype(np.int32)
    c = BlockAllocator(nb, bs, order)
    o = SequenceManager(nb, bs, order)
    live = []
    next_id = 0
    for step in range(600):
        kind = rng.choice(["add", "append", "append", "append", "share", "cow", "free", "bad"])
        if kind == "add" or not live:
            pair = (_do(c, "add_seq", next_id), _do(o, "add_seq", next_id))
            live.append(next_id)
            next_id += 1
        elif kind == "append":
            s = int(rng.choice(live))
            n = int(rng.integers(0, 3 * bs + 2))
            rc, ro = _do(c, "append_slots", s, n), _do(o, "append_slots", s, n)
            if rc[0] == "ok" and ro[0] == "ok":
                assert rc[1].tolist() == ro[1]
            pair = (rc, ro)
        elif kind == "share":
            src = int(rng.choice(live))
            n = int(rng.integers(0, o.num_tokens[src] + 1))
            _do(c, "add_seq", next_id), _do(o, "add_seq", next_id)
            pair = (_do(c, "share", next_id, src, n), _do(o, "share", next_id, src, n))
            live.append(next_id)
            next_id += 1
        elif kind == "cow":
            s = int(rng.choice(live))
            lb = int(rng.integers(-1, len(o.tables[s]) + 1))
            rc, ro = _do(c, "cow", s, lb), _do(o, "cow", s, lb)
            if rc[0] == "ok" and ro[0] == "ok":
                assert tuple(rc[1]) == tuple(ro[1])
            pair = (rc, ro)
        elif kind == "free":
            s = int(rng.choice(live))
            pair = (_do(c, "free_seq", s), _do(o, "free_seq", s))
            live.remove(s)
        else:  # invalid requests: unknown sequence, double free, bad block id
            s = next_id + 1000
            pair = (_do(c, "free_seq", s), _do(o, "free_seq", s))
            assert _do(c, "ref", nb)[0] == "err" and _do(o, "ref", nb)[0] == "err"
        assert pair[0][0] == pair[1][0], (step, kind, pair)
        assert_same(c, o)


def test_pool_exhaustion_is_all_or_nothing():
    c = BlockAllocator(4, 4)
    c.add_seq(0)
    c.append_slots(0, 10)
    with pytest.raises(CNoFree):
        c.append_slots(0, 7)
    assert c.block_table(0) == [0, 1, 2] and c.seq_len(0) == 10 and c.num_free() == 1
    assert c.stats()["alloc_failures"] == 1


def test_many_requests_cross_a_block_boundary_in_one_step():
    """Every request's next token needs a new block at once; the pool covers exactly that."""
    n = 32
    c = BlockAllocator(2 * n, 16)
    for s in range(n):
        c.add_seq(s)
        c.append_slots(s, 16)
    for s in range(n):
        assert c.append_slots(s, 1).tolist() == [c.block_table(s)[1] * 16]
    assert c.num_free() == 0
    c.add_seq(n)
    with pytest.raises(CNoFree):
        c.append_slots(n, 1)


def test_prefill_burst_exhausts_then_immediate_reuse():
    c = BlockAllocator(8, 16)
    c.add_seq(0)
    c.append_slots(0, 128)                    # all 8 blocks
    c.add_seq(1)
    with pytest.raises(CNoFree):
        c.append_slots(1, 1)
    tab = c.block_table(0)
    c.free_seq(0)
    assert c.free_list() == tab[::-1]        # reused tail-first, contents not cleared
    assert c.append_slots(1, 1).tolist() == [tab[-1] * 16]


def test_shared_append_needs_cow_first():
    c = BlockAllocator(10, 4)
    c.add_seq(0)
    c.append_slots(0, 6)
    c.add_seq(1)
    c.share(1, 0, 6)
    with pytest.raises(_lib.PAError) as e:
        c.append_slots(1, 1)
    assert e.value.status == _lib.PA_ERR_SHARED_BLOCK
    assert c.cow(1, 1) == (1, 2)
    assert c.append_slots(1, 2).tolist() == [10, 11]


def test_build_tables_pads_with_minus_one():
    c = BlockAllocator(10, 4)
    for s, n in ((3, 9), (5, 1)):
        c.add_seq(s)
        c.append_slots(s, n)
    t, lens = c.build_tables([5, 3], 4)
    assert t.tolist() == [[3, -1, -1, -1], [0, 1, 2, -1]] and lens.tolist() == [1, 9]
    with pytest.raises(_lib.PAError):
        c.build_tables([3], 2)


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host compiler")
def test_allocator_under_address_and_ub_sanitizers(tmp_path):
    exe = tmp_path / "alloc_fuzz"
    src = os.path.join(ROOT, "tests", "alloc_fuzz.cpp")
    alloc = os.path.join(ROOT, "paged_kv_cache_76_gb300", "csrc", "block_alloc.cpp")
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
                        "-I", os.path.join(ROOT, "include"), src, alloc, "-o", str(exe)],
                       capture_output=True, text=True)
    if r.returncode and "sanitize" in r.stderr:
        pytest.skip("sanitizer runtime unavailable: " + r.stderr[-200:])
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe), "8000"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok" in r.stdout


def test_common_prefix_counts_shared_full_blocks():
    c = BlockAllocator(64, 4)
    c.add_seq(0)
    c.append_slots(0, 22)                 # 5 full blocks + 2 tokens
    for s, n in ((1, 22), (2, 16), (3, 9)):
        c.add_seq(s)
        c.share(s, 0, n)
    assert c.common_prefix([0, 1]) == 5                # the partial 6th block does not count
    assert c.common_prefix([0, 1, 2]) == 4
    assert c.common_prefix([0, 3]) == 2
    assert c.common_prefix([1]) == 5
    c.cow(1, 1)                                        # seq 1's second block becomes private
    assert c.common_prefix([0, 1]) == 1
    c.add_seq(9)
    c.append_slots(9, 8)
    assert c.common_prefix([0, 9]) == 0
    with pytest.raises(_lib.PAError):
        c.common_prefix([0, 12345])


# ---------------------------------------------------------------- prefix caching
def test_block_hash_matches_the_oracle():
    from oracle.block_pool import block_hash
    rng = np.random.default_rng(7)
    L = _lib.lib()
    for _ in range(50):
        parent = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        toks = rng.integers(-2**31, 2**31, size=int(rng.integers(0, 20)), dtype=np.int64).astype(np.int32)
        ptr = toks.ctypes.data_as(_lib.C.POINTER(_lib.C.c_int32)) if toks.size else None
        assert L.pa_block_hash(parent, ptr, int(toks.size)) == block_hash(parent, toks.tolist())


def assert_same_cache(c: BlockAllocator, o: SequenceManager):
    assert_same(c, o)
    for b in range(c.num_blocks):
        assert c.block_hash(b) == o.pool.block_hash[b]
    st = c.prefix_cache_stats()
    assert st == {"lookup_blocks": o.lookup_blocks, "hit_blocks": o.hit_blocks, "evictions": o.pool.evictions,
                  "cached_blocks": len(o.pool.cached_block_hash_to_block)}


@pytest.mark.parametrize("seed", range(8))
def test_prefix_cache_scripts_match_the_oracle_bit_exactly(seed):
    rng = np.random.default_rng(100 + seed)
    nb = int(rng.integers(12, 60))
    bs = int(rng.choice([1, 2, 4, 16]))
    order = rng.permutation(nb).astype(np.int32)
    c = BlockAllocator(nb, bs, order)
    o = SequenceManager(nb, bs, order)
    if seed % 4 != 3:  # one script in four runs with caching off
        c.enable_prefix_caching()
        o.enable_prefix_caching()
    prompts = [rng.integers(0, 3, size=int(rng.integers(1, 4 * bs + 3))).tolist() for _ in range(5)]
    live, next_id = [], 0
    for step in range(500):
        kind = rng.choice(["add_cached", "add_cached", "append_tokens", "append_tokens", "append", "share",
                           "cow", "free", "free"])
        if kind == "add_cached" or not live:
            p = prompts[int(rng.integers(len(prompts)))] + rng.integers(0, 3, size=int(rng.integers(0, 3))).tolist()
            salt = int(rng.integers(0, 2))
            rc, ro = _do(c, "add_seq_cached", next_id, p, salt), _do(o, "add_seq_cached", next_id, p, salt)
            assert rc == ro, (step, rc, ro)
            live.append(next_id)
            next_id += 1
            if rc[0] == "ok":  # the prompt's uncached tokens
                rest = p[rc[1]:]
                rc, ro = _do(c, "append_tokens", next_id - 1, rest), _do(o, "append_tokens", next_id - 1, rest)
                if rc[0] == "ok" and ro[0] == "ok":
                    assert rc[1].tolist() == ro[1]
            pair = (rc, ro)
        elif kind == "append_tokens":
            s = int(rng.choice(live))
            t = rng.integers(0, 3, size=int(rng.integers(0, 2 * bs + 2))).tolist()
            rc, ro = _do(c, "append_tokens", s, t), _do(o, "append_tokens", s, t)
            if rc[0] == "ok" and ro[0] == "ok":
                assert rc[1].tolist() == ro[1]
            pair = (rc, ro)
        elif kind == "append":
            s = int(rng.choice(live))
            n = int(rng.integers(0, bs + 2))
            pair = (_do(c, "append_slots", s, n), _do(o, "append_slots", s, n))
        elif kind == "share":
            src = int(rng.choice(live))
            n = int(rng.integers(0, o.num_tokens[src] + 1))
            _do(c, "add_seq", next_id), _do(o, "add_seq", next_id)
            pair = (_do(c, "share", next_id, src, n), _do(o, "share", next_id, src, n))
            live.append(next_id)
            next_id += 1
        elif kind == "cow":
            s = int(rng.choice(live))
            lb = int(rng.integers(0, len(o.tables[s]) + 1))
            rc, ro = _do(c, "cow", s, lb), _do(o, "cow", s, lb)
            if rc[0] == "ok" and ro[0] == "ok":
                assert tuple(rc[1]) == tuple(ro[1])
            pair = (rc, ro)
        else:
            s = int(rng.choice(live))
            pair = (_do(c, "free_seq", s), _do(o, "free_seq", s))
            live.remove(s)
        assert pair[0][0] == pair[1][0], (step, kind, pair)
        assert_same_cache(c, o)


# ---------------------------------------------------------------- swapping
def assert_same_swap(c: BlockAllocator, o: SequenceManager):
    assert_same(c, o)
    assert c.num_free_cpu() == o.num_free_cpu()
    for s in o.tables:
        assert c.is_swapped(s) == (s in o.on_cpu)


@pytest.mark.parametrize("seed", range(8))
def test_swap_scripts_match_the_oracle_bit_exactly(seed):
    rng = np.random.default_rng(300 + seed)
    nb = int(rng.integers(8, 48))
    ncpu = int(rng.integers(2, 40))
    bs = int(rng.choice([1, 2, 4, 16]))
    order = rng.permutation(nb).astype(np.int32)
    c = BlockAllocator(nb, bs, order)
    o = SequenceManager(nb, bs, order)
    caching = seed % 2 == 0
    for m in (c, o):
        if caching:
            m.enable_prefix_caching()
        m.enable_swap(ncpu)
    prompts = [rng.integers(0, 3, size=int(rng.integers(1, 3 * bs + 3))).tolist() for _ in range(4)]
    live, next_id = [], 0
    for step in range(500):
        kind = rng.choice(["add", "append", "append", "share", "cow", "free", "swap_out", "swap_out",
                           "swap_in", "swap_in"])
        if kind == "add" or not live:
            p = prompts[int(rng.integers(len(prompts)))] + rng.integers(0, 3, size=int(rng.integers(0, 3))).tolist()
            rc, ro = _do(c, "add_seq_cached", next_id, p), _do(o, "add_seq_cached", next_id, p)
            assert rc == ro
            live.append(next_id)
            next_id += 1
            if rc[0] == "ok":
                rest = p[rc[1]:]
                rc, ro = _do(c, "append_tokens", next_id - 1, rest), _do(o, "append_tokens", next_id - 1, rest)
                if rc[0] == "ok" and ro[0] == "ok":
                    assert rc[1].tolist() == ro[1]
            pair = (rc, ro)
        elif kind == "append":
            s = int(rng.choice(live))
            t = rng.integers(0, 3, size=int(rng.integers(0, 2 * bs + 2))).tolist()
            rc, ro = _do(c, "append_tokens", s, t), _do(o, "append_tokens", s, t)
            if rc[0] == "ok" and ro[0] == "ok":
                assert rc[1].tolist() == ro[1]
            pair = (rc, ro)
        elif kind == "share":
            src = int(rng.choice(live))
            n = int(rng.integers(0, o.num_tokens[src] + 1))
            _do(c, "add_seq", next_id), _do(o, "add_seq", next_id)
            pair = (_do(c, "share", next_id, src, n), _do(o, "share", next_id, src, n))
            live.append(next_id)
            next_id += 1
        elif kind == "cow":
            s = int(rng.choice(live))
            lb = int(rng.integers(0, len(o.tables[s]) + 1))
            rc, ro = _do(c, "cow", s, lb), _do(o, "cow", s, lb)
            if rc[0] == "ok" and ro[0] == "ok":
                assert tuple(rc[1]) == tuple(ro[1])
            pair = (rc, ro)
        elif kind in ("swap_out", "swap_in"):
            s = int(rng.choice(live))
            rc, ro = _do(c, kind, s), _do(o, kind, s)
            if rc[0] == "ok" and ro[0] == "ok":
                assert rc[1].tolist() == [list(p) for p in ro[1]]
            pair = (rc, ro)
        else:
            s = int(rng.choice(live))
            pair = (_do(c, "free_seq", s), _do(o, "free_seq", s))
            live.remove(s)
        assert pair[0][0] == pair[1][0], (step, kind, pair)
        assert_same_swap(c, o)
        if caching:
            for b in range(nb):
                assert c.block_hash(b) == o.pool.block_hash[b]


def test_swap_needs_a_pool_and_a_large_enough_pairs_buffer():
    c = BlockAllocator(8, 4)
    c.add_seq(0)
    c.append_slots(0, 9)
    with pytest.raises(_lib.PAError):
        c.swap_out(0)                                  # no swap pool yet
    c.enable_swap(4)
    with pytest.raises(_lib.PAError):
        c.enable_swap(4)                               # set once
    L = _lib.lib()
    n = _lib.C.c_int(0)
    out = np.empty((2, 2), dtype=np.int32)
    st = L.pa_alloc_swap_out(c._h, 0, out.ctypes.data_as(_lib.C.POINTER(_lib.C.c_int32)), 2, _lib.C.byref(n))
    assert st == _lib.PA_ERR_INVALID and n.value == 3   # three pairs needed, nothing changed
    assert not c.is_swapped(0) and c.num_free() == 5 and c.num_free_cpu() == 4
    pairs = c.swap_out(0)
    assert pairs.shape == (3, 2) and c.is_swapped(0) and c.num_free() == 8 and c.num_free_cpu() == 1
