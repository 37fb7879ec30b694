"""Checkpoint and resume of the C++ host allocator (pa_alloc_export /
pa_alloc_import), on the CPU.

An allocator rebuilt from another's words must behave as the original for
every later call: seeded random scripts (sequences, appends, sharing,
copy-on-write, frees, prefix caching, swapping) run on both in lockstep after
a checkpoint, with equal results and equal exported words after every
operation.  Malformed words are refused without building an allocator."""
import numpy as np
import pytest

from paged_kv_cache_76_gb300 import _lib
from paged_kv_cache_76_gb300.allocator import BlockAllocator


@pytest.fixture(scope="module", autouse=True)
def built():
    try:
        _lib.lib()
    except _lib.LibraryMissing:
        from paged_kv_cache_76_gb300 import build
        build.build()


def _do(alloc, op, *args):
    try:
        r = getattr(alloc, op)(*args)
    except _lib.PAError as e:
        return ("err", type(e).__name__)
    if isinstance(r, np.ndarray):
        r = r.tolist()
    return ("ok", r)


def _script_op(rng, live, prompts, next_id, caching, swapping, bs):
    """One random operation: (name, args, new live ids, removed id)."""
    kinds = ["add", "append", "append", "share", "cow", "free"]
    if caching:
        kinds += ["add_cached", "append_tokens", "append_tokens"]
    if swapping:
        kinds += ["swap_out", "swap_in"]
    kind = str(rng.choice(kinds)) if live else ("add_cached" if caching else "add")
    if kind == "add":
        return "add_seq", (next_id,), [next_id], None
    if kind == "add_cached":
        p = prompts[int(rng.integers(len(prompts)))] + rng.integers(0, 3, size=int(rng.integers(0, 3))).tolist()
        return "add_seq_cached", (next_id, p, int(rng.integers(0, 2))), [next_id], None
    s = int(rng.choice(live))
    if kind == "append":
        return "append_slots", (s, int(rng.integers(0, bs + 2))), [], None
    if kind == "append_tokens":
        return "append_tokens", (s, rng.integers(0, 3, size=int(rng.integers(0, 2 * bs + 2))).tolist()), [], None
    if kind == "share":
        return "share_new", (next_id, s, int(rng.integers(0, 4 * bs))), [next_id], None
    if kind == "cow":
        return "cow", (s, int(rng.integers(0, 6))), [], None
    if kind == "swap_out":
        return "swap_out", (s,), [], None
    if kind == "swap_in":
        return "swap_in", (s,), [], None
    return "free_seq", (s,), [], s


def _apply(alloc, name, args):
    if name == "share_new":  # a fresh sequence sharing the first n tokens of another
        r1 = _do(alloc, "add_seq", args[0])
        return (r1, _do(alloc, "share", *args))
    return _do(alloc, name, *args)


@pytest.mark.parametrize("seed", range(8))
def test_a_restored_allocator_behaves_as_the_original(seed):
    rng = np.random.default_rng(900 + seed)
    nb = int(rng.integers(10, 50))
    bs = int(rng.choice([1, 2, 4, 16]))
    caching, swapping = seed % 2 == 0, seed % 4 < 2
    order = rng.permutation(nb).astype(np.int32)
    a = BlockAllocator(nb, bs, order)
    if caching:
        a.enable_prefix_caching()
    if swapping:
        a.enable_swap(int(rng.integers(4, 30)))
    prompts = [rng.integers(0, 3, size=int(rng.integers(1, 4 * bs + 3))).tolist() for _ in range(4)]
    b = None
    live, next_id = [], 0
    restores = 0
    for step in range(400):
        if step % 53 == 17:  # checkpoint the original, resume a fresh copy from the words
            w = a.export()
            if b is not None:
                assert np.array_equal(w, b.export())
                b.close()
            b = BlockAllocator.from_words(w)
            assert np.array_equal(b.export(), w)
            restores += 1
        name, args, new, gone = _script_op(rng, live, prompts, next_id, caching, swapping, bs)
        ra = _apply(a, name, args)
        if b is not None:
            assert _apply(b, name, args) == ra, (step, name, args)
            assert np.array_equal(a.export(), b.export()), (step, name)
        live += new
        next_id += len(new)
        if gone is not None:
            live.remove(gone)
    assert restores >= 7
    # observable state agrees too
    assert a.free_list() == b.free_list() and a.stats() == b.stats()
    for s in live:
        assert a.block_table(s) == b.block_table(s)


def _valid_words():
    a = BlockAllocator(12, 4, np.arange(12, dtype=np.int32)[::-1].copy())
    a.enable_prefix_caching()
    a.enable_swap(8)
    a.add_seq_cached(0, [1, 2, 1, 0, 2, 2, 1, 0, 1], 0)
    a.append_tokens(0, [1, 2, 1, 0, 2, 2, 1, 0, 1])
    a.add_seq(1)
    a.share(1, 0, 6)
    a.add_seq(2)
    a.append_slots(2, 5)
    a.swap_out(2)
    return a.export()


def test_malformed_words_are_refused():
    w = _valid_words()
    BlockAllocator.from_words(w)  # the untouched words import
    bad = []
    bad.append(w[:-1])                         # truncated
    bad.append(np.concatenate([w, [0]]))       # trailing word
    x = w.copy(); x[0] += 1; bad.append(x)     # magic
    x = w.copy(); x[1] = 2; bad.append(x)      # version
    x = w.copy(); x[2] = 0; bad.append(x)      # no blocks
    x = w.copy(); x[11] = 13; bad.append(x)    # more free blocks than blocks
    x = w.copy(); x[12] = x[13]; bad.append(x)  # a block twice in the free queue
    x = w.copy(); x[12] = 12; bad.append(x)    # a block id past the pool
    nfree = int(w[11])
    x = w.copy(); x[12 + nfree] += 1; bad.append(x)  # a refcount that no table accounts for
    # a swap pool larger than the words could describe: refused before the
    # pool's bookkeeping is sized (a 2^31-block pool would be gigabytes)
    x = w.copy(); x[5] = 2**31 - 1; bad.append(x)
    x = w.copy(); x[5] = len(w) + 1; bad.append(x)
    for v in bad:
        with pytest.raises(_lib.PAError):
            BlockAllocator.from_words(v)


def _seq_words(w):
    """Index of each sequence's record in exported words: {seq id: (index of its
    block count, index of its pending count)}, following the export layout."""
    nb = int(w[2])
    i = 11
    nfree = int(w[i]); i += 1 + nfree
    i += 3 * nb                                   # refcounts, hash flags, hashes
    ncached = int(w[i]); i += 1 + 2 * ncached
    ncpu_free = int(w[i]); i += 1 + ncpu_free
    nseq = int(w[i]); i += 1
    out = {}
    for _ in range(nseq):
        sid = int(w[i])
        nblk_at = i + 6
        nblk = int(w[nblk_at])
        np_at = nblk_at + 1 + nblk
        out[sid] = (nblk_at, np_at)
        i = np_at + 1 + int(w[np_at])
    assert i == len(w)
    return out


def test_a_swap_block_held_twice_is_refused():
    """Two swapped-out sequences must not hold the same swap block, and no
    swap block may be neither free nor held (it would leak, and the next two
    swap-outs would both get the other one)."""
    a = BlockAllocator(8, 4)
    a.enable_swap(4)
    for s in (1, 2):
        a.add_seq(s)
        a.append_slots(s, 3)
        a.swap_out(s)
    w = a.export()
    BlockAllocator.from_words(w)
    at = _seq_words(w)
    b1, b2 = int(w[at[1][0] + 1]), int(w[at[2][0] + 1])
    assert b1 != b2
    x = w.copy()
    x[at[2][0] + 1] = b1                          # sequence 2 now claims sequence 1's swap block
    with pytest.raises(_lib.PAError):
        BlockAllocator.from_words(x)


def test_pending_tokens_of_a_full_block_are_refused():
    w = _valid_words()
    at = _seq_words(w)
    sid = next(s for s, (_, p) in at.items() if int(w[p]) > 0)
    p = at[sid][1]
    n = int(w[p])
    x = np.concatenate([w[:p], [4], w[p + 1:p + 1 + n], np.zeros(4 - n, w.dtype), w[p + 1 + n:]])
    assert len(x) == len(w) + 4 - n
    with pytest.raises(_lib.PAError):             # block_size 4: at most 3 pending token ids
        BlockAllocator.from_words(x)
    y = np.concatenate([w[:p], [3], w[p + 1:p + 1 + n], np.zeros(3 - n, w.dtype), w[p + 1 + n:]])
    BlockAllocator.from_words(y)                  # 3 is still a valid count


def test_random_corruptions_never_crash_and_what_imports_round_trips():
    w = _valid_words()
    rng = np.random.default_rng(4)
    accepted = 0
    for _ in range(2000):
        x = w.copy()
        k = int(rng.integers(len(x)))
        x[k] = int(rng.choice([x[k] + 1, x[k] - 1, -1, 0, 1 << 40, int(rng.integers(-5, 50))]))
        try:
            b = BlockAllocator.from_words(x)
        except _lib.PAError:
            continue
        accepted += 1
        assert np.array_equal(BlockAllocator.from_words(b.export()).export(), b.export())
    assert accepted < 2000
