"""Block allocator of a paged KV cache, restated from the pages' design.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"2.1 PagedAttention" §9.1-9.3 splits the work in two:

* a global pool of physical blocks (BlockPool) with a free queue that is a
  doubly linked list (FreeKVCacheBlockQueue: O(1) popleft and O(1) removal
  from the middle, §9.2) and a reference count per block (§9.3);
* a per-request manager (KVCacheManager, §9.1) that grows a request's Block
  Table on demand (a new block only when the last one is full, §3), and frees
  its blocks in reverse order when it ends (tail blocks first).

BlockPool's get_new_blocks, free_blocks and touch take the steps of the
pages' BlockPool listing (§9.3) in the listing's order, and keep its names
for the lists they build (to_free, no_hash, has_hash), by design: the listing
is the only definition of the allocator's semantics that the pages give, and
this module is the oracle that restates it.  The product allocator is a
separate design and does not follow the listing's structure.

Sharing and Copy-on-Write follow §6: tables may point at the same physical
block (refcount = number of tables), and a request about to write a shared
block first copies it into a private one, repoints its table entry and drops
one reference on the original.

Readings (the pages disagree or are silent):

* free_blocks: the Vietnamese edition's pseudocode puts freed blocks with
  no hash at the head of the free queue (reused first) and hashed ones at
  the tail; the Chinese edition's pseudocode appends every freed block at the
  tail, while its own prose describes head/tail placement.  We follow the
  head/tail rule.  No block carries a hash here, so every freed block goes to
  the head, in the order given: freeing a request hands the list
  [b_last, ..., b_0] to prepend_n, so b_last is reused first.
* The initial free queue is the given order (ascending ids by default).
* A request may only append into its partially filled last block if no other
  table shares that block; otherwise the caller copies it first (cow).
* cow on a block with refcount 1 is a no-op that returns (b, b).
* Every operation either succeeds fully or leaves the state unchanged.

Automatic prefix caching ("Khám phá vLLM … phần 2", prefix caching;
"2.1 PagedAttention" §9.2-9.3), when enabled:

* only full blocks are cached.  Block i of a request gets the hash
  H(h_{i-1}, its token ids), chained from the previous block's hash, with a
  per-request salt in place of h_{-1} (the pages fold a cache salt into the
  first block's hash so that only requests with the same salt share blocks).
  H is 64-bit FNV-1a over the parent hash (8 bytes, little-endian) followed
  by the token ids (4 bytes each, little-endian, two's complement); the pages
  leave the function open (Python's hash or SHA-256), FNV-1a is a published
  one that a C implementation can reproduce exactly.
* a new request looks its prompt's full blocks up in order and stops at the
  first miss (find_longest_cache_hit); hits are touched.  Reading: the hit
  is capped at floor((n-1)/bs) blocks of an n-token prompt, so that at least
  one prompt token is computed (the model needs it to produce the next
  token); the pages' example always continues past the cached prefix.
* a block is registered (hash -> block) when it becomes full through an
  append that carries token ids; if that hash is already cached by another
  block, the new block stays unregistered (the first one remains the cached
  copy).  Appends without token ids end the request's hashing.
* a freed zero-count block with a hash goes to the tail of the free queue,
  without one to the head (the free_blocks rule above), so cached blocks are
  evicted in release order, the first block of a request last.
* a cached block loses its hash only when the free queue hands it out again
  (popleft): its map entry is removed then.

Swapping ("2.1 PagedAttention" §7, preemption by swapping), when a swap pool
of CPU blocks is set up:

* swap_out copies every block of a request into CPU blocks taken from the
  head of the swap pool's free queue (one per logical block, in order, shared
  blocks included) and then releases its GPU blocks exactly as free_seq
  would.  The request keeps its id and token count; its table now lists its
  CPU blocks and it can neither grow nor be shared or copied until swap_in.
* swap_in takes one GPU block per CPU block from the head of the free queue
  (new private blocks: sharing is not restored, cached hashes are not
  carried over) and returns the CPU blocks to the head of the swap pool's
  queue in reverse order.  Both return the (source, destination) pairs the
  caller copies with swap_blocks before reusing the source blocks.
* free_seq on a swapped-out request returns its CPU blocks.
"""
from __future__ import annotations

__all__ = ["NoFreeBlocks", "AllocError", "FreeBlockQueue", "BlockPool", "SequenceManager", "fnv1a64",
           "block_hash"]

FNV64_OFFSET = 0xCBF29CE484222325
FNV64_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """64-bit FNV-1a: for each byte, xor it in, then multiply by the FNV prime."""
    h = FNV64_OFFSET
    for byte in data:
        h ^= byte
        h = (h * FNV64_PRIME) & MASK64
    return h


def block_hash(parent: int, tokens) -> int:
    """Chained hash of one full block: FNV-1a of parent (8 bytes LE) + token ids (4 bytes LE each)."""
    data = (parent & MASK64).to_bytes(8, "little") + b"".join(
        (int(t) & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return fnv1a64(data)


class NoFreeBlocks(Exception):
    """Not enough free blocks; the scheduler above would preempt (§7, §9.1)."""


class AllocError(Exception):
    """Invalid request (unknown sequence, bad index, shared partial block...)."""


class FreeBlockQueue:
    """Doubly linked list of free block ids (head = next to be allocated)."""

    def __init__(self, order):
        self.prev = {}
        self.next = {}
        self.head = None
        self.tail = None
        self.n = 0
        for b in order:
            self._push_back(int(b))

    def __len__(self):
        return self.n

    def __contains__(self, b):
        return b in self.prev

    def _push_back(self, b):
        self.prev[b] = self.tail
        self.next[b] = None
        if self.tail is None:
            self.head = b
        else:
            self.next[self.tail] = b
        self.tail = b
        self.n += 1

    def _push_front(self, b):
        self.next[b] = self.head
        self.prev[b] = None
        if self.head is None:
            self.tail = b
        else:
            self.prev[self.head] = b
        self.head = b
        self.n += 1

    def remove(self, b):
        p, nx = self.prev.pop(b), self.next.pop(b)
        if p is None:
            self.head = nx
        else:
            self.next[p] = nx
        if nx is None:
            self.tail = p
        else:
            self.prev[nx] = p
        self.n -= 1

    def popleft_n(self, n):
        out = []
        for _ in range(n):
            b = self.head
            self.remove(b)
            out.append(b)
        return out

    def prepend_n(self, blocks):
        """Put ``blocks`` at the head, keeping their order (blocks[0] first)."""
        for b in reversed(list(blocks)):
            self._push_front(b)

    def append_n(self, blocks):
        for b in blocks:
            self._push_back(b)

    def to_list(self):
        out, b = [], self.head
        while b is not None:
            out.append(b)
            b = self.next[b]
        return out


class BlockPool:
    """Global physical blocks: refcounts and the free queue (§9.3 pseudocode)."""

    def __init__(self, num_blocks, initial_free_order=None):
        order = list(range(num_blocks)) if initial_free_order is None else [int(x) for x in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise AllocError("initial free order must be a permutation of the block ids")
        self.num_blocks = num_blocks
        self.ref_cnt = [0] * num_blocks
        self.block_hash = [None] * num_blocks
        self.free_block_queue = FreeBlockQueue(order)
        self.caching = False
        self.cached_block_hash_to_block = {}
        self.evictions = 0

    def get_num_free_blocks(self):
        return len(self.free_block_queue)

    def get_new_blocks(self, num_blocks):
        if num_blocks > self.get_num_free_blocks():
            raise NoFreeBlocks(f"need {num_blocks}, have {self.get_num_free_blocks()}")
        blocks = self.free_block_queue.popleft_n(num_blocks)
        for b in blocks:
            assert self.ref_cnt[b] == 0
            self.ref_cnt[b] += 1
            h = self.block_hash[b]
            if h is not None:
                # a cached block about to be overwritten: it leaves the cache
                if self.cached_block_hash_to_block.get(h) == b:
                    del self.cached_block_hash_to_block[h]
                self.block_hash[b] = None
                self.evictions += 1
        return blocks

    def free_blocks(self, ordered_blocks):
        for b in ordered_blocks:
            self.ref_cnt[b] -= 1
        to_free = [b for b in ordered_blocks if self.ref_cnt[b] == 0]
        no_hash = [b for b in to_free if self.block_hash[b] is None]
        has_hash = [b for b in to_free if self.block_hash[b] is not None]
        self.free_block_queue.prepend_n(no_hash)
        self.free_block_queue.append_n(has_hash)

    def touch(self, blocks):
        for b in blocks:
            if self.ref_cnt[b] == 0:
                self.free_block_queue.remove(b)
            self.ref_cnt[b] += 1


class SequenceManager:
    """Per-request Block Tables on top of a :class:`BlockPool` (§9.1, §3, §6)."""

    def __init__(self, num_blocks, block_size, initial_free_order=None):
        if block_size <= 0 or num_blocks <= 0:
            raise AllocError("num_blocks and block_size must be positive")
        self.block_size = block_size
        self.pool = BlockPool(num_blocks, initial_free_order)
        self.tables = {}
        self.num_tokens = {}
        self.cow_copies = 0
        self.alloc_failures = 0
        # prefix caching: per request the salt, the hash of its last full
        # block (the salt before the first) and the token ids of its partial
        # last block (None: its tokens are not known, nothing more is hashed)
        self.salt = {}
        self.parent = {}
        self.pending = {}
        self.lookup_blocks = 0
        self.hit_blocks = 0
        # swapping: the swap pool's free queue and the swapped-out requests
        self.cpu_free = None
        self.on_cpu = set()

    def enable_prefix_caching(self):
        self.pool.caching = True

    def enable_swap(self, num_cpu_blocks):
        if num_cpu_blocks <= 0 or self.cpu_free is not None:
            raise AllocError("swap pool: positive size, set once")
        self.cpu_free = FreeBlockQueue(range(num_cpu_blocks))

    def num_free_cpu(self):
        return len(self.cpu_free) if self.cpu_free is not None else 0

    def _resident(self, seq):
        self._need(seq)
        if seq in self.on_cpu:
            raise AllocError(f"sequence {seq} is swapped out")

    def swap_out(self, seq):
        """Move ``seq`` to the swap pool; returns its (gpu, cpu) block pairs."""
        self._resident(seq)
        if self.cpu_free is None:
            raise AllocError("no swap pool")
        table = self.tables[seq]
        if len(table) > len(self.cpu_free):
            self.alloc_failures += 1
            raise NoFreeBlocks(f"need {len(table)} swap blocks, have {len(self.cpu_free)}")
        cpu = self.cpu_free.popleft_n(len(table))
        pairs = list(zip(table, cpu))
        self.pool.free_blocks(list(reversed(table)))
        self.tables[seq] = cpu
        self.on_cpu.add(seq)
        return pairs

    def swap_in(self, seq):
        """Bring ``seq`` back into GPU blocks; returns its (cpu, gpu) block pairs."""
        self._need(seq)
        if seq not in self.on_cpu:
            raise AllocError(f"sequence {seq} is not swapped out")
        cpu = self.tables[seq]
        if len(cpu) > self.num_free():
            self.alloc_failures += 1
            raise NoFreeBlocks(f"need {len(cpu)}, have {self.num_free()}")
        gpu = self.pool.get_new_blocks(len(cpu))
        pairs = list(zip(cpu, gpu))
        self.cpu_free.prepend_n(list(reversed(cpu)))
        self.tables[seq] = gpu
        self.on_cpu.discard(seq)
        return pairs

    # -- queries -----------------------------------------------------------
    def num_free(self):
        return self.pool.get_num_free_blocks()

    def ref(self, b):
        if not 0 <= b < self.pool.num_blocks:
            raise AllocError("block id out of range")
        return self.pool.ref_cnt[b]

    def block_table(self, seq):
        self._need(seq)
        return list(self.tables[seq])

    def free_list(self):
        return self.pool.free_block_queue.to_list()

    def waste(self, seq):
        """Allocated but unused slots of ``seq`` (all in its last block)."""
        self._need(seq)
        return len(self.tables[seq]) * self.block_size - self.num_tokens[seq]

    # -- operations ----------------------------------------------------------
    def _need(self, seq):
        if seq not in self.tables:
            raise AllocError(f"unknown sequence {seq}")

    def add_seq(self, seq, salt=0):
        if seq in self.tables:
            raise AllocError(f"sequence {seq} exists")
        self.tables[seq] = []
        self.num_tokens[seq] = 0
        self.salt[seq] = salt
        self.parent[seq] = salt
        self.pending[seq] = []

    def add_seq_cached(self, seq, tokens, salt=0):
        """New request with prompt ``tokens``: its table starts with the longest
        run of cached full blocks of the prompt (at most floor((n-1)/bs)).
        Returns the number of prompt tokens covered (a multiple of bs)."""
        self.add_seq(seq, salt)
        if not self.pool.caching:
            return 0
        bs = self.block_size
        nfull = (len(tokens) - 1) // bs if len(tokens) > 0 else 0
        parent, hits = salt, []
        for i in range(nfull):
            h = block_hash(parent, tokens[i * bs:(i + 1) * bs])
            self.lookup_blocks += 1
            b = self.pool.cached_block_hash_to_block.get(h)
            if b is None:
                break
            hits.append(b)
            parent = h
        self.hit_blocks += len(hits)
        self.pool.touch(hits)
        self.tables[seq] = hits
        self.num_tokens[seq] = len(hits) * bs
        self.parent[seq] = parent
        return len(hits) * bs

    def append_slots(self, seq, n):
        """Give the next ``n`` tokens of ``seq`` their slots, growing on demand."""
        self._resident(seq)
        slots = self._grow(seq, n)
        if n > 0:
            self.pending[seq] = None  # token ids unknown: no more hashing for seq
        return slots

    def append_tokens(self, seq, tokens):
        """append_slots for tokens whose ids are known: every block they fill is
        hashed and, with prefix caching on, registered unless its hash is
        already cached."""
        tokens = [int(t) for t in tokens]
        self._resident(seq)
        slots = self._grow(seq, len(tokens))
        pend = self.pending[seq]
        if pend is None:
            return slots
        bs = self.block_size
        first = self.num_tokens[seq] - len(tokens)  # index of tokens[0] in seq
        for i, t in enumerate(tokens):
            pend.append(t)
            if len(pend) == bs:
                h = block_hash(self.parent[seq], pend)
                b = self.tables[seq][(first + i) // bs]
                if self.pool.caching and h not in self.pool.cached_block_hash_to_block:
                    self.pool.cached_block_hash_to_block[h] = b
                    self.pool.block_hash[b] = h
                self.parent[seq] = h
                pend.clear()
        return slots

    def _grow(self, seq, n):
        self._need(seq)
        if n < 0:
            raise AllocError("negative token count")
        bs = self.block_size
        table = self.tables[seq]
        cur = self.num_tokens[seq]
        if n > 0 and cur % bs != 0 and self.pool.ref_cnt[table[-1]] > 1:
            raise AllocError("last block is shared: copy it before writing")
        need = -(-(cur + n) // bs) - len(table)
        if need > self.num_free():
            self.alloc_failures += 1
            raise NoFreeBlocks(f"need {need}, have {self.num_free()}")
        table.extend(self.pool.get_new_blocks(need))
        slots = []
        for t in range(cur, cur + n):
            slots.append(table[t // bs] * bs + t % bs)
        self.num_tokens[seq] = cur + n
        return slots

    def share(self, dst, src, n_tokens):
        """``dst`` (empty) starts with the first ``n_tokens`` of ``src``'s KV."""
        self._resident(dst)
        self._resident(src)
        if self.tables[dst] or self.num_tokens[dst]:
            raise AllocError("share target must be empty")
        if not 0 <= n_tokens <= self.num_tokens[src]:
            raise AllocError("share length out of range")
        nblk = -(-n_tokens // self.block_size)
        blocks = self.tables[src][:nblk]
        self.pool.touch(blocks)
        self.tables[dst] = list(blocks)
        self.num_tokens[dst] = n_tokens
        # dst continues the hash chain only from a full, hashed last block
        self.salt[dst] = self.salt[src]
        if n_tokens == 0:
            self.parent[dst], self.pending[dst] = self.salt[src], []
        elif n_tokens % self.block_size == 0 and self.pool.block_hash[blocks[-1]] is not None:
            self.parent[dst], self.pending[dst] = self.pool.block_hash[blocks[-1]], []
        else:
            self.pending[dst] = None

    def cow(self, seq, logical_block):
        """Make ``seq``'s logical block private; return (src, dst) to copy."""
        self._resident(seq)
        table = self.tables[seq]
        if not 0 <= logical_block < len(table):
            raise AllocError("logical block out of range")
        b = table[logical_block]
        if self.pool.ref_cnt[b] == 1:
            return (b, b)
        if self.num_free() < 1:
            self.alloc_failures += 1
            raise NoFreeBlocks("no block for the private copy")
        (nb,) = self.pool.get_new_blocks(1)
        self.pool.ref_cnt[b] -= 1
        table[logical_block] = nb
        self.cow_copies += 1
        return (b, nb)

    def free_seq(self, seq):
        """Release ``seq``: its blocks in reverse order, tail block first."""
        self._need(seq)
        if seq in self.on_cpu:
            self.cpu_free.prepend_n(list(reversed(self.tables[seq])))
            self.on_cpu.discard(seq)
        else:
            self.pool.free_blocks(list(reversed(self.tables[seq])))
        del self.tables[seq]
        del self.num_tokens[seq]
        del self.salt[seq], self.parent[seq], self.pending[seq]

    # -- workload scripts ------------------------------------------------------
    def run(self, ops):
        """Replay an allocator script; returns (slots of appends, cow pairs)."""
        slots, pairs = [], []
        for op in ops:
            kind = op[0]
            if kind == "add":
                self.add_seq(op[1])
            elif kind == "append":
                slots.extend(self.append_slots(op[1], op[2]))
            elif kind == "enable_caching":
                self.enable_prefix_caching()
            elif kind == "add_cached":  # (kind, seq, prompt tokens, salt)
                self.add_seq_cached(op[1], op[2], op[3] if len(op) > 3 else 0)
            elif kind == "append_tokens":  # (kind, seq, token ids)
                slots.extend(self.append_tokens(op[1], op[2]))
            elif kind == "swap_out":
                self.swap_out(op[1])
            elif kind == "swap_in":
                self.swap_in(op[1])
            elif kind == "share":
                self.share(op[1], op[2], op[3])
            elif kind == "cow":
                s, d = self.cow(op[1], op[2])
                if s != d:
                    pairs.append((s, d))
            elif kind == "free":
                self.free_seq(op[1])
            else:
                raise AllocError(f"unknown op {kind}")
        return slots, pairs
