"""Block allocator of a paged KV cache, restated from the pages' design.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"2.1 PagedAttention" §9.1-9.3 splits the work in two:

* a global pool of physical blocks (BlockPool) with a free queue that is a
  doubly linked list (FreeKVCacheBlockQueue: O(1) popleft and O(1) removal
  from the middle, §9.2) and a reference count per block (§9.3);
* a per-request manager (KVCacheManager, §9.1) that grows a request's Block
  Table on demand (a new block only when the last one is full, §3), and frees
  its blocks in reverse order when it ends (tail blocks first).

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
"""
from __future__ import annotations

__all__ = ["NoFreeBlocks", "AllocError", "FreeBlockQueue", "BlockPool", "SequenceManager"]


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

    def get_num_free_blocks(self):
        return len(self.free_block_queue)

    def get_new_blocks(self, num_blocks):
        if num_blocks > self.get_num_free_blocks():
            raise NoFreeBlocks(f"need {num_blocks}, have {self.get_num_free_blocks()}")
        blocks = self.free_block_queue.popleft_n(num_blocks)
        for b in blocks:
            assert self.ref_cnt[b] == 0
            self.ref_cnt[b] += 1
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

    def add_seq(self, seq):
        if seq in self.tables:
            raise AllocError(f"sequence {seq} exists")
        self.tables[seq] = []
        self.num_tokens[seq] = 0

    def append_slots(self, seq, n):
        """Give the next ``n`` tokens of ``seq`` their slots, growing on demand."""
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
        self._need(dst)
        self._need(src)
        if self.tables[dst] or self.num_tokens[dst]:
            raise AllocError("share target must be empty")
        if not 0 <= n_tokens <= self.num_tokens[src]:
            raise AllocError("share length out of range")
        nblk = -(-n_tokens // self.block_size)
        blocks = self.tables[src][:nblk]
        self.pool.touch(blocks)
        self.tables[dst] = list(blocks)
        self.num_tokens[dst] = n_tokens

    def cow(self, seq, logical_block):
        """Make ``seq``'s logical block private; return (src, dst) to copy."""
        self._need(seq)
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
        self.pool.free_blocks(list(reversed(self.tables[seq])))
        del self.tables[seq]
        del self.num_tokens[seq]

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
