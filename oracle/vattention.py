"""Bookkeeping of a vAttention-style KV memory manager (no memory is touched).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"vAttention 完全拆解" (pinghaoyang.com.cn): every K and V tensor of every
layer is one contiguous *virtual* range ``[B][L][H][D]``; request slot
``reqId`` owns the sub-range at offset reqId * L*H*D*P.  Physical pages of
``G`` bytes are created up front into a pool and mapped onto a slot's range
only when the slot's sequence grows into it (section "the core abstraction",
figure 2; section "from request to page mapping", steps 1-4):

* ``step(lens)`` maps, for every active slot, the pages its current length
  needs, in every sub-tensor (2 x layers of them), and nothing else;
* a finished slot keeps its pages (deferred reclamation); a new request that
  takes the slot reuses them and overwrites the old data;
* pages are returned to the pool only when a step cannot be covered
  otherwise (the low-watermark reclamation of that section), taken from
  slots that are not active.

Readings where the page is silent (each stated):

* pages needed for length ``n``: ceil(roundup(n, tile) * h / G) with
  h = H*D*P bytes per token of one sub-tensor.  The page's formula is
  ceil(q*h / G); the attention kernel that reads the slot fetches whole
  ``tile``-token tiles (16), so the mapped range must cover the rounded
  length.  With ``tile`` = 1 this is the page's formula exactly.
* ``alloc_slot`` hands out the free slot holding the most mapped pages,
  lowest id on ties (figure 2 (e): the new request takes over the finished
  request's id and its pages).
* reclamation takes whole slots in increasing id order among inactive slots
  holding pages, and only as many as the step needs; a step that cannot be
  covered even after reclaiming every inactive slot fails and changes
  nothing.
"""
from __future__ import annotations


class NoPages(Exception):
    """The page pool cannot cover a step; nothing changed."""


class VAttnError(Exception):
    """Invalid request (bad slot, length past the reservation, ...)."""


def pages_for(length: int, bytes_per_token: int, page_bytes: int, tile: int = 16) -> int:
    """Pages one sub-tensor needs to back the first ``length`` tokens of a slot."""
    if length <= 0:
        return 0
    covered = -(-length // tile) * tile
    return -(-(covered * bytes_per_token) // page_bytes)


def tail_commit_bytes(layers: int, page_bytes: int) -> int:
    """W_max = 2 N' G: physical bytes one page-boundary crossing commits (K and V of each layer)."""
    return 2 * layers * page_bytes


class VirtualKV:
    def __init__(self, num_slots: int, max_len: int, layers: int, kv_heads: int, head_dim: int,
                 elem_bytes: int, page_bytes: int, max_pages: int, tile: int = 16):
        if num_slots <= 0 or max_len <= 0 or layers <= 0 or page_bytes <= 0 or max_pages < 0:
            raise VAttnError("bad sizes")
        self.B, self.L, self.layers = num_slots, max_len, layers
        self.h = kv_heads * head_dim * elem_bytes           # bytes per token of one sub-tensor
        self.G = page_bytes
        self.tile = tile
        self.tensors = 2 * layers
        self.slot_pages = -(-(max_len * self.h) // page_bytes)  # virtual pages per slot per sub-tensor
        self.max_pages = max_pages
        self.mapped = [0] * num_slots                        # pages mapped per slot (per sub-tensor)
        self.active = [False] * num_slots
        self.map_calls = 0
        self.unmap_calls = 0

    # -- queries -------------------------------------------------------------
    def pages_in_use(self) -> int:
        return sum(self.mapped) * self.tensors

    def pool_free(self) -> int:
        return self.max_pages - self.pages_in_use()

    def mapped_tokens(self, slot: int) -> int:
        """Tokens of whole tiles backed by mapped pages in ``slot``."""
        tok = self.mapped[slot] * self.G // self.h
        return min(tok // self.tile * self.tile, self.L)

    def virtual_offset(self, slot: int) -> int:
        """offset(reqId) = reqId * L * H * D * P (bytes from the sub-tensor's base)."""
        return slot * self.L * self.h

    # -- slots ---------------------------------------------------------------
    def alloc_slot(self) -> int:
        free = [s for s in range(self.B) if not self.active[s]]
        if not free:
            raise NoPages("no free slot")
        s = max(free, key=lambda x: (self.mapped[x], -x))
        self.active[s] = True
        return s

    def free_slot(self, slot: int):
        if not 0 <= slot < self.B or not self.active[slot]:
            raise VAttnError("slot not active")
        self.active[slot] = False          # its pages stay mapped

    # -- the per-iteration call ----------------------------------------------
    def step(self, lens):
        """Map what every active slot's length needs; returns the pages mapped this step."""
        if len(lens) != self.B:
            raise VAttnError("one length per slot")
        need = [0] * self.B
        for s, n in enumerate(lens):
            n = int(n)
            if n < 0 or n > self.L or (n > 0 and not self.active[s]):
                raise VAttnError(f"bad length {n} for slot {s}")
            need[s] = pages_for(n, self.h, self.G, self.tile)
        extra = sum(max(0, need[s] - self.mapped[s]) for s in range(self.B)) * self.tensors
        short = extra - self.pool_free()
        if short > 0:
            donors = [s for s in range(self.B) if not self.active[s] and self.mapped[s] > 0]
            if sum(self.mapped[s] for s in donors) * self.tensors < short:
                raise NoPages(f"need {extra} pages, {self.pool_free()} free")
            for s in donors:
                if short <= 0:
                    break
                short -= self.mapped[s] * self.tensors
                self.unmap_calls += self.mapped[s] * self.tensors
                self.mapped[s] = 0
        for s in range(self.B):
            if need[s] > self.mapped[s]:
                self.map_calls += (need[s] - self.mapped[s]) * self.tensors
                self.mapped[s] = need[s]
        return extra

    def committed_bytes(self) -> int:
        return self.pages_in_use() * self.G

    def run(self, ops):
        """Replay a script of ("alloc",) / ("free", slot) / ("step", lens) ops; returns alloc results."""
        got = []
        for op in ops:
            if op[0] == "alloc":
                got.append(self.alloc_slot())
            elif op[0] == "free":
                self.free_slot(op[1])
            elif op[0] == "step":
                self.step(op[1])
            else:
                raise VAttnError(f"unknown op {op[0]}")
        return got


def slot_row(slot: int, token: int, max_len: int) -> int:
    """Row of token ``token`` of slot ``slot`` in the contiguous [B*L] token axis."""
    return slot * max_len + token

