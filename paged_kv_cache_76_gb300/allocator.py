"""Python handle over the C++ block allocator (``pa_alloc_*`` in include/pa.h)."""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import _lib
from ._lib import PA_ERR_NO_FREE_BLOCKS, PAError, check

__all__ = ["BlockAllocator", "NoFreeBlocks"]


class NoFreeBlocks(PAError):
    """The pool cannot cover the request; the allocator state is unchanged."""


def _chk(st, what):
    if st == PA_ERR_NO_FREE_BLOCKS:
        raise NoFreeBlocks(st, what)
    return check(st, what)


def _i32p(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


class BlockAllocator:
    """Free queue + refcounts + per-sequence Block Tables, in C++."""

    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        self._L = _lib.lib()
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        h = C.c_void_p()
        order = None
        if initial_free_order is not None:
            order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
            if order.shape != (self.num_blocks,):
                raise ValueError("initial_free_order must list every block once")
        _chk(self._L.pa_alloc_create(self.num_blocks, self.block_size,
                                     _i32p(order) if order is not None else None, C.byref(h)),
             "pa_alloc_create")
        self._h = h
        self._order_keepalive = order

    def export(self) -> np.ndarray:
        """The allocator's whole state as int64 words (pa_alloc_export)."""
        n = C.c_int64(0)
        _chk(self._L.pa_alloc_export(self._h, None, 0, C.byref(n)), "pa_alloc_export")
        words = np.zeros(n.value, dtype=np.int64)
        _chk(self._L.pa_alloc_export(self._h, words.ctypes.data_as(C.c_void_p), n.value, C.byref(n)),
             "pa_alloc_export")
        return words

    @classmethod
    def from_words(cls, words) -> "BlockAllocator":
        """A new allocator with the state exported as `words` (pa_alloc_import)."""
        w = np.ascontiguousarray(words, dtype=np.int64)
        obj = cls.__new__(cls)
        obj._L = _lib.lib()
        h = C.c_void_p()
        _chk(obj._L.pa_alloc_import(w.ctypes.data_as(C.c_void_p), int(w.size), C.byref(h)), "pa_alloc_import")
        obj._h = h
        obj.num_blocks = int(w[2])
        obj.block_size = int(w[3])
        obj._order_keepalive = None
        return obj

    def close(self):
        if getattr(self, "_h", None):
            self._L.pa_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq: int):
        _chk(self._L.pa_alloc_add_seq(self._h, int(seq)), "pa_alloc_add_seq")

    def append_slots(self, seq: int, n: int) -> np.ndarray:
        out = np.empty(int(n), dtype=np.int32)
        _chk(self._L.pa_alloc_append_slots(self._h, int(seq), int(n), _i32p(out)), "pa_alloc_append_slots")
        return out

    def share(self, dst: int, src: int, n_tokens: int):
        _chk(self._L.pa_alloc_share(self._h, int(dst), int(src), int(n_tokens)), "pa_alloc_share")

    def cow(self, seq: int, logical_block: int):
        out = np.empty(2, dtype=np.int32)
        _chk(self._L.pa_alloc_cow(self._h, int(seq), int(logical_block), _i32p(out)), "pa_alloc_cow")
        return int(out[0]), int(out[1])

    def free_seq(self, seq: int):
        _chk(self._L.pa_alloc_free_seq(self._h, int(seq)), "pa_alloc_free_seq")

    def block_table(self, seq: int) -> list:
        n = C.c_int(0)
        self._L.pa_alloc_block_table(self._h, int(seq), None, 0, C.byref(n))
        out = np.empty(max(n.value, 1), dtype=np.int32)
        _chk(self._L.pa_alloc_block_table(self._h, int(seq), _i32p(out), out.shape[0], C.byref(n)),
             "pa_alloc_block_table")
        return out[:n.value].tolist()

    def build_tables(self, seqs, max_blocks_per_seq: int):
        ids = np.ascontiguousarray(seqs, dtype=np.int32).astype(np.intc)
        n = ids.shape[0]
        tables = np.empty((n, int(max_blocks_per_seq)), dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        _chk(self._L.pa_alloc_build_tables(self._h, ids.ctypes.data_as(C.POINTER(C.c_int)), n, _i32p(tables),
                                           int(max_blocks_per_seq), _i32p(lens)), "pa_alloc_build_tables")
        return tables, lens

    def common_prefix(self, seqs) -> int:
        """Leading full blocks all of ``seqs`` share (same physical ids)."""
        ids = np.ascontiguousarray(seqs, dtype=np.intc)
        n = C.c_int(0)
        _chk(self._L.pa_alloc_common_prefix(self._h, ids.ctypes.data_as(C.POINTER(C.c_int)), ids.shape[0],
                                            C.byref(n)), "pa_alloc_common_prefix")
        return int(n.value)

    # -- automatic prefix caching -------------------------------------------
    def enable_prefix_caching(self):
        _chk(self._L.pa_alloc_enable_prefix_caching(self._h), "pa_alloc_enable_prefix_caching")

    def add_seq_cached(self, seq: int, tokens, salt: int = 0) -> int:
        """New sequence whose table starts with its prompt's cached blocks; returns the tokens covered."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = C.c_int(0)
        _chk(self._L.pa_alloc_add_seq_cached(self._h, int(seq), _i32p(t) if t.size else None, int(t.size),
                                             int(salt) & 0xFFFFFFFFFFFFFFFF, C.byref(n)), "pa_alloc_add_seq_cached")
        return int(n.value)

    def append_tokens(self, seq: int, tokens) -> np.ndarray:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty(t.size, dtype=np.int32)
        _chk(self._L.pa_alloc_append_tokens(self._h, int(seq), _i32p(t) if t.size else None, int(t.size),
                                            _i32p(out)), "pa_alloc_append_tokens")
        return out

    def block_hash(self, block: int):
        """The block's cached hash, or None if it is not in the cache."""
        h, c = C.c_uint64(0), C.c_int(0)
        _chk(self._L.pa_alloc_block_hash(self._h, int(block), C.byref(h), C.byref(c)), "pa_alloc_block_hash")
        return int(h.value) if c.value else None

    def prefix_cache_stats(self) -> dict:
        s = _lib.PrefixCacheStats()
        _chk(self._L.pa_alloc_get_prefix_cache_stats(self._h, C.byref(s)), "pa_alloc_get_prefix_cache_stats")
        return {name: int(getattr(s, name)) for name, _ in s._fields_}

    # -- preemption by swapping ----------------------------------------------
    def enable_swap(self, num_cpu_blocks: int):
        _chk(self._L.pa_alloc_enable_swap(self._h, int(num_cpu_blocks)), "pa_alloc_enable_swap")

    def num_free_cpu(self) -> int:
        return _chk(self._L.pa_alloc_num_free_cpu(self._h), "pa_alloc_num_free_cpu")

    def is_swapped(self, seq: int) -> bool:
        return bool(_chk(self._L.pa_alloc_is_swapped(self._h, int(seq)), "pa_alloc_is_swapped"))

    def _swap(self, fn, seq, what):
        n = C.c_int(0)
        cap = len(self.block_table(seq))
        out = np.empty((max(cap, 1), 2), dtype=np.int32)
        _chk(fn(self._h, int(seq), _i32p(out), cap, C.byref(n)), what)
        return out[:n.value]

    def swap_out(self, seq: int) -> np.ndarray:
        """Move ``seq`` to the swap pool; int32 [n, 2] (gpu block, swap block) pairs."""
        return self._swap(self._L.pa_alloc_swap_out, seq, "pa_alloc_swap_out")

    def swap_in(self, seq: int) -> np.ndarray:
        """Bring ``seq`` back into new GPU blocks; int32 [n, 2] (swap block, gpu block) pairs."""
        return self._swap(self._L.pa_alloc_swap_in, seq, "pa_alloc_swap_in")

    def seq_len(self, seq: int) -> int:
        v = C.c_int64(0)
        _chk(self._L.pa_alloc_seq_len(self._h, int(seq), C.byref(v)), "pa_alloc_seq_len")
        return int(v.value)

    def num_free(self) -> int:
        return _chk(self._L.pa_alloc_num_free(self._h), "pa_alloc_num_free")

    def ref(self, block: int) -> int:
        return _chk(self._L.pa_alloc_ref(self._h, int(block)), "pa_alloc_ref")

    def free_list(self) -> list:
        out = np.empty(self.num_blocks, dtype=np.int32)
        n = _chk(self._L.pa_alloc_free_list(self._h, _i32p(out), self.num_blocks), "pa_alloc_free_list")
        return out[:n].tolist()

    def stats(self) -> dict:
        s = _lib.AllocStats()
        _chk(self._L.pa_alloc_get_stats(self._h, C.byref(s)), "pa_alloc_get_stats")
        return {name: int(getattr(s, name)) for name, _ in s._fields_}

    def run(self, ops):
        """Replay an allocator script (see ``workloads``); returns (slots, cow pairs)."""
        slots, pairs = [], []
        for op in ops:
            kind = op[0]
            if kind == "add":
                self.add_seq(op[1])
            elif kind == "append":
                slots.extend(self.append_slots(op[1], op[2]).tolist())
            elif kind == "share":
                self.share(op[1], op[2], op[3])
            elif kind == "cow":
                s, d = self.cow(op[1], op[2])
                if s != d:
                    pairs.append((s, d))
            elif kind == "free":
                self.free_seq(op[1])
            elif kind == "enable_caching":
                self.enable_prefix_caching()
            elif kind == "add_cached":
                self.add_seq_cached(op[1], op[2], op[3] if len(op) > 3 else 0)
            elif kind == "append_tokens":
                slots.extend(self.append_tokens(op[1], op[2]).tolist())
            elif kind == "swap_out":
                self.swap_out(op[1])
            elif kind == "swap_in":
                self.swap_in(op[1])
            else:
                raise ValueError(f"unknown op {kind}")
        return slots, pairs
