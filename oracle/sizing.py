"""KV byte counts.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""
from __future__ import annotations


def kv_cache_bytes(layers: int, length: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """M_KV = 2 * N * L * H * D * P.

    "vAttention 完全拆解", first section: a worker holding N layers with H
    local KV heads of dimension D at P bytes per element keeps 2NLHDP bytes
    of KV for a request of current length L (the 2 is K and V).
    """
    return 2 * layers * length * kv_heads * head_dim * elem_bytes


def kv_slot_bytes(length: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """S = L * H * D * P: one layer's K (or V) for one request slot (same page)."""
    return length * kv_heads * head_dim * elem_bytes


def decode_step_bytes(context_lens, q_heads: int, kv_heads: int, head_dim: int,
                      block_size: int, elem_bytes: int = 2) -> int:
    """Algorithmic bytes one paged decode step must move (one query per request).

    Per request: the K and V of its context (2 * L * Hkv * D * P), its query
    and output rows (Hq * D * P each), its block-table entries (4 bytes per
    logical block) and its context length (4 bytes).
    """
    total = 0
    for L in context_lens:
        L = int(L)
        nblk = -(-L // block_size)
        total += 2 * L * kv_heads * head_dim * elem_bytes
        total += 2 * q_heads * head_dim * elem_bytes
        total += 4 * nblk + 4
    return total


def unique_block_bytes(block_ids, block_size: int, kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """K+V bytes of a set of physical blocks, each counted once."""
    return len(set(int(b) for b in block_ids)) * 2 * block_size * kv_heads * head_dim * elem_bytes
