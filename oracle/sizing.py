"""KV byte counts.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Pins (``tests/test_oracle_pins.py``): ``kv_cache_bytes`` and
``kv_slot_bytes`` against the worked numbers of "vAttention 完全拆解";
``decode_step_bytes`` and ``unique_kv_bytes`` against a brute-force count of
the array elements one decode step touches (numpy ``nbytes`` of the slices
actually read and written, marked element by element), and against the
prefix-shared decode's closed form (the shared prefix counted once).
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
                      block_size: int, elem_bytes: int = 2, q_len: int = 1) -> int:
    """Algorithmic bytes one paged decode step must move.

    Per request of context L ("2.1 PagedAttention" §5: the kernel walks the
    request's Block Table and reads each logical token's K and V once): the K
    and V of its L tokens (all KV heads), its q_len query rows and q_len
    output rows (Hq * D elements each), the block-table entries that cover L
    tokens (one int32 per logical block) and its int32 context length.
    """
    total = 0
    for L in context_lens:
        L = int(L)
        blocks = -(-L // block_size)
        kv = 2 * L * kv_heads * head_dim * elem_bytes
        qo = 2 * q_len * q_heads * head_dim * elem_bytes
        total += kv + qo + 4 * blocks + 4
    return total


def unique_kv_bytes(block_tables, context_lens, q_heads: int, kv_heads: int, head_dim: int,
                    block_size: int, elem_bytes: int = 2, q_len: int = 1) -> int:
    """Bytes a decode step must move when every cache row is read only once.

    "2.1 PagedAttention" §6: several Block Tables may point at the same
    physical blocks (a shared prefix).  The cache rows a batch reads are the
    distinct (physical block, offset) pairs over all requests' first L
    tokens; each costs one K and one V row (Hkv * D elements each).  The
    per-request terms (q, o, table entries, length) are as in
    ``decode_step_bytes``.
    """
    rows = set()
    per_request = 0
    for table, L in zip(block_tables, context_lens):
        L = int(L)
        for t in range(L):
            rows.add((int(table[t // block_size]), t % block_size))
        per_request += 2 * q_len * q_heads * head_dim * elem_bytes + 4 * (-(-L // block_size)) + 4
    return len(rows) * 2 * kv_heads * head_dim * elem_bytes + per_request
