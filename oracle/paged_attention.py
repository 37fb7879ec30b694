"""Paged KV cache: float64 reference of every device operation.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Layout (the one the library uses, stated here independently): a cache tensor
is ``[num_blocks, block_size, kv_heads, head_dim]``; a block table row lists,
for each logical block of a request, the id of the physical block holding it.

Conventions where the pages are silent (each is a stated reading):

* GQA: query head ``h`` reads KV head ``h // (q_heads // kv_heads)``
  (contiguous groups).  The pages only name ``kv_head_idx``.
* A context length counts every token the request has, including the ones
  this step writes; zero context gives a zero output.
* A slot below zero marks a padding token that is not written.
* Chunked prefill: query ``i`` of a chunk that starts at absolute position
  ``p0`` attends keys ``0 .. p0 + i`` (all history plus causal inside the
  chunk).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "token_location",
    "slots_for",
    "reshape_and_cache",
    "copy_blocks",
    "swap_blocks",
    "gather_context",
    "decode",
    "decode_split_partials",
    "lse_merge",
    "decode_split",
    "chunked_prefill",
    "verify_decode",
]


def token_location(block_table_row, t: int, block_size: int):
    """Logical token ``t`` -> (physical_block_number, physical_block_offset).

    "2.1 PagedAttention" §3 and §5: the kernel looks the token's logical
    block up in the request's Block Table to get the physical block number,
    and the position inside the block is the offset.
    """
    logical_block = t // block_size
    return int(block_table_row[logical_block]), t % block_size


def slots_for(block_table_row, positions, block_size: int) -> np.ndarray:
    """Flat slot index ``pbn * block_size + offset`` for each logical position."""
    out = []
    for t in positions:
        pbn, off = token_location(block_table_row, int(t), block_size)
        out.append(pbn * block_size + off)
    return np.asarray(out, dtype=np.int64)


def reshape_and_cache(k, v, slot_mapping, k_cache, v_cache):
    """Write token ``i``'s K/V into slot ``slot_mapping[i]`` (skip slots < 0).

    New tokens fill the next free slots of their request's blocks ("2.1
    PagedAttention" §3, decode growth); the forward pass fills the KV of the
    allocated blocks ("Khám phá vLLM … phần 2", prefix caching walk-through).
    Works on any element type, so the copy is bit-exact.  Returns new arrays.
    """
    k_cache = np.array(k_cache, copy=True)
    v_cache = np.array(v_cache, copy=True)
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    for i, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s < 0:
            continue
        if s >= nb * bs:
            raise IndexError(f"slot {s} outside a pool of {nb * bs} slots")
        k_cache[s // bs, s % bs] = k[i]
        v_cache[s // bs, s % bs] = v[i]
    return k_cache, v_cache


def copy_blocks(k_cache, v_cache, pairs):
    """Copy-on-Write device step: block ``dst`` becomes a copy of block ``src``.

    "2.1 PagedAttention" §6: before a request writes a shared block it copies
    the block into a private one.  ``pairs`` is a sequence of (src, dst);
    a dst may not repeat nor be another pair's src.  Returns new arrays.
    """
    k_cache = np.array(k_cache, copy=True)
    v_cache = np.array(v_cache, copy=True)
    pairs = [(int(s), int(d)) for s, d in pairs]
    dsts = [d for _, d in pairs]
    if len(set(dsts)) != len(dsts) or set(dsts) & {s for s, _ in pairs}:
        raise ValueError("copy_blocks pairs must have distinct dsts that are not srcs")
    for s, d in pairs:
        k_cache[d] = k_cache[s]
        v_cache[d] = v_cache[s]
    return k_cache, v_cache


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs):
    """Swap step of preemption: block ``d`` of the destination pool becomes a
    copy of block ``s`` of the source pool, for each (s, d).

    "2.1 PagedAttention" §7: a preempted request's KV blocks are copied from
    GPU memory to CPU memory (swap out) and back when it resumes (swap in),
    each time into whatever blocks the other pool hands out.  Destinations may
    not repeat.  Returns new destination arrays; the source is not changed.
    """
    dst_k = np.array(dst_k, copy=True)
    dst_v = np.array(dst_v, copy=True)
    pairs = [(int(s), int(d)) for s, d in pairs]
    dsts = [d for _, d in pairs]
    if len(set(dsts)) != len(dsts):
        raise ValueError("swap_blocks pairs must have distinct destinations")
    for s, d in pairs:
        dst_k[d] = src_k[s]
        dst_v[d] = src_v[s]
    return dst_k, dst_v


def gather_context(cache, block_table_row, length: int, block_size: int) -> np.ndarray:
    """The request's keys (or values) in logical order, ``[length, kv_heads, D]``.

    Token by token through the Block Table ("2.1 PagedAttention" §3, §5):
    physical storage scattered over blocks is read as one logical context.
    """
    rows = []
    for t in range(length):
        pbn, off = token_location(block_table_row, t, block_size)
        rows.append(np.asarray(cache[pbn, off], dtype=np.float64))
    if not rows:
        return np.zeros((0,) + tuple(cache.shape[2:]), dtype=np.float64)
    return np.stack(rows)


def _softmax_attend(q, K, V, scale):
    """Textbook softmax attention of one query vector over ``K``/``V`` rows."""
    s = scale * (K @ q)
    p = np.exp(s - s.max())
    p = p / p.sum()
    return p @ V


def decode(q, k_cache, v_cache, block_tables, context_lens, scale):
    """Paged decode attention, one query token per request; float64 output.

    ``q``: [B, q_heads, D]; ``block_tables``: [B, max_blocks]; the output row
    for (request r, head h) is softmax(scale * K_r q) V_r over the request's
    ``context_lens[r]`` tokens, gathered through its Block Table.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    bs = k_cache.shape[1]
    group = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for r in range(B):
        L = int(context_lens[r])
        if L == 0:
            continue
        K = gather_context(k_cache, block_tables[r], L, bs)
        V = gather_context(v_cache, block_tables[r], L, bs)
        for h in range(Hq):
            g = h // group
            out[r, h] = _softmax_attend(q[r, h], K[:, g, :], V[:, g, :], scale)
    return out


def decode_split_partials(q, k_cache, v_cache, block_tables, context_lens, scale, split_tokens):
    """Per-partition partial results of decode (the context-split order).

    The context of request r is cut into partitions [c*S, min((c+1)*S, L)).
    For each partition: m_c = max score, l_c = sum exp(score - m_c),
    o_c = sum exp(score - m_c) v (unnormalised).  Returns a list over
    requests of (o [n_c, Hq, D], m [n_c, Hq], l [n_c, Hq]), natural-log units.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    bs = k_cache.shape[1]
    group = Hq // Hkv
    res = []
    for r in range(B):
        L = int(context_lens[r])
        n_c = -(-L // split_tokens)
        K = gather_context(k_cache, block_tables[r], L, bs)
        V = gather_context(v_cache, block_tables[r], L, bs)
        o = np.zeros((n_c, Hq, D))
        m = np.zeros((n_c, Hq))
        l = np.zeros((n_c, Hq))
        for c in range(n_c):
            lo, hi = c * split_tokens, min((c + 1) * split_tokens, L)
            for h in range(Hq):
                g = h // group
                s = scale * (K[lo:hi, g, :] @ q[r, h])
                m[c, h] = s.max()
                p = np.exp(s - m[c, h])
                l[c, h] = p.sum()
                o[c, h] = p @ V[lo:hi, g, :]
        res.append((o, m, l))
    return res


def lse_merge(o_parts, m_parts, l_parts):
    """Log-sum-exp merge of partition partials into the normalised output.

    M = max_c m_c; w_c = exp(m_c - M); out = sum_c w_c o_c / sum_c w_c l_c.
    Arrays are [n_c, ...] with the partition axis first.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    m_parts = np.asarray(m_parts, dtype=np.float64)
    l_parts = np.asarray(l_parts, dtype=np.float64)
    M = m_parts.max(axis=0)
    w = np.exp(m_parts - M)
    denom = (w * l_parts).sum(axis=0)
    num = (w[..., None] * o_parts).sum(axis=0)
    return num / denom[..., None]


def decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, split_tokens):
    """Decode by partitions then merge; must equal :func:`decode`."""
    parts = decode_split_partials(q, k_cache, v_cache, block_tables, context_lens, scale, split_tokens)
    B, Hq, D = np.asarray(q).shape
    out = np.zeros((B, Hq, D))
    for r, (o, m, l) in enumerate(parts):
        if o.shape[0] == 0:
            continue
        out[r] = lse_merge(o, m, l)
    return out


def chunked_prefill(q, q_start, context_lens, k_cache, v_cache, block_tables, scale, rows=None):
    """Attention of a chunk of queries per request over its paged history.

    "Khám phá vLLM … phần 2", chunked prefill: a long prompt is processed a
    chunk of tokens per engine step; this step's chunk attends the history
    already in the cache plus itself.  Request r's queries are rows
    ``q_start[r] .. q_start[r+1]-1`` of ``q`` ([T, q_heads, D]);
    ``context_lens[r]`` includes the chunk, so the chunk starts at
    p0 = context_lens[r] - chunk and query i sees keys 0 .. p0 + i.
    ``rows`` optionally restricts the work to those rows of ``q`` (the others
    stay zero), for sampled checks of large inputs.
    """
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    bs = k_cache.shape[1]
    group = Hq // Hkv
    out = np.zeros((T, Hq, D))
    R = len(q_start) - 1
    wanted = None if rows is None else set(int(x) for x in rows)
    for r in range(R):
        a, b = int(q_start[r]), int(q_start[r + 1])
        chunk = b - a
        L = int(context_lens[r])
        p0 = L - chunk
        if chunk == 0:
            continue
        K = gather_context(k_cache, block_tables[r], L, bs)
        V = gather_context(v_cache, block_tables[r], L, bs)
        for i in range(chunk):
            if wanted is not None and a + i not in wanted:
                continue
            visible = p0 + i + 1
            for h in range(Hq):
                g = h // group
                out[a + i, h] = _softmax_attend(q[a + i, h], K[:visible, g, :], V[:visible, g, :], scale)
    return out


def verify_decode(q, k_cache, v_cache, block_tables, context_lens, scale):
    """Verify step of speculative decoding over the paged cache.

    "Khám phá vLLM … phần 2", speculative decoding: the large model runs once
    over the context plus the k draft tokens and yields a distribution for
    each of the k+1 positions.  Here ``q`` is [B, k+1, q_heads, D]: the
    queries of the last k+1 positions of each request, whose K/V are already
    in the cache, so ``context_lens[r]`` = L counts them.  Query ``i`` sits at
    position L-(k+1)+i and attends keys 0 .. L-(k+1)+i (causal), i.e. it is
    plain decode with context L-k+i.  A query that sees no key (L < k+1-i)
    gives a zero row.  Float64 output [B, k+1, q_heads, D].
    """
    q = np.asarray(q, dtype=np.float64)
    B, Q, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    bs = k_cache.shape[1]
    group = Hq // Hkv
    out = np.zeros((B, Q, Hq, D), dtype=np.float64)
    for r in range(B):
        L = int(context_lens[r])
        for i in range(Q):
            visible = L - (Q - 1 - i)
            if visible <= 0:
                continue
            K = gather_context(k_cache, block_tables[r], visible, bs)
            V = gather_context(v_cache, block_tables[r], visible, bs)
            for h in range(Hq):
                g = h // group
                out[r, i, h] = _softmax_attend(q[r, i, h], K[:, g, :], V[:, g, :], scale)
    return out
