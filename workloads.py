"""Seeded synthetic inputs for the paged-KV attention path.

This module is shared by the oracle-side tests and the CUDA-side tests and
bench.  It only draws random numbers and describes workloads: it holds none of
the method's arithmetic.  In particular it never computes a slot, a block-table
entry or an attention value.  Each workload is described as

* shapes (heads, head_dim, block_size, pool size, dtype, softmax scale);
* ``free_order``: the initial order of the block allocator's free list (a
  seeded permutation of the pool's block ids);
* ``setup_ops``: an allocator script that builds the history before the step
  (``("add", seq)``, ``("append", seq, n)``, ``("share", dst, src, n)``,
  ``("cow", seq, logical_block)``, ``("free", seq)``);
* ``step_ops``: the allocator script of the measured step (the ``append``s
  that give the new tokens their slots, the ``cow``s whose pairs feed
  ``copy_blocks``);
* ``decode_seqs`` / ``prefill``: which sequences decode one token and which
  run a prefill chunk of how many tokens this step.

Both allocator implementations (the C++ one behind the C ABI and the Python
one in the oracle) replay the same scripts independently.  Values (queries,
new keys/values, the pre-step contents of the whole pool, stale data included)
come from :func:`make_values`.

Workloads follow the shapes of the pages' subject (Llama-8B / Yi-34B-TP2 style
GQA decode, block_size 16, long contexts, shared system prompts, chunked
prefill); the pages measure on text datasets that are not available here, and
these synthetic shapes stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = [
    "Workload",
    "tiny_paged_decode",
    "llama8b_gqa_decode",
    "long_context_splitk_decode",
    "prefix_shared_cow_decode",
    "mixed_prefill_decode",
    "custom_decode",
    "make_values",
    "WORKLOADS",
]


@dataclass
class Workload:
    name: str
    dtype: str                      # "fp16" | "bf16"
    q_heads: int
    kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    free_order: np.ndarray          # int32 [num_blocks]
    setup_ops: list = field(default_factory=list)
    step_ops: list = field(default_factory=list)
    decode_seqs: list = field(default_factory=list)     # seq ids, one query each
    decode_lens: list = field(default_factory=list)     # context length incl. the new token
    prefill: list = field(default_factory=list)         # (seq id, chunk tokens, context len incl. chunk)
    split_tokens: int = 0           # 0 = let the library choose
    q_len: int = 1                  # queries per decode request (k+1 for a speculative verify)
    value_dist: str = "normal"      # "normal" N(0,1) | "uniform" U[-1,1]
    seed: int = 0
    note: str = ""

    # sizes derived from the description, for reports and buffer sizing
    @property
    def new_tokens(self) -> int:
        """Tokens whose K/V this step writes (the step script's appends)."""
        return sum(op[2] for op in self.step_ops if op[0] == "append")

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16

    @property
    def max_context(self) -> int:
        lens = list(self.decode_lens) + [l for _, _, l in self.prefill]
        return max(lens) if lens else 0


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _pool(rng, needed_blocks: int, factor: float = 1.5):
    nb = int(math.ceil(factor * needed_blocks))
    return nb, rng.permutation(nb).astype(np.int32)


def _decode_scripts(seqs, lens, new: int = 1):
    """History of len-new tokens per sequence, then `new` tokens this step."""
    setup, step = [], []
    for s, L in zip(seqs, lens):
        setup.append(("add", s))
        if L - new > 0:
            setup.append(("append", s, L - new))
        step.append(("append", s, min(new, L)))
    return setup, step


def tiny_paged_decode(seed: int = 1) -> Workload:
    """2 requests with contexts 9 and 5, block_size 4, a pool of 16 blocks.

    Request 0's three blocks are #7, #2, #5 as in the worked Block Table
    example of "2.1 PagedAttention" (§3); request 1's two blocks come from a
    seeded permutation of the other 13 ids.  All 14 tokens are written by
    reshape_and_cache in this step (no history), fp16 U[-1,1].
    """
    rng = _rng(seed)
    rest = np.array([b for b in range(16) if b not in (7, 2, 5)], dtype=np.int32)
    free_order = np.concatenate([np.array([7, 2, 5], np.int32), rng.permutation(rest).astype(np.int32)])
    lens = [9, 5]
    setup = [("add", 0), ("add", 1)]
    step = [("append", 0, 9), ("append", 1, 5)]
    return Workload(
        name="tiny_paged_decode", dtype="fp16", q_heads=2, kv_heads=1, head_dim=64,
        block_size=4, num_blocks=16, scale=1.0 / 8.0, free_order=free_order,
        setup_ops=setup, step_ops=step, decode_seqs=[0, 1], decode_lens=lens,
        prefill=[], value_dist="uniform", seed=seed,
        note="all 14 tokens written by reshape_and_cache; decode of one query per request",
    )


def custom_decode(batch: int, len_lo: int, len_hi: int, q_heads: int, kv_heads: int,
                  head_dim: int = 128, block_size: int = 16, dtype: str = "bf16",
                  seed: int = 0, split_tokens: int = 0, lens=None, pool_factor: float = 1.5,
                  name: str = "custom_decode") -> Workload:
    """Decode-only workload: lens uniform in [len_lo, len_hi] (inclusive).

    The pool is 1.5x the blocks the requests need and its free list is
    shuffled, so block tables are scattered with holes left free.
    """
    rng = _rng(seed)
    if lens is None:
        lens = rng.integers(len_lo, len_hi, size=batch, endpoint=True).astype(int).tolist()
    else:
        lens = [int(x) for x in lens]
    needed = sum(_cdiv(L, block_size) for L in lens)
    nb, order = _pool(rng, max(needed, 1), pool_factor)
    seqs = list(range(len(lens)))
    setup, step = _decode_scripts(seqs, lens)
    return Workload(
        name=name, dtype=dtype, q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim,
        block_size=block_size, num_blocks=nb, scale=1.0 / math.sqrt(head_dim), free_order=order,
        setup_ops=setup, step_ops=step, decode_seqs=seqs, decode_lens=lens,
        split_tokens=split_tokens, seed=seed,
    )


def llama8b_gqa_decode(seed: int = 0, batch: int = 64, len_lo: int = 512, len_hi: int = 4096,
                       block_size: int = 16) -> Workload:
    """Batch 64, 32 q heads / 8 KV heads, D=128, bs=16, bf16 N(0,1), lens U{512..4096}.

    ``block_size`` other than 16 gives the same contexts in blocks of another
    size (the block-size trade-off of "2.1 PagedAttention" §4 and §10)."""
    wl = custom_decode(batch, len_lo, len_hi, 32, 8, 128, block_size, "bf16", seed, name="llama8b_gqa_decode")
    wl.note = "one query token per request; pool 1.5x needed, shuffled free list"
    return wl


def spec_verify_decode(seed: int = 0, batch: int = 64, len_lo: int = 512, len_hi: int = 4096,
                       k: int = 3, block_size: int = 16) -> Workload:
    """Verify step of speculative decoding on the llama8b_gqa_decode shape.

    Batch 64, 32 q heads / 8 KV heads, D=128, bs=16, bf16 N(0,1); each
    request's context is U{512..4096} tokens including its k=3 draft tokens,
    whose K/V this step writes; k+1 = 4 queries per request (the last
    accepted token and the drafts), 16 query rows per KV head.
    """
    wl = custom_decode(batch, len_lo, len_hi, 32, 8, 128, block_size, "bf16", seed, name="spec_verify_decode")
    wl.q_len = k + 1
    wl.setup_ops, wl.step_ops = _decode_scripts(wl.decode_seqs, wl.decode_lens, k + 1)
    wl.note = f"k={k} draft tokens per request written this step; k+1 causal queries per request"
    return wl


def _renamed(wl: Workload, name: str) -> Workload:
    wl.name = name
    return wl


def long_context_splitk_decode(seed: int = 0, batch: int = 8, len_lo: int = 32768,
                               len_hi: int = 131072, block_size: int = 16) -> Workload:
    """Batch 8, 64 q heads / 8 KV heads, D=128, bs=16, lens U{32768..131072}, 512-token splits."""
    wl = custom_decode(batch, len_lo, len_hi, 64, 8, 128, block_size, "bf16", seed, split_tokens=512,
                       name="long_context_splitk_decode")
    wl.note = "context partitioned into 512-token chunks merged by log-sum-exp"
    return wl


def prefix_shared_cow_decode(seed: int = 0, batch: int = 256, prefix_tokens: int = 2048,
                             suffix_lo: int = 16, suffix_hi: int = 512, cow_frac: float = 0.1,
                             q_heads: int = 32, kv_heads: int = 8, head_dim: int = 128,
                             block_size: int = 16) -> Workload:
    """256 requests sharing a 2048-token prefix (128 blocks, refcount 256).

    A holder sequence writes the prefix, every request shares it, and the
    holder is freed, leaving each prefix block with refcount == batch.
    round(0.1 * batch) requests, chosen by the seeded generator, copy-on-write
    the last shared block before appending (with a 2048-token prefix that
    block is full, so their suffix then goes to fresh blocks).  Every request
    then holds a private suffix of U{16..512} tokens, the last of which is this
    step's new token.
    """
    if prefix_tokens % block_size:
        raise ValueError("the measured workload shares whole blocks only; a partial shared "
                         "block would make every writer copy it first")
    rng = _rng(seed)
    suffix = rng.integers(suffix_lo, suffix_hi, size=batch, endpoint=True).astype(int).tolist()
    n_cow = int(round(cow_frac * batch))
    cow_seqs = sorted(rng.choice(batch, size=n_cow, replace=False).astype(int).tolist())
    shared_blocks = prefix_tokens // block_size
    last_shared = shared_blocks - 1
    needed = shared_blocks + n_cow + sum(_cdiv(s, block_size) for s in suffix)
    nb, order = _pool(rng, needed)
    holder = batch  # sequence id of the prefix writer
    setup = [("add", holder), ("append", holder, prefix_tokens)]
    for r in range(batch):
        setup.append(("add", r))
        setup.append(("share", r, holder, prefix_tokens))
    setup.append(("free", holder))
    for r in range(batch):
        if suffix[r] - 1 > 0:
            setup.append(("append", r, suffix[r] - 1))
    step = [("cow", r, last_shared) for r in cow_seqs]
    step += [("append", r, 1) for r in range(batch)]
    lens = [prefix_tokens + s for s in suffix]
    return Workload(
        name="prefix_shared_cow_decode", dtype="bf16", q_heads=q_heads, kv_heads=kv_heads,
        head_dim=head_dim, block_size=block_size, num_blocks=nb, scale=1.0 / math.sqrt(head_dim),
        free_order=order, setup_ops=setup, step_ops=step, decode_seqs=list(range(batch)),
        decode_lens=lens, seed=seed,
        note=f"prefix {prefix_tokens} tokens shared by {batch}; {n_cow} requests copy-on-write block {last_shared}",
    )


def mixed_prefill_decode(seed: int = 0, n_prefill: int = 4, chunk: int = 512, hist_lo: int = 0,
                         hist_hi: int = 8192, n_decode: int = 192, dec_lo: int = 256,
                         dec_hi: int = 16384) -> Workload:
    """Yi-34B-TP2-like step: 28 q heads / 4 KV heads, D=128, bs=16, bf16 N(0,1).

    4 prefill requests each run a 512-token chunk (causal within the chunk)
    over U{0..8192} tokens of paged history; 192 decode requests have contexts
    U{256..16384}.  K/V of all 4*512 + 192 new tokens are written by
    reshape_and_cache in the same step.
    """
    rng = _rng(seed)
    hist = rng.integers(hist_lo, hist_hi, size=n_prefill, endpoint=True).astype(int).tolist()
    dlens = rng.integers(dec_lo, dec_hi, size=n_decode, endpoint=True).astype(int).tolist()
    bs = 16
    needed = sum(_cdiv(h + chunk, bs) for h in hist) + sum(_cdiv(L, bs) for L in dlens)
    nb, order = _pool(rng, needed)
    setup, step = [], []
    prefill = []
    for i, h in enumerate(hist):
        s = 10000 + i
        setup.append(("add", s))
        if h > 0:
            setup.append(("append", s, h))
        step.append(("append", s, chunk))
        prefill.append((s, chunk, h + chunk))
    dsetup, dstep = _decode_scripts(list(range(n_decode)), dlens)
    return Workload(
        name="mixed_prefill_decode", dtype="bf16", q_heads=28, kv_heads=4, head_dim=128,
        block_size=bs, num_blocks=nb, scale=1.0 / math.sqrt(128), free_order=order,
        setup_ops=setup + dsetup, step_ops=step + dstep, decode_seqs=list(range(n_decode)),
        decode_lens=dlens, prefill=prefill, seed=seed,
        note="prefill chunks and decode in the same step, one stream",
    )


def mixed_prefill_part(seed: int = 0) -> Workload:
    """The prefill half of mixed_prefill_decode alone (same 4 chunks and
    histories; pool sized for them): a tensor-core workload for profiling."""
    wl = mixed_prefill_decode(seed=seed, n_decode=0)
    wl.name = "mixed_prefill_part"
    wl.note = "prefill chunks of the mixed step only"
    return wl


def mixed_decode_part_small(seed: int = 0) -> Workload:
    """A 24-request decode shaped like mixed_prefill_decode's decode half
    (28/4 heads, D=128, bs=16, contexts U{256..16384}), with a pool small
    enough for multi-pass profiler captures."""
    wl = mixed_prefill_decode(seed=seed, n_prefill=0, n_decode=24)
    wl.name = "mixed_decode_part_small"
    wl.note = "decode of the mixed step's shape, 24 requests"
    return wl


WORKLOADS = {
    "tiny_paged_decode": tiny_paged_decode,
    "llama8b_gqa_decode": llama8b_gqa_decode,
    "long_context_splitk_decode": long_context_splitk_decode,
    "spec_verify_decode": spec_verify_decode,
    "spec_verify_decode_k7": lambda seed=0: _renamed(spec_verify_decode(seed, k=7), "spec_verify_decode_k7"),
    "prefix_shared_cow_decode": prefix_shared_cow_decode,
    "mixed_prefill_decode": mixed_prefill_decode,
    "mixed_prefill_part": mixed_prefill_part,
    "mixed_decode_part_small": mixed_decode_part_small,
}


def make_values(wl: Workload, device="cpu", seed: int | None = None, poison_pool: bool = False):
    """Random tensors for one step of ``wl``.

    Returns a dict of torch tensors in ``wl``'s dtype:

    * ``k_cache``, ``v_cache``: [num_blocks, block_size, kv_heads, head_dim],
      the pool's contents before the step (history and stale data alike);
    * ``q_decode``: [len(decode_seqs), q_heads, head_dim], or
      [len(decode_seqs), q_len, q_heads, head_dim] when q_len > 1;
    * ``q_prefill``: [sum of chunks, q_heads, head_dim];
    * ``k_new``, ``v_new``: [new_tokens, kv_heads, head_dim], ordered as the
      step's ``append`` ops list their tokens.

    On "cpu" the values come from numpy's PCG64; on a CUDA device from a
    seeded torch generator on that device (much faster for multi-GB pools).
    ``poison_pool`` fills every pool slot with NaN instead, so that any read
    of a slot the step does not own shows up in the output.
    """
    seed = wl.seed if seed is None else seed
    dt = wl.torch_dtype
    pool_shape = (wl.num_blocks, wl.block_size, wl.kv_heads, wl.head_dim)
    nq_pref = sum(c for _, c, _ in wl.prefill)
    shapes = {
        "k_cache": pool_shape,
        "v_cache": pool_shape,
        "q_decode": ((len(wl.decode_seqs), wl.q_heads, wl.head_dim) if wl.q_len == 1 else
                     (len(wl.decode_seqs), wl.q_len, wl.q_heads, wl.head_dim)),
        "q_prefill": (nq_pref, wl.q_heads, wl.head_dim),
        "k_new": (wl.new_tokens, wl.kv_heads, wl.head_dim),
        "v_new": (wl.new_tokens, wl.kv_heads, wl.head_dim),
    }
    out = {}
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = _rng(seed + 7919)
        for name, shp in shapes.items():
            n = int(np.prod(shp))
            if wl.value_dist == "uniform":
                a = rng.uniform(-1.0, 1.0, size=n).astype(np.float32)
            else:
                a = rng.standard_normal(size=n, dtype=np.float32)
            out[name] = torch.from_numpy(a).reshape(shp).to(dt)
    else:
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 7919)
        for name, shp in shapes.items():
            if wl.value_dist == "uniform":
                t = torch.rand(shp, generator=g, device=dev, dtype=torch.float32) * 2.0 - 1.0
            else:
                t = torch.randn(shp, generator=g, device=dev, dtype=torch.float32)
            out[name] = t.to(dt)
    if poison_pool:
        out["k_cache"].fill_(float("nan"))
        out["v_cache"].fill_(float("nan"))
    return out
