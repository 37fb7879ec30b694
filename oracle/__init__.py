"""CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the paged-KV path computes, in float64 NumPy (allocator
state in plain Python).  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  The library itself never
does: it shares no code with this package, and this package imports nothing
from the library.

Sources (web pages on the subject, cited by title and section):

* "2.1 PagedAttention" (Vietnamese edition, infra-guide): §3 Block Table and
  its worked example, §5 the kernel's view (physical_block_number /
  physical_block_offset), §6 sharing and Copy-on-Write, §9.1-9.3 the
  KVCacheManager / BlockPool / free-queue design and pseudocode.
* "2.1 PagedAttention：像操作系统管理内存一样管理 KV Cache" (Chinese edition,
  aiinfraguide): the same sections; its free_blocks pseudocode differs (see
  ``block_pool``).
* "Khám phá vLLM … phần 2" (gpuhub.net): chunked prefill.
* "vAttention 完全拆解" (pinghaoyang.com.cn): the KV size closed form and the
  rule that stale KV past a request's valid length is never visible.

Modules:

* ``paged_attention``: slot translation, reshape_and_cache, copy_blocks,
  paged decode (direct and context-split + log-sum-exp merge), chunked
  prefill.  Pinned by the tests in ``tests/test_oracle_pins.py``.
* ``block_pool``: free queue, block pool and per-sequence manager.  Pinned by
  ``tests/test_oracle_allocator.py``.
* ``sizing``: KV byte counts (the vAttention page's closed form; the bytes
  a decode step moves, logical and with shared rows counted once).  Pinned
  by the page's worked numbers and by a brute-force count of the array
  elements a step touches.
* ``vattention``: the vAttention-style manager's bookkeeping.  Pinned by
  ``tests/test_oracle_vattention.py`` (the page's formulas, numbers and
  figure 2 walk-through; numpy's own row-major addressing for slot rows).

Parity status: every public function here has at least one pin that does not
restate its own formula (a printed value, a library routine, a brute-force
count or an invariant); ``tests/`` names it beside each test.  The one part
the pages leave undecided is the free-queue placement of released blocks,
where the two editions' listings disagree; the reading taken is stated in
``block_pool`` and pinned by the allocator tests.
"""
from . import block_pool, paged_attention, sizing, vattention  # noqa: F401
