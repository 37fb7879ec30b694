"""Paged-KV-cache attention for NVIDIA GB300 (sm_103a).

The compute path is ``libpa.so`` (hand-written CUDA behind the C ABI of
``include/pa.h``); this package is its ctypes binding:

* :mod:`.ops` - reshape_and_cache, copy_blocks, decode (partial + lse_merge),
  chunked_prefill, device error word;
* :mod:`.allocator` - the C++ block allocator (free queue, refcounts, share,
  copy-on-write);
* :mod:`.build` - compiles the library in-tree.

Importing the package does not load the library; the first call does, and
raises :class:`LibraryMissing` if it has not been built.
"""
from ._lib import LibraryMissing, PAError  # noqa: F401

__version__ = "0.1.0"
