"""pa_decode_noalloc: decode whose split-K scratch lives inside the library.

For callers that cannot allocate device memory (a plugin in a framework that
owns all of the GPU's memory, or a loop where cudaMalloc/cudaFree would
synchronise the device).  The entry point is called through the C ABI and its
output is compared with pa_decode's (caller-provided workspace) on two calls in
a row with different shapes, within the attention tolerance of the other
tests.  Collected last on purpose: a failure here comes after every other test.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.paged_step import TOL_MAX, TOL_MEAN, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_76_gb300 import _lib
    try:
        return _lib.lib()
    except _lib.LibraryMissing:
        from paged_kv_cache_76_gb300 import build
        build.build()
        return _lib.lib()


def _case(batch, lo, hi, seed):
    """Device-resident decode inputs from the C++ allocator (C ABI)."""
    from paged_kv_cache_76_gb300.allocator import BlockAllocator
    wl = W.custom_decode(batch, lo, hi, 32, 8, 128, 16, "bf16", seed=seed)
    vals = W.make_values(wl)
    a = BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
    a.run(wl.setup_ops)
    slots, _ = a.run(wl.step_ops)
    maxblk = max(len(a.block_table(s)) for s in wl.decode_seqs)
    tables, lens = a.build_tables(wl.decode_seqs, maxblk)
    d = "cuda"
    kc, vc = vals["k_cache"].to(d), vals["v_cache"].to(d)
    from paged_kv_cache_76_gb300 import ops
    ops.reshape_and_cache(vals["k_new"].to(d), vals["v_new"].to(d), torch.tensor(slots, dtype=torch.int32, device=d),
                          kc, vc)
    return wl, vals["q_decode"].to(d), kc, vc, torch.from_numpy(tables).to(d), torch.from_numpy(lens).to(d)


def _call_noalloc(lib, wl, q, kc, vc, tables, lens, out):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.pa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), tables.data_ptr(), tables.shape[1],
                                 lens.data_ptr(), q.shape[0], wl.q_heads, wl.kv_heads, wl.head_dim, wl.block_size,
                                 wl.num_blocks, wl.scale, wl.split_tokens, out.data_ptr(), 1, stream)


def test_noalloc_decode_matches_pa_decode_on_two_calls_in_a_row(lib):
    from paged_kv_cache_76_gb300 import ops
    for batch, lo, hi, seed in [(16, 600, 3000, 5), (9, 100, 1500, 6)]:
        wl, q, kc, vc, tables, lens = _case(batch, lo, hi, seed)
        need = ops.decode_workspace_size(q.shape[0], wl.q_heads, wl.head_dim, tables.shape[1], wl.block_size)
        assert 0 < need <= lib.pa_decode_workspace_size(q.shape[0], wl.q_heads, wl.head_dim, tables.shape[1], 16, 0)
        ref = ops.decode(q, kc, vc, tables, lens, wl.scale)            # pa_decode, torch-allocated workspace
        out = torch.full_like(q, float("nan"))
        assert _call_noalloc(lib, wl, q, kc, vc, tables, lens, out) == 0
        torch.cuda.synchronize()
        a, b = to_f64(out), to_f64(ref)
        assert np.isfinite(a).all()
        err = np.abs(a - b)
        assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN
        assert ops.get_device_error() == 0


def test_noalloc_decode_rejects_scratch_beyond_its_limit(lib):
    from paged_kv_cache_76_gb300 import _lib
    wl, q, kc, vc, tables, lens = _case(4, 100, 200, 7)
    # a table width that would need more than 16 MiB of partials: rejected before any launch
    wide = torch.full((q.shape[0], 1 << 17), -1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    assert _call_noalloc(lib, wl, q, kc, vc, wide, lens, out) == _lib.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
