"""pa_decode_noalloc: decode whose split-K scratch lives inside the library.

For callers that cannot allocate device memory (a plugin in a framework that
owns all of the GPU's memory, or a loop where cudaMalloc/cudaFree would
synchronise the device).  The entry point is called through the C ABI and its
output is compared with pa_decode's (caller-provided workspace) on calls in a
row with different shapes.  Both run the same kernels over the same
partitions, so the outputs must agree bit for bit.  A smaller call follows a
larger one whose partials are huge (V scaled by 2^12), so a read of the
previous call's leftovers would show.  Collected last on purpose: a failure
here comes after every other test.
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


def _case(batch, lo, hi, seed, v_scale=1.0):
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
    kc, vc = vals["k_cache"].to(d), (vals["v_cache"] * v_scale).to(d)
    from paged_kv_cache_76_gb300 import ops
    ops.reshape_and_cache(vals["k_new"].to(d), (vals["v_new"] * v_scale).to(d),
                          torch.tensor(slots, dtype=torch.int32, device=d), kc, vc)
    return wl, vals["q_decode"].to(d), kc, vc, torch.from_numpy(tables).to(d), torch.from_numpy(lens).to(d)


def _call_noalloc(lib, wl, q, kc, vc, tables, lens, out):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.pa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), tables.data_ptr(), tables.shape[1],
                                 lens.data_ptr(), q.shape[0], wl.q_heads, wl.kv_heads, wl.head_dim, wl.block_size,
                                 wl.num_blocks, wl.scale, wl.split_tokens, out.data_ptr(), 1, stream)


def _reference(wl, q, kc, vc, tables, lens):
    """pa_decode with a torch-allocated workspace that starts as NaN."""
    from paged_kv_cache_76_gb300 import ops
    ws = ops.make_workspace(q, tables, wl.block_size)
    if ws is not None:
        ws.view(torch.float32)[: ws.numel() // 4].fill_(float("nan"))
    return ops.decode(q, kc, vc, tables, lens, wl.scale, workspace=ws)


def test_noalloc_decode_matches_pa_decode_on_calls_in_a_row(lib):
    from paged_kv_cache_76_gb300 import ops
    # (batch, context range, seed, V scale): the large first call fills the
    # scratch with partials about 2^12 times the size of the next call's
    for batch, lo, hi, seed, vs in [(16, 600, 3000, 5, 4096.0), (9, 100, 1500, 6, 1.0), (12, 2000, 5000, 8, 1.0)]:
        wl, q, kc, vc, tables, lens = _case(batch, lo, hi, seed, vs)
        need = ops.decode_workspace_size(q.shape[0], wl.q_heads, wl.head_dim, tables.shape[1], wl.block_size)
        assert 0 < need <= lib.pa_decode_workspace_size(q.shape[0], wl.q_heads, wl.head_dim, tables.shape[1], 16, 0)
        ref = _reference(wl, q, kc, vc, tables, lens)
        out = torch.full_like(q, float("nan"))
        assert _call_noalloc(lib, wl, q, kc, vc, tables, lens, out) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"batch {batch}: differs from pa_decode"
        assert np.isfinite(to_f64(out)).all()
        if vs == 1.0:  # and both within the attention tolerance of the float64 oracle on a few rows
            from oracle import paged_attention as opa
            for r in (0, batch - 1):
                L = int(lens[r])
                nblk = -(-L // wl.block_size)
                ids = tables[r, :nblk].long()
                want = opa.decode(to_f64(q[r:r + 1]), to_f64(kc[ids]), to_f64(vc[ids]),
                                  np.arange(nblk)[None], [L], wl.scale)
                err = np.abs(to_f64(out[r:r + 1]) - want)
                assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN
        assert ops.get_device_error() == 0


def test_noalloc_decode_with_no_scratch_needed(lib):
    """Every context fits one partition: no scratch is used, and the call still
    matches pa_decode bit for bit (right after calls that did use it)."""
    from paged_kv_cache_76_gb300 import ops
    wl, q, kc, vc, tables, lens = _case(8, 100, 384, 9)
    assert lib.pa_decode_workspace_size(q.shape[0], wl.q_heads, wl.head_dim, tables.shape[1], 16, 0) == 0
    ref = _reference(wl, q, kc, vc, tables, lens)
    out = torch.full_like(q, float("nan"))
    assert _call_noalloc(lib, wl, q, kc, vc, tables, lens, out) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
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
