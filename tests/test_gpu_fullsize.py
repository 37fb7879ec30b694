"""Parity at the full sizes of the five measured workloads (GPU).

The device runs the whole step exactly as bench.py times it (same kernels,
partitions and launch configuration: copy_blocks -> reshape_and_cache ->
chunked prefill -> decode partial -> merge); pools are generated on the GPU.
The float64 oracle checks sampled outputs on a compacted copy of the blocks
they read; bitwise properties (physical relabelling, copy-on-write vs shared)
are checked on every output.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.paged_step import DeviceStep, assert_close, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_76_gb300 import _lib
    try:
        _lib.lib()
    except _lib.LibraryMissing:
        from paged_kv_cache_76_gb300 import build
        build.build()


def _no_err():
    from paged_kv_cache_76_gb300 import ops
    assert ops.get_device_error() == 0


def test_llama8b_gqa_decode_full_size():
    wl = W.llama8b_gqa_decode()
    vals = W.make_values(wl, device="cuda")
    dev = DeviceStep(wl, vals)
    dev.run()
    rows = list(range(0, 64, 4))
    ref = oracle_step(wl, vals, decode_rows=rows, compact=True)
    assert_close(dev.out_decode[rows], ref["decode"], "llama8b sampled")
    _no_err()


def test_spec_verify_decode_full_size():
    """The verify workload as bench.py times it: reshape_and_cache of the k=3
    drafts, then pa_verify_decode; sampled requests against the oracle."""
    wl = W.spec_verify_decode()
    vals = W.make_values(wl, device="cuda")
    dev = DeviceStep(wl, vals)
    dev.run()
    rows = list(range(0, 64, 8))
    ref = oracle_step(wl, vals, decode_rows=rows, compact=True)
    assert_close(dev.out_decode[rows], ref["decode"], "verify sampled")
    _no_err()


def test_spec_verify_decode_k7_tensor_core_form_full_size():
    """The k = 7 verify workload as bench.py times it by default (32 query
    columns per KV head: pa_verify_decode_tc), sampled requests against the
    oracle, and every row against the warp-MMA form within the tolerance."""
    from paged_kv_cache_76_gb300 import ops
    wl = W.WORKLOADS["spec_verify_decode_k7"]()
    vals = W.make_values(wl, device="cuda")
    dev = DeviceStep(wl, vals)
    dev.run()                                   # reshape_and_cache + pa_verify_decode
    tc = ops.verify_decode_tc(dev.q_decode, dev.k_cache, dev.v_cache, dev.dec_tables, dev.dec_lens, wl.scale)
    torch.cuda.synchronize()
    rows = list(range(3, 64, 8))
    ref = oracle_step(wl, vals, decode_rows=rows, compact=True)
    assert_close(tc[rows], ref["decode"], "verify k7 tensor-core form sampled")
    d = (tc.float() - dev.out_decode.float()).abs()
    assert d.max().item() <= 2e-2 and d.mean().item() <= 1e-3
    _no_err()


def test_long_context_splitk_decode_full_size():
    wl = W.long_context_splitk_decode()
    vals = W.make_values(wl, device="cuda")
    dev = DeviceStep(wl, vals)
    dev.run()
    # the shortest and the longest request (up to 256 partitions merged by
    # the block-per-row merge) against the oracle
    for row in (int(np.argmin(wl.decode_lens)), int(np.argmax(wl.decode_lens))):
        ref = oracle_step(wl, vals, decode_rows=[row], compact=True)
        assert_close(dev.out_decode[[row]], ref["decode"], f"long context request {row}")
    # every output: a random relabelling of all physical blocks gives the same bits
    out = dev.out_decode.clone()
    pi = torch.randperm(wl.num_blocks, generator=torch.Generator().manual_seed(1)).cuda()
    k2, v2 = torch.empty_like(dev.k_cache), torch.empty_like(dev.v_cache)
    k2[pi] = dev.k_cache
    v2[pi] = dev.v_cache
    t2 = torch.where(dev.dec_tables >= 0, pi[dev.dec_tables.clamp(min=0).long()].int(), dev.dec_tables)
    from paged_kv_cache_76_gb300 import ops
    out2 = ops.decode(dev.q_decode, k2, v2, t2, dev.dec_lens, wl.scale, split_tokens=wl.split_tokens)
    assert torch.equal(out, out2)
    _no_err()


def test_prefix_shared_cow_decode_full_size():
    wl = W.prefix_shared_cow_decode()
    vals = W.make_values(wl, device="cuda")
    dev = DeviceStep(wl, vals)
    assert len(dev.pairs_host) == 26
    dev.run()
    cow_rows = sorted({int(op[1]) for op in wl.step_ops if op[0] == "cow"})[:8]
    rows = sorted(set(cow_rows + list(range(0, 256, 16))))
    ref = oracle_step(wl, vals, decode_rows=rows, compact=True)
    assert_close(dev.out_decode[rows], ref["decode"], "prefix sampled")
    # every output: the same step without the copies reads the shared block instead
    wl2 = W.Workload(**{**wl.__dict__, "step_ops": [op for op in wl.step_ops if op[0] != "cow"]})
    dev2 = DeviceStep(wl2, vals)
    dev2.run()
    assert torch.equal(dev.out_decode, dev2.out_decode)
    _no_err()


def test_mixed_prefill_decode_full_size():
    wl = W.mixed_prefill_decode()
    vals = W.make_values(wl, device="cuda")
    dev = DeviceStep(wl, vals)
    dev.run()
    dec_rows = list(range(0, 192, 24))
    # prefill rows: first, last and a spread inside each 512-query chunk
    pre_rows = sorted({512 * r + i for r in range(4) for i in (0, 1, 63, 64, 255, 256, 510, 511)})
    ref = oracle_step(wl, vals, decode_rows=dec_rows, prefill_rows=pre_rows, compact=True)
    assert_close(dev.out_decode[dec_rows], ref["decode"], "mixed decode sampled")
    assert_close(dev.out_prefill[pre_rows], ref["prefill"][pre_rows], "mixed prefill sampled")
    _no_err()


def test_mixed_step_as_the_bench_launches_it_equals_the_single_stream_step():
    """bench.py's mixed step: the prefill on a second, highest-priority stream
    over a capped set of persistent CTAs, beside the decode.  Every unit
    computes exactly as with one CTA per unit on one stream, so the outputs
    are the same bits."""
    import bench
    wl = W.mixed_prefill_decode()
    vals = W.make_values(wl, device="cuda")
    dev = DeviceStep(wl, vals)
    dev.run()
    step = bench.Step(wl, torch.device("cuda", 0), value_seed=wl.seed)
    assert step.side is not None
    step.prefill_ctas = 57
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.run(s)
    s.synchronize()
    assert torch.equal(step.out_pre, dev.out_prefill)
    assert torch.equal(step.out_dec, dev.out_decode)
    _no_err()


@pytest.mark.parametrize("name", ["prefix_shared_cow_decode", "mixed_prefill_decode"])
def test_bench_step_recorded_once_replays_to_the_same_bits(name):
    """bench.py's end-to-end loop can issue a step from launches marshalled
    once (ops.recording), including the event fork and join of a second
    stream: replaying the plan gives the bits of the step run directly."""
    import bench
    wl = W.WORKLOADS[name]()
    step = bench.Step(wl, torch.device("cuda", 0), value_seed=wl.seed)
    assert step.side is not None or step.prefix_side is not None
    if step.side is not None:
        step.prefill_ctas = 57
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.run(s)
    s.synchronize()
    outs = [t.clone() for t in (step.out_dec, step.out_pre) if t is not None]
    plan = step.record_plan(s)
    for t in (step.out_dec, step.out_pre):
        if t is not None:
            t.zero_()
    with torch.cuda.stream(s):
        plan()
    s.synchronize()
    got = [t for t in (step.out_dec, step.out_pre) if t is not None]
    assert all(torch.equal(a, b) for a, b in zip(got, outs))
    _no_err()
